// Decode attention over a TurboQuant-compressed KV cache (sm_103a): device
// error word, launch dispatch over the query-group size, and the
// allocation-free entry point.  The kernel itself is in tq_decode_kernel.cuh,
// instantiated in tq_decode_g{1,2,4,8}.cu.
#include <cuda_runtime.h>
#include <stdint.h>

#include "tq_decode_kernel.cuh"

namespace tq {

__device__ unsigned g_decode_err;

int launch_decode_g1(const DecodeArgs& a, cudaStream_t s);
int launch_decode_g2(const DecodeArgs& a, cudaStream_t s);
int launch_decode_g4(const DecodeArgs& a, cudaStream_t s);
int launch_decode_g8(const DecodeArgs& a, cudaStream_t s);

int launch_decode(const DecodeArgs& a, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (a.Hkv > 65535 || a.B > 65535) return 1;
  switch (a.G) {
    case 1: return launch_decode_g1(a, s);
    case 2: return launch_decode_g2(a, s);
    case 4: return launch_decode_g4(a, s);
    case 8: return launch_decode_g8(a, s);
  }
  return 1;
}

unsigned* decode_error_ptr() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_decode_err) != cudaSuccess) return nullptr;
  return (unsigned*)p;
}

int decode_read_error(unsigned* out) {
  unsigned zero = 0;
  if (cudaMemcpyFromSymbol(out, g_decode_err, sizeof(unsigned)) != cudaSuccess) return 1;
  if (cudaMemcpyToSymbol(g_decode_err, &zero, sizeof(unsigned)) != cudaSuccess) return 1;
  return 0;
}

}  // namespace tq

// ------------------------------------------------ allocation-free decode entry
// Some callers cannot hand this library a workspace: a plugin inside a
// serving engine that owns every device allocation and passes only tensor
// pointers, or a latency-bound decode loop that must not call the CUDA
// allocator (cudaMalloc can synchronize the whole device).  For them the
// decode split partials and split counters live in one fixed array in device
// memory that this library reserves when it is loaded.
#include <mutex>

namespace tq {

constexpr size_t kStaticScratchBytes = 8u << 20;   // 8 MiB per GPU
constexpr int kMaxDevices = 64;

// Reserved on every GPU that loads the library, held until the process exits.
// In host code this name is only a stand-in for the device object: its device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

static void* g_static_scratch_addr[kMaxDevices];
static std::mutex g_static_scratch_mu;

// Device address of the array on the current device, looked up once per device.
static tq_status static_scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return TQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_static_scratch_mu);
  if (!g_static_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return TQ_ERR_CUDA;
    g_static_scratch_addr[dev] = p;
  }
  *out = g_static_scratch_addr[dev];
  return TQ_OK;
}

}  // namespace tq

extern "C" tq_status tq_decode_attention_noalloc(
    const tq_config* cfg, const void* tables, int layer, const void* q, int q_dtype,
    float softmax_scale, int batch, int n_q_heads, int n_kv_heads, tq_planes k, tq_planes v,
    const uint16_t* k_win, const uint16_t* v_win, const int32_t* seq_lens, int max_seq_len,
    float* out, void* stream) {
  if (!cfg || batch < 0 || n_kv_heads < 1 || n_q_heads < n_kv_heads || max_seq_len < 0)
    return TQ_ERR_INVALID_ARG;
  const size_t need = tq_workspace_bytes(cfg, batch, n_q_heads, n_kv_heads, max_seq_len);
  if (need > tq::kStaticScratchBytes) return TQ_ERR_BUFFER_TOO_SMALL;
  void* scratch = nullptr;
  tq_status st = tq::static_scratch_address(&scratch);
  if (st != TQ_OK) return st;
  // the array keeps whatever the previous call left (another call's partials
  // may lie where this call's split counters go); the counters must start at
  // zero, so clear them.  The partials are written before they are read.
  size_t coff = 0, cbytes = 0;
  tq_status cst = tq::decode_counters_range(cfg, layer, batch, n_q_heads, n_kv_heads,
                                            max_seq_len, &coff, &cbytes);
  if (cst != TQ_OK) return cst;
  if (cbytes > 0 && cudaMemsetAsync((unsigned char*)scratch + coff, 0, cbytes,
                                    (cudaStream_t)stream) != cudaSuccess)
    return TQ_ERR_CUDA;
  return tq_decode_attention(cfg, tables, layer, q, q_dtype, softmax_scale, batch, n_q_heads,
                             n_kv_heads, k, v, k_win, v_win, seq_lens, max_seq_len, out, scratch,
                             tq::kStaticScratchBytes, stream);
}
