// Private declarations shared by the host code (tq_host.cpp) and the CUDA
// translation units of the TurboQuant library.  Not part of the C ABI.
#pragma once

#include <stdint.h>
#include <stddef.h>

#include <cuda_runtime.h>

#include "../../include/tq.h"

namespace tq {

constexpr int kHeadDim = 128;          // the head_dim the kernels implement
constexpr int kQjlM = 128;             // the QJL projection count the kernels implement
constexpr int kDecodeSms = 152;         // decode grid target: one wave over the GB300's SMs
constexpr int kPartialStride = 4 + kHeadDim;   // floats per (split, head): m, l, pad, pad, o[d]

// ---- decode CTA shape, shared by the host's split plan and the kernel --------
// words per head row of the V-sum weight buffer (16 used): the B-operand
// reads of the 8 heads x 4 lanes fall into 32 different banks
constexpr int kWsStride = 20;
// 32-token chunks in each warp's staging ring: enough bytes in flight per SM
// to cover the HBM latency (3 slots of 12 warps hold about 120 KB for 3- and
// 4-bit keys); formats with 2-bit keys and narrow rows keep 4.
__host__ __device__ constexpr int ring_slots(int kb, int vb) {
  return kb <= 2 && kb + vb <= 8 ? 4 : 3;
}

// Byte layout of the dynamic shared memory of a decode CTA with nw warps
// (G query columns per kv-head; res 0 = MSE keys, 1 = QJL, 2 = Direct Sign).
struct DecodeSmem {
  int qr = 0, qo = 0, sv = 0, qjlb = 0, sq = 0, lutk4 = 0, warps = 0, warp_stride = 0;
  int kbuf = 0, vbuf = 0, kn = 0, vn = 0, sbuf = 0, rn = 0, ws = 0, bar = 0;   // inside one warp's region
  int comb = 0, total = 0;
  __host__ __device__ constexpr DecodeSmem(int G, int res, int kb, int vb, int nw) {
    const bool qjl = res == 1, sres = res != 0;
    int off = 0;
    qr = off; off += kHeadDim * G * 4;            // [128][G] rotated, scaled queries
    qo = off; off += kHeadDim * G * 4;            // [128][G] original-domain queries
    sv = off; off += kHeadDim * 4;
    qjlb = off; off += qjl ? 32 * 8 * 16 : 0;     // per lane, per k-tile: S q hi/lo operands
    sq = off; off += qjl ? G * kQjlM * 4 : 0;     // [G][m] S q_rot (QJL)
    // pair table: 256-byte rows, 16 key replicas then 16 value replicas (2-bit values)
    lutk4 = off; off += vb == 2 || kb == 4 ? 256 * 256 : kb == 3 ? 64 * 256 : 0;
    warps = off;
    const int ns = ring_slots(kb, vb);
    int w = 0;
    kbuf = w; w += ns * 32 * 16 * kb;
    vbuf = w; w += ns * 32 * 16 * vb;
    kn = w; w += ns * 128;
    vn = w; w += ns * 128;
    sbuf = w; w += sres ? ns * 32 * 16 : 0;       // 128 sign bits per token
    rn = w; w += sres ? ns * 128 : 0;             // gamma (QJL) or scale (Direct Sign)
    ws = w; w += 8 * kWsStride * 4;               // [8 heads][16 token pairs] fp16 weights
    bar = w; w += 8 * ns;
    w = (w + 15) & ~15;
    warp_stride = w;
    int region = nw * w;
    const int comb_need = nw * G * (2 + kHeadDim) * 4;   // cm, cl, co
    const int merge_need = nw * (4 + 2 * kHeadDim) * 4;  // the last CTA's per-warp merges
    if (region < comb_need) region = comb_need;
    if (region < merge_need) region = merge_need;
    comb = warps;
    off += region;
    total = off + 16;                             // + is-last flag
  }
};

// dynamic shared memory a decode CTA may use (227 KB per CTA, less the
// kernel's static tables and a fused decode step's scratch)
constexpr int kDecodeSmemBudget = 216 * 1024;
// a fused decode step's scratch after the CTA's dynamic shared memory (see
// step_leaving_token): 128-byte alignment slack, two codebooks' boundaries,
// 32 words of packing scratch and 128 floats of residual scratch
constexpr int kFusedScratchBytes = 128 + 2 * 256 * 4 + 32 * 4 + 128 * 4;

// Warps of a decode CTA.  G <= 4 query columns with MSE keys (about 168
// registers a thread): one CTA per SM of 12 warps, or 8 when 12 staging
// rings do not fit.  G = 8 with MSE keys (about 240 registers): one CTA of 8
// warps.  Keys with a residual term: two or three CTAs of 4 warps per SM, so that one
// CTA's prologue runs beside the other's main loop (measured faster for these
// formats).  Fewer, wider CTAs build the SM's lookup tables once and leave
// half as many splits to merge.
__host__ __device__ constexpr int decode_warps(int G, int kb, int vb, int res) {
  return res != 0                                                        ? 4
         : G > 4 ? (DecodeSmem(G, res, kb, vb, 8).total <= kDecodeSmemBudget ? 8 : 4)
         : DecodeSmem(G, res, kb, vb, 12).total <= kDecodeSmemBudget ? 12
         : DecodeSmem(G, res, kb, vb, 8).total <= kDecodeSmemBudget  ? 8
                                                                       : 4;
}
// resident decode CTAs per SM: CTAs of 4 warps three (or two) to an SM when
// they fit in its 228 KB of shared memory, each with its dynamic shared memory,
// a decode step's scratch, up to 4.5 KB of static tables and 1 KB the system
// reserves per CTA; else one.  Three CTAs (G <= 4 query heads) cap a thread
// at 168 registers, which the 2-bit-key, 3-bit-value formats with a residual
// term meet without spills (measured faster than two CTAs); with G = 8 the
// register cap would spill.
__host__ __device__ constexpr int decode_ctas_per_sm(int G, int kb, int vb, int res) {
  return decode_warps(G, kb, vb, res) != 4 ? 1
         : G <= 4 && 3 * (DecodeSmem(G, res, kb, vb, 4).total + kFusedScratchBytes + 5632) <=
                         228 * 1024
             ? 3
         : 2 * (DecodeSmem(G, res, kb, vb, 4).total + 4 * 1024) <= 227 * 1024 ? 2
                                                                             : 1;
}

// ---- device tables (built on the host by tq_build_tables) -------------------
// [0, 256)                 header, int32 words (see kTbl*)
// [256, 256 + 8*2048)      codebook slot for bits 1..8: 256 centroids then
//                          256 boundaries (fp32; unused tail = +inf)
// signs                    (2*layer + kind) * d fp32 (+1 / -1)
// qjl                      one m*d bf16 matrix per QJL layer, in layer order
constexpr size_t kTblHeader = 256;
constexpr size_t kTblCodebook = 256;
constexpr size_t kTblCodebookSlot = 2048;
constexpr uint32_t kTblMagic = 0x42545154u;  // "TQTB"

struct TableOffsets {
  size_t signs;     // byte offset of the sign vectors
  size_t qjl;       // byte offset of the QJL matrices
  size_t total;     // total bytes
};

// ---- kernel argument blocks ----------------------------------------------------
struct QuantArgs {
  // source rows
  const void* src;      // new rows (dtype src_f32 ? fp32 : bf16)
  int src_f32;
  int64_t sb, sh, st;   // element strides of src (batch, head, token)
  int B, H, n;          // n rows per (b, h)
  const int32_t* dst_pos;        // plain mode: first plane row per sequence (or null)
  // append mode (rows come from the window ring or the new input)
  int append;
  const int32_t* seq_before;     // T0 per sequence
  int W;
  uint16_t* win;                 // bf16 ring [B][H][W][d]: leaving tokens are read from it,
                                 // the new tokens that stay are written into it
  // destination planes
  uint8_t* codes;
  float* norms;
  uint8_t* qjl_signs;
  float* qjl_rnorm;
  int64_t cap;
  // codec
  int bits;
  const float* centroids;        // [256]
  const float* boundaries;       // [256]
  const float* rot_signs;        // [d]
  int qjl;                       // 0 | 1
  int dsign;                     // keys in Direct Sign mode: 0 | 1
  const uint16_t* S;             // bf16 [m][d]
  int m;
  unsigned* err;                 // device error word
  uint32_t wait_limit;           // polls per bounded wait (0 = default)
  // code search grid (see SearchGrid) and the rotation signs as fp32 sign-bit
  // masks, kept in the parameter block so the kernel reads them as operands
  float grid_scale;              // cells per unit of y
  float grid_magic;              // 1.5 * 2^23 + grid_cells / 2
  float grid_clamp;              // |y| clamp before the cell index (0: none)
  int grid_cells;
  uint32_t smask[kHeadDim];
};

// Code search by a uniform grid over y: cell k = round(y * scale) + cells / 2.
// The cell width is a quarter of the smallest gap between two boundaries, so
// any three neighbouring cells hold at most one boundary, and the entry of
// cell k (the number of boundaries below the lower edge of cells k-1..k+1 and
// the first boundary above it) gives the code with one comparison.
struct SearchGrid {
  float scale, magic, clamp;
  int cells;
};
constexpr int kMaxGridCells = 2560;

// tq_append_kv for a few new tokens per sequence: one launch does the K and
// V quantize of the tokens leaving the window and the window ring update.
struct AppendArgs {
  const void* src[2];            // k_new, v_new
  int src_f32;
  int64_t sb, sh, st;            // element strides of both sources
  int B, H, n;
  const int32_t* seq_before;
  int W;
  uint16_t* win[2];              // bf16 rings (W > 0)
  uint8_t* codes[2];
  float* norms[2];
  int64_t cap[2];
  uint8_t* qjl_signs;            // K only
  float* qjl_rnorm;
  int bits[2];
  const float* centroids[2];
  const float* boundaries[2];
  const float* rot_signs[2];
  int qjl;                       // K in MSE+QJL mode
  int dsign;                     // K in Direct Sign mode
  const uint16_t* S;             // bf16 [m][d]
  unsigned* err;
};
constexpr int kAppendFusedMaxNew = 8;   // larger appends take the bulk quantize kernel

struct DequantArgs {
  const uint8_t* codes;
  const float* norms;
  const uint8_t* qjl_signs;
  const float* qjl_rnorm;
  int64_t cap;
  int B, H, n;
  int bits;
  const float* centroids;
  const float* rot_signs;
  int qjl;
  int dsign;                     // add the Direct Sign residual a (2 bits - 1)
  const uint16_t* S;
  int m;
  float* dst;
  unsigned* err;                 // device error word (bounds-checked build)
};

struct DecodeArgs {
  const void* q;
  int q_f32;
  float qscale;                  // softmax_scale * log2(e)
  int B, Hq, Hkv, G;
  // planes
  const uint8_t* kc; const float* kn; const uint8_t* ks; const float* kr; int64_t kcap;
  const uint8_t* vc; const float* vn; int64_t vcap;
  int kb, vb, qjl, m;
  int dsign;                     // keys in Direct Sign mode
  float sparse_thr;              // skip a chunk's V sum below this weight (0: never)
  int n_q;                       // query tokens per sequence (columns g: token g % n_q)
  int step_new;                  // decode step (1, with fused_step): seq_lens are the
                                 // lengths before the step's token; T = seq_lens + step_new
  const uint16_t* kwin; const uint16_t* vwin; int W;
  const int32_t* seq_lens;
  int max_seq_len;               // host bound on every T: a T outside [0, max_seq_len]
                                 // sets kErrBounds and is decoded as an empty sequence
  int n_qsplits;                 // splits over the quantized tokens
  int n_splits;                  // n_qsplits + the window splits
  int split_tokens;              // tokens per quantized split (multiple of 32)
  int wsplit_tokens;             // window tokens per window split
  int long_first;                // CTA order: all quantized splits before the window
                                 // splits (several waves), else split-major per pair
  int pdl_trigger;               // one wave of one CTA per SM: let the next decode's
                                 // CTAs start early (griddepcontrol.launch_dependents)
  // decode step in one launch (fused_step = 1, step_new = 1): the kernel also
  // appends the step's token.  The quantized splits stop before plane row
  // T - 1 - W (the token leaving the window; with W = 0 the new token itself);
  // the pair's first window split (with W = 0 a split of its own) quantizes
  // that token into the planes, attends to its dequantized key and value, and
  // with W > 0 writes the new token into the ring slot it leaves; the window
  // splits read the new token from knew / vnew.
  int fused_step;
  const void* knew; const void* vnew;   // [B][Hkv][.][d] rows
  int new_f32;                   // knew / vnew are fp32 (W = 0 only: the ring is bf16)
  int64_t nsb, nsh;              // element strides of knew / vnew (batch, head)
  // codec
  const float* ck; const float* cv;
  const float* sk; const float* sv;
  const uint16_t* S;
  // outputs / workspace
  float* out;
  float* partials;               // [B][Hkv][n_splits][G][4 + d]
  unsigned* counters;            // [B][Hkv]
  unsigned* err;
  uint32_t wait_limit;           // polls per bounded wait (0 = default)
  uint32_t extra_tx;             // test hook (tq_set_fault_injection), normally 0
};

// ---- launchers (defined in the .cu files) -------------------------------------
int launch_quantize(const QuantArgs& a, void* stream);
// keys and values of an append in one launch: bf16 rows, neither kind in QJL
// mode, the same bit width and search grid (tq_append_kv checks)
int launch_quantize_kv(const QuantArgs& ak, const QuantArgs& av, void* stream);
int launch_quantize_qjl(const QuantArgs& a, cudaStream_t stream);   // keys in MSE+QJL mode
int sm_count();
int launch_append(const AppendArgs& a, void* stream);
int launch_dequantize(const DequantArgs& a, void* stream);
int launch_decode(const DecodeArgs& a, void* stream);

// the split counters' byte range in a decode workspace (tq_host.cpp)
tq_status decode_counters_range(const tq_config* cfg, int layer, int batch, int n_q_heads,
                                int n_kv_heads, int max_seq_len, size_t* off, size_t* bytes);

// device error words: each .cu owns one; these read-and-clear them
int quant_read_error(unsigned* out);
int decode_read_error(unsigned* out);
unsigned* quant_error_ptr();
unsigned* decode_error_ptr();

extern uint32_t g_wait_limit;
extern uint32_t g_fault_injection;

// error bits written by the kernels
constexpr unsigned kErrTimeout = 1u;
constexpr unsigned kErrBounds = 2u;

}  // namespace tq
