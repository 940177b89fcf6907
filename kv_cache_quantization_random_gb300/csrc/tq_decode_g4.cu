// Decode-attention kernels for 4 query head(s) per kv-head: every
// (key bits, value bits, QJL) storage format of the library.
#include "tq_decode_kernel.cuh"

namespace tq {
int launch_decode_g4(const DecodeArgs& a, cudaStream_t s) { return launch_decode_g<4>(a, s); }
}  // namespace tq
