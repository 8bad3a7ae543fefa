// Decode kernels for head dim 512 (one translation unit per head dim, compiled in parallel).
#include "tq_decode_wide.cuh"

namespace tqd {

bool dispatch_decode_wide_d512(int kb, int vb, int vq, const DecodeParams& p, dim3 g, cudaStream_t s,
                              cudaError_t* e) {
  TQ_WIDE_CASES(512)
}
}  // namespace tqd
