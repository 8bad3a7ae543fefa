// Instantiation of the decode kernel for SQU-KV (spectral keys and values, head dim 128).
#include "tq_decode_kernel.cuh"

namespace tqd {

bool dispatch_decode_ksq(int kq, int kh, int vb, int vq, const DecodeParams& p, dim3 g, cudaStream_t s,
                         cudaError_t* e) {
  TQ_DECODE_CASE(kSQ, 0, 0, kSQ, 0)
  return false;
}

}  // namespace tqd
