// Instantiations of the decode and logits kernels for 2-bit key codes.  The codec
// combinations built are those of the schemes at n bits (Plain-KV, TQ-KV, KQV, QKQV) and the
// HeadQ key side; other combinations report "not built".
#include "tq_decode_kernel.cuh"

namespace tqd {

bool dispatch_decode_k2(int kq, int kh, int vb, int vq, const DecodeParams& p, dim3 g, cudaStream_t s,
                        cudaError_t* e) {
  TQ_DECODE_CASE(2, 0, 0, 2, 0)
  TQ_DECODE_CASE(2, 0, 0, 1, 1)
  TQ_DECODE_CASE(2, 1, 0, 2, 1)
  TQ_DECODE_CASE(2, 0, 1, 2, 0)
  TQ_DECODE_CASE(2, 0, 1, 4, 0)
  TQ_DECODE_CASE(2, 0, 1, 1, 1)
  return false;
}

bool dispatch_logits_k2(int kq, int kh, const LogitsParams& p, dim3 g, cudaStream_t s, cudaError_t* e) {
  TQ_LOGITS_CASE(2, 0, 0)
  TQ_LOGITS_CASE(2, 1, 0)
  TQ_LOGITS_CASE(2, 0, 1)
  return false;
}

}  // namespace tqd
