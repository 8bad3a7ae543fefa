// Decode kernels for head dim 1024 (one translation unit per head dim, compiled in parallel).
#include "tq_decode_wide.cuh"

namespace tqd {

bool dispatch_decode_wide_d1024(int kb, int vb, int vq, const DecodeParams& p, dim3 g, cudaStream_t s,
                              cudaError_t* e) {
  TQ_WIDE_CASES(1024)
}

cudaError_t launch_finalize_sketch(int D, const float* T, const float* sk, float* part, float* out, int H, int m,
                                   float scale, cudaStream_t s) {
  const int slices = m / kSkRows;
  const dim3 g1(D / kSkCols, (H + kSkHeads - 1) / kSkHeads, slices);
  const dim3 g2((unsigned)(((long long)H * D + 255) / 256));
  switch (D) {
    case 256:
      sketch_partial_kernel<256><<<g1, 256, 0, s>>>(T, sk, part, H, m);
      sketch_reduce_kernel<256><<<g2, 256, 0, s>>>(part, out, H, slices, scale);
      break;
    case 512:
      sketch_partial_kernel<512><<<g1, 256, 0, s>>>(T, sk, part, H, m);
      sketch_reduce_kernel<512><<<g2, 256, 0, s>>>(part, out, H, slices, scale);
      break;
    case 1024:
      sketch_partial_kernel<1024><<<g1, 256, 0, s>>>(T, sk, part, H, m);
      sketch_reduce_kernel<1024><<<g2, 256, 0, s>>>(part, out, H, slices, scale);
      break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace tqd
