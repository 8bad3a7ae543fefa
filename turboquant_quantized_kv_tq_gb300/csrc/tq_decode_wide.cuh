// Fused decode attention for head dims 256, 512 and 1024 (no key-side QJL, no HeadQ).
//
// The same rotated-domain decode as the head-dim-128 kernel ([HEADQ] "Espaço de Pontuação da
// Chave" / "Geometria de Leitura de Valores"; [TQ-KV] "Contribuciones Clave" 1 for the value
// sketch), with each 16-token tile shared by a group of D / 128 warps: warp `sl` of a group owns
// coordinates [128 sl, 128 sl + 128) of every code stream, the query and the accumulators.  Per
// tile, each warp computes its slice's partial key scores with the head-dim-128 building blocks,
// the group adds the D / 128 partials through a shared-memory exchange (one named barrier per
// tile; every warp sums them in the same order, so all warps hold identical scores and identical
// softmax state), and each warp accumulates the value readout of its own slice.  With a QJL value
// side the sketch readout rides in query columns G .. 2 G - 1 of the value MMA, as in the
// head-dim-128 kernel, so every variant runs the same 16 warps per block.
//
// Loads: per group, a ring of single-tile stages (K block then V block, one bulk copy each)
// issued by the group's first lane and refilled once the exchange barrier shows that every warp
// of the group has read the stage.  Work split: the stream-K tile partition of the head-dim-128
// kernel, a block's segment cut into one contiguous sub-range per group.  The last block of a
// slab merges the partials and writes o = R_V^T acc / l; with a QJL value side it also leaves
// acc_sk / l in the workspace for the sketch kernels, which add
// sqrt(pi/2)/m (S_V R_V)^T acc_sk / l = sqrt(pi/2)/m R_V^T S_V^T acc_sk / l for all heads at once
// (one pass over the m x d table instead of one per slab).
#pragma once

#include "tq_decode_kernel.cuh"

namespace tqd {

template <int D, int KB, int VB, bool VQ>
struct WideCfg {
  static constexpr int DS = D / kDecD;                  // warps per group
  static constexpr int NG = 512 / (DS * 32);             // groups per block
  static constexpr int NW = DS * NG;
  static constexpr int kSlots = 3;                       // single-tile stages per group
  using S = Stage<KB, false, false, VB, VQ, D>;
  static constexpr int PS = 4 + D + (VQ ? D : 0);        // per head: m, l, pad, pad, acc, (acc_sk)
  static constexpr uint32_t lutK = LutEntries<KB>::value * kLutStride;
  static constexpr uint32_t lutV = KB == VB ? 0 : LutEntries<VB>::value * kLutStride;
  static constexpr bool sepV = lutV > 0;
  static constexpr uint32_t ring = kSlots * S::bytes;
  static constexpr uint32_t xch = 2 * DS * 32 * 16;       // partial-score exchange, double-buffered
  static constexpr int kHeads = 4;                         // query heads per KV head (G <= 4 here)
  static constexpr uint32_t mslot = kHeads * PS * 4;       // merge slot of the group
  static constexpr uint32_t RS0 = ring + xch > mslot ? ring + xch : mslot;
  static constexpr uint32_t RS = (RS0 + 15) / 16 * 16;
  using Plan = RegionPlan<lutK, lutV, RS, NG>;
  static constexpr uint32_t bytes = Plan::bars + NG * kSlots * 8;
  static_assert(S::bytes % 16 == 0, "stages must keep 16-byte alignment");
  static_assert(2 * D * 4 <= RS, "the final merge buffer does not fit a region");
};

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

// Bulk copies of one 16-token tile (K block, V block) into the stage at shared address `st`.
template <int D, int KB, int VB, bool VQ>
__device__ __forceinline__ void issue_tile(uint32_t st, uint32_t bar, const SlabPtrs& s, int tile) {
  using S = Stage<KB, false, false, VB, VQ, D>;
  constexpr uint32_t KBL = S::VC, VBL = S::bytes - S::VC;
  mbar_arrive_expect_tx(bar, KBL + VBL);
  bulk_g2s(st, s.kb + (unsigned long long)tile * KBL, KBL, bar);
  bulk_g2s(st + KBL, s.vb + (unsigned long long)tile * VBL, VBL, bar);
}

template <int D, int KB, int VB, bool VQ>
__global__ void __launch_bounds__(WideCfg<D, KB, VB, VQ>::NW * 32, 1) decode_wide_kernel(const DecodeParams p) {
  using C = WideCfg<D, KB, VB, VQ>;
  using SG = typename C::S;
  using PL = typename C::Plan;
  constexpr int PS = C::PS;
  constexpr int DS = C::DS;
  constexpr int E = D / 32;  // coordinates per lane in the final transform
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int lg = lane >> 2, lt = lane & 3;
  const int grp = warp / DS, sl = warp % DS;

  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(smem);
  if (sbase > kDynBaseMax) {
    if (threadIdx.x == 0) atomicExch(p.err, kErrSmemPlan);
    return;
  }
  unsigned char* const win = smem - sbase;
  if constexpr (KB != 1) build_lut<KB>(win + kLutAddrK, p.tab.k_c);
  if constexpr (C::sepV && VB != 1) build_lut<VB>(win + kLutAddrV, p.tab.v_c);
  const uint32_t k_m0 = pack_half2(__ldg(p.tab.k_c + 1), __ldg(p.tab.k_c + 1));
  const uint32_t v_m0 = pack_half2(__ldg(p.tab.v_c + 1), __ldg(p.tab.v_c + 1));
  const uint32_t lxK = kLutAddrK | (4u * lane);
  const uint32_t lxV = (C::sepV ? kLutAddrV : kLutAddrK) | (4u * lane);
  const uint32_t gbars = PL::bars + grp * C::kSlots * 8;
  if (sl == 0 && lane < C::kSlots) mbar_init(gbars + 8 * lane, 1);
  fence_mbar_init();
  __syncthreads();

  const uint32_t ring_s = PL::region(grp);
  unsigned char* ring = win + ring_s;
  float4* xch = reinterpret_cast<float4*>(ring + C::ring);  // [2][DS][32]
  const bool leader = sl == 0 && lane == 0;
  const int G = p.G;
  const int Hq = p.Hkv * G;
  const int N = p.nblocks;
  long long x = (long long)blockIdx.x * p.W / N;
  const long long x_end = (long long)(blockIdx.x + 1) * p.W / N;
  unsigned seq = 0;  // tiles this group has streamed so far: slot seq % S, phase (seq / S) & 1
  bool timed_out = false;
  const uint32_t zero16[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
  const uint32_t zero2[2] = {0u, 0u};

  while (x < x_end) {
    // ---- locate the slab segment that starts at tile x
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.batch_start[mid] <= x) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int L = p.seq_len[b];
    const int ntb = (L + kTile - 1) / kTile;
    const long long off = x - p.batch_start[b];
    const int kvh = (int)(off / ntb);
    const int ts = (int)(off % ntb);
    const long long slab_start = p.batch_start[b] + (long long)kvh * ntb;
    const long long seg_end = min(x_end, slab_start + ntb);
    const int te = ts + (int)(seg_end - x);
    const int pair = b * p.Hkv + kvh;

    // ---- query fragments of this warp's slice: column lg of KV head kvh (columns G .. 2 G - 1
    // hold the lo terms), dims 128 sl + [32 lt, 32 lt + 32)
    const bool hv = lg < 2 * G;
    const long long qrow = (long long)(b * p.Hkv + kvh) * kQCols + (hv ? lg : 0);
    uint32_t qf[16];
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
      const uint4 v = hv ? *reinterpret_cast<const uint4*>(p.q_rot + qrow * (D / 2) + 64 * sl + 16 * lt + i)
                         : make_uint4(0, 0, 0, 0);
      qf[i] = v.x; qf[i + 1] = v.y; qf[i + 2] = v.z; qf[i + 3] = v.w;
    }

    // ---- this group's tiles of the segment
    const int n = te - ts;
    const int per = (n + C::NG - 1) / C::NG;
    const int m0t = min(te, ts + grp * per);
    const int m1t = min(te, m0t + per);
    const int nt = m1t - m0t;
    SlabPtrs sp;
    sp.init(p.cache, b, kvh);
    WarpState<false> st;  // a value sketch's readout shares the value MMA (columns G .. 2 G - 1)
    st.reset();
    if (leader) {
      for (int i = 0; i < C::kSlots && i < nt; ++i) {
        const unsigned slot = (seq + i) % C::kSlots;
        issue_tile<D, KB, VB, VQ>(ring_s + slot * SG::bytes, gbars + 8 * slot, sp, m0t + i);
      }
    }
    for (int i = 0; i < nt; ++i) {
      const unsigned cur = seq + i, slot = cur % C::kSlots;
      if (!mbar_wait(gbars + 8 * slot, (cur / C::kSlots) & 1u, kWaitLimit)) timed_out = true;
      const unsigned char* stg = ring + slot * SG::bytes;
      TileData<KB, false, false, VB, VQ> d[2];
      read_stage<KB, false, false, VB, VQ, D>(d[0], stg, stg, lg, lt, sl);
      fence_proxy_async_shared();
      float s[1][4];
      key_scores(d[0], s[0], qf, zero16, zero2, lxK, k_m0, p.qjl_scale, p.score_scale, zero16, zero16, p.lo_xor);
      float4* xb = xch + (i & 1) * DS * 32;
      xb[sl * 32 + lane] = make_float4(s[0][0], s[0][1], s[0][2], s[0][3]);
      named_barrier(1 + grp, DS * 32);  // every warp of the group has read the stage and written
      if (leader && i + C::kSlots < nt)
        issue_tile<D, KB, VB, VQ>(ring_s + slot * SG::bytes, gbars + 8 * slot, sp, m0t + i + C::kSlots);
      float4 t = xb[lane];
#pragma unroll
      for (int w = 1; w < DS; ++w) {
        const float4 u = xb[w * 32 + lane];
        t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
      }
      s[0][0] = t.x; s[0][1] = t.y; s[0][2] = t.z; s[0][3] = t.w;
      const int t0 = (m0t + i) * kTile;
      if (t0 + kTile <= L)
        softmax_readout<1, false, VQ>(d, s, st, lxV, v_m0, t0, L, L, G, G, lg);
      else
        softmax_readout<1, true, VQ>(d, s, st, lxV, v_m0, t0, L, L, G, G, lg);
    }
    seq += nt;

    // ---- merge the groups of this block for this segment
    float l0 = st.l0, l1 = st.l1;
#pragma unroll
    for (int m = 4; m <= 16; m <<= 1) {
      l0 += __shfl_xor_sync(kFull, l0, m);
      l1 += __shfl_xor_sync(kFull, l1, m);
    }
    __syncthreads();  // every group is done with its ring and exchange: reuse them for the merge
    float* mg = reinterpret_cast<float*>(win + PL::region(grp));
    // column c < G: head c's m, l and code readout; G <= c < 2 G (QJL value side): head c - G's
    // sketch readout; other columns carry nothing
    const int c0 = 2 * lt, c1 = 2 * lt + 1;
    if (sl == 0 && lg == 0) {
      if (c0 < G) { mg[c0 * PS + 0] = st.m0; mg[c0 * PS + 1] = l0; }
      if (c1 < G) { mg[c1 * PS + 0] = st.m1; mg[c1 * PS + 1] = l1; }
    }
    const int o0 = c0 < G ? c0 * PS + 4 : (VQ && c0 < 2 * G ? (c0 - G) * PS + 4 + D : -1);
    const int o1 = c1 < G ? c1 * PS + 4 : (VQ && c1 < 2 * G ? (c1 - G) * PS + 4 + D : -1);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int d0 = kDecD * sl + 16 * lg + 2 * mt;
      if (o0 >= 0) {
        mg[o0 + d0] = st.acc[mt][0];
        mg[o0 + d0 + 1] = st.acc[mt][2];
      }
      if (o1 >= 0) {
        mg[o1 + d0] = st.acc[mt][1];
        mg[o1 + d0 + 1] = st.acc[mt][3];
      }
    }
    __syncthreads();
    float* part_out = p.part + ((long long)(pair + blockIdx.x) * G) * PS;
    for (int idx = threadIdx.x; idx < G * PS; idx += blockDim.x) {
      const int h = idx / PS, e = idx % PS;
      float M = -INFINITY;
#pragma unroll
      for (int g = 0; g < C::NG; ++g) M = fmaxf(M, reinterpret_cast<const float*>(win + PL::region(g))[h * PS]);
      float v;
      if (e == 0) {
        v = M;
      } else if (e == 2 || e == 3) {
        v = 0.f;
      } else {
        v = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int g = 0; g < C::NG; ++g) {
            const float* mgg = reinterpret_cast<const float*>(win + PL::region(g)) + h * PS;
            v = fmaf(exp2f(mgg[0] - M), mgg[e], v);
          }
        }
      }
      part_out[h * PS + e] = v;
    }

    // ---- the last block of this slab merges all its partials
    const int c_first = owner_block(slab_start, p.W, N);
    const int c_last = owner_block(slab_start + ntb - 1, p.W, N);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const int prev = atomicAdd(p.tickets + pair, 1);
      s_last = prev == c_last - c_first;
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      float* fin = reinterpret_cast<float*>(win + PL::region(0));  // acc [D], then acc_sk [D]
      const long long sstride = (long long)G * PS;
      const int ns = c_last - c_first + 1;
      for (int h = 0; h < G; ++h) {
        const float* base = p.part + (long long)(pair + c_first) * sstride + h * PS;
        float M = -INFINITY;
        for (int s2 = 0; s2 < ns; ++s2) M = fmaxf(M, __ldcg(base + s2 * sstride));
        float L2 = 0.f;
        if (M != -INFINITY)
          for (int s2 = 0; s2 < ns; ++s2) L2 = fmaf(exp2f(__ldcg(base + s2 * sstride) - M), __ldcg(base + s2 * sstride + 1), L2);
        const float invL = L2 > 0.f ? 1.f / L2 : 0.f;
        for (int i = threadIdx.x; i < (VQ ? 2 * D : D); i += blockDim.x) {
          float v = 0.f;
          if (M != -INFINITY)
            for (int s2 = 0; s2 < ns; ++s2)
              v = fmaf(exp2f(__ldcg(base + s2 * sstride) - M), __ldcg(base + s2 * sstride + 4 + i), v);
          fin[i] = v;
        }
        __syncthreads();
        const long long head = (long long)b * Hq + kvh * G + h;
        if constexpr (VQ) {
          for (int i = threadIdx.x; i < D; i += blockDim.x) p.sk_final[head * D + i] = fin[D + i] * invL;
        }
        if (warp == 0) {
          float o[E];
#pragma unroll
          for (int e = 0; e < E; ++e) o[e] = fin[lane * E + e];
          if (p.v_rotate) {
            wht_warp<E>(o);
            const float rs = 1.f / sqrtf((float)D);
#pragma unroll
            for (int e = 0; e < E; ++e) o[e] = o[e] * rs * __ldg(p.tab.v_sign + lane * E + e) * invL;
          } else {
#pragma unroll
            for (int e = 0; e < E; ++e) o[e] *= invL;
          }
          float* dst = p.out + head * D + lane * E;
#pragma unroll
          for (int e = 0; e < E; e += 4) *reinterpret_cast<float4*>(dst + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
        }
        __syncthreads();
      }
      if (threadIdx.x == 0) p.tickets[pair] = 0;
    }
    __syncthreads();  // the merge area becomes the next segment's stages
    x = seg_end;
  }
  if (timed_out) atomicExch(p.err, kErrWaitTimeout);
}

// The value-sketch term for all H heads at once: out[h][i] += scale * sum_j T[j][i] sk[h][j]
// (T = S_V R_V, [m][D]; sk = acc_sk / l, [H][m]).  Stage 1: block (x, y, z) multiplies the
// 32-head x 64-row tile of sk by the 64-row x 64-column tile of T (both staged in shared
// memory; each thread owns 2 heads x 4 columns) and writes a partial for its row slice z.
// Stage 2 adds the m / 64 partials in slice order, so the result does not depend on timing.
constexpr int kSkRows = 64, kSkCols = 64, kSkHeads = 32;

template <int D>
__global__ void __launch_bounds__(256) sketch_partial_kernel(const float* __restrict__ T,
                                                             const float* __restrict__ sk,
                                                             float* __restrict__ part, int H, int m) {
  __shared__ float As[kSkHeads][kSkRows + 1];
  __shared__ float Bs[kSkRows][kSkCols];
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int c0 = blockIdx.x * kSkCols, h0 = blockIdx.y * kSkHeads, k0 = blockIdx.z * kSkRows;
  for (int idx = tid; idx < kSkHeads * kSkRows; idx += 256) {
    const int hh = idx / kSkRows, kk = idx % kSkRows;
    As[hh][kk] = h0 + hh < H ? __ldg(sk + (long long)(h0 + hh) * m + k0 + kk) : 0.f;
  }
  for (int idx = tid; idx < kSkRows * kSkCols; idx += 256) {
    const int kk = idx / kSkCols, cc = idx % kSkCols;
    Bs[kk][cc] = __ldg(T + (long long)(k0 + kk) * D + c0 + cc);
  }
  __syncthreads();
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 8
  for (int kk = 0; kk < kSkRows; ++kk) {
    const float a0 = As[ty][kk], a1 = As[ty + 16][kk];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float bv = Bs[kk][tx + 16 * i];
      acc[0][i] = fmaf(a0, bv, acc[0][i]);
      acc[1][i] = fmaf(a1, bv, acc[1][i]);
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int h = h0 + ty + 16 * r;
    if (h < H) {
#pragma unroll
      for (int i = 0; i < 4; ++i) part[((long long)blockIdx.z * H + h) * D + c0 + tx + 16 * i] = acc[r][i];
    }
  }
}

template <int D>
__global__ void __launch_bounds__(256) sketch_reduce_kernel(const float* __restrict__ part, float* out, int H,
                                                            int slices, float scale) {
  const long long i = (long long)blockIdx.x * 256 + threadIdx.x;
  if (i >= (long long)H * D) return;
  float v = 0.f;
  for (int z = 0; z < slices; ++z) v += part[(long long)z * H * D + i];
  out[i] = fmaf(scale, v, out[i]);
}

template <int D, int KB, int VB, bool VQ>
cudaError_t launch_decode_wide_t(const DecodeParams& p, dim3 grid, cudaStream_t s) {
  using C = WideCfg<D, KB, VB, VQ>;
  static_assert(C::bytes <= 227 * 1024, "decode shared memory exceeds the per-block limit");
  cudaError_t e = check_dyn_base(decode_wide_kernel<D, KB, VB, VQ>);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_wide_kernel<D, KB, VB, VQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)C::bytes);
  if (e != cudaSuccess) return e;
  decode_wide_kernel<D, KB, VB, VQ><<<grid, C::NW * 32, C::bytes, s>>>(p);
  return cudaGetLastError();
}

// Per-head-dim dispatchers (one translation unit each); false when the codecs are not built.
bool dispatch_decode_wide_d256(int kb, int vb, int vq, const DecodeParams& p, dim3 g, cudaStream_t s, cudaError_t* e);
bool dispatch_decode_wide_d512(int kb, int vb, int vq, const DecodeParams& p, dim3 g, cudaStream_t s, cudaError_t* e);
bool dispatch_decode_wide_d1024(int kb, int vb, int vq, const DecodeParams& p, dim3 g, cudaStream_t s, cudaError_t* e);
cudaError_t launch_finalize_sketch(int D, const float* T, const float* sk, float* part, float* out, int H, int m,
                                   float scale, cudaStream_t s);

#define TQ_WIDE_CASES(D_)                                                                   \
  if (kb == 1 && vb == 1 && !vq) { if (e) *e = launch_decode_wide_t<D_, 1, 1, false>(p, g, s); return true; } \
  if (kb == 2 && vb == 2 && !vq) { if (e) *e = launch_decode_wide_t<D_, 2, 2, false>(p, g, s); return true; } \
  if (kb == 3 && vb == 3 && !vq) { if (e) *e = launch_decode_wide_t<D_, 3, 3, false>(p, g, s); return true; } \
  if (kb == 4 && vb == 4 && !vq) { if (e) *e = launch_decode_wide_t<D_, 4, 4, false>(p, g, s); return true; } \
  if (kb == 2 && vb == 1 && vq) { if (e) *e = launch_decode_wide_t<D_, 2, 1, true>(p, g, s); return true; }   \
  if (kb == 3 && vb == 2 && vq) { if (e) *e = launch_decode_wide_t<D_, 3, 2, true>(p, g, s); return true; }   \
  if (kb == 4 && vb == 3 && vq) { if (e) *e = launch_decode_wide_t<D_, 4, 3, true>(p, g, s); return true; }   \
  return false;

}  // namespace tqd
