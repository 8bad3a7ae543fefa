// Chunked-prefill attention over the packed cache (head dim 128): many queries per KV head.
//
// [ABL] "Recomendações Práticas" 2 names prefill workloads; [HEADQ] "Espaço de Pontuação da
// Chave" / "Geometria de Leitura de Valores" give the scores q^T k / sqrt(d) and the weighted
// value sum; [TQ-KV] "Contribuciones Clave" 1 the QJL estimate of a residual inner product.
//
// The rows of one (batch, KV head) slab are the chunk's (query, head) pairs, r = i G + g, and
// row r attends to the first L - nq + 1 + r / G tokens.  A block takes 128 rows (8 warps x 16)
// and walks the slab's tokens in 32-token tiles.  Each tile's packed K and V are unpacked once
// per block into shared memory as fp16 rows of the rotated domain -- C[c], and on a QJL side
// rho (2 sigma - 1) (keys) or 2 sigma - 1 (values) -- so the scores and the readout are dense
// tensor-core products (mma.sync m16n8k16, fp32 accumulation):
//   S[16 rows x 32 tok]  = Q_hi K_hi^T + Q_lo K_hi^T + Q_hi K_lo^T (+ (c S_K q_rot) (rho (2 sigma - 1))^T)
//   acc[16 x 128]       += (p nu_V) V_hat,   acc_sk[16 x 128] += (p nu_V rho_V) (2 sigma_V - 1)
// with an online softmax (log2 domain) in between.  The epilogue forms
// o = R_V^T (acc + c S_V^T acc_sk) / l in the accumulator layout: the sketch product is one more
// MMA against S_V^T staged as fp16, and the inverse Walsh-Hadamard transform's stages run in
// registers (two of its seven stages cross lanes).  The queries and the key centroids enter as
// fp16 hi + lo terms: a single rounding of q is a score error common to every token of a row,
// and one of a centroid an error common to every token with that code; with peaked attention
// (outlier channels) either reaches the output undiluted.
#include <algorithm>
#include <string>

#include "tq_device.cuh"
#include "tq_tc05.cuh"

namespace tqd {
namespace {

constexpr int kPfWarps = 8;
constexpr int kPfRows = 16 * kPfWarps;  // rows per block
constexpr int kPfTok = 32;              // tokens per tile
constexpr int kPfPitch = 272;           // bytes per fp16 row of 128 (+ 8 halves: ldmatrix rows on distinct banks)
constexpr int kPfD = 128;
constexpr float kPfLog2e = 1.4426950408889634f;
constexpr float kPfFloor = -1e30f;      // running maximum of a row that has seen no token yet
constexpr uint32_t kPfWaitLimit = 1u << 20;  // polls of a stage's mbarrier before giving up

struct PrefillPrepParams {
  Tables tab;
  const float* q;  // [B][nq][Hq][128]
  __half* qhi;     // [B*Hkv][R_pad][128]
  __half* qlo;
  __half* qsk;     // c S_K q_rot (QJL key side)
  int B, Hkv, G, nq, rows, R_pad;
  int k_rotate, kq;
  float qjl_scale;
  int* err;        // cleared here, before the prefill kernel runs
};

struct PrefillParams {
  Tables tab;
  Cache cache;
  const __half* qhi;
  const __half* qlo;
  const __half* qsk;
  float* out;  // [B][nq][Hq][128]
  int B, Hkv, G, nq, rows, R_pad;
  int kbits, vbits, v_rotate;
  unsigned kblk, vblk;  // bytes of one 16-token block of each side
  int* err;             // device error word (the workspace's first bytes)
  float score_scale;  // log2(e) / sqrt(d)
  float qjl_scale;    // sqrt(pi/2) / m
  int seq_len[TQ_MAX_BATCH];
};

// Shared-memory plan of a prefill block: the block's query rows (hi, lo, and the key-sketch
// products), the tile's unpacked key and value rows, and per-token scalars.
template <bool KQ, bool VQ>
struct PfSmem {
  static constexpr int QHI = 0;
  static constexpr int QLO = QHI + kPfRows * kPfPitch;
  static constexpr int QSK = QLO + kPfRows * kPfPitch;
  static constexpr int KC = QSK + (KQ ? kPfRows * kPfPitch : 0);
  static constexpr int KL = KC + kPfTok * kPfPitch;
  static constexpr int KS = KL + kPfTok * kPfPitch;
  static constexpr int VC = KS + (KQ ? kPfTok * kPfPitch : 0);
  static constexpr int VS = VC + kPfTok * kPfPitch;
  static constexpr int NUK = VS + (VQ ? kPfTok * kPfPitch : 0);
  static constexpr int NUV = NUK + kPfTok * 4;
  static constexpr int FV = NUV + kPfTok * 4;
  // two stages of packed tiles (bulk copies of two 16-token blocks per side) follow
  static constexpr int STG = (FV + kPfTok * 4 + 127) / 128 * 128;
  // the epilogue's S_V^T (fp16, 128 rows) reuses the query rows
  static_assert(QLO >= 0 && kPfD * kPfPitch <= KC, "S_V^T staging overlaps the tile");
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ float pf_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// The 4 W bits of coordinates 4 lane .. 4 lane + 3 of a W-bit stream (W = 1, 2, 4): a whole
// record at src (pos < 0), or a value-side stream stored by 16-coordinate groups at block
// position pos.
template <int W>
__device__ __forceinline__ uint32_t lane_bits(const unsigned char* src, int pos) {
  const unsigned lane = threadIdx.x & 31;
  if constexpr (W == 4) {
    const unsigned j = 2 * lane;  // even, and so is its grouped position
    return *reinterpret_cast<const unsigned short*>(pos < 0 ? src + j : src + grouped_byte(j, (unsigned)pos, 4));
  } else if constexpr (W == 2) {
    return pos < 0 ? src[lane] : src[grouped_byte(lane, (unsigned)pos, 2)];
  } else {
    const unsigned j = lane >> 1;
    const uint32_t byte = pos < 0 ? src[j] : src[grouped_byte(j, (unsigned)pos, 1)];
    return (byte >> (4 * (lane & 1))) & 0xFu;
  }
}

// Centroids C[c] of this lane's four coordinates of one code record (sign-magnitude symbols: a
// sign bit s and a magnitude rank k give c = s ? 2^(b-1) + k : 2^(b-1) - 1 - k).
__device__ __forceinline__ void unpack_codes(const unsigned char* codes, int bits, int pos, int second,
                                             const float* cent, float (&y)[4]) {
  uint32_t mag = 0, sgn = 0;
  if (bits == 4) {
    const uint32_t v = lane_bits<4>(codes, pos);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      sgn |= ((v >> (4 * e + 3)) & 1u) << e;
      mag |= ((v >> (4 * e)) & 7u) << (4 * e);
    }
  } else if (bits == 3) {
    const uint32_t v = lane_bits<2>(codes, pos);
#pragma unroll
    for (int e = 0; e < 4; ++e) mag |= ((v >> (2 * e)) & 3u) << (4 * e);
    sgn = lane_bits<1>(codes + second, pos);
  } else if (bits == 2) {
    const uint32_t v = lane_bits<2>(codes, pos);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      sgn |= ((v >> (2 * e + 1)) & 1u) << e;
      mag |= ((v >> (2 * e)) & 1u) << (4 * e);
    }
  } else {
    sgn = lane_bits<1>(codes, pos);
  }
  const uint32_t half = 1u << (bits - 1);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const uint32_t k = (mag >> (4 * e)) & 7u;
    const uint32_t c = ((sgn >> e) & 1u) ? half + k : half - 1u - k;
    y[e] = __ldg(cent + c);
  }
}

// The packed blocks of tile `tile` of slab (b, h) -- nb 16-token blocks from block nb * tile --
// into a stage: the K blocks at dst, the V blocks at dst + nb * kblk.  The copy stops at the
// slab's last block, and the mbarrier expects the bytes actually copied.
__device__ __forceinline__ void pf_issue_stage(const Cache& C, int b, int h, int tile, int nb, unsigned kblk,
                                               unsigned vblk, uint32_t dst, uint32_t bar) {
  const int first = tile * nb;
  const int n = max(0, min(nb, C.tiles_per_slab - first));
  mbar_arrive_expect_tx(bar, (uint32_t)n * (kblk + vblk));
  if (n > 0) {
    bulk_g2s(dst, C.blockp(0, b, h, first), (uint32_t)n * kblk, bar);
    bulk_g2s(dst + (uint32_t)nb * kblk, C.blockp(1, b, h, first), (uint32_t)n * vblk, bar);
  }
}

__device__ __forceinline__ void st_half4(unsigned char* dst, const float (&v)[4]) {
  const uint32_t a = pack_half2(v[0], v[1]), b = pack_half2(v[2], v[3]);
  *reinterpret_cast<uint2*>(dst) = make_uint2(a, b);
}

// One warp per padded row of every slab: q_rot = R_K q, its fp16 hi and lo terms, and on a QJL
// key side c S_K q_rot (S_K^T staged in shared memory).  Padding rows are zero.
__global__ void __launch_bounds__(256) prefill_prep_kernel(const PrefillPrepParams p) {
  extern __shared__ __align__(16) float st[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (blockIdx.x == 0 && threadIdx.x == 0) *p.err = 0;
  if (p.kq) {
    stage_table<256>(st, p.tab.S_K_T, kPfD * kPfD);
    __syncthreads();
  }
  const int Hq = p.Hkv * p.G;
  const long long total = (long long)p.B * p.Hkv * p.R_pad;
  const float rs = 1.f / sqrtf((float)kPfD);
  for (long long w = (long long)blockIdx.x * 8 + warp; w < total; w += (long long)gridDim.x * 8) {
    const int slab = (int)(w / p.R_pad), r = (int)(w % p.R_pad);
    const int b = slab / p.Hkv, h = slab % p.Hkv;
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if (r < p.rows) {
      const int i = r / p.G, g = r % p.G;
      const float4 v = *reinterpret_cast<const float4*>(p.q + (((long long)b * p.nq + i) * Hq + h * p.G + g) * kPfD + 4 * lane);
      x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
      if (p.k_rotate) {
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] *= __ldg(p.tab.k_sign + 4 * lane + e);
        wht_warp<4>(x);
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] *= rs;
      }
    }
    float hi[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      hi[e] = __half2float(__float2half_rn(x[e]));
      lo[e] = x[e] - hi[e];
    }
    st_half4(reinterpret_cast<unsigned char*>(p.qhi + w * kPfD + 4 * lane), hi);
    st_half4(reinterpret_cast<unsigned char*>(p.qlo + w * kPfD + 4 * lane), lo);
    if (p.kq) {  // a_i = c sum_j S_K[i][j] q_rot[j], i = 4 lane + e
      float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
      for (int j = 0; j < kPfD; ++j) {
        const float xj = __shfl_sync(kFull, x[j & 3], j >> 2);
        const float4 s4 = *reinterpret_cast<const float4*>(st + j * kPfD + 4 * lane);
        a[0] = fmaf(s4.x, xj, a[0]); a[1] = fmaf(s4.y, xj, a[1]);
        a[2] = fmaf(s4.z, xj, a[2]); a[3] = fmaf(s4.w, xj, a[3]);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) a[e] *= p.qjl_scale;
      st_half4(reinterpret_cast<unsigned char*>(p.qsk + w * kPfD + 4 * lane), a);
    }
  }
}

template <bool KQ, bool VQ>
__global__ void __launch_bounds__(kPfWarps * 32, 1) prefill_kernel(const PrefillParams p) {
  using SM = PfSmem<KQ, VQ>;
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int slab = blockIdx.y;
  const int b = slab / p.Hkv, h = slab % p.Hkv;
  const int r0 = blockIdx.x * kPfRows;
  const int L = p.seq_len[b];
  const int Lmin = L - p.nq + 1;  // causal end of the chunk's first query
  const int rlast = min(r0 + kPfRows, p.rows) - 1;
  const int eblk = max(0, min(L, Lmin + rlast / p.G));  // tokens any row of the block sees
  const uint32_t sb = (uint32_t)__cvta_generic_to_shared(smem);

  // ---- the block's query rows into shared memory (16-byte pieces)
  {
    const long long row0 = (long long)slab * p.R_pad + r0;
    const int n16 = kPfRows * (kPfD * 2 / 16);
    for (int i = threadIdx.x; i < n16; i += blockDim.x) {
      const int rr = i >> 4, c = i & 15;
      const long long src = (row0 + rr) * kPfD + 8 * c;
      *reinterpret_cast<uint4*>(smem + SM::QHI + rr * kPfPitch + 16 * c) = *reinterpret_cast<const uint4*>(p.qhi + src);
      *reinterpret_cast<uint4*>(smem + SM::QLO + rr * kPfPitch + 16 * c) = *reinterpret_cast<const uint4*>(p.qlo + src);
      if constexpr (KQ)
        *reinterpret_cast<uint4*>(smem + SM::QSK + rr * kPfPitch + 16 * c) = *reinterpret_cast<const uint4*>(p.qsk + src);
    }
  }

  // ---- this warp's rows: lane rows g (A) and g + 8 (B) of the warp's 16
  const int rw0 = r0 + 16 * warp;
  const int rA = rw0 + g, rB = rA + 8;
  const int eA = rA < p.rows ? Lmin + rA / p.G : 0;
  const int eB = rB < p.rows ? Lmin + rB / p.G : 0;
  const int ew = rw0 < p.rows ? max(0, min(L, Lmin + (min(rw0 + 15, p.rows - 1)) / p.G)) : 0;
  float mA = kPfFloor, mB = kPfFloor, lA = 0.f, lB = 0.f;
  float acc[16][4], accs[VQ ? 16 : 1][4];
#pragma unroll
  for (int n = 0; n < 16; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc[n][e] = 0.f;
      if constexpr (VQ) accs[n][e] = 0.f;
    }
  const Cache& C = p.cache;
  const float* kcent = p.tab.k_c;
  const float* vcent = p.tab.v_c;
  float* nuK = reinterpret_cast<float*>(smem + SM::NUK);
  float* nuV = reinterpret_cast<float*>(smem + SM::NUV);
  float* fV = reinterpret_cast<float*>(smem + SM::FV);
  // ldmatrix lane addressing: matrix mi = lane / 8, row lane % 8 of it
  const int mi = lane >> 3, mr = lane & 7;

  // packed tiles stream through two shared-memory stages: one bulk copy per side brings the
  // tile's two 16-token blocks (adjacent in the slab), completing on the stage's mbarrier
  __shared__ __align__(8) unsigned long long s_bars[2];
  const uint32_t bar0 = (uint32_t)__cvta_generic_to_shared(&s_bars[0]);
  const unsigned kblk = p.kblk, vblk = p.vblk, SB = 2 * (kblk + vblk);
  const int ntiles = (eblk + kPfTok - 1) / kPfTok;
  if (threadIdx.x == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8, 1);
    fence_mbar_init();
    for (int k = 0; k < 2 && k < ntiles; ++k) {
      const uint32_t dst = sb + SM::STG + k * SB;
      pf_issue_stage(C, b, h, k, 2, kblk, vblk, dst, bar0 + 8 * k);
    }
  }
  bool timed_out = false;

  for (int k = 0; k < ntiles; ++k) {
    const int t0 = k * kPfTok, stage = k & 1;
    __syncthreads();  // the previous tile's rows are consumed (and the queries are in place)
    if (!mbar_wait(bar0 + 8 * stage, (uint32_t)(k >> 1) & 1u, kPfWaitLimit)) timed_out = true;
    const unsigned char* stg = smem + SM::STG + stage * SB;
    // ---- unpack the tile: warp w takes token rows 4 w .. 4 w + 3 of each side
#pragma unroll 1
    for (int jj = 0; jj < 4; ++jj) {
      const int j = 4 * warp + jj, tok = t0 + j;
      const bool ok = tok < L;
      const int pos = j & (tqi::kTileTokens - 1);
      const unsigned char* kp = stg + (j >> 4) * kblk;             // the token's K block
      const unsigned char* vp = stg + 2 * kblk + (j >> 4) * vblk;  // and V block
      float y[4] = {0.f, 0.f, 0.f, 0.f};
      float nu = 0.f;
      if (ok) {
        unpack_codes(kp + C.off[tqi::R_K_CODES] + pos * C.rec[tqi::R_K_CODES], p.kbits, -1, kPfD / 4, kcent, y);
        nu = *reinterpret_cast<const float*>(kp + C.off[tqi::R_K_NORM] + 4 * pos);
      }
      float yl[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float hi = __half2float(__float2half_rn(y[e]));
        yl[e] = y[e] - hi;
      }
      st_half4(smem + SM::KC + j * kPfPitch + 8 * lane, y);
      st_half4(smem + SM::KL + j * kPfPitch + 8 * lane, yl);
      if (lane == 0) nuK[j] = nu;
      if constexpr (KQ) {
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        if (ok) {
          const uint32_t sg = lane_bits<1>(kp + C.off[tqi::R_K_SIGNS] + pos * C.rec[tqi::R_K_SIGNS], -1);
          const float rho = __half2float(*reinterpret_cast<const __half*>(kp + C.off[tqi::R_K_RHO] + 2 * pos));
#pragma unroll
          for (int e = 0; e < 4; ++e) s[e] = ((sg >> e) & 1u) ? rho : -rho;
        }
        st_half4(smem + SM::KS + j * kPfPitch + 8 * lane, s);
      }
      // value row: streams by coordinate groups at block position pos
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      float nv = 0.f, fv = 0.f;
      if (ok) {
        unpack_codes(vp + C.off[tqi::R_V_CODES], p.vbits, pos, tqi::kTileTokens * (kPfD / 4), vcent, v);
        nv = *reinterpret_cast<const float*>(vp + C.off[tqi::R_V_NORM] + 4 * pos);
        if constexpr (VQ) fv = nv * __half2float(*reinterpret_cast<const __half*>(vp + C.off[tqi::R_V_RHO] + 2 * pos));
      }
      st_half4(smem + SM::VC + j * kPfPitch + 8 * lane, v);
      if (lane == 0) {
        nuV[j] = nv;
        fV[j] = fv;
      }
      if constexpr (VQ) {
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        if (ok) {
          const uint32_t sg = lane_bits<1>(vp + C.off[tqi::R_V_SIGNS], pos);
#pragma unroll
          for (int e = 0; e < 4; ++e) s[e] = ((sg >> e) & 1u) ? 1.f : -1.f;
        }
        st_half4(smem + SM::VS + j * kPfPitch + 8 * lane, s);
      }
    }
    __syncthreads();
    // the stage is read: refill it with tile k + 2
    if (threadIdx.x == 0 && k + 2 < ntiles) {
      fence_proxy_async_shared();
      const uint32_t dst = sb + SM::STG + stage * SB;
      pf_issue_stage(C, b, h, k + 2, 2, kblk, vblk, dst, bar0 + 8 * stage);
    }
    if (t0 >= ew) continue;  // every row of this warp is past its causal end (warp-uniform)

    // ---- scores of the warp's 16 rows against the tile's 32 tokens (4 n-tiles of 8)
    float s[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[n][e] = 0.f;
    const uint32_t qa = sb + (16 * warp + mr + 8 * (mi & 1)) * kPfPitch + 16 * (mi >> 1);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t a0, a1, a2, a3, l0, l1, l2, l3;
      ldsm_x4(qa + SM::QHI + 32 * ks, a0, a1, a2, a3);
      ldsm_x4(qa + SM::QLO + 32 * ks, l0, l1, l2, l3);
      uint32_t z0, z1, z2, z3;
      if constexpr (KQ) ldsm_x4(qa + SM::QSK + 32 * ks, z0, z1, z2, z3);
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        const uint32_t kb = sb + (16 * np + mr + 8 * (mi >> 1)) * kPfPitch + 32 * ks + 16 * (mi & 1);
        uint32_t b0, b1, b2, b3, d0, d1, d2, d3;
        ldsm_x4(kb + SM::KC, b0, b1, b2, b3);
        ldsm_x4(kb + SM::KL, d0, d1, d2, d3);
        mma16816(s[2 * np], a0, a1, a2, a3, b0, b1);
        mma16816(s[2 * np], l0, l1, l2, l3, b0, b1);
        mma16816(s[2 * np], a0, a1, a2, a3, d0, d1);
        mma16816(s[2 * np + 1], a0, a1, a2, a3, b2, b3);
        mma16816(s[2 * np + 1], l0, l1, l2, l3, b2, b3);
        mma16816(s[2 * np + 1], a0, a1, a2, a3, d2, d3);
        if constexpr (KQ) {
          uint32_t c0, c1, c2, c3;
          ldsm_x4(kb + SM::KS, c0, c1, c2, c3);
          mma16816(s[2 * np], z0, z1, z2, z3, c0, c1);
          mma16816(s[2 * np + 1], z0, z1, z2, z3, c2, c3);
        }
      }
    }
    // ---- key norms, causal masks, online softmax (log2 domain)
    float mxA = kPfFloor, mxB = kPfFloor;
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = 8 * n + 2 * t + e, tok = t0 + j;
        const float nu = nuK[j] * p.score_scale;
        s[n][e] = tok < eA ? s[n][e] * nu : -INFINITY;
        s[n][2 + e] = tok < eB ? s[n][2 + e] * nu : -INFINITY;
        mxA = fmaxf(mxA, s[n][e]);
        mxB = fmaxf(mxB, s[n][2 + e]);
      }
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
      mxA = fmaxf(mxA, __shfl_xor_sync(kFull, mxA, m));
      mxB = fmaxf(mxB, __shfl_xor_sync(kFull, mxB, m));
    }
    const float nA = fmaxf(mA, mxA), nB = fmaxf(mB, mxB);
    const float aA = pf_ex2(mA - nA), aB = pf_ex2(mB - nB);
    mA = nA;
    mB = nB;
    lA *= aA;
    lB *= aB;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      acc[n][0] *= aA; acc[n][1] *= aA; acc[n][2] *= aB; acc[n][3] *= aB;
      if constexpr (VQ) {
        accs[n][0] *= aA; accs[n][1] *= aA; accs[n][2] *= aB; accs[n][3] *= aB;
      }
    }
    // ---- readout: per 16-token chunk, P (times nu_V, and nu_V rho_V for the sketch) as the A
    // operand straight from the score layout; V_hat rows transposed by ldmatrix
#pragma unroll
    for (int kc = 0; kc < 2; ++kc) {
      float pw[2][4], ps[2][4];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int n = 2 * kc + hh;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = 8 * n + 2 * t + e;
          const float pa = pf_ex2(s[n][e] - nA), pb = pf_ex2(s[n][2 + e] - nB);
          lA += pa;
          lB += pb;
          const float nv = nuV[j];
          pw[hh][e] = pa * nv;
          pw[hh][2 + e] = pb * nv;
          if constexpr (VQ) {
            const float f = fV[j];
            ps[hh][e] = pa * f;
            ps[hh][2 + e] = pb * f;
          }
        }
      }
      const uint32_t p0 = pack_half2(pw[0][0], pw[0][1]), p1 = pack_half2(pw[0][2], pw[0][3]);
      const uint32_t p2 = pack_half2(pw[1][0], pw[1][1]), p3 = pack_half2(pw[1][2], pw[1][3]);
      uint32_t q0 = 0, q1 = 0, q2 = 0, q3 = 0;
      if constexpr (VQ) {
        q0 = pack_half2(ps[0][0], ps[0][1]); q1 = pack_half2(ps[0][2], ps[0][3]);
        q2 = pack_half2(ps[1][0], ps[1][1]); q3 = pack_half2(ps[1][2], ps[1][3]);
      }
      const uint32_t vb0 = sb + (16 * kc + mr + 8 * (mi & 1)) * kPfPitch + 16 * (mi >> 1);
#pragma unroll
      for (int dt = 0; dt < 8; ++dt) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb0 + SM::VC + 32 * dt, b0, b1, b2, b3);
        mma16816(acc[2 * dt], p0, p1, p2, p3, b0, b1);
        mma16816(acc[2 * dt + 1], p0, p1, p2, p3, b2, b3);
        if constexpr (VQ) {
          uint32_t c0, c1, c2, c3;
          ldsm_x4_t(vb0 + SM::VS + 32 * dt, c0, c1, c2, c3);
          mma16816(accs[2 * dt], q0, q1, q2, q3, c0, c1);
          mma16816(accs[2 * dt + 1], q0, q1, q2, q3, c2, c3);
        }
      }
    }
  }

  // ---- epilogue: o = R_V^T (acc + c S_V^T acc_sk) / l, in the accumulator layout
#pragma unroll
  for (int m = 1; m <= 2; m <<= 1) {
    lA += __shfl_xor_sync(kFull, lA, m);
    lB += __shfl_xor_sync(kFull, lB, m);
  }
  const float iA = lA > 0.f ? 1.f / lA : 0.f, iB = lB > 0.f ? 1.f / lB : 0.f;
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    acc[n][0] *= iA; acc[n][1] *= iA; acc[n][2] *= iB; acc[n][3] *= iB;
  }
  if constexpr (VQ) {
    // S_V^T [128 i][128 j] as fp16 rows over the query rows (every warp is past its last tile)
    __syncthreads();
    for (int idx = threadIdx.x; idx < kPfD * kPfD / 4; idx += blockDim.x) {
      const int i = idx >> 5, c4 = idx & 31;
      const float4 v = __ldg(reinterpret_cast<const float4*>(p.tab.S_V_T + i * kPfD + 4 * c4));
      const float vv[4] = {v.x, v.y, v.z, v.w};
      st_half4(smem + i * kPfPitch + 8 * c4, vv);
    }
    __syncthreads();
    // acc[r][i] += sum_j (c acc_sk[r][j] / l_r) S_V^T[i][j]: A = the scaled sketch accumulator
    // (score layout -> A operand, as P above), B = S_V^T rows (n = i, k = j)
    const float cA = iA * p.qjl_scale, cB = iB * p.qjl_scale;
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) {
      const uint32_t a0 = pack_half2(accs[2 * kc][0] * cA, accs[2 * kc][1] * cA);
      const uint32_t a1 = pack_half2(accs[2 * kc][2] * cB, accs[2 * kc][3] * cB);
      const uint32_t a2 = pack_half2(accs[2 * kc + 1][0] * cA, accs[2 * kc + 1][1] * cA);
      const uint32_t a3 = pack_half2(accs[2 * kc + 1][2] * cB, accs[2 * kc + 1][3] * cB);
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        const uint32_t sa = sb + (16 * np + mr + 8 * (mi >> 1)) * kPfPitch + 32 * kc + 16 * (mi & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sa, b0, b1, b2, b3);
        mma16816(acc[2 * np], a0, a1, a2, a3, b0, b1);
        mma16816(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
    }
  }
  // inverse rotation x = D_V H o_rot / sqrt(d).  Lane (g, t) holds, for each of its two rows,
  // coordinates 8 n + 2 t + e (n = 0..15, e = 0..1): butterflies over bit 0 (e) and bits 3-6 (n)
  // are local, over bits 1-2 (t) lane shuffles
  if (p.v_rotate) {
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      float x0 = acc[n][0], x1 = acc[n][1];
      acc[n][0] = x0 + x1; acc[n][1] = x0 - x1;
      x0 = acc[n][2]; x1 = acc[n][3];
      acc[n][2] = x0 + x1; acc[n][3] = x0 - x1;
    }
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
#pragma unroll
      for (int n = 0; n < 16; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float o = __shfl_xor_sync(kFull, acc[n][e], m);
          acc[n][e] = (t & m) ? (o - acc[n][e]) : (acc[n][e] + o);
        }
    }
#pragma unroll
    for (int hb = 1; hb < 16; hb <<= 1) {
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        if ((n & hb) == 0) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x0 = acc[n][e], x1 = acc[n + hb][e];
            acc[n][e] = x0 + x1;
            acc[n + hb][e] = x0 - x1;
          }
        }
      }
    }
    const float rs = 1.f / sqrtf((float)kPfD);
#pragma unroll
    for (int n = 0; n < 16; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float sg = __ldg(p.tab.v_sign + 8 * n + 2 * t + e) * rs;
        acc[n][e] *= sg;
        acc[n][2 + e] *= sg;
      }
  }
  const int Hq = p.Hkv * p.G;
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int r = rr ? rB : rA;
    if (r >= p.rows) continue;
    const int i = r / p.G, gg = r % p.G;
    float* dst = p.out + (((long long)b * p.nq + i) * Hq + h * p.G + gg) * kPfD;
#pragma unroll
    for (int n = 0; n < 16; ++n)
      *reinterpret_cast<float2*>(dst + 8 * n + 2 * t) = make_float2(acc[n][2 * rr], acc[n][2 * rr + 1]);
  }
  if (timed_out) atomicExch(p.err, TQ_DEVERR_WAIT_TIMEOUT);
}

// ---- The same product on the 5th-generation tensor cores (sides without a QJL sketch) ------
// A block takes 128 rows, one per tensor-memory lane, and the slab's tokens in 64-token tiles:
//   S[128 x 64]   = Q_hi K_hi^T + Q_lo K_hi^T + Q_hi K_lo^T      (tcgen05.mma, M = 128, N = 64)
//   O[128 x 128] += P V,  P = 2^(s - m) nu_V as fp16               (tcgen05.mma, M = 128, N = 128)
// Q_hi, Q_lo, S (two buffers), P and O live in tensor memory; the unpacked K and V tiles in
// shared memory (three buffers).  Warps 0-7 own the rows: warp w takes the rows of tensor-memory
// lanes 32 (w % 4) .. + 31 and tokens 32 (w / 4) .. + 31 of every tile.  They load the queries
// into tensor memory, run the online softmax on S (the two threads of a row share their maxima
// through shared memory) and write P, rescale O when a row's maximum rises, and finish
// o = R_V^T O / l.  Warps 8-15 unpack the tiles, which bulk copies bring into packed stages; with
// three tile buffers the unpacking runs up to two tiles ahead.  One thread of warp 16 issues the
// MMAs, each as soon as its inputs are ready: a tile's scores when it is unpacked, its readout
// when its P is written.  The stages hand
// over through mbarriers: a tile unpacked (U), its scores done (S), its P written (P), its
// readout done (O, which frees the tile's buffers and P).
constexpr int kTcTok = 64;                       // tokens per tile
constexpr int kTcBlk = kTcTok / 16;              // 16-token cache blocks per tile
constexpr int kTcNB = 3;                         // tile buffers (and packed stages): unpacking runs two tiles ahead
constexpr int kTcThreads = 544;                  // warps 0-7 rows, 8-15 unpack, 16 MMA issue
constexpr int kTcRowThreads = 256;               // two threads per row, 32 of a tile's tokens each
constexpr int kTcUnpack = 256;                   // unpacking threads
constexpr int kTcIssueWarp = 16;
constexpr uint32_t kTcCols = 512;  // the whole tensor memory: one block per SM
constexpr uint32_t kTcQhi = 0, kTcQlo = 64, kTcS = 128, kTcO = 256;  // tensor-memory columns
// Without a value sketch: S in two buffers (128 .. 255), P at 384 (32 columns).  With one: S in
// one buffer (128 .. 191), P at 192, P_sk at 224, O at 256 and O_sk at 384 (the whole memory).
template <bool VQ> struct TcCols {
  static constexpr int NS = VQ ? 1 : 2;  // score buffers
  static constexpr uint32_t P = VQ ? 192 : 384, PSK = 224, OSK = 384;
};
constexpr int kTcSmemMin = 116 * 1024;  // asking for more than half the shared memory keeps one block per SM
constexpr int kTcSmemMax = 227 * 1024;  // a block's shared memory

// Shared-memory plan.  Tiles are token-major core matrices: element (token j, dim d) at
// (j / 8) * 2048 + (d / 8) * 128 + (j % 8) * 16 + (d % 8) * 2 -- a K-major B operand for the
// scores (LBO 128, SBO 2048) and an MN-major B operand for the readout (LBO 2048, SBO 128).
template <bool VQ, bool KQ>
struct TcSmem {
  static constexpr int NB = KQ ? 2 : kTcNB;                       // tile buffers (the key sketch's tiles need the room)
  static constexpr int TILE = kTcTok * kPfD * 2;                 // 16 KiB
  static constexpr int KHI = 0, KLO = NB * TILE, VV = 2 * NB * TILE;  // NB buffers each
  static constexpr int VS = 3 * NB * TILE;                        // value signs 2 sigma - 1 (VQ)
  static constexpr int KS = (VQ ? 4 : 3) * NB * TILE;             // key sketch rows rho (2 sigma - 1) (KQ)
  static constexpr int QSK = ((VQ ? 4 : 3) + (KQ ? 1 : 0)) * NB * TILE;  // c S_K q_rot, 128 rows (KQ), K-major A
  static constexpr int NUK = QSK + (KQ ? kPfRows * kPfD * 2 : 0); // float [NB][kTcTok]
  static constexpr int NUV = NUK + NB * kTcTok * 4;               // float [NB][kTcTok]
  static constexpr int FV = NUV + NB * kTcTok * 4;                // nu_V rho_V, float [NB][kTcTok] (VQ)
  static constexpr int CENT = FV + (VQ ? NB * kTcTok * 4 : 0);    // [16] (K hi | K lo << 16), [16] V fp16
  static constexpr int XCH = CENT + 128;  // float [3][2 halves][128 rows]: maxima (by tile parity), then l
  static constexpr int STG = (XCH + 3 * 2 * 128 * 4 + 127) / 128 * 128;  // NB packed stages
};

// Spread the 2-bit fields of a 16-bit value into the low bits of 8 nibbles, and the 8 bits of a
// byte into bit 0 of 8 nibbles.
__device__ __forceinline__ uint32_t spread2(uint32_t x) {
  x = (x | (x << 8)) & 0x00FF00FFu;
  x = (x | (x << 4)) & 0x0F0F0F0Fu;
  return (x | (x << 2)) & 0x33333333u;
}
__device__ __forceinline__ uint32_t spread1(uint32_t x) {
  x = (x | (x << 12)) & 0x000F000Fu;
  x = (x | (x << 6)) & 0x03030303u;
  return (x | (x << 3)) & 0x11111111u;
}

// Codebook indices (one per nibble, dim 8 c + e in nibble e) of 8 coordinates of a b-bit
// sign-magnitude stream whose bytes for those coordinates start at `src` (4-bit: 4 bytes;
// 3-bit: 2 magnitude bytes at src, the sign byte at sgn; 2-bit: 2 bytes; 1-bit: 1 byte).  A sign
// bit s and magnitude rank k give index s ? 2^(b-1) + k : 2^(b-1) - 1 - k, i.e. the stored
// symbol with its magnitude bits inverted when s = 0.
template <int BITS = 0>
__device__ __forceinline__ uint32_t codes8(const unsigned char* src, const unsigned char* sgn, int rbits) {
  const int bits = BITS ? BITS : rbits;
  if (bits == 4) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(src);
    return w ^ (((~w >> 3) & 0x11111111u) * 7u);
  }
  if (bits == 3) {
    const uint32_t m = spread2(*reinterpret_cast<const unsigned short*>(src));
    const uint32_t s = spread1(*sgn);
    return (m | (s << 2)) ^ ((~s & 0x11111111u) * 3u);
  }
  if (bits == 2) {
    const uint32_t x = spread2(*reinterpret_cast<const unsigned short*>(src));
    return x ^ ((~x >> 1) & 0x11111111u);
  }
  return spread1(*src);
}

__device__ __forceinline__ void tc_out_row(const PrefillParams& p, int b, int h, int rr, uint32_t t_o, float il, int hf,
                                           uint32_t t_add);

// KB, VB: the key and value code widths as compile-time constants (0: read from the parameters).
// VQ: a QJL value side -- its sketch readout O_sk += P_sk (2 sigma_V - 1), P_sk = p nu_V rho_V,
// rides beside the code readout, and the epilogue adds c S_V^T O_sk / l as one more MMA.
template <int KB, int VB, bool VQ, bool KQ>
__global__ void __launch_bounds__(kTcThreads, 1) prefill_tc_kernel(const PrefillParams p) {
  using SM = TcSmem<VQ, KQ>;
  using TC = TcCols<VQ>;
  constexpr int NB = SM::NB;
  extern __shared__ __align__(128) unsigned char smem[];
  // mbarriers: packed stages [3], unpacked tiles U [3], scores S [2], readouts O [3], P, scores
  // consumed (one score buffer), the epilogue's sketch product
  __shared__ __align__(8) unsigned long long s_bars[14];
  __shared__ uint32_t s_tmem;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slab = blockIdx.y;
  const int b = slab / p.Hkv, h = slab % p.Hkv;
  const int r0 = blockIdx.x * kPfRows;
  const int L = p.seq_len[b];
  const int Lmin = L - p.nq + 1;
  const int rlast = min(r0 + kPfRows, p.rows) - 1;
  const int eblk = max(0, min(L, Lmin + rlast / p.G));
  const int ntiles = (eblk + kTcTok - 1) / kTcTok;
  const uint32_t sb = (uint32_t)__cvta_generic_to_shared(smem);
  const uint32_t bar = (uint32_t)__cvta_generic_to_shared(s_bars);
  const uint32_t B_STG = bar, B_U = bar + 24, B_S = bar + 48, B_O = bar + 64, B_P = bar + 88;
  const uint32_t B_SC = bar + 96, B_E = bar + 104;
  const Cache& C = p.cache;
  const unsigned kblk = p.kblk, vblk = p.vblk, SB = kTcBlk * (kblk + vblk);
  bool timed_out = false;

  if (warp == kTcIssueWarp) tc_alloc((uint32_t)__cvta_generic_to_shared(&s_tmem), kTcCols);
  if (tid == 0) {
    for (int i = 0; i < NB; ++i) {
      mbar_init(B_STG + 8 * i, 1);
      mbar_init(B_U + 8 * i, kTcUnpack);
      mbar_init(B_O + 8 * i, 1);
    }
    mbar_init(B_S, 1);
    mbar_init(B_S + 8, 1);
    mbar_init(B_P, kTcRowThreads);
    mbar_init(B_SC, kTcRowThreads);
    mbar_init(B_E, 1);
    fence_mbar_init();
    for (int k = 0; k < NB && k < ntiles; ++k) {
      const uint32_t dst = sb + SM::STG + k * SB;
      pf_issue_stage(C, b, h, k, kTcBlk, kblk, vblk, dst, B_STG + 8 * k);
    }
  }
  // codebooks: key centroids as fp16 hi | lo << 16, value centroids as fp16
  if (tid < 16) {
    const float c = __ldg(p.tab.k_c + tid);
    const __half hi = __float2half_rn(c);
    const __half lo = __float2half_rn(c - __half2float(hi));
    reinterpret_cast<uint32_t*>(smem + SM::CENT)[tid] =
        (uint32_t)__half_as_ushort(hi) | ((uint32_t)__half_as_ushort(lo) << 16);
  } else if (tid < 32) {
    reinterpret_cast<__half*>(smem + SM::CENT + 64)[tid - 16] = __float2half_rn(__ldg(p.tab.v_c + tid - 16));
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp < 4) {
    // ---- row owners: the row's queries (fp16 pairs) into tensor memory
    const int r = tid;
    const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);
    const uint32_t* qh = reinterpret_cast<const uint32_t*>(p.qhi + ((long long)slab * p.R_pad + r0 + r) * kPfD);
    const uint32_t* ql = reinterpret_cast<const uint32_t*>(p.qlo + ((long long)slab * p.R_pad + r0 + r) * kPfD);
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 32) {
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const uint4 x = *reinterpret_cast<const uint4*>(qh + c0 + i);
        v[i] = __uint_as_float(x.x); v[i + 1] = __uint_as_float(x.y);
        v[i + 2] = __uint_as_float(x.z); v[i + 3] = __uint_as_float(x.w);
      }
      tc_st32(trow + kTcQhi + c0, v);
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const uint4 x = *reinterpret_cast<const uint4*>(ql + c0 + i);
        v[i] = __uint_as_float(x.x); v[i + 1] = __uint_as_float(x.y);
        v[i + 2] = __uint_as_float(x.z); v[i + 3] = __uint_as_float(x.w);
      }
      tc_st32(trow + kTcQlo + c0, v);
    }
  }
  if constexpr (KQ) {
    if (warp < 8) {  // c S_K q_rot of the block's rows: a K-major A operand in shared memory
#pragma unroll 1
      for (int it = 0; it < 8; ++it) {
        const int item = tid + kTcRowThreads * it, rw = item >> 4, cc = item & 15;
        const uint4 x = *reinterpret_cast<const uint4*>(p.qsk + ((long long)slab * p.R_pad + r0 + rw) * kPfD + 8 * cc);
        *reinterpret_cast<uint4*>(smem + SM::QSK + (rw >> 3) * 2048 + cc * 128 + (rw & 7) * 16) = x;
      }
      tc_fence_smem();
    }
  }
  tc_fence_before();
  __syncthreads();  // the queries are in tensor memory before the first score MMA
  tc_fence_after();

  if (warp >= 8 && warp < 16) {
    // ---- unpack: thread pt takes 8-coordinate chunk c of tokens 8 jg + t8 (jg = pt / 128 + 2 i,
    // i = 0..3), so the eight threads of a quarter warp write the eight 16-byte rows of one core
    // matrix
    const int pt = tid - 256, c = (pt >> 3) & 15, t8 = pt & 7, jg0 = pt >> 7;
    const int kbits = KB ? KB : p.kbits, vbits = VB ? VB : p.vbits, vW = vbits == 3 ? 2 : vbits;
    const unsigned kc_off = C.off[tqi::R_K_CODES], kc_rec = C.rec[tqi::R_K_CODES];
    const unsigned kn_off = C.off[tqi::R_K_NORM], vc_off = C.off[tqi::R_V_CODES], vn_off = C.off[tqi::R_V_NORM];
    const unsigned vs_off = C.off[tqi::R_V_SIGNS], vr_off = C.off[tqi::R_V_RHO];
    const unsigned ks_off = C.off[tqi::R_K_SIGNS], ks_rec = C.rec[tqi::R_K_SIGNS], kr_off = C.off[tqi::R_K_RHO];
    const int kbyte = kbits == 1 ? c : kbits == 4 ? 4 * c : 2 * c;  // the chunk's first code byte in a key record
    const float kscale = p.score_scale;
    const uint32_t* kcent = reinterpret_cast<const uint32_t*>(smem + SM::CENT);
    const unsigned short* vcent = reinterpret_cast<const unsigned short*>(smem + SM::CENT + 64);
    const int g = c >> 1, hv = c & 1;  // the chunk's 16-coordinate value group and half of it
    for (int k = 0; k < ntiles; ++k) {
      const int bf = k % NB, t0 = k * kTcTok;
      // the tile NB back has been read out: its buffers are free
      if (k >= NB && !mbar_wait(B_O + 8 * bf, (uint32_t)(k / NB - 1) & 1u, kPfWaitLimit)) timed_out = true;
      if (!mbar_wait(B_STG + 8 * bf, (uint32_t)(k / NB) & 1u, kPfWaitLimit)) timed_out = true;
      const unsigned char* stg = smem + SM::STG + bf * SB;
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int j = 8 * (jg0 + 2 * it) + t8, pos = j & (tqi::kTileTokens - 1);
        const bool ok = t0 + j < L;
        const unsigned char* kp = stg + (j >> 4) * kblk;             // the token's K block
        const unsigned char* vp = stg + kTcBlk * kblk + (j >> 4) * vblk;  // and V block
        // (tokens past the sequence: the stage holds stale bytes there, read but replaced by zeros)
        uint4 khi, klo, vv;
        float nk, nv;
        {
          const unsigned char* kr = kp + kc_off + pos * kc_rec;
          const uint32_t kc = codes8<KB>(kr + kbyte, kr + kPfD / 4 + c, kbits);
          // value streams by 16-coordinate groups: W bytes of the W-bit stream per chunk
          const unsigned char* vr = vp + vc_off;
          const uint32_t vc = codes8<VB>(vr + g * 32 * vW + pos * 2 * vW + hv * vW,
                                         vr + tqi::kTileTokens * (kPfD / 4) + g * 32 + pos * 2 + hv, vbits);
          uint32_t kh[4], kl[4], vw[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t a = kcent[(kc >> (8 * e)) & 15u], bq = kcent[(kc >> (8 * e + 4)) & 15u];
            kh[e] = __byte_perm(a, bq, 0x5410);
            kl[e] = __byte_perm(a, bq, 0x7632);
            vw[e] = (uint32_t)vcent[(vc >> (8 * e)) & 15u] | ((uint32_t)vcent[(vc >> (8 * e + 4)) & 15u] << 16);
          }
          const uint32_t z = ok ? 0xffffffffu : 0u;
          khi = make_uint4(kh[0] & z, kh[1] & z, kh[2] & z, kh[3] & z);
          klo = make_uint4(kl[0] & z, kl[1] & z, kl[2] & z, kl[3] & z);
          vv = make_uint4(vw[0] & z, vw[1] & z, vw[2] & z, vw[3] & z);
          nk = ok ? *reinterpret_cast<const float*>(kp + kn_off + 4 * pos) * kscale : 0.f;  // nu_K log2(e) / sqrt(d)
          nv = ok ? *reinterpret_cast<const float*>(vp + vn_off + 4 * pos) : 0.f;
        }
        if constexpr (KQ) {  // the key sketch's rows rho_K (2 sigma - 1): token-major 16-byte sign records
          const uint32_t sgb = kp[ks_off + pos * ks_rec + c];
          const uint32_t rh = (uint32_t)__half_as_ushort(*reinterpret_cast<const __half*>(kp + kr_off + 2 * pos));
          uint32_t sw[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            sw[e] = ((rh | rh << 16) | ((~sgb >> (2 * e)) & 1u) << 15 | ((~sgb >> (2 * e + 1)) & 1u) << 31) &
                    (ok ? 0xffffffffu : 0u);
          const int off = (j >> 3) * 2048 + c * 128 + (j & 7) * 16;
          *reinterpret_cast<uint4*>(smem + SM::KS + bf * SM::TILE + off) = make_uint4(sw[0], sw[1], sw[2], sw[3]);
        }
        if constexpr (VQ) {  // the value sketch's signs as +-1 (stream by 16-coordinate groups) and nu_V rho_V
          const uint32_t sgb = vp[vs_off + g * 32 + pos * 2 + hv];
          uint32_t sw[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            sw[e] = (0x3C003C00u | ((~sgb >> (2 * e)) & 1u) << 15 | ((~sgb >> (2 * e + 1)) & 1u) << 31) &
                    (ok ? 0xffffffffu : 0u);
          const int off = (j >> 3) * 2048 + c * 128 + (j & 7) * 16;
          *reinterpret_cast<uint4*>(smem + SM::VS + bf * SM::TILE + off) = make_uint4(sw[0], sw[1], sw[2], sw[3]);
          if (c == 0)
            reinterpret_cast<float*>(smem + SM::FV)[kTcTok * bf + j] =
                ok ? nv * __half2float(*reinterpret_cast<const __half*>(vp + vr_off + 2 * pos)) : 0.f;
        }
        const int off = (j >> 3) * 2048 + c * 128 + (j & 7) * 16;
        *reinterpret_cast<uint4*>(smem + SM::KHI + bf * SM::TILE + off) = khi;
        *reinterpret_cast<uint4*>(smem + SM::KLO + bf * SM::TILE + off) = klo;
        *reinterpret_cast<uint4*>(smem + SM::VV + bf * SM::TILE + off) = vv;
        if (c == 0) {
          reinterpret_cast<float*>(smem + SM::NUK)[kTcTok * bf + j] = nk;
          reinterpret_cast<float*>(smem + SM::NUV)[kTcTok * bf + j] = nv;
        }
      }
      tc_fence_smem();  // the tile's rows are visible to the tensor cores' operand reads
      tc_mbar_arrive(B_U + 8 * bf);
      asm volatile("bar.sync 1, 256;\n" ::: "memory");  // every unpacking thread is done with the stage
      if (pt == 0 && k + NB < ntiles) {
        fence_proxy_async_shared();
        const uint32_t dst = sb + SM::STG + bf * SB;
        pf_issue_stage(C, b, h, k + NB, kTcBlk, kblk, vblk, dst, B_STG + 8 * bf);
      }
    }
  }

  if (warp == kTcIssueWarp && lane == 0) {
    // ---- MMA issue, each as soon as its inputs are ready: the readout of tile kr once its P is
    // written (checked first: it is what the rows wait for), the scores of tile ks once it is
    // unpacked and at most one tile ahead of the readouts (S(ks) reuses S(ks - 2)'s columns, free
    // once P(ks - 2) has been read).  A tile's 24 score MMAs go back to back.
    constexpr uint32_t idS = tc_idesc_f16(128, kTcTok), idO = tc_idesc_f16(128, kPfD, true);
    int ks = 0, kr = 0;
    uint32_t idle = 0;
    while (kr < ntiles) {
      bool moved = false;
      if (kr < ks && tc_mbar_test(B_P, (uint32_t)kr & 1u)) {
        tc_fence_after();
        const uint32_t vb = sb + SM::VV + (kr % NB) * SM::TILE;
#pragma unroll
        for (int kk = 0; kk < kTcTok / 16; ++kk)
          tc_mma_f16_ta(tmem + kTcO, tmem + TC::P + 8 * kk, tc_sdesc(vb + 4096 * kk, 2048, 128), idO,
                        (kr > 0 || kk > 0) ? 1u : 0u);
        if constexpr (VQ) {
          const uint32_t vsb = sb + SM::VS + (kr % NB) * SM::TILE;
#pragma unroll
          for (int kk = 0; kk < kTcTok / 16; ++kk)
            tc_mma_f16_ta(tmem + TC::OSK, tmem + TC::PSK + 8 * kk, tc_sdesc(vsb + 4096 * kk, 2048, 128), idO,
                          (kr > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(B_O + 8 * (kr % NB));
        ++kr;
        moved = true;
      }
      // one score buffer: S(ks) only after the rows have read S(ks - 1)
      if (ks < ntiles && ks <= kr + 1 && (TC::NS == 2 || ks == 0 || tc_mbar_test(B_SC, (uint32_t)(ks - 1) & 1u)) &&
          tc_mbar_test(B_U + 8 * (ks % NB), (uint32_t)(ks / NB) & 1u)) {
        tc_fence_after();
        const int bf = ks % NB;
        const uint32_t kh = sb + SM::KHI + bf * SM::TILE, kl = sb + SM::KLO + bf * SM::TILE;
        const uint32_t dS = tmem + kTcS + kTcTok * (TC::NS == 2 ? (ks & 1) : 0);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          tc_mma_f16_ta(dS, tmem + kTcQhi + 8 * kk, tc_sdesc(kh + 256 * kk, 128, 2048), idS, kk > 0 ? 1u : 0u);
          tc_mma_f16_ta(dS, tmem + kTcQlo + 8 * kk, tc_sdesc(kh + 256 * kk, 128, 2048), idS, 1u);
          tc_mma_f16_ta(dS, tmem + kTcQhi + 8 * kk, tc_sdesc(kl + 256 * kk, 128, 2048), idS, 1u);
        }
        if constexpr (KQ) {  // + (c S_K q_rot) (rho_K (2 sigma - 1))^T, A from shared memory
          const uint32_t kss = sb + SM::KS + bf * SM::TILE;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc_mma_f16(dS, tc_sdesc(sb + SM::QSK + 256 * kk, 128, 2048), tc_sdesc(kss + 256 * kk, 128, 2048), idS, 1u);
        }
        tc_commit(B_S + 8 * (TC::NS == 2 ? (ks & 1) : 0));
        ++ks;
        moved = true;
      }
      if (moved) {
        idle = 0;
      } else if (++idle > 4u * kPfWaitLimit) {  // nothing became ready: give up (the error word says so)
        timed_out = true;
        break;
      } else {
        __nanosleep(32);  // a short back-off keeps the poll from taking issue slots from the other warps
      }
    }
  }

  if (warp < 8) {
    // ---- row owners: online softmax (log2 domain) over the tiles, then o = R_V^T O / l.  Thread
    // (q, hf) of row r = 32 q + lane takes tokens 32 hf .. 32 hf + 31 of each tile.
    const int q = warp & 3, hf = warp >> 2, r = 32 * q + lane, rr = r0 + r;
    const int er = rr < p.rows ? Lmin + rr / p.G : 0;  // row rr sees tokens [0, er)
    const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
    float* xch = reinterpret_cast<float*>(smem + SM::XCH);  // [tile parity][half][row]
    float m = kPfFloor, l = 0.f;  // l: this thread's share of the row sum
    for (int k = 0; k < ntiles; ++k) {
      const int bf = k % NB, sbf = TC::NS == 2 ? (k & 1) : 0, t0 = k * kTcTok + 32 * hf;
      if (!mbar_wait(B_S + 8 * sbf, (uint32_t)(TC::NS == 2 ? (k >> 1) : k) & 1u, kPfWaitLimit)) timed_out = true;
      if (!mbar_wait(B_U + 8 * bf, (uint32_t)(k / NB) & 1u, kPfWaitLimit)) timed_out = true;  // the norms
      tc_fence_after();
      float s[32];
      tc_ld32(trow + kTcS + kTcTok * sbf + 32 * hf, s);
      if constexpr (TC::NS == 1) {  // the score columns may take the next tile's scores
        tc_fence_before();
        tc_mbar_arrive(B_SC);
      }
      const float4* nk4 = reinterpret_cast<const float4*>(smem + SM::NUK) + (kTcTok * bf + 32 * hf) / 4;
      float mx = kPfFloor;
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        const float4 n = nk4[j / 4];  // nu_K log2(e) / sqrt(d)
        s[j] *= n.x; s[j + 1] *= n.y; s[j + 2] *= n.z; s[j + 3] *= n.w;
      }
      if (t0 + 32 > er) {  // the tile reaches this row's end
#pragma unroll
        for (int j = 0; j < 32; ++j) s[j] = t0 + j < er ? s[j] : -INFINITY;
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) mx = fmaxf(mx, s[j]);
      // the row's maximum over both halves (two exchange slots by tile parity)
      xch[((k & 1) * 2 + hf) * 128 + r] = mx;
      asm volatile("bar.sync 2, 256;\n" ::: "memory");
      const float mn = fmaxf(m, fmaxf(mx, xch[((k & 1) * 2 + (hf ^ 1)) * 128 + r]));
      const float alpha = pf_ex2(m - mn);
      const float4* nv4 = reinterpret_cast<const float4*>(smem + SM::NUV) + (kTcTok * bf + 32 * hf) / 4;
      const float4* fv4 = reinterpret_cast<const float4*>(smem + SM::FV) + (kTcTok * bf + 32 * hf) / 4;
      float ps = 0.f;
      uint32_t pw[16], pk[16];
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        const float4 n = nv4[j / 4];
        const float p0 = pf_ex2(s[j] - mn), p1 = pf_ex2(s[j + 1] - mn);
        const float p2 = pf_ex2(s[j + 2] - mn), p3 = pf_ex2(s[j + 3] - mn);
        ps += (p0 + p1) + (p2 + p3);
        pw[j / 2] = pack_half2(p0 * n.x, p1 * n.y);
        pw[j / 2 + 1] = pack_half2(p2 * n.z, p3 * n.w);
        if constexpr (VQ) {  // P_sk = p nu_V rho_V
          const float4 f = fv4[j / 4];
          pk[j / 2] = pack_half2(p0 * f.x, p1 * f.y);
          pk[j / 2 + 1] = pack_half2(p2 * f.z, p3 * f.w);
        }
      }
      l = l * alpha + ps;
      m = mn;
      if (k >= 1) {  // the readout of tile k - 1 is done: O is settled and P's columns are free
        if (!mbar_wait(B_O + 8 * ((k - 1) % NB), (uint32_t)((k - 1) / NB) & 1u, kPfWaitLimit)) timed_out = true;
        tc_fence_after();
        if (__any_sync(kFull, alpha != 1.f)) {  // this thread's half of the row's accumulator
#pragma unroll 1
          for (int c4 = 0; c4 < (VQ ? 4 : 2); ++c4) {  // O's half, then (VQ) O_sk's half
            const uint32_t col = (c4 < 2 ? kTcO : TC::OSK) + 64 * hf + 32 * (c4 & 1);
            float o[32];
            tc_ld32(trow + col, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tc_st32(trow + col, o);
          }
        }
      }
      tc_st16(trow + TC::P + 16 * hf, pw);
      if constexpr (VQ) tc_st16(trow + TC::PSK + 16 * hf, pk);
      tc_fence_before();
      tc_mbar_arrive(B_P);
    }
    if (ntiles > 0) {
      if (!mbar_wait(B_O + 8 * ((ntiles - 1) % NB), (uint32_t)((ntiles - 1) / NB) & 1u, kPfWaitLimit))
        timed_out = true;
      tc_fence_after();
    }
    // the row sum over both halves
    xch[(4 + hf) * 128 + r] = l;
    asm volatile("bar.sync 2, 256;\n" ::: "memory");
    const float lt = l + xch[(4 + (hf ^ 1)) * 128 + r];
    const float il = lt > 0.f ? 1.f / lt : 0.f;
    if constexpr (VQ) {
      if (ntiles > 0) {
        // c S_V^T O_sk / l: S_V^T as fp16 rows (K-major B, row i, k = j) in the free tile buffers,
        // c O_sk / l as fp16 pairs (the A operand) in the free score columns, one MMA chain into
        // O_sk's columns
        for (int it = 0; it < 8; ++it) {
          const int item = tid + kTcRowThreads * it, i = item >> 4, cc = item & 15;
          const float4 x0 = __ldg(reinterpret_cast<const float4*>(p.tab.S_V_T + i * kPfD + 8 * cc));
          const float4 x1 = __ldg(reinterpret_cast<const float4*>(p.tab.S_V_T + i * kPfD + 8 * cc + 4));
          *reinterpret_cast<uint4*>(smem + SM::KHI + (i >> 3) * 2048 + cc * 128 + (i & 7) * 16) =
              make_uint4(pack_half2(x0.x, x0.y), pack_half2(x0.z, x0.w), pack_half2(x1.x, x1.y), pack_half2(x1.z, x1.w));
        }
        const float cs = p.qjl_scale * il;
#pragma unroll 1
        for (int c2 = 0; c2 < 2; ++c2) {
          float o[32];
          tc_ld32(trow + TC::OSK + 64 * hf + 32 * c2, o);
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) w[i] = pack_half2(o[2 * i] * cs, o[2 * i + 1] * cs);
          tc_st16(trow + kTcS + 32 * hf + 16 * c2, w);
        }
        tc_fence_smem();
        tc_fence_before();
        asm volatile("bar.sync 2, 256;\n" ::: "memory");
        if (tid == 0) {
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc_mma_f16_ta(tmem + TC::OSK, tmem + kTcS + 8 * kk, tc_sdesc(sb + SM::KHI + 256 * kk, 128, 2048),
                          tc_idesc_f16(128, kPfD), kk > 0 ? 1u : 0u);
          tc_commit(B_E);
        }
        if (!mbar_wait(B_E, 0, kPfWaitLimit)) timed_out = true;
        tc_fence_after();
      }
    }
    tc_out_row(p, b, h, rr, ntiles > 0 ? trow + kTcO : 0u, il, hf, (VQ && ntiles > 0) ? trow + TC::OSK : 0u);
  }

  tc_fence_before();
  __syncthreads();  // every MMA has completed (the row owners waited for the last readout)
  if (warp == kTcIssueWarp) {
    tc_fence_after();
    tc_dealloc(tmem, kTcCols);
  }
  if (timed_out) atomicExch(p.err, TQ_DEVERR_WAIT_TIMEOUT);
}

__device__ __forceinline__ void tc_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// Row rr of the slab's output from its accumulator (128 columns from t_o; t_o = 0: no token,
// the row is zero): o = O il, then, when the value side is rotated, x = D_V H o / sqrt(d) --
// butterflies over coordinate bits 0 .. 4 within each 32-column piece (written back), then over
// bits 5 and 6 across the four pieces, 8 columns at a time -- stored to out.  The row's two
// threads (hf = 0, 1) split the work: pieces 2 hf, 2 hf + 1, then columns 16 hf .. 16 hf + 15 of
// every piece, with the row owners' barrier between.  t_add (when not 0): 128 more columns added
// to O il before the transform (the value sketch's term).  Every thread of the 8 row-owner warps
// calls (tensor-memory loads are warp-wide); rows past the chunk store nothing.
__device__ __forceinline__ void tc_out_row(const PrefillParams& p, int b, int h, int rr, uint32_t t_o, float il, int hf,
                                           uint32_t t_add) {
  const bool store = rr < p.rows;
  const int Hq = p.Hkv * p.G;
  float* dst = store ? p.out + (((long long)b * p.nq + rr / p.G) * Hq + h * p.G + rr % p.G) * kPfD : nullptr;
  const bool have = __any_sync(kFull, t_o != 0u);  // uniform: every row of the block shares the tiles
#pragma unroll 1
  for (int c4 = 2 * hf; c4 < 2 * hf + 2; ++c4) {
    float v[32];
    if (have) tc_ld32(t_o + 32 * c4, v);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = have ? v[i] * il : 0.f;
    if (t_add != 0u && have) {
      float a[32];
      tc_ld32(t_add + 32 * c4, a);
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] += a[i];
    }
    if (p.v_rotate) {
#pragma unroll
      for (int hb = 1; hb < 32; hb <<= 1) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if ((i & hb) == 0) {
            const float x0 = v[i], x1 = v[i + hb];
            v[i] = x0 + x1;
            v[i + hb] = x0 - x1;
          }
        }
      }
      if (have) tc_st32(t_o + 32 * c4, v);
    } else if (store) {
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        *reinterpret_cast<float4*>(dst + 32 * c4 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    }
  }
  if (!p.v_rotate) return;
  tc_fence_before();
  asm volatile("bar.sync 2, 256;\n" ::: "memory");  // both threads' pieces are back in tensor memory
  tc_fence_after();
  const float rs = 1.f / sqrtf((float)kPfD);
#pragma unroll 1
  for (int i0 = 16 * hf; i0 < 16 * hf + 16; i0 += 8) {
    float v[4][8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (have) {
        tc_ld8(t_o + 32 * q + i0, v[q]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[q][i] = 0.f;
      }
    }
#pragma unroll
    for (int hq = 1; hq < 4; hq <<= 1) {  // coordinate bits 5 (hq = 1) and 6 (hq = 2)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if ((q & hq) == 0) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float x0 = v[q][i], x1 = v[q + hq][i];
            v[q][i] = x0 + x1;
            v[q + hq][i] = x0 - x1;
          }
        }
      }
    }
    if (store) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int d0 = 32 * q + i0;
        float w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = v[q][i] * (__ldg(p.tab.v_sign + d0 + i) * rs);
        *reinterpret_cast<float4*>(dst + d0) = make_float4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<float4*>(dst + d0 + 4) = make_float4(w[4], w[5], w[6], w[7]);
      }
    }
  }
}

size_t pf_align(size_t x) { return (x + 255) / 256 * 256; }

tq_status pf_fail(const char* what, cudaError_t e) {
  tqi::set_error(std::string(what) + ": " + cudaGetErrorString(e));
  return TQ_ERR_CUDA;
}

int pf_rows_padded(const tq_context* ctx, int nq) {
  const int rows = nq * (ctx->cfg.num_q_heads / ctx->cfg.num_kv_heads);
  return (rows + kPfRows - 1) / kPfRows * kPfRows;
}

template <bool KQ, bool VQ>
cudaError_t launch_pf(const PrefillParams& p, dim3 grid, cudaStream_t s) {
  const int smem = PfSmem<KQ, VQ>::STG + 4 * (int)(p.kblk + p.vblk);
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<KQ, VQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  prefill_kernel<KQ, VQ><<<grid, kPfWarps * 32, smem, s>>>(p);
  return cudaGetLastError();
}

template <bool VQ, bool KQ>
int pf_tc_smem(const PrefillParams& p) {  // the packed stages: NB of kTcBlk K blocks and kTcBlk V blocks each
  using SM = TcSmem<VQ, KQ>;
  return std::max(SM::STG + SM::NB * kTcBlk * (int)(p.kblk + p.vblk), kTcSmemMin);
}

template <bool VQ, bool KQ>
cudaError_t launch_pf_tc(const PrefillParams& p, dim3 grid, cudaStream_t s) {
  const int smem = pf_tc_smem<VQ, KQ>(p);
  auto go = [&](auto kern) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kTcThreads, smem, s>>>(p);
    return cudaGetLastError();
  };
  if constexpr (KQ) {  // QKQV at n = 4 / 3 / 2 (one code width on both sides)
    if (p.kbits == p.vbits) {
      switch (p.kbits) {
        case 3: return go(prefill_tc_kernel<3, 3, VQ, true>);
        case 2: return go(prefill_tc_kernel<2, 2, VQ, true>);
        case 1: return go(prefill_tc_kernel<1, 1, VQ, true>);
      }
    }
    return go(prefill_tc_kernel<0, 0, VQ, true>);
  } else if constexpr (VQ) {  // KQV at n = 4 / 3 / 2 (keys one bit wider than the value codes)
    if (p.kbits == 4 && p.vbits == 3) return go(prefill_tc_kernel<4, 3, true, false>);
    if (p.kbits == 3 && p.vbits == 2) return go(prefill_tc_kernel<3, 2, true, false>);
    if (p.kbits == 2 && p.vbits == 1) return go(prefill_tc_kernel<2, 1, true, false>);
    return go(prefill_tc_kernel<0, 0, true, false>);
  } else {  // one code width on both sides (Plain-KV, TQ-KV)
    if (p.kbits == p.vbits) {
      switch (p.kbits) {
        case 4: return go(prefill_tc_kernel<4, 4, false, false>);
        case 3: return go(prefill_tc_kernel<3, 3, false, false>);
        case 2: return go(prefill_tc_kernel<2, 2, false, false>);
        case 1: return go(prefill_tc_kernel<1, 1, false, false>);
      }
    }
    return go(prefill_tc_kernel<0, 0, false, false>);
  }
}

}  // namespace
}  // namespace tqd

namespace tqi {

size_t prefill_workspace_bytes(const tq_context* ctx, int nq) {
  const size_t rows = (size_t)ctx->cfg.batch * ctx->cfg.num_kv_heads * tqd::pf_rows_padded(ctx, nq);
  const size_t arr = tqd::pf_align(rows * tqd::kPfD * 2);
  return 256 + arr * (ctx->cfg.k.qjl ? 3 : 2);  // error word, then the query arrays
}

tq_status launch_prefill(const tq_context* ctx, const void* cache, const float* q, int nq,
                         const int32_t* seq_len, float* out, void* ws, Stream stream) {
  using namespace tqd;
  const cudaStream_t s = (cudaStream_t)stream;
  const int B = ctx->cfg.batch, Hkv = ctx->cfg.num_kv_heads, Hq = ctx->cfg.num_q_heads;
  const int G = Hq / Hkv;
  const int R_pad = pf_rows_padded(ctx, nq);
  const size_t rows_all = (size_t)B * Hkv * R_pad;
  const size_t arr = pf_align(rows_all * kPfD * 2);
  int* err = (int*)ws;
  unsigned char* base = (unsigned char*)ws + 256;

  PrefillPrepParams pp;
  pp.tab = make_tables(ctx);
  pp.q = q;
  pp.qhi = (__half*)base;
  pp.qlo = (__half*)(base + arr);
  pp.qsk = ctx->cfg.k.qjl ? (__half*)(base + 2 * arr) : nullptr;
  pp.B = B;
  pp.Hkv = Hkv;
  pp.G = G;
  pp.nq = nq;
  pp.rows = nq * G;
  pp.R_pad = R_pad;
  pp.k_rotate = ctx->cfg.k.rotate;
  pp.kq = ctx->cfg.k.qjl;
  pp.qjl_scale = (float)(1.2533141373155003 / ctx->m);
  pp.err = err;
  const int psmem = pp.kq ? kPfD * kPfD * 4 : 0;
  cudaError_t e = cudaSuccess;
  if (psmem) {
    e = cudaFuncSetAttribute(prefill_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, psmem);
    if (e != cudaSuccess) return tqd::pf_fail("prefill prep", e);
  }
  const long long warps = (long long)rows_all;
  long long blocks = (warps + 7) / 8;
  if (pp.kq && blocks > 4 * 152) blocks = 4 * 152;  // each block stages S_K^T once: reuse it
  if (blocks > 65535) blocks = 65535;
  prefill_prep_kernel<<<(unsigned)blocks, 256, psmem, s>>>(pp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return tqd::pf_fail("prefill prep", e);

  PrefillParams p;
  p.tab = pp.tab;
  p.cache = make_cache(ctx, cache);
  p.qhi = pp.qhi;
  p.qlo = pp.qlo;
  p.qsk = pp.qsk;
  p.out = out;
  p.B = B;
  p.Hkv = Hkv;
  p.G = G;
  p.nq = nq;
  p.rows = nq * G;
  p.R_pad = R_pad;
  p.kbits = ctx->cfg.k.bits;
  p.vbits = ctx->cfg.v.bits;
  p.v_rotate = ctx->cfg.v.rotate;
  p.kblk = (unsigned)ctx->layout.block[0];
  p.vblk = (unsigned)ctx->layout.block[1];
  p.err = err;
  p.score_scale = kPfLog2e / sqrtf((float)kPfD);
  p.qjl_scale = pp.qjl_scale;
  for (int b = 0; b < TQ_MAX_BATCH; ++b) p.seq_len[b] = b < B ? seq_len[b] : 0;
  const dim3 grid(R_pad / kPfRows, B * Hkv);
  const bool kq = ctx->cfg.k.qjl != 0, vq = ctx->cfg.v.qjl != 0;
  if (kq && vq && pf_tc_smem<true, true>(p) <= kTcSmemMax) e = launch_pf_tc<true, true>(p, grid, s);  // tcgen05
  else if (kq && vq) e = launch_pf<true, true>(p, grid, s);
  else if (kq) e = launch_pf<true, false>(p, grid, s);
  else if (vq && pf_tc_smem<true, false>(p) <= kTcSmemMax) e = launch_pf_tc<true, false>(p, grid, s);  // tcgen05
  else if (vq) e = launch_pf<false, true>(p, grid, s);
  else e = launch_pf_tc<false, false>(p, grid, s);  // no sketch: the tcgen05 kernel
  if (e != cudaSuccess) return tqd::pf_fail("prefill", e);
  return TQ_OK;
}

}  // namespace tqi
