// Chunked-prefill attention over the packed cache (head dim 128): many queries per KV head.
//
// [ABL] "Recomendações Práticas" 2 names prefill workloads; [HEADQ] "Espaço de Pontuação da
// Chave" / "Geometria de Leitura de Valores" give the scores q^T k / sqrt(d) and the weighted
// value sum; [TQ-KV] "Contribuciones Clave" 1 the QJL estimate of a residual inner product.
//
// The rows of one (batch, KV head) slab are the chunk's (query, head) pairs, r = i G + g, and
// row r attends to the first L - nq + 1 + r / G tokens.  A block takes 128 rows and walks the
// slab's tokens in 64-token tiles.  Each tile's packed K and V are unpacked once per block into
// shared memory as fp16 rows of the rotated domain -- C[c], and on a QJL side rho (2 sigma - 1)
// (keys) or 2 sigma - 1 (values) -- so the scores and the readout are dense products on the
// 5th-generation tensor cores (tcgen05.mma, fp16 operands, fp32 accumulators in tensor memory):
//   S[128 rows x 64 tok] = Q_hi K_hi^T + Q_lo K_hi^T + Q_hi K_lo^T (+ (c S_K q_rot) (rho (2 sigma - 1))^T)
//   O[128 x 128]        += (p nu_V) V_hat,   O_sk[128 x 128] += (p nu_V rho_V) (2 sigma_V - 1)
// with an online softmax (log2 domain) in between.  The epilogue forms
// o = R_V^T (O + c S_V^T O_sk) / l: the sketch product is one more MMA against S_V^T staged as
// fp16, and the inverse Walsh-Hadamard transform runs on 32-column pieces of the accumulator.
// The queries and the key centroids enter as fp16 hi + lo terms: a single rounding of q is a
// score error common to every token of a row, and one of a centroid an error common to every
// token with that code; with peaked attention (outlier channels) either reaches the output
// undiluted.
#include <algorithm>
#include <string>
#include <type_traits>

#include "tq_device.cuh"
#include "tq_tc05.cuh"

namespace tqd {
namespace {

constexpr int kPfRows = 128;            // rows per block (one per tensor-memory lane)
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

__device__ __forceinline__ float pf_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
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

// ---- The prefill kernel ---------------------------------------------------------------------
// Q_hi, Q_lo, S, P and O (and with a QJL value side P_sk and O_sk) live in tensor memory; the
// unpacked tiles in shared memory (three buffers, two with a QJL key side, whose c S_K q_rot is a
// shared-memory A operand).  Warps 0-7 own the rows: warp w takes the rows of tensor-memory
// lanes 32 (w % 4) .. + 31 and tokens 32 (w / 4) .. + 31 of every tile.  They load the queries
// into tensor memory, run the online softmax on S (the two threads of a row share their maxima
// through shared memory) and write P, rescale the accumulators when a row's maximum rises, and
// finish o.  Warps 8-15 unpack the tiles, which bulk copies bring into packed stages; with three
// tile buffers the unpacking runs up to two tiles ahead.  One thread of warp 16 issues the MMAs,
// each as soon as its inputs are ready: a tile's scores when it is unpacked, its readout when its
// P is written.  The stages hand over through mbarriers: a tile unpacked (U), its scores done
// (S), its scores read (one score buffer), its P written (P), its readout done (O, which frees
// the tile's buffers and P).
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
// One score buffer.  Without a value sketch it is 128 columns wide (WIDE): a tile's K_hi and K_lo
// rows sit side by side in shared memory, so Q_hi [K_hi | K_lo]^T is one N = 128 MMA per k-step
// (full tensor rate, where N = 64 runs at about 70 %) and Q_lo K_hi^T one N = 64 MMA into the first
// half; the rows add the halves.  With a value sketch the columns hold P_sk and O_sk instead, and
// the three products run as N = 64 MMAs into a 64-column buffer.
template <bool VQ> struct TcCols {
  static constexpr int NS = 1;  // score buffers
  static constexpr bool WIDE = !VQ;
  static constexpr uint32_t P = VQ ? 192 : 384, PSK = 224, OSK = 384;
  static_assert(!VQ || (PSK == P + 32 && OSK == kTcO + 128), "tensor-memory plan");
  static_assert(VQ || kTcS + 128 <= kTcO, "tensor-memory plan");
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
  // buffer bf: K hi at KHI + bf KSTR, K lo right after it (the wide score operand), V at VV + bf TILE
  static constexpr int KSTR = 2 * TILE, KHI = 0, KLO = TILE, VV = 2 * NB * TILE;
  static constexpr int VS = 3 * NB * TILE;                        // value signs 2 sigma - 1 (VQ)
  static constexpr int KS = (VQ ? 4 : 3) * NB * TILE;             // key sketch rows rho (2 sigma - 1) (KQ)
  static constexpr int QSK = ((VQ ? 4 : 3) + (KQ ? 1 : 0)) * NB * TILE;  // c S_K q_rot, 128 rows (KQ), K-major A
  static constexpr int NUK = QSK + (KQ ? kPfRows * kPfD * 2 : 0); // float [NB][kTcTok]
  static constexpr int NUV = NUK + NB * kTcTok * 4;               // float [NB][kTcTok]
  static constexpr int FV = NUV + NB * kTcTok * 4;                // nu_V rho_V, float [NB][kTcTok] (VQ)
  static constexpr int CENT = FV + (VQ ? NB * kTcTok * 4 : 0);    // [16] (K hi | K lo << 16), [16] V fp16
  static constexpr int SGN = CENT + 128;  // uint2 [16]: the fp16 sign fields of four signs (a nibble)
  static constexpr int XCH = SGN + 128;   // float [3][2 halves][128 rows]: maxima (by tile parity), then l
  static constexpr int STG = (XCH + 3 * 2 * 128 * 4 + 127) / 128 * 128;  // NB packed stages
  static_assert(VS == VV + NB * TILE && KS >= VS && QSK >= KS, "shared-memory plan");
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

// 3-bit codes without shared-memory lookups: a pair's two 2-bit magnitudes select its two fp16
// magnitudes from a four-entry table held in two registers (t0 = mag0 | mag1 << 16, t1 = mag2 |
// mag3 << 16) with one byte permute.  m: spread2 of the chunk's magnitude bytes (coordinate i's
// magnitude in bits 4 i, 4 i + 1); the selector of pair e has nibbles 2 m0, 2 m0 + 1, 2 m1, 2 m1 + 1.
__device__ __forceinline__ uint32_t mag_pair(uint32_t t0, uint32_t t1, uint32_t m, int e) {
  const uint32_t t = (m >> (8 * e)) & 0x33u;            // m0 in bits 0-1, m1 in bits 4-5
  const uint32_t u = (t & 0x3u) | ((t & 0x30u) << 4);   // m1 to bits 8-9
  return __byte_perm(t0, t1, u * 0x22u + 0x1010u);
}

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
  } else if (tid < 48) {  // nibble n: signs 0..3 (a set bit is +) as the sign fields of two fp16 pairs
    const uint32_t n = (uint32_t)tid - 32;
    reinterpret_cast<uint2*>(smem + SM::SGN)[n] =
        make_uint2((~n & 1u) << 15 | ((~n >> 1) & 1u) << 31, ((~n >> 2) & 1u) << 15 | ((~n >> 3) & 1u) << 31);
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
    // 3-bit sides: the upper half of the symmetric codebook (the magnitudes) in registers, fp16 hi
    // and lo terms for the keys, fp16 for the values
    auto mag2 = [&](const float* cent, int m0, bool lo_term) {
      const float a = __ldg(cent + 4 + m0), b2 = __ldg(cent + 5 + m0);
      const __half ha = __float2half_rn(a), hb = __float2half_rn(b2);
      const __half xa = lo_term ? __float2half_rn(a - __half2float(ha)) : ha;
      const __half xb = lo_term ? __float2half_rn(b2 - __half2float(hb)) : hb;
      return (uint32_t)__half_as_ushort(xa) | ((uint32_t)__half_as_ushort(xb) << 16);
    };
    uint32_t kmh0 = 0, kmh1 = 0, kml0 = 0, kml1 = 0, vm0 = 0, vm1 = 0;
    if constexpr (KB == 3) {
      kmh0 = mag2(p.tab.k_c, 0, false); kmh1 = mag2(p.tab.k_c, 2, false);
      kml0 = mag2(p.tab.k_c, 0, true);  kml1 = mag2(p.tab.k_c, 2, true);
    }
    if constexpr (VB == 3) {
      vm0 = mag2(p.tab.v_c, 0, false); vm1 = mag2(p.tab.v_c, 2, false);
    }
    const uint2* sgn = reinterpret_cast<const uint2*>(smem + SM::SGN);
    const unsigned short* vcent = reinterpret_cast<const unsigned short*>(smem + SM::CENT + 64);
    const int g = c >> 1, hv = c & 1;  // the chunk's 16-coordinate value group and half of it
    for (int k = 0; k < ntiles; ++k) {
      const int bf = k % NB, t0 = k * kTcTok;
      // the tile NB back has been read out: its buffers are free
      if (k >= NB && !mbar_wait(B_O + 8 * bf, (uint32_t)(k / NB - 1) & 1u, kPfWaitLimit)) timed_out = true;
      if (!mbar_wait(B_STG + 8 * bf, (uint32_t)(k / NB) & 1u, kPfWaitLimit)) timed_out = true;
      const unsigned char* stg = smem + SM::STG + bf * SB;
      // FULL: every token of the tile is inside the sequence (all but a sequence's last tile), so
      // nothing is masked
      auto unpack_tile = [&](auto full_c) {
      constexpr bool FULL = decltype(full_c)::value;
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int j = 8 * (jg0 + 2 * it) + t8, pos = j & (tqi::kTileTokens - 1);
        const bool ok = FULL || t0 + j < L;
        const unsigned char* kp = stg + (j >> 4) * kblk;             // the token's K block
        const unsigned char* vp = stg + kTcBlk * kblk + (j >> 4) * vblk;  // and V block
        // (tokens past the sequence: the stage holds stale bytes there, read but replaced by zeros)
        uint4 khi, klo, vv;
        float nk, nv;
        {
          const unsigned char* kr = kp + kc_off + pos * kc_rec;
          // value streams by 16-coordinate groups: W bytes of the W-bit stream per chunk
          const unsigned char* vr = vp + vc_off;
          const unsigned char* vsrc = vr + g * 32 * vW + pos * 2 * vW + hv * vW;
          const unsigned char* vsgn = vr + tqi::kTileTokens * (kPfD / 4) + g * 32 + pos * 2 + hv;
          uint32_t kh[4], kl[4], vw[4];
          if constexpr (KB == 3) {  // magnitudes from registers, signs (a set bit is +) by nibble table
            const uint32_t m = spread2(*reinterpret_cast<const unsigned short*>(kr + kbyte));
            const uint32_t sb = kr[kPfD / 4 + c];
            const uint2 s0 = sgn[sb & 15u], s1 = sgn[sb >> 4];
            const uint32_t sf[4] = {s0.x, s0.y, s1.x, s1.y};
#pragma unroll
            for (int e = 0; e < 4; ++e) {  // (the lo term of -c is -lo(c): the sign flips both)
              kh[e] = mag_pair(kmh0, kmh1, m, e) ^ sf[e];
              kl[e] = mag_pair(kml0, kml1, m, e) ^ sf[e];
            }
          } else {
            const uint32_t kc = codes8<KB>(kr + kbyte, kr + kPfD / 4 + c, kbits);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t a = kcent[(kc >> (8 * e)) & 15u], bq = kcent[(kc >> (8 * e + 4)) & 15u];
              kh[e] = __byte_perm(a, bq, 0x5410);
              kl[e] = __byte_perm(a, bq, 0x7632);
            }
          }
          if constexpr (VB == 3) {
            const uint32_t m = spread2(*reinterpret_cast<const unsigned short*>(vsrc));
            const uint32_t sb = *vsgn;
            const uint2 s0 = sgn[sb & 15u], s1 = sgn[sb >> 4];
            vw[0] = mag_pair(vm0, vm1, m, 0) ^ s0.x;
            vw[1] = mag_pair(vm0, vm1, m, 1) ^ s0.y;
            vw[2] = mag_pair(vm0, vm1, m, 2) ^ s1.x;
            vw[3] = mag_pair(vm0, vm1, m, 3) ^ s1.y;
          } else {
            const uint32_t vc = codes8<VB>(vsrc, vsgn, vbits);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              vw[e] = (uint32_t)vcent[(vc >> (8 * e)) & 15u] | ((uint32_t)vcent[(vc >> (8 * e + 4)) & 15u] << 16);
          }
          const uint32_t z = ok ? 0xffffffffu : 0u;
          khi = make_uint4(kh[0] & z, kh[1] & z, kh[2] & z, kh[3] & z);
          klo = make_uint4(kl[0] & z, kl[1] & z, kl[2] & z, kl[3] & z);
          vv = make_uint4(vw[0] & z, vw[1] & z, vw[2] & z, vw[3] & z);
          nk = ok ? *reinterpret_cast<const float*>(kp + kn_off + 4 * pos) * kscale : 0.f;  // nu_K log2(e) / sqrt(d)
          nv = ok ? *reinterpret_cast<const float*>(vp + vn_off + 4 * pos) : 0.f;
        }
        // the sign fields of a byte of sketch signs: two table entries, one per nibble
        auto sign_fields = [&](uint32_t sgb, uint32_t mag2) {
          const uint2 a = sgn[sgb & 15u], bq = sgn[sgb >> 4];
          const uint32_t z = ok ? 0xffffffffu : 0u;
          return make_uint4((a.x | mag2) & z, (a.y | mag2) & z, (bq.x | mag2) & z, (bq.y | mag2) & z);
        };
        if constexpr (KQ) {  // the key sketch's rows rho_K (2 sigma - 1): token-major 16-byte sign records
          const uint32_t sgb = kp[ks_off + pos * ks_rec + c];
          const uint32_t rh = (uint32_t)__half_as_ushort(*reinterpret_cast<const __half*>(kp + kr_off + 2 * pos));
          const int off = (j >> 3) * 2048 + c * 128 + (j & 7) * 16;
          *reinterpret_cast<uint4*>(smem + SM::KS + bf * SM::TILE + off) = sign_fields(sgb, rh | rh << 16);
        }
        if constexpr (VQ) {  // the value sketch's signs as +-1 (stream by 16-coordinate groups) and nu_V rho_V
          const uint32_t sgb = vp[vs_off + g * 32 + pos * 2 + hv];
          const int off = (j >> 3) * 2048 + c * 128 + (j & 7) * 16;
          *reinterpret_cast<uint4*>(smem + SM::VS + bf * SM::TILE + off) = sign_fields(sgb, 0x3C003C00u);
          if (c == 0)
            reinterpret_cast<float*>(smem + SM::FV)[kTcTok * bf + j] =
                ok ? nv * __half2float(*reinterpret_cast<const __half*>(vp + vr_off + 2 * pos)) : 0.f;
        }
        const int off = (j >> 3) * 2048 + c * 128 + (j & 7) * 16;
        *reinterpret_cast<uint4*>(smem + SM::KHI + bf * SM::KSTR + off) = khi;
        *reinterpret_cast<uint4*>(smem + SM::KLO + bf * SM::KSTR + off) = klo;
        *reinterpret_cast<uint4*>(smem + SM::VV + bf * SM::TILE + off) = vv;
        if (c == 0) {
          reinterpret_cast<float*>(smem + SM::NUK)[kTcTok * bf + j] = nk;
          reinterpret_cast<float*>(smem + SM::NUV)[kTcTok * bf + j] = nv;
        }
      }
      };
      if (t0 + kTcTok <= L) unpack_tile(std::true_type());
      else unpack_tile(std::false_type());
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

  // The issue form per variant (measured): with a key sketch (both operands of its MMAs in shared
  // memory) the whole warp runs the issue loop and one elected lane issues, which keeps every
  // descriptor warp-uniform (QKQV n=4 11.27 -> 10.08 ms); without one a single lane issues
  // (warp-wide was 0.8 % slower for Plain / TQ and 5 % for KQV).
  constexpr bool kWarpIssue = KQ;
  if (warp == kTcIssueWarp && (kWarpIssue || lane == 0)) {
    // ---- MMA issue, each as soon as its inputs are ready: the readout of tile kr once its P is
    // written (checked first: it is what the rows wait for), the scores of tile ks once it is
    // unpacked, at most one tile ahead of the readouts, and once the rows have read S(ks - 1) (one
    // score buffer).  A tile's score MMAs go back to back.
    // Warp-wide (kWarpIssue): one elected lane issues each MMA and commit, and every poll takes
    // lane 0's answer, so the warp never diverges.
    constexpr uint32_t idS = tc_idesc_f16(128, kTcTok), idO = tc_idesc_f16(128, kPfD, true);
    constexpr uint32_t idS2 = tc_idesc_f16(128, 2 * kTcTok);
    auto test = [&](uint32_t bar, uint32_t parity) {
      if constexpr (kWarpIssue) return __shfl_sync(kFull, tc_mbar_test(bar, parity) ? 1 : 0, 0) != 0;
      else return tc_mbar_test(bar, parity);
    };
    auto mma_ta = [&](uint32_t d, uint32_t a, uint64_t bd, uint32_t id, uint32_t acc) {
      if constexpr (kWarpIssue) tc_mma_f16_ta_w(d, a, bd, id, acc);
      else tc_mma_f16_ta(d, a, bd, id, acc);
    };
    auto mma = [&](uint32_t d, uint64_t ad, uint64_t bd, uint32_t id, uint32_t acc) {
      if constexpr (kWarpIssue) tc_mma_f16_w(d, ad, bd, id, acc);
      else tc_mma_f16(d, ad, bd, id, acc);
    };
    auto commit = [&](uint32_t bar) {
      if constexpr (kWarpIssue) tc_commit_w(bar);
      else tc_commit(bar);
    };
    int ks = 0, kr = 0;
    uint32_t idle = 0;
    while (kr < ntiles) {
      bool moved = false;
      if (kr < ks && test(B_P, (uint32_t)kr & 1u)) {
        tc_fence_after();
        // each batch's descriptors from one base: a step of 256 (4096) bytes adds 16 (256) to the
        // address field, which stays below 2^14 for every shared-memory address
        const uint64_t dv = tc_sdesc(sb + SM::VV + (kr % NB) * SM::TILE, 2048, 128);
#pragma unroll
        for (int kk = 0; kk < kTcTok / 16; ++kk)
          mma_ta(tmem + kTcO, tmem + TC::P + 8 * kk, dv + 256u * kk, idO, (kr > 0 || kk > 0) ? 1u : 0u);
        if constexpr (VQ) {
          const uint64_t dvs = tc_sdesc(sb + SM::VS + (kr % NB) * SM::TILE, 2048, 128);
#pragma unroll
          for (int kk = 0; kk < kTcTok / 16; ++kk)
            mma_ta(tmem + TC::OSK, tmem + TC::PSK + 8 * kk, dvs + 256u * kk, idO,
                          (kr > 0 || kk > 0) ? 1u : 0u);
        }
        commit(B_O + 8 * (kr % NB));
        ++kr;
        moved = true;
      }
      // one score buffer: S(ks) only after the rows have read S(ks - 1)
      if (ks < ntiles && ks <= kr + 1 && (TC::NS == 2 || ks == 0 || test(B_SC, (uint32_t)(ks - 1) & 1u)) &&
          test(B_U + 8 * (ks % NB), (uint32_t)(ks / NB) & 1u)) {
        tc_fence_after();
        const int bf = ks % NB;
        const uint64_t dkh = tc_sdesc(sb + SM::KHI + bf * SM::KSTR, 128, 2048);
        const uint64_t dkl = tc_sdesc(sb + SM::KLO + bf * SM::KSTR, 128, 2048);
        const uint32_t dS = tmem + kTcS + kTcTok * (TC::NS == 2 ? (ks & 1) : 0);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          if constexpr (TC::WIDE) {  // [K_hi | K_lo]: 128 rows from dkh
            mma_ta(dS, tmem + kTcQhi + 8 * kk, dkh + 16u * kk, idS2, kk > 0 ? 1u : 0u);
            mma_ta(dS, tmem + kTcQlo + 8 * kk, dkh + 16u * kk, idS, 1u);
          } else {
            mma_ta(dS, tmem + kTcQhi + 8 * kk, dkh + 16u * kk, idS, kk > 0 ? 1u : 0u);
            mma_ta(dS, tmem + kTcQlo + 8 * kk, dkh + 16u * kk, idS, 1u);
            mma_ta(dS, tmem + kTcQhi + 8 * kk, dkl + 16u * kk, idS, 1u);
          }
        }
        if constexpr (KQ) {  // + (c S_K q_rot) (rho_K (2 sigma - 1))^T, A from shared memory
          const uint64_t dq = tc_sdesc(sb + SM::QSK, 128, 2048), dks = tc_sdesc(sb + SM::KS + bf * SM::TILE, 128, 2048);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) mma(dS, dq + 16u * kk, dks + 16u * kk, idS, 1u);
        }
        commit(B_S + 8 * (TC::NS == 2 ? (ks & 1) : 0));
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
      if constexpr (TC::WIDE) {  // + Q_hi K_lo^T from the second half
        float s2[32];
        tc_ld32(trow + kTcS + kTcTok + 32 * hf, s2);
#pragma unroll
        for (int j = 0; j < 32; ++j) s[j] += s2[j];
      }
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
    if constexpr (VQ) {
      if (p.kbits == p.vbits) {
        switch (p.kbits) {
          case 3: return go(prefill_tc_kernel<3, 3, true, true>);
          case 2: return go(prefill_tc_kernel<2, 2, true, true>);
          case 1: return go(prefill_tc_kernel<1, 1, true, true>);
        }
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

  const bool kq = ctx->cfg.k.qjl != 0, vq = ctx->cfg.v.qjl != 0;
  {  // the kernel's packed stages must fit next to its tiles (they do for every record of head dim 128)
    PrefillParams q0;
    q0.kblk = (unsigned)ctx->layout.block[0];
    q0.vblk = (unsigned)ctx->layout.block[1];
    const int need = kq ? (vq ? pf_tc_smem<true, true>(q0) : pf_tc_smem<false, true>(q0))
                        : (vq ? pf_tc_smem<true, false>(q0) : pf_tc_smem<false, false>(q0));
    if (need > kTcSmemMax) {
      set_error("prefill: the cache records are too large for the prefill kernel's shared memory");
      return TQ_ERR_UNSUPPORTED;
    }
  }
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
  if (kq && vq) e = launch_pf_tc<true, true>(p, grid, s);
  else if (kq) e = launch_pf_tc<false, true>(p, grid, s);
  else if (vq) e = launch_pf_tc<true, false>(p, grid, s);
  else e = launch_pf_tc<false, false>(p, grid, s);
  if (e != cudaSuccess) return tqd::pf_fail("prefill", e);
  return TQ_OK;
}

}  // namespace tqi
