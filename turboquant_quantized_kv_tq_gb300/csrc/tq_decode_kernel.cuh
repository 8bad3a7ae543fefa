// Fused decode attention over the packed cache (head dim 128), templated on the two codecs.
//
// [HEADQ] "Espaço de Pontuação da Chave" / "Geometria de Leitura de Valores": keys enter through
// scores q^T k / sqrt(d), values through the attention-weighted sum.  [TQ-KV] "Contribuciones
// Clave" 1: the QJL estimate sqrt(pi/2)/m * ||r|| * <S a, sign(S r)> of a residual inner
// product.  [HEADQ] "Leitura do Cache": s_hat = q^T k_base / sqrt(d) + q^T U z_hat / sqrt(d).
//
// Everything happens in the rotated domain: with q_rot = R_K q, the key score is
// nu_K * <q_rot, C[c]> (+ nu_K * rho_K * sqrt(pi/2)/m * <S_K q_rot, 2 sigma - 1>) (+ scale *
// <U^T q, zeta>), and the value readout accumulates acc = sum p nu_V C[c] and, on a QJL value
// side, acc_sk = sum p nu_V rho_V (2 sigma - 1); the merge applies
// o = R_V^T (acc + sqrt(pi/2)/m S_V^T acc_sk) / l once per head.
//
// Work split: grid (splits, H_kv, B); each block covers one contiguous token range of one
// (batch, KV head) slab for all G <= 8 query heads of the group; each warp streams its own
// sub-range in tiles of 16 tokens.  Per tile:
//   scores  S[16 tok x 8 heads] = K_hat[16 x 128] Q[128 x 8]   (8 mma.m16n8k16)
//   readout O^T[128 dims x 8 heads] += V_hat^T[128 x 16] P[16 x 8]  (8 mma), P moved from the
//           score accumulator layout to the B operand layout with movmatrix.trans.
// Packed codes go straight from global memory (16-byte coalesced loads) to registers and are
// expanded to fp16 pairs through lane-replicated lookup tables in shared memory (entry e for
// lane l at word 32 e + l: conflict-free) or, for sign bits, by moving the bit into the fp16
// sign position.  Token order inside a tile is permuted so that each thread's value operands
// come from four consecutive tokens: score row r <-> token pi(r) = 4((r&7)>>1) + 2(r>>3) + (r&1).
#pragma once

#include <cfloat>

#include "tq_device.cuh"

namespace tqd {

constexpr int kDecD = 128;
constexpr int kDecWarps = 8;
constexpr int kTile = 16;
constexpr int kHeadsPad = 8;

struct DecodeParams {
  Tables tab;
  Cache cache;
  const uint32_t* q_rot;  // fp16 pairs [B][Hq][D/2]
  const uint32_t* q_sk;   // fp16 pairs [B][Hq][m/2]
  const uint32_t* q_u;    // fp16 pairs [B][Hq][8]
  float* part;            // [B][Hkv][splits][8][PS]
  int* tickets;           // [B][Hkv]
  float* out;             // [B][Hq][D]
  int B, Hkv, G, splits, chunk, v_rotate;
  float score_scale;  // log2(e) / sqrt(d)
  float qjl_scale;    // sqrt(pi/2) / m
  int seq_len[TQ_MAX_BATCH];
};

template <int B>
struct LutEntries { static constexpr int value = B == 4 ? 256 : (B == 1 ? 0 : 16); };

// Lane-replicated pair table for a b-bit codebook (sign-magnitude symbols).
template <int B>
__device__ __forceinline__ void build_lut(uint32_t* lut, const float* cent) {
  constexpr int N = LutEntries<B>::value;
  for (int i = threadIdx.x; i < N * 32; i += blockDim.x) {
    const int e = i >> 5;
    float lo, hi;
    if constexpr (B == 4) {
      const int a = e & 15, c = e >> 4;
      lo = (a & 8 ? 1.f : -1.f) * __ldg(cent + 8 + (a & 7));
      hi = (c & 8 ? 1.f : -1.f) * __ldg(cent + 8 + (c & 7));
    } else if constexpr (B == 3) {  // magnitudes only
      lo = __ldg(cent + 4 + (e & 3));
      hi = __ldg(cent + 4 + (e >> 2));
    } else {  // B == 2: field (s << 1) | k
      const int a = e & 3, c = e >> 2;
      lo = (a & 2 ? 1.f : -1.f) * __ldg(cent + 2 + (a & 1));
      hi = (c & 2 ? 1.f : -1.f) * __ldg(cent + 2 + (c & 1));
    }
    lut[i] = pack_half2(lo, hi);
  }
}

__device__ __forceinline__ uint32_t lut_get(const uint32_t* lut_lane, uint32_t idx) {
  return lut_lane[idx << 5];
}

// half2 with the sign bits taken from bits 15 and 31 of ~xsh (bit set in xsh = positive).
__device__ __forceinline__ uint32_t signed_pair(uint32_t mag, uint32_t xsh) {
  return mag | (~xsh & 0x80008000u);
}

// ---------------------------------------------------------------------------------------------
// Key side: per thread, the 32-coordinate chunk [32 lt, 32 lt + 32) of the two tokens of its
// score rows.
template <int KB>
struct KChunk;

template <>
struct KChunk<4> {
  uint4 c;
  __device__ __forceinline__ void load(const unsigned char* rec, int lt) { c = ldg_stream16(rec + 16 * lt); }
  __device__ __forceinline__ void prepare() {}
  __device__ __forceinline__ uint32_t pair(const uint32_t* lut, uint32_t, int p) const {
    const uint32_t w = p < 4 ? c.x : p < 8 ? c.y : p < 12 ? c.z : c.w;
    return lut_get(lut, (w >> (8 * (p & 3))) & 0xffu);
  }
};

template <>
struct KChunk<3> {
  uint2 k;
  uint32_t s;
  __device__ __forceinline__ void load(const unsigned char* rec, int lt) {
    k = ldg_stream8(rec + 8 * lt);
    s = ldg_stream4(rec + kDecD / 4 + 4 * lt);
  }
  __device__ __forceinline__ void prepare() { s = unshuffle_bits(s); }
  __device__ __forceinline__ uint32_t pair(const uint32_t* lut, uint32_t, int p) const {
    const uint32_t w = p < 8 ? k.x : k.y;
    const uint32_t mag = lut_get(lut, (w >> (4 * (p & 7))) & 0xfu);
    return signed_pair(mag, s << (15 - p));
  }
};

template <>
struct KChunk<2> {
  uint2 k;
  __device__ __forceinline__ void load(const unsigned char* rec, int lt) { k = ldg_stream8(rec + 8 * lt); }
  __device__ __forceinline__ void prepare() {}
  __device__ __forceinline__ uint32_t pair(const uint32_t* lut, uint32_t, int p) const {
    const uint32_t w = p < 8 ? k.x : k.y;
    return lut_get(lut, (w >> (4 * (p & 7))) & 0xfu);
  }
};

template <>
struct KChunk<1> {
  uint32_t s;
  __device__ __forceinline__ void load(const unsigned char* rec, int lt) { s = ldg_stream4(rec + 4 * lt); }
  __device__ __forceinline__ void prepare() { s = unshuffle_bits(s); }
  __device__ __forceinline__ uint32_t pair(const uint32_t*, uint32_t m0, int p) const {
    return signed_pair(m0, s << (15 - p));
  }
};

// Sign chunk of a QJL key: 32 bits per token, as +-1 pairs.
struct KSign {
  uint32_t s;
  __device__ __forceinline__ void load(const unsigned char* rec, int lt) { s = ldg_stream4(rec + 4 * lt); }
  __device__ __forceinline__ void prepare() { s = unshuffle_bits(s); }
  __device__ __forceinline__ uint32_t pair(int p) const { return signed_pair(0x3C003C00u, s << (15 - p)); }
};

// ---------------------------------------------------------------------------------------------
// Value side: per thread, dims [16 lg, 16 lg + 16) of the four tokens 4 lt .. 4 lt + 3.
template <int VB>
struct VChunk;

template <>
struct VChunk<4> {
  uint2 w[4];
  uint32_t e01[2], o01[2], e23[2], o23[2];
  __device__ __forceinline__ void load(const unsigned char* const (&rec)[4], int lg) {
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = ldg_stream8(rec[j] + 8 * lg);
  }
  __device__ __forceinline__ void prepare() {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t a = h ? w[0].y : w[0].x, b = h ? w[1].y : w[1].x;
      const uint32_t c = h ? w[2].y : w[2].x, d = h ? w[3].y : w[3].x;
      e01[h] = (a & 0x0F0F0F0Fu) | ((b & 0x0F0F0F0Fu) << 4);
      o01[h] = ((a >> 4) & 0x0F0F0F0Fu) | (b & 0xF0F0F0F0u);
      e23[h] = (c & 0x0F0F0F0Fu) | ((d & 0x0F0F0F0Fu) << 4);
      o23[h] = ((c >> 4) & 0x0F0F0F0Fu) | (d & 0xF0F0F0F0u);
    }
  }
  __device__ __forceinline__ void frag(const uint32_t* lut, uint32_t, int mt, uint32_t (&a)[4]) const {
    const int h = mt >> 2, sh = 8 * (mt & 3);
    a[0] = lut_get(lut, (e01[h] >> sh) & 0xffu);
    a[1] = lut_get(lut, (o01[h] >> sh) & 0xffu);
    a[2] = lut_get(lut, (e23[h] >> sh) & 0xffu);
    a[3] = lut_get(lut, (o23[h] >> sh) & 0xffu);
  }
};

template <>
struct VChunk<3> {
  uint32_t k[4], s[4];
  uint32_t e01, o01, e23, o23, x01, x23;
  __device__ __forceinline__ void load(const unsigned char* const (&rec)[4], int lg) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      k[j] = ldg_stream4(rec[j] + 4 * lg);
      s[j] = ldg_stream2(rec[j] + kDecD / 4 + 2 * lg);
    }
  }
  __device__ __forceinline__ void prepare() {
    e01 = (k[0] & 0x33333333u) | ((k[1] & 0x33333333u) << 2);
    o01 = ((k[0] >> 2) & 0x33333333u) | (k[1] & 0xCCCCCCCCu);
    e23 = (k[2] & 0x33333333u) | ((k[3] & 0x33333333u) << 2);
    o23 = ((k[2] >> 2) & 0x33333333u) | (k[3] & 0xCCCCCCCCu);
    x01 = (s[0] & 0xffffu) | (s[1] << 16);
    x23 = (s[2] & 0xffffu) | (s[3] << 16);
  }
  __device__ __forceinline__ void frag(const uint32_t* lut, uint32_t, int mt, uint32_t (&a)[4]) const {
    const int sh = 4 * mt;
    a[0] = signed_pair(lut_get(lut, (e01 >> sh) & 0xfu), x01 << (15 - 2 * mt));
    a[1] = signed_pair(lut_get(lut, (o01 >> sh) & 0xfu), x01 << (14 - 2 * mt));
    a[2] = signed_pair(lut_get(lut, (e23 >> sh) & 0xfu), x23 << (15 - 2 * mt));
    a[3] = signed_pair(lut_get(lut, (o23 >> sh) & 0xfu), x23 << (14 - 2 * mt));
  }
};

template <>
struct VChunk<2> {
  uint32_t k[4];
  uint32_t e01, o01, e23, o23;
  __device__ __forceinline__ void load(const unsigned char* const (&rec)[4], int lg) {
#pragma unroll
    for (int j = 0; j < 4; ++j) k[j] = ldg_stream4(rec[j] + 4 * lg);
  }
  __device__ __forceinline__ void prepare() {
    e01 = (k[0] & 0x33333333u) | ((k[1] & 0x33333333u) << 2);
    o01 = ((k[0] >> 2) & 0x33333333u) | (k[1] & 0xCCCCCCCCu);
    e23 = (k[2] & 0x33333333u) | ((k[3] & 0x33333333u) << 2);
    o23 = ((k[2] >> 2) & 0x33333333u) | (k[3] & 0xCCCCCCCCu);
  }
  __device__ __forceinline__ void frag(const uint32_t* lut, uint32_t, int mt, uint32_t (&a)[4]) const {
    const int sh = 4 * mt;
    a[0] = lut_get(lut, (e01 >> sh) & 0xfu);
    a[1] = lut_get(lut, (o01 >> sh) & 0xfu);
    a[2] = lut_get(lut, (e23 >> sh) & 0xfu);
    a[3] = lut_get(lut, (o23 >> sh) & 0xfu);
  }
};

// 1-bit stream of 16 dims per token: values (+-M0) or QJL signs (+-1) depending on `base`.
struct VBits {
  uint32_t s[4];
  uint32_t x01, x23;
  __device__ __forceinline__ void load(const unsigned char* const (&rec)[4], int lg) {
#pragma unroll
    for (int j = 0; j < 4; ++j) s[j] = ldg_stream2(rec[j] + 2 * lg);
  }
  __device__ __forceinline__ void prepare() {
    x01 = (s[0] & 0xffffu) | (s[1] << 16);
    x23 = (s[2] & 0xffffu) | (s[3] << 16);
  }
  __device__ __forceinline__ void frag(uint32_t base, int mt, uint32_t (&a)[4]) const {
    a[0] = signed_pair(base, x01 << (15 - 2 * mt));
    a[1] = signed_pair(base, x01 << (14 - 2 * mt));
    a[2] = signed_pair(base, x23 << (15 - 2 * mt));
    a[3] = signed_pair(base, x23 << (14 - 2 * mt));
  }
};

template <>
struct VChunk<1> {
  VBits bits;
  __device__ __forceinline__ void load(const unsigned char* const (&rec)[4], int lg) { bits.load(rec, lg); }
  __device__ __forceinline__ void prepare() { bits.prepare(); }
  __device__ __forceinline__ void frag(const uint32_t*, uint32_t m0, int mt, uint32_t (&a)[4]) const {
    bits.frag(m0, mt, a);
  }
};

// ---------------------------------------------------------------------------------------------
// One tile's raw data for one thread.
template <int KB, bool KQ, bool KH, int VB, bool VQ>
struct TileData {
  KChunk<KB> kA, kB;
  KSign sA, sB;             // KQ
  uint2 zA, zB;             // KH: side code bytes lt, lt + 4 (as two words)
  float nuKA, nuKB, rhoKA, rhoKB, zsA, zsB;
  VChunk<VB> v;
  VBits vs;                 // VQ
  float nuVA, nuVB, rhoVA, rhoVB;
};

__device__ __forceinline__ float ld_f32(const unsigned char* p) {
  return __uint_as_float(ldg_stream4(p));
}
__device__ __forceinline__ float ld_f16(const unsigned char* p) {
  const unsigned short h = (unsigned short)ldg_stream2(p);
  return __half2float(__ushort_as_half(h));
}

// Signed 4-bit pairs (two's complement) -> exact fp16 integers, low nibble first.
__device__ __forceinline__ uint32_t side_pair(uint32_t byte) {
  uint32_t x = (byte & 0xFu) | ((byte & 0xF0u) << 12);
  x = (x ^ 0x00080008u) | 0x64006400u;  // 1024 + (n ^ 8), i.e. 1032 + n
  const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&x), __floats2half2_rn(1032.f, 1032.f));
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ int tile_row_token(int r) {
  return 4 * ((r & 7) >> 1) + 2 * (r >> 3) + (r & 1);
}

template <int KB, bool KQ, bool KH, int VB, bool VQ>
__device__ __forceinline__ void load_ktile(TileData<KB, KQ, KH, VB, VQ>& d, const Cache& C, int b,
                                           int kvh, int t0, int last, int lg, int lt) {
  const int tA = min(t0 + tile_row_token(lg), last);
  const int tB = min(t0 + tile_row_token(lg + 8), last);
  d.kA.load(C.ptr(tqi::R_K_CODES, b, kvh, tA), lt);
  d.kB.load(C.ptr(tqi::R_K_CODES, b, kvh, tB), lt);
  d.nuKA = ld_f32(C.ptr(tqi::R_K_NORM, b, kvh, tA));
  d.nuKB = ld_f32(C.ptr(tqi::R_K_NORM, b, kvh, tB));
  if constexpr (KQ) {
    d.sA.load(C.ptr(tqi::R_K_SIGNS, b, kvh, tA), lt);
    d.sB.load(C.ptr(tqi::R_K_SIGNS, b, kvh, tB), lt);
    d.rhoKA = ld_f16(C.ptr(tqi::R_K_RHO, b, kvh, tA));
    d.rhoKB = ld_f16(C.ptr(tqi::R_K_RHO, b, kvh, tB));
  }
  if constexpr (KH) {
    const uint2 sa = ldg_stream8(C.ptr(tqi::R_K_SIDE, b, kvh, tA));
    const uint2 sb = ldg_stream8(C.ptr(tqi::R_K_SIDE, b, kvh, tB));
    d.zA = make_uint2((sa.x >> (8 * lt)) & 0xffu, (sa.y >> (8 * lt)) & 0xffu);
    d.zB = make_uint2((sb.x >> (8 * lt)) & 0xffu, (sb.y >> (8 * lt)) & 0xffu);
    d.zsA = ld_f16(C.ptr(tqi::R_K_SIDE_SCALE, b, kvh, tA));
    d.zsB = ld_f16(C.ptr(tqi::R_K_SIDE_SCALE, b, kvh, tB));
  }
}

// Unscaled key scores of the thread's four accumulator slots (tokens pi(lg), pi(lg+8) x heads
// 2 lt, 2 lt + 1): nu <q_rot, C[c]> (+ nu rho sqrt(pi/2)/m <S q_rot, 2 sigma - 1>)
// (+ scale <U^T q, zeta>).  Multiply by 1/sqrt(d) for the logit.
template <int KB, bool KQ, bool KH, int VB, bool VQ>
__device__ __forceinline__ void key_scores(TileData<KB, KQ, KH, VB, VQ>& d, float (&s)[4],
                                           const uint32_t (&qf)[16], const uint32_t (&qs)[16],
                                           const uint32_t (&qu)[2], const uint32_t* lutK,
                                           uint32_t k_m0, float qjl_scale) {
  d.kA.prepare();
  d.kB.prepare();
  float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    mma16816(sc, d.kA.pair(lutK, k_m0, 2 * ks), d.kB.pair(lutK, k_m0, 2 * ks),
             d.kA.pair(lutK, k_m0, 2 * ks + 1), d.kB.pair(lutK, k_m0, 2 * ks + 1), qf[2 * ks],
             qf[2 * ks + 1]);
  }
  s[0] = sc[0] * d.nuKA;
  s[1] = sc[1] * d.nuKA;
  s[2] = sc[2] * d.nuKB;
  s[3] = sc[3] * d.nuKB;
  if constexpr (KQ) {
    d.sA.prepare();
    d.sB.prepare();
    float sq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      mma16816(sq, d.sA.pair(2 * ks), d.sB.pair(2 * ks), d.sA.pair(2 * ks + 1), d.sB.pair(2 * ks + 1),
               qs[2 * ks], qs[2 * ks + 1]);
    }
    const float fa = d.nuKA * d.rhoKA * qjl_scale, fb = d.nuKB * d.rhoKB * qjl_scale;
    s[0] = fmaf(sq[0], fa, s[0]);
    s[1] = fmaf(sq[1], fa, s[1]);
    s[2] = fmaf(sq[2], fb, s[2]);
    s[3] = fmaf(sq[3], fb, s[3]);
  }
  if constexpr (KH) {
    float sz[4] = {0.f, 0.f, 0.f, 0.f};
    mma16816(sz, side_pair(d.zA.x), side_pair(d.zB.x), side_pair(d.zA.y), side_pair(d.zB.y), qu[0], qu[1]);
    s[0] = fmaf(sz[0], d.zsA, s[0]);
    s[1] = fmaf(sz[1], d.zsA, s[1]);
    s[2] = fmaf(sz[2], d.zsB, s[2]);
    s[3] = fmaf(sz[3], d.zsB, s[3]);
  }
}

template <int KB, bool KQ, bool KH, int VB, bool VQ>
__device__ __forceinline__ void load_tile(TileData<KB, KQ, KH, VB, VQ>& d, const DecodeParams& p,
                                          int b, int kvh, int t0, int last, int lg, int lt) {
  const Cache& C = p.cache;
  load_ktile(d, C, b, kvh, t0, last, lg, lt);
  const int tA = min(t0 + tile_row_token(lg), last);
  const int tB = min(t0 + tile_row_token(lg + 8), last);
  const unsigned char* vrec[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) vrec[j] = C.ptr(tqi::R_V_CODES, b, kvh, min(t0 + 4 * lt + j, last));
  d.v.load(vrec, lg);
  d.nuVA = ld_f32(C.ptr(tqi::R_V_NORM, b, kvh, tA));
  d.nuVB = ld_f32(C.ptr(tqi::R_V_NORM, b, kvh, tB));
  if constexpr (VQ) {
    const unsigned char* srec[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) srec[j] = C.ptr(tqi::R_V_SIGNS, b, kvh, min(t0 + 4 * lt + j, last));
    d.vs.load(srec, lg);
    d.rhoVA = ld_f16(C.ptr(tqi::R_V_RHO, b, kvh, tA));
    d.rhoVB = ld_f16(C.ptr(tqi::R_V_RHO, b, kvh, tB));
  }
}

// Per-warp running state.
template <bool VQ>
struct WarpState {
  float m0, m1;  // running max (log2 domain) of heads 2 lt, 2 lt + 1
  float l0, l1;  // this thread's partial softmax denominators
  float acc[8][4];
  float accs[VQ ? 8 : 1][4];
};

template <int KB, bool KQ, bool KH, int VB, bool VQ>
__device__ __forceinline__ void compute_tile(TileData<KB, KQ, KH, VB, VQ>& d, WarpState<VQ>& st,
                                             const uint32_t (&qf)[16], const uint32_t (&qs)[16],
                                             const uint32_t (&qu)[2], const uint32_t* lutK,
                                             const uint32_t* lutV, uint32_t k_m0, uint32_t v_m0,
                                             const DecodeParams& p, int t0, int end, int lg) {
  // ---- scores
  float s[4];
  key_scores(d, s, qf, qs, qu, lutK, k_m0, p.qjl_scale);
  const bool va = t0 + tile_row_token(lg) < end;
  const bool vb = t0 + tile_row_token(lg + 8) < end;
  s[0] = va ? s[0] * p.score_scale : -INFINITY;
  s[1] = va ? s[1] * p.score_scale : -INFINITY;
  s[2] = vb ? s[2] * p.score_scale : -INFINITY;
  s[3] = vb ? s[3] * p.score_scale : -INFINITY;

  // ---- online softmax (log2 domain)
  float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
  for (int m = 4; m <= 16; m <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, m));
    mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, m));
  }
  const float n0 = fmaxf(st.m0, mx0), n1 = fmaxf(st.m1, mx1);
  if (__any_sync(kFull, n0 > st.m0 || n1 > st.m1)) {
    const float a0 = exp2f(st.m0 - n0), a1 = exp2f(st.m1 - n1);
    st.l0 *= a0;
    st.l1 *= a1;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      st.acc[mt][0] *= a0; st.acc[mt][1] *= a1; st.acc[mt][2] *= a0; st.acc[mt][3] *= a1;
      if constexpr (VQ) {
        st.accs[mt][0] *= a0; st.accs[mt][1] *= a1; st.accs[mt][2] *= a0; st.accs[mt][3] *= a1;
      }
    }
    st.m0 = n0;
    st.m1 = n1;
  }
  const float p0 = exp2f(s[0] - n0), p1 = exp2f(s[1] - n1);
  const float p2 = exp2f(s[2] - n0), p3 = exp2f(s[3] - n1);
  st.l0 += p0 + p2;
  st.l1 += p1 + p3;

  // ---- value readout
  const uint32_t bv0 = movmatrix_trans(pack_half2(p0 * d.nuVA, p1 * d.nuVA));
  const uint32_t bv1 = movmatrix_trans(pack_half2(p2 * d.nuVB, p3 * d.nuVB));
  d.v.prepare();
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    uint32_t a[4];
    d.v.frag(lutV, v_m0, mt, a);
    mma16816(st.acc[mt], a[0], a[1], a[2], a[3], bv0, bv1);
  }
  if constexpr (VQ) {
    const float fa = d.nuVA * d.rhoVA, fb = d.nuVB * d.rhoVB;
    const uint32_t bs0 = movmatrix_trans(pack_half2(p0 * fa, p1 * fa));
    const uint32_t bs1 = movmatrix_trans(pack_half2(p2 * fb, p3 * fb));
    d.vs.prepare();
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      uint32_t a[4];
      d.vs.frag(0x3C003C00u, mt, a);
      mma16816(st.accs[mt], a[0], a[1], a[2], a[3], bs0, bs1);
    }
  }
}

template <int KB, int VB, bool VQ>
struct DecodeSmem {
  static constexpr int lutK = LutEntries<KB>::value * 32;
  static constexpr int lutV = LutEntries<VB>::value * 32;
  // partial record per head: m, l, 2 pad words, acc[D], (acc_sk[m])
  static constexpr int PS = 4 + kDecD + (VQ ? kDecD : 0);
  static constexpr int merge = kDecWarps * kHeadsPad * PS;
  static constexpr int words = (lutK + lutV) > merge ? (lutK + lutV) : merge;
  static constexpr int bytes = words * 4 + 64;
};

template <int KB, bool KQ, bool KH, int VB, bool VQ>
__global__ void __launch_bounds__(kDecWarps * 32, 1) decode_kernel(const DecodeParams p) {
  using SM = DecodeSmem<KB, VB, VQ>;
  constexpr int PS = SM::PS;
  extern __shared__ __align__(16) uint32_t smem[];
  __shared__ int s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int lg = lane >> 2, lt = lane & 3;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;

  uint32_t* lutK = smem;
  uint32_t* lutV = smem + SM::lutK;
  if constexpr (KB != 1) build_lut<KB>(lutK, p.tab.k_c);
  if constexpr (VB != 1) build_lut<VB>(lutV, p.tab.v_c);
  const uint32_t k_m0 = pack_half2(__ldg(p.tab.k_c + 1), __ldg(p.tab.k_c + 1));
  const uint32_t v_m0 = pack_half2(__ldg(p.tab.v_c + 1), __ldg(p.tab.v_c + 1));
  __syncthreads();

  // query fragments: head kvh * G + lg, dims [32 lt, 32 lt + 32)
  const int G = p.G;
  const int Hq = p.Hkv * G;
  const bool hv = lg < G;
  const long long qrow = (long long)b * Hq + kvh * G + (hv ? lg : 0);
  uint32_t qf[16], qs[16], qu[2];
#pragma unroll
  for (int i = 0; i < 16; i += 4) {
    const uint4 v = hv ? *reinterpret_cast<const uint4*>(p.q_rot + qrow * (kDecD / 2) + 16 * lt + i)
                       : make_uint4(0, 0, 0, 0);
    qf[i] = v.x; qf[i + 1] = v.y; qf[i + 2] = v.z; qf[i + 3] = v.w;
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) qs[i] = 0;
  if constexpr (KQ) {
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
      const uint4 v = hv ? *reinterpret_cast<const uint4*>(p.q_sk + qrow * (kDecD / 2) + 16 * lt + i)
                         : make_uint4(0, 0, 0, 0);
      qs[i] = v.x; qs[i + 1] = v.y; qs[i + 2] = v.z; qs[i + 3] = v.w;
    }
  }
  qu[0] = qu[1] = 0;
  if constexpr (KH) {
    if (hv) {
      qu[0] = p.q_u[qrow * 8 + lt];
      qu[1] = p.q_u[qrow * 8 + lt + 4];
    }
  }

  // this warp's token range
  const int T = p.seq_len[b];
  const int c0 = split * p.chunk;
  const int c1 = min(T, c0 + p.chunk);
  const int n = max(0, c1 - c0);
  const int per = ((n + kDecWarps - 1) / kDecWarps + kTile - 1) / kTile * kTile;
  const int w0 = c0 + warp * per;
  const int w1 = min(c1, w0 + per);

  WarpState<VQ> st;
  st.m0 = st.m1 = -INFINITY;
  st.l0 = st.l1 = 0.f;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      st.acc[mt][j] = 0.f;
      if constexpr (VQ) st.accs[mt][j] = 0.f;
    }

  if (w0 < w1) {
    const int last = w1 - 1;
    TileData<KB, KQ, KH, VB, VQ> cur, nxt;
    load_tile(cur, p, b, kvh, w0, last, lg, lt);
    for (int t0 = w0; t0 < w1; t0 += kTile) {
      const bool more = t0 + kTile < w1;
      if (more) load_tile(nxt, p, b, kvh, t0 + kTile, last, lg, lt);
      compute_tile(cur, st, qf, qs, qu, lutK + lane, lutV + lane, k_m0, v_m0, p, t0, w1, lg);
      if (more) cur = nxt;
    }
  }

  // ---- merge the warps of this block
  float l0 = st.l0, l1 = st.l1;
#pragma unroll
  for (int m = 4; m <= 16; m <<= 1) {
    l0 += __shfl_xor_sync(kFull, l0, m);
    l1 += __shfl_xor_sync(kFull, l1, m);
  }
  __syncthreads();  // tables no longer needed: reuse shared memory for the merge
  float* mb = reinterpret_cast<float*>(smem) + warp * kHeadsPad * PS;
  if (lg == 0) {
    mb[(2 * lt) * PS + 0] = st.m0;
    mb[(2 * lt) * PS + 1] = l0;
    mb[(2 * lt + 1) * PS + 0] = st.m1;
    mb[(2 * lt + 1) * PS + 1] = l1;
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int d0 = 16 * lg + 2 * mt;
    mb[(2 * lt) * PS + 4 + d0] = st.acc[mt][0];
    mb[(2 * lt + 1) * PS + 4 + d0] = st.acc[mt][1];
    mb[(2 * lt) * PS + 4 + d0 + 1] = st.acc[mt][2];
    mb[(2 * lt + 1) * PS + 4 + d0 + 1] = st.acc[mt][3];
    if constexpr (VQ) {
      mb[(2 * lt) * PS + 4 + kDecD + d0] = st.accs[mt][0];
      mb[(2 * lt + 1) * PS + 4 + kDecD + d0] = st.accs[mt][1];
      mb[(2 * lt) * PS + 4 + kDecD + d0 + 1] = st.accs[mt][2];
      mb[(2 * lt + 1) * PS + 4 + kDecD + d0 + 1] = st.accs[mt][3];
    }
  }
  __syncthreads();
  const float* all = reinterpret_cast<const float*>(smem);
  float* part_out = p.part + ((((long long)b * p.Hkv + kvh) * p.splits + split) * kHeadsPad) * PS;
  for (int idx = threadIdx.x; idx < G * PS; idx += blockDim.x) {
    const int h = idx / PS, e = idx % PS;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, all[(w * kHeadsPad + h) * PS]);
    float v;
    if (e == 0) {
      v = M;
    } else if (e == 2 || e == 3) {
      v = 0.f;
    } else {
      v = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) {
          const float mw = all[(w * kHeadsPad + h) * PS];
          v = fmaf(exp2f(mw - M), all[(w * kHeadsPad + h) * PS + e], v);
        }
      }
    }
    part_out[h * PS + e] = v;
  }

  // ---- the last block of this (batch, KV head) merges all splits
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(p.tickets + b * p.Hkv + kvh, 1);
    s_last = prev == p.splits - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (warp < G) {
    const int h = warp;
    const float* base = p.part + (((long long)b * p.Hkv + kvh) * p.splits * kHeadsPad + h) * PS;
    const long long sstride = (long long)kHeadsPad * PS;
    float M = -INFINITY;
    for (int s = 0; s < p.splits; ++s) M = fmaxf(M, __ldcg(base + s * sstride));
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f), accs = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
      for (int s = 0; s < p.splits; ++s) {
        const float* ps = base + s * sstride;
        const float w = exp2f(__ldcg(ps) - M);
        L = fmaf(w, __ldcg(ps + 1), L);
        const float4 a = __ldcg(reinterpret_cast<const float4*>(ps + 4 + 4 * lane));
        acc.x = fmaf(w, a.x, acc.x); acc.y = fmaf(w, a.y, acc.y);
        acc.z = fmaf(w, a.z, acc.z); acc.w = fmaf(w, a.w, acc.w);
        if constexpr (VQ) {
          const float4 c = __ldcg(reinterpret_cast<const float4*>(ps + 4 + kDecD + 4 * lane));
          accs.x = fmaf(w, c.x, accs.x); accs.y = fmaf(w, c.y, accs.y);
          accs.z = fmaf(w, c.z, accs.z); accs.w = fmaf(w, c.w, accs.w);
        }
      }
    }
    float o[4] = {acc.x, acc.y, acc.z, acc.w};
    if constexpr (VQ) {
      // o_rot += sqrt(pi/2)/m * S_V^T acc_sk
      const float sv[4] = {accs.x, accs.y, accs.z, accs.w};
      float corr[4] = {0.f, 0.f, 0.f, 0.f};
      for (int r4 = 0; r4 < 32; ++r4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float ar = __shfl_sync(kFull, sv[i], r4);
          const float4 srow =
              __ldg(reinterpret_cast<const float4*>(p.tab.S_V + (4 * r4 + i) * kDecD + 4 * lane));
          corr[0] = fmaf(srow.x, ar, corr[0]); corr[1] = fmaf(srow.y, ar, corr[1]);
          corr[2] = fmaf(srow.z, ar, corr[2]); corr[3] = fmaf(srow.w, ar, corr[3]);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = fmaf(p.qjl_scale, corr[i], o[i]);
    }
    const float invL = L > 0.f ? 1.f / L : 0.f;
    if (p.v_rotate) {
      wht_warp<4>(o);
      const float rs = 1.f / sqrtf((float)kDecD);
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = o[i] * rs * __ldg(p.tab.v_sign + 4 * lane + i) * invL;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] *= invL;
    }
    float* dst = p.out + ((long long)b * Hq + kvh * G + h) * kDecD + 4 * lane;
    *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
  }
  if (threadIdx.x == 0) p.tickets[b * p.Hkv + kvh] = 0;
}

// ---------------------------------------------------------------------------------------------
// Corrected logits for every stored token ([HEADQ] "Leitura do Cache"), without the softmax.
struct LogitsParams {
  Tables tab;
  Cache cache;
  const float* q;  // [B][Hq][D] fp32
  float* logits;   // [B][Hq][stride]
  int B, Hkv, G, stride, tokens_per_block, k_rotate;
  float qjl_scale, inv_sqrt_d;
  int seq_len[TQ_MAX_BATCH];
};

template <int KB>
struct LogitsSmem {
  static constexpr int lut = LutEntries<KB>::value * 32;
  static constexpr int words = lut + kHeadsPad * (kDecD / 2) * 2 + kHeadsPad * 8;
  static constexpr int bytes = words * 4;
};

template <int KB, bool KQ, bool KH>
__global__ void __launch_bounds__(kDecWarps * 32) logits_kernel(const LogitsParams p) {
  extern __shared__ __align__(16) uint32_t smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int lg = lane >> 2, lt = lane & 3;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int T = p.seq_len[b];
  const int c0 = blockIdx.x * p.tokens_per_block;
  if (c0 >= T) return;  // the whole block leaves together
  const int G = p.G, Hq = p.Hkv * G;
  uint32_t* lutK = smem;
  uint32_t* qrot = smem + LogitsSmem<KB>::lut;
  uint32_t* qsk = qrot + kHeadsPad * (kDecD / 2);
  uint32_t* qus = qsk + kHeadsPad * (kDecD / 2);
  if constexpr (KB != 1) build_lut<KB>(lutK, p.tab.k_c);
  const uint32_t k_m0 = pack_half2(__ldg(p.tab.k_c + 1), __ldg(p.tab.k_c + 1));
  if (warp < G) {
    const float4 q4 = *reinterpret_cast<const float4*>(p.q + ((long long)b * Hq + kvh * G + warp) * kDecD + 4 * lane);
    float x[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] *= __ldg(p.tab.k_sign + 4 * lane + i);
    if (p.k_rotate) {
      wht_warp<4>(x);
      const float rs = 1.f / sqrtf((float)kDecD);
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] *= rs;
    }
    qrot[warp * (kDecD / 2) + 2 * lane] = pack_half2(x[0], x[1]);
    qrot[warp * (kDecD / 2) + 2 * lane + 1] = pack_half2(x[2], x[3]);
    if constexpr (KQ) {
      float a[4] = {0.f, 0.f, 0.f, 0.f};
      for (int jl = 0; jl < 32; ++jl) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float xj = __shfl_sync(kFull, x[e], jl);
          const float4 s4 = __ldg(reinterpret_cast<const float4*>(p.tab.S_K_T + (4 * jl + e) * kDecD + 4 * lane));
          a[0] = fmaf(s4.x, xj, a[0]); a[1] = fmaf(s4.y, xj, a[1]);
          a[2] = fmaf(s4.z, xj, a[2]); a[3] = fmaf(s4.w, xj, a[3]);
        }
      }
      qsk[warp * (kDecD / 2) + 2 * lane] = pack_half2(a[0], a[1]);
      qsk[warp * (kDecD / 2) + 2 * lane + 1] = pack_half2(a[2], a[3]);
    }
    if constexpr (KH) {
      const float* Ur = p.tab.U_rot + (long long)kvh * kDecD * 16;
      float z[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) z[k] = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
#pragma unroll
        for (int k = 0; k < 16; ++k) z[k] = fmaf(__ldg(Ur + (4 * lane + e) * 16 + k), x[e], z[k]);
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) z[k] = warp_sum(z[k]);
      if (lane < 8) {
        float lo = 0.f, hi = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (k == lane) { lo = z[2 * k]; hi = z[2 * k + 1]; }
        }
        qus[warp * 8 + lane] = pack_half2(lo, hi);
      }
    }
  }
  __syncthreads();
  const bool hv = lg < G;
  uint32_t qf[16], qs[16], qu[2];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    qf[i] = hv ? qrot[lg * (kDecD / 2) + 16 * lt + i] : 0u;
    qs[i] = (KQ && hv) ? qsk[lg * (kDecD / 2) + 16 * lt + i] : 0u;
  }
  qu[0] = (KH && hv) ? qus[lg * 8 + lt] : 0u;
  qu[1] = (KH && hv) ? qus[lg * 8 + lt + 4] : 0u;

  const int c1 = min(T, c0 + p.tokens_per_block);
  const int per = ((c1 - c0 + kDecWarps - 1) / kDecWarps + kTile - 1) / kTile * kTile;
  const int w0 = c0 + warp * per;
  const int w1 = min(c1, w0 + per);
  for (int t0 = w0; t0 < w1; t0 += kTile) {
    TileData<KB, KQ, KH, 1, false> d;
    load_ktile(d, p.cache, b, kvh, t0, w1 - 1, lg, lt);
    float s[4];
    key_scores(d, s, qf, qs, qu, lutK + lane, k_m0, p.qjl_scale);
    const int tA = t0 + tile_row_token(lg), tB = t0 + tile_row_token(lg + 8);
    const long long r0 = ((long long)b * Hq + kvh * G + 2 * lt) * p.stride;
    const long long r1 = r0 + p.stride;
    if (tA < w1) {
      if (2 * lt < G) p.logits[r0 + tA] = s[0] * p.inv_sqrt_d;
      if (2 * lt + 1 < G) p.logits[r1 + tA] = s[1] * p.inv_sqrt_d;
    }
    if (tB < w1) {
      if (2 * lt < G) p.logits[r0 + tB] = s[2] * p.inv_sqrt_d;
      if (2 * lt + 1 < G) p.logits[r1 + tB] = s[3] * p.inv_sqrt_d;
    }
  }
}

// Launch helpers used by the per-bit-width instantiation units.
template <int KB, bool KQ, bool KH, int VB, bool VQ>
cudaError_t launch_decode_t(const DecodeParams& p, dim3 grid, cudaStream_t s) {
  using SM = DecodeSmem<KB, VB, VQ>;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<KB, KQ, KH, VB, VQ>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SM::bytes);
  if (e != cudaSuccess) return e;
  decode_kernel<KB, KQ, KH, VB, VQ><<<grid, kDecWarps * 32, SM::bytes, s>>>(p);
  return cudaGetLastError();
}

template <int KB, bool KQ, bool KH>
cudaError_t launch_logits_t(const LogitsParams& p, dim3 grid, cudaStream_t s) {
  using SM = LogitsSmem<KB>;
  cudaError_t e = cudaFuncSetAttribute(logits_kernel<KB, KQ, KH>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SM::bytes);
  if (e != cudaSuccess) return e;
  logits_kernel<KB, KQ, KH><<<grid, kDecWarps * 32, SM::bytes, s>>>(p);
  return cudaGetLastError();
}

// Per-bit-width dispatchers (one translation unit each).  Return false when the codec
// combination is not built.
bool dispatch_decode_k1(int kq, int kh, int vb, int vq, const DecodeParams& p, dim3 g, cudaStream_t s, cudaError_t* e);
bool dispatch_decode_k2(int kq, int kh, int vb, int vq, const DecodeParams& p, dim3 g, cudaStream_t s, cudaError_t* e);
bool dispatch_decode_k3(int kq, int kh, int vb, int vq, const DecodeParams& p, dim3 g, cudaStream_t s, cudaError_t* e);
bool dispatch_decode_k4(int kq, int kh, int vb, int vq, const DecodeParams& p, dim3 g, cudaStream_t s, cudaError_t* e);
bool dispatch_logits_k1(int kq, int kh, const LogitsParams& p, dim3 g, cudaStream_t s, cudaError_t* e);
bool dispatch_logits_k2(int kq, int kh, const LogitsParams& p, dim3 g, cudaStream_t s, cudaError_t* e);
bool dispatch_logits_k3(int kq, int kh, const LogitsParams& p, dim3 g, cudaStream_t s, cudaError_t* e);
bool dispatch_logits_k4(int kq, int kh, const LogitsParams& p, dim3 g, cudaStream_t s, cudaError_t* e);

#define TQ_DECODE_CASE(KB_, KQ_, KH_, VB_, VQ_)                                           \
  if (kq == KQ_ && kh == KH_ && vb == VB_ && vq == VQ_) {                                 \
    *e = launch_decode_t<KB_, KQ_ != 0, KH_ != 0, VB_, VQ_ != 0>(p, g, s);                \
    return true;                                                                          \
  }
#define TQ_LOGITS_CASE(KB_, KQ_, KH_)                                                     \
  if (kq == KQ_ && kh == KH_) {                                                           \
    *e = launch_logits_t<KB_, KQ_ != 0, KH_ != 0>(p, g, s);                               \
    return true;                                                                          \
  }

}  // namespace tqd
