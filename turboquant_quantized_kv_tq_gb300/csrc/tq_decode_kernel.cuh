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
// Work split (balanced, "stream-K"): the (batch, KV head, token) positions of all sequences are
// laid end to end and cut into one equal contiguous range per block, one block per SM, counting
// a fixed allowance of virtual tiles before each slab so that a block whose range crosses a slab
// boundary takes fewer real tiles.  A block walks the slab segments of its range; for each, its
// warps stream contiguous sub-ranges in
// tiles of 16 tokens and the block merges them into one partial per (slab, block).  The last
// block to finish a slab (atomic ticket) merges that slab's partials in block order and writes
// the output.  Per tile:
//   scores  S[16 tok x 8 heads] = K_hat[16 x 128] Q[128 x 8]   (8 mma.m16n8k16)
//   readout O^T[128 dims x 8 heads] += V_hat^T[128 x 16] P[16 x 8]  (8 mma), P moved from the
//           score accumulator layout to the B operand layout with movmatrix.trans.
// Loads: each warp streams its tiles, two at a time, through a ring of two shared-memory stages;
// a stage holds two adjacent 16-token K blocks and the two matching V blocks of the cache (one
// bulk copy per side, completing on the stage's mbarrier) and is refilled as soon as its
// operands are in registers.  Codes become fp16 pairs
// through lane-replicated tables (entry e, lane l at byte 256 e + 4 l, the address built by one
// byte permute) or, for sign bits, by moving the bit to the fp16 sign position.  Token order
// inside a tile is permuted so each thread's value operands come from four consecutive tokens:
// score row r <-> token pi(r) = 4((r&7)>>1) + 2(r>>3) + (r&1).
#pragma once

#include <cfloat>

#include "tq_device.cuh"

namespace tqd {

constexpr int kDecD = 128;
constexpr int kSQ = 5;  // code-width tag of a spectral (SQU-KV) side in the decode templates
constexpr int kLogitsWarps = 8;
// Warps per decode block: 16 (4 per scheduler, 128 registers a thread), or 12 (170 registers)
// when the query's lo terms take their own MMAs (QLO): their fragments, and with a QJL value
// side a second accumulator (32 registers), do not fit 128.  Without QLO a QJL value side's
// readout shares the value MMA and its accumulator.
template <bool KQ, bool VQ, bool QLO>
struct DecWarps { static constexpr int value = (QLO || KQ || VQ) ? 12 : 16; };
constexpr int kQCols = 8;  // query columns per KV head in the prepared query arrays
constexpr int kTile = 16;
constexpr int kHeadsPad = 8;
constexpr int kPairStages = 2;  // per-warp ring of 32-token (two-tile) stages
constexpr int kMaxBlocks = 256;  // partial slots reserved for blocks (>= SM count)
constexpr int kLutStride = 256;  // bytes between table entries

struct DecodeParams {
  Tables tab;
  Cache cache;
  // Query columns: column c of KV head h is query i = c / G of the chunk, head h G + c % G
  // (nq queries per sequence, Gc = G nq <= 8 columns; nq = 1 is plain decode).
  // Queries are split into two fp16 terms, hi + lo (one rounding of q alone is a systematic
  // score error that long contexts turn into an output error of ~3e-3).  With 2 Gc <= 8 the lo
  // terms ride in columns Gc .. 2 Gc - 1 of the same MMA and are added back by a shuffle
  // (lo_xor); otherwise they sit in q_rot_lo / q_sk_lo and get their own MMA.
  const uint32_t* q_rot;  // fp16 pairs [B][Hkv][8 columns][D/2]
  const uint32_t* q_sk;   // fp16 pairs [B][Hkv][8][m/2]
  const uint32_t* q_u;    // fp16 pairs [B][Hkv][8][8] (hi term only: a small correction)
  const uint32_t* q_rot_lo;  // [B][Hkv][8][D/2], separate lo terms
  const uint32_t* q_sk_lo;
  float* part;            // [B*Hkv + kMaxBlocks][G][PS]; slab p's partial from block c at p + c
  int* tickets;           // [B*Hkv]
  int* err;               // device error word
  float* out;             // [B][nq][Hq][D]
  float* sk_final;        // [B][Hq][m]: acc_sk / l (head dim > 128 with a QJL value side)
  int B, Hkv, G, v_rotate, nblocks;
  int nq, Gc;             // queries per sequence (query i sees tokens [0, seq_len - nq + 1 + i))
  int lo_xor;             // lo columns: lane xor to add them back (Gc / 2), -1 when Gc = 1
  int n_fresh;            // each sequence's last n_fresh tokens are being written by the step's
                          // append until grid_dependency_wait returns (0: none)
  long long W;            // number of 16-token tiles over all (batch, KV head) slabs
  float score_scale;      // log2(e) / sqrt(d)
  float qjl_scale;        // sqrt(pi/2) / m
  int seq_len[TQ_MAX_BATCH];
  long long batch_start[TQ_MAX_BATCH + 1];  // first tile of batch b: Hkv * sum of ceil(len/16)
  // paged pool: lengths in device memory (clamped to [0, lmax]); each block then computes W,
  // seq_len and batch_start itself (paged_plan) in place of the copies above
  const int* dev_seq_len;
  int lmax;
};

template <int B>
struct LutEntries { static constexpr int value = (B == 4 || B == kSQ) ? 256 : B == 3 ? 64 : (B == 1 ? 0 : 16); };

// Lane-replicated pair table for a b-bit codebook (sign-magnitude symbols).
template <int B>
__device__ __forceinline__ void build_lut(unsigned char* lut, const float* cent) {
  constexpr int N = LutEntries<B>::value;
  for (int i = threadIdx.x; i < N * 32; i += blockDim.x) {
    const int e = i >> 5, l = i & 31;
    float lo, hi;
    if constexpr (B == 4) {
      const int a = e & 15, c = e >> 4;
      lo = (a & 8 ? 1.f : -1.f) * __ldg(cent + 8 + (a & 7));
      hi = (c & 8 ? 1.f : -1.f) * __ldg(cent + 8 + (c & 7));
    } else if constexpr (B == kSQ) {  // magnitudes of the 4-bit codebook, two 3-bit fields
      lo = __ldg(cent + 8 + (e & 7));
      hi = __ldg(cent + 8 + ((e >> 4) & 7));
    } else if constexpr (B == 3) {  // magnitudes in bits 0-1 / 2-3, their signs in bits 4 / 5
      lo = (e & 16 ? 1.f : -1.f) * __ldg(cent + 4 + (e & 3));
      hi = (e & 32 ? 1.f : -1.f) * __ldg(cent + 4 + ((e >> 2) & 3));
    } else {  // B == 2: field (s << 1) | k
      const int a = e & 3, c = e >> 2;
      lo = (a & 2 ? 1.f : -1.f) * __ldg(cent + 2 + (a & 1));
      hi = (c & 2 ? 1.f : -1.f) * __ldg(cent + 2 + (c & 1));
    }
    *reinterpret_cast<uint32_t*>(lut + e * kLutStride + 4 * l) = pack_half2(lo, hi);
  }
}

// Tables sit at fixed shared-window addresses that are multiples of 64 KiB, so the full address
// of entry e for lane l, A + 256 e + 4 l, is one byte permute of the code word with
// lx = A | 4 l (bytes: 4 l, e, A >> 16, 0), and a lookup is two instructions.
constexpr uint32_t kLutAddrK = 0x10000u;  // key table (and the value table when shared)
constexpr uint32_t kLutAddrV = 0x20000u;  // value table when its codebook differs
constexpr uint32_t kDynBaseMax = 0x1000u; // highest dynamic shared-memory start the plan allows

__device__ __forceinline__ uint32_t lut_get(uint32_t lx, uint32_t w, int j) {
  const uint32_t addr = __byte_perm(w, lx, 0x7604u | ((uint32_t)j << 4));
  uint32_t v;
  asm("ld.shared.u32 %0, [%1];\n" : "=r"(v) : "r"(addr));
  return v;
}

// half2 with the sign bits taken from bits 15 and 31 of ~xsh (bit set in xsh = positive).
__device__ __forceinline__ uint32_t signed_pair(uint32_t mag, uint32_t xsh) {
  return mag | (~xsh & 0x80008000u);
}

// Byte j of the result = nibble j of x (low half) | nibble 4 + j of x << 4.
__device__ __forceinline__ uint32_t nibble_pairs(uint32_t x) {
  x = __byte_perm(x, 0, 0x3120);  // nibbles 0 1 4 5 2 3 6 7
  const uint32_t t = (x ^ (x >> 4)) & 0x00F000F0u;
  return x ^ t ^ (t << 4);
}

// Outer perfect shuffle: bit i of the low half -> bit 2 i, bit i of the high half -> 2 i + 1.
__device__ __forceinline__ uint32_t shuffle_halves(uint32_t x) {
  uint32_t t;
  x = __byte_perm(x, 0, 0x3120);
  t = (x ^ (x >> 4)) & 0x00F000F0u; x ^= t ^ (t << 4);
  t = (x ^ (x >> 2)) & 0x0C0C0C0Cu; x ^= t ^ (t << 2);
  t = (x ^ (x >> 1)) & 0x22222222u; x ^= t ^ (t << 1);
  return x;
}

// Sign bits of 16 coordinate pairs (bit 2 p, 2 p + 1 of s for pair p) as two words in which pair
// p's bits sit at 2 (p & 7) and 2 (p & 7) + 16: lo for p < 8, hi for p >= 8.
struct PairSigns {
  uint32_t lo, hi;
  __device__ __forceinline__ void build(uint32_t s) {
    lo = __byte_perm(s, s << 15, 0x7610);
    hi = __byte_perm(s, s >> 1, 0x7632);
  }
  __device__ __forceinline__ uint32_t at(int p) const { return (p < 8 ? lo : hi) << (15 - 2 * (p & 7)); }
};

// Nibbles 0,2,4,6 / 1,3,5,7 of w, one per byte.
__device__ __forceinline__ uint32_t nib_even(uint32_t w) { return w & 0x0F0F0F0Fu; }
__device__ __forceinline__ uint32_t nib_odd(uint32_t w) { return (w >> 4) & 0x0F0F0F0Fu; }

// ---------------------------------------------------------------------------------------------
// Key side: per thread, the 32-coordinate chunk [32 lt, 32 lt + 32) of the two tokens of its
// score rows.  pair(p) is the fp16 pair of coordinates (2p, 2p+1) of the chunk.
template <int KB>
struct KChunk;

template <>
struct KChunk<4> {
  uint4 c;
  __device__ __forceinline__ void prepare() {}
  __device__ __forceinline__ uint32_t pair(uint32_t lx, uint32_t, int p) const {
    const uint32_t w = p < 4 ? c.x : p < 8 ? c.y : p < 12 ? c.z : c.w;
    return lut_get(lx, w, p & 3);
  }
};

// 3-bit keys: the magnitude nibble of a pair (two 2-bit fields) and its two sign bits form one
// 6-bit table index, so a signed pair is one lookup.  With t = nibble_pairs(s), byte j of t holds
// the signs of coordinates 4j .. 4j + 3 (bits 0-3) and 16 + 4j .. 16 + 4j + 3 (bits 4-7), so one
// shift per index word brings a pair's two signs to bits 4 and 5 of its byte.
template <>
struct KChunk<3> {
  uint2 k;
  uint32_t s;
  uint32_t xe, xo, ye, yo;
  __device__ __forceinline__ void prepare() {
    const uint32_t t = nibble_pairs(s);
    xe = nib_even(k.x) | ((t << 4) & 0x30303030u);
    xo = nib_odd(k.x) | ((t << 2) & 0x30303030u);
    ye = nib_even(k.y) | (t & 0x30303030u);
    yo = nib_odd(k.y) | ((t >> 2) & 0x30303030u);
  }
  __device__ __forceinline__ uint32_t pair(uint32_t lx, uint32_t, int p) const {
    const uint32_t w = p < 8 ? (p & 1 ? xo : xe) : (p & 1 ? yo : ye);
    return lut_get(lx, w, (p & 7) >> 1);
  }
};

template <>
struct KChunk<2> {
  uint2 k;
  uint32_t xe, xo, ye, yo;
  __device__ __forceinline__ void prepare() {
    xe = nib_even(k.x); xo = nib_odd(k.x); ye = nib_even(k.y); yo = nib_odd(k.y);
  }
  __device__ __forceinline__ uint32_t pair(uint32_t lx, uint32_t, int p) const {
    const uint32_t w = p < 8 ? (p & 1 ? xo : xe) : (p & 1 ? yo : ye);
    return lut_get(lx, w, (p & 7) >> 1);
  }
};

template <>
struct KChunk<1> {
  uint32_t s;
  PairSigns ps;
  __device__ __forceinline__ void prepare() { ps.build(s); }
  __device__ __forceinline__ uint32_t pair(uint32_t, uint32_t m0, int p) const {
    return signed_pair(m0, ps.at(p));
  }
};

// SQU-KV key chunk: the chunk's first 8 coordinates are modeled (4-bit magnitudes in mg, byte p
// = coordinates 2p, 2p + 1), the other 24 the 1-bit floor (magnitude m0 = the 1-bit centroid);
// s holds the 32 signs.
template <>
struct KChunk<kSQ> {
  uint32_t mg;
  uint32_t s;
  PairSigns ps;
  __device__ __forceinline__ void prepare() { ps.build(s); }
  __device__ __forceinline__ uint32_t pair(uint32_t lx, uint32_t m0, int p) const {
    return signed_pair(p < 4 ? lut_get(lx, mg, p) : m0, ps.at(p));
  }
};

// Sign chunk of a QJL key: 32 bits per token, as +-1 pairs.
struct KSign {
  uint32_t s;
  PairSigns ps;
  __device__ __forceinline__ void prepare() { ps.build(s); }
  __device__ __forceinline__ uint32_t pair(int p) const { return signed_pair(0x3C003C00u, ps.at(p)); }
};

// ---------------------------------------------------------------------------------------------
// Value side: per thread, dims [16 lg, 16 lg + 16) of the four tokens 4 lt .. 4 lt + 3.
// frag(mt) gives the A operand of M-tile mt: rows = dims 16 lg + 2 mt (+1), columns = tokens.
template <int VB>
struct VChunk;

template <>
struct VChunk<4> {
  uint2 w[4];
  uint32_t e01[2], o01[2], e23[2], o23[2];
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
  __device__ __forceinline__ void frag(uint32_t lx, uint32_t, int mt,
                                       uint32_t (&a)[4]) const {
    const int h = mt >> 2, j = mt & 3;
    a[0] = lut_get(lx, e01[h], j);
    a[1] = lut_get(lx, o01[h], j);
    a[2] = lut_get(lx, e23[h], j);
    a[3] = lut_get(lx, o23[h], j);
  }
};

// 2-bit fields of two tokens interleaved into nibbles (first token low), split into even / odd
// nibble bytes: index nibble for dim 2 mt (e) and 2 mt + 1 (o).
struct Pair2 {
  uint32_t e01[2], o01[2], e23[2], o23[2];
  __device__ __forceinline__ void build(const uint32_t (&k)[4]) {
    const uint32_t e0 = (k[0] & 0x33333333u) | ((k[1] & 0x33333333u) << 2);
    const uint32_t o0 = ((k[0] >> 2) & 0x33333333u) | (k[1] & 0xCCCCCCCCu);
    const uint32_t e1 = (k[2] & 0x33333333u) | ((k[3] & 0x33333333u) << 2);
    const uint32_t o1 = ((k[2] >> 2) & 0x33333333u) | (k[3] & 0xCCCCCCCCu);
    e01[0] = nib_even(e0); e01[1] = nib_odd(e0);
    o01[0] = nib_even(o0); o01[1] = nib_odd(o0);
    e23[0] = nib_even(e1); e23[1] = nib_odd(e1);
    o23[0] = nib_even(o1); o23[1] = nib_odd(o1);
  }
  __device__ __forceinline__ void mags(uint32_t lx, int mt, uint32_t (&a)[4]) const {
    const int h = mt & 1, j = mt >> 1;
    a[0] = lut_get(lx, e01[h], j);
    a[1] = lut_get(lx, o01[h], j);
    a[2] = lut_get(lx, e23[h], j);
    a[3] = lut_get(lx, o23[h], j);
  }
};

// 1-bit stream, 16 dims per token: bit i of token j for dims 16 lg + i; x01 holds tokens 0 (low
// half) and 1, x23 tokens 2 and 3 (the stream's group layout stores them that way).
struct Bits16 {
  uint32_t x01, x23;
  __device__ __forceinline__ void build(const uint32_t (&s)[2]) {
    x01 = s[0];
    x23 = s[1];
  }
  __device__ __forceinline__ void apply(int mt, uint32_t (&a)[4]) const {
    a[0] = signed_pair(a[0], x01 << (15 - 2 * mt));
    a[1] = signed_pair(a[1], x01 << (14 - 2 * mt));
    a[2] = signed_pair(a[2], x23 << (15 - 2 * mt));
    a[3] = signed_pair(a[3], x23 << (14 - 2 * mt));
  }
  // The bits of dims 16 lg + 2 mt (+1) as masked operands.  A word holds the bit of dim offset k
  // at k (first token) and k + 16 (second token).  Shifted left by s(k) = 0 (k >= 10), 6 (k >= 4)
  // or 12 (k < 4) -- three shifted copies of the word serve all 16 dims -- it sits at
  // pos(k) = k + s(k) in [10, 15], and masking it there gives an fp16 number 0 or 2^e(pos), all
  // normal (tensor cores flush subnormal inputs): 2^-14, 2^-13, 2^-11, 2^-7, 2^1 for pos 10 .. 14.
  // The readout's row k is then 2^e sum_j w_j sigma_j, and sum_j w_j (2 sigma_j - 1) =
  // 2 2^-e row - sum_j w_j.  pos 15 is the fp16 sign: those dims (k = 3, 9, 15) take +-1 instead.
  // One LOP3 per operand plus two shifts per word, where moving each bit to the sign position
  // takes a shift and a LOP3 per operand.
  __device__ __forceinline__ static uint32_t mask_bit(uint32_t x, int k) {
    const int sft = k >= 10 ? 0 : (k >= 4 ? 6 : 12), pos = k + sft;
    const uint32_t y = x << sft;
    // (a set bit is sigma = 1: +1, so the sign field takes the complement)
    return pos == 15 ? ((~y & 0x80008000u) | 0x3C003C00u) : (y & (0x00010001u << pos));
  }
  __device__ __forceinline__ void mask(int mt, uint32_t (&a)[4]) const {
    a[0] = mask_bit(x01, 2 * mt);
    a[1] = mask_bit(x01, 2 * mt + 1);
    a[2] = mask_bit(x23, 2 * mt);
    a[3] = mask_bit(x23, 2 * mt + 1);
  }
};

// Whether dim offset k's masked operand is +-1 (its bit lands on the fp16 sign) rather than
// sigma 2^e, and 2^-e for the others (Bits16::mask_bit).
__device__ __forceinline__ bool mask_is_pm1(int k) { return k == 3 || k == 9 || k == 15; }
__device__ __forceinline__ float mask_unscale(int k) {
  const int pos = k + (k >= 10 ? 0 : (k >= 4 ? 6 : 12));
  const int e = pos == 10 ? -14 : pos == 11 ? -13 : pos == 12 ? -11 : pos == 13 ? -7 : 1;
  return __int_as_float((127 - e) << 23);
}

// 3-bit values: as on the key side the two sign bits join the magnitude nibble in the table
// index.  After shuffle_halves, byte j of a sign word holds dims 4 j .. 4 j + 3 of the two tokens
// interleaved (token 0 at even bits), so one shift per index word places them at bits 4 and 5.
template <>
struct VChunk<3> {
  uint32_t k[4], s[2];
  Pair2 m;
  __device__ __forceinline__ static void fold(uint32_t x, uint32_t (&e)[2], uint32_t (&o)[2]) {
    x = shuffle_halves(x);
    e[0] |= (x << 4) & 0x30303030u;
    o[0] |= (x << 2) & 0x30303030u;
    e[1] |= x & 0x30303030u;
    o[1] |= (x >> 2) & 0x30303030u;
  }
  __device__ __forceinline__ void prepare() {
    m.build(k);
    fold(s[0], m.e01, m.o01);
    fold(s[1], m.e23, m.o23);
  }
  __device__ __forceinline__ void frag(uint32_t lx, uint32_t, int mt,
                                       uint32_t (&a)[4]) const {
    m.mags(lx, mt, a);
  }
};

template <>
struct VChunk<2> {
  uint32_t k[4];
  Pair2 m;
  __device__ __forceinline__ void prepare() { m.build(k); }
  __device__ __forceinline__ void frag(uint32_t lx, uint32_t, int mt,
                                       uint32_t (&a)[4]) const {
    m.mags(lx, mt, a);
  }
};

template <>
struct VChunk<1> {
  uint32_t s[2];
  Bits16 sg;
  __device__ __forceinline__ void prepare() { sg.build(s); }
  __device__ __forceinline__ void frag(uint32_t, uint32_t m0, int mt, uint32_t (&a)[4]) const {
    a[0] = a[1] = a[2] = a[3] = m0;
    sg.apply(mt, a);
  }
  // sign bits as masked operands (Bits16::mask); the centroid magnitude is applied at the merge
  __device__ __forceinline__ void frag_mask(int mt, uint32_t (&a)[4]) const { sg.mask(mt, a); }
};

// SQU-KV value chunk: dims 16 lg .. 16 lg + 3 of the group are modeled.  m[0] holds the 4-bit
// magnitudes of those dims for tokens 0 (low half) and 1, m[1] for tokens 2 and 3; s the signs.
// e01 / e23: byte d = magnitude of dim d of the first token | that of the second << 4.
__device__ __forceinline__ uint32_t nibbles_to_bytes(uint32_t x16) {
  x16 = (x16 | (x16 << 8)) & 0x00FF00FFu;
  return (x16 | (x16 << 4)) & 0x0F0F0F0Fu;
}
template <>
struct VChunk<kSQ> {
  uint32_t m[2], s[2];
  uint32_t e01, e23;
  Bits16 sg;
  __device__ __forceinline__ void prepare() {
    e01 = nibbles_to_bytes(m[0] & 0xffffu) | (nibbles_to_bytes(m[0] >> 16) << 4);
    e23 = nibbles_to_bytes(m[1] & 0xffffu) | (nibbles_to_bytes(m[1] >> 16) << 4);
    sg.build(s);
  }
  __device__ __forceinline__ void frag(uint32_t lx, uint32_t m0, int mt, uint32_t (&a)[4]) const {
    if (mt < 2) {
      a[0] = lut_get(lx, e01, 2 * mt);
      a[1] = lut_get(lx, e01, 2 * mt + 1);
      a[2] = lut_get(lx, e23, 2 * mt);
      a[3] = lut_get(lx, e23, 2 * mt + 1);
    } else {
      a[0] = a[1] = a[2] = a[3] = m0;
    }
    sg.apply(mt, a);
  }
};

// QJL value signs: +-1 pairs.
struct VSign {
  uint32_t s[2];
  Bits16 sg;
  __device__ __forceinline__ void prepare() { sg.build(s); }
  __device__ __forceinline__ void frag(int mt, uint32_t (&a)[4]) const {
    a[0] = a[1] = a[2] = a[3] = 0x3C003C00u;
    sg.apply(mt, a);
  }
  __device__ __forceinline__ void frag_mask(int mt, uint32_t (&a)[4]) const { sg.mask(mt, a); }
};

// ---------------------------------------------------------------------------------------------
// One tile's raw data for one thread.
template <int KB, bool KQ, bool KH, int VB, bool VQ>
struct TileData {
  KChunk<KB> kA, kB;
  KSign sA, sB;  // KQ
  uint2 zA, zB;  // KH: side code bytes lt, lt + 4
  float nuKA, nuKB, rhoKA, rhoKB, zsA, zsB;
  VChunk<VB> v;
  VSign vs;  // VQ
  float nuVA, nuVB, rhoVA, rhoVB;
};

__device__ __forceinline__ float half_of(uint32_t word, int hi) {
  return __half2float(__ushort_as_half((unsigned short)(hi ? word >> 16 : word & 0xffffu)));
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

// Block bases of one (batch, KV head) slab: block `tile` of a side at base + tile * bytes.
// A paged pool instead keeps the pages of the warp's tiles (below t_end) in windows of 32 tiles
// -- lane l holds the page of tile t_base + l in pg0 and of tile t_base + 32 + l in pg1 -- so the
// window after the current one is already loaded and a copy's issue does not wait on its
// block-table entry.
struct SlabPtrs {
  const unsigned char* kb;
  const unsigned char* vb;
  unsigned int kbytes, vbytes;
  int t_base, t_end, pg0, pg1;
  __device__ __forceinline__ void init(const Cache& C, int b, int h) {
    kb = C.blockp(0, b, h, 0);
    vb = C.blockp(1, b, h, 0);
    kbytes = C.block[0];
    vbytes = C.block[1];
  }
  int* err;  // where a bad table entry is recorded
  __device__ __forceinline__ int load_page(const Cache& C, int b, int t) const {
    return t < t_end ? C.page_of(b, t, err) : 0;
  }
  __device__ __forceinline__ void init_pages(const Cache& C, int b, int m0t, int m1t, int lane, int* e) {
    t_base = m0t;
    t_end = m1t;
    err = e;
    pg0 = load_page(C, b, m0t + lane);
    pg1 = load_page(C, b, m0t + 32 + lane);
  }
  // page of `tile` (warp-uniform and non-decreasing from call to call; every lane calls)
  __device__ __forceinline__ int page(const Cache& C, int b, int tile, int lane) {
    const int w = (tile - t_base) >> 5;
    if (w != 0) {  // a later window: shift (the next one is in pg1) and load the one after it
      pg0 = w == 1 ? pg1 : load_page(C, b, t_base + 32 * w + lane);
      t_base += 32 * w;
      pg1 = load_page(C, b, t_base + 32 + lane);
    }
    return __shfl_sync(kFull, pg0, (tile - t_base) & 31);
  }
};

template <int KB, int D = kDecD> struct KRec { static constexpr int value = KB == kSQ ? D / 4 : D * KB / 8; };

// Shared-memory stage of one 16-token tile: the tile's K block then its V block, in the cache's
// block layout for head dim D (QJL rows m = D; field offsets are multiples of 16 bytes).
template <int KB, bool KQ, bool KH, int VB, bool VQ, int D = kDecD>
struct Stage {
  static constexpr int KC = 0;
  static constexpr int KN = KC + kTile * KRec<KB, D>::value;
  static constexpr int KS = KN + kTile * 4;
  static constexpr int KRH = KS + (KQ ? kTile * (D / 8) : 0);
  static constexpr int KZ = KRH + (KQ ? kTile * 2 : 0);
  static constexpr int KZS = KZ + (KH ? kTile * 8 : 0);
  static constexpr int VC = KZS + (KH ? kTile * 2 : 0);
  static constexpr int VN = VC + kTile * KRec<VB, D>::value;
  static constexpr int VS = VN + kTile * 4;
  static constexpr int VRH = VS + (VQ ? kTile * (D / 8) : 0);
  static constexpr int bytes = VRH + (VQ ? kTile * 2 : 0);
};

// Start the bulk copies of tiles [tile, tile + nt) (nt = 1 or 2: adjacent 16-token blocks of the
// slab (b, h), so each side is one contiguous copy) into the pair stage at shared address `st`:
// K blocks at st, V blocks at st + 2 * (K block bytes).  Lane 0 registers the byte count on `bar`
// and issues the copies; a paged pool (PAGED) takes one copy per block (its pages are not
// adjacent), its blocks looked up through the block table.
template <int KB, bool KQ, bool KH, int VB, bool VQ, bool PAGED>
__device__ __forceinline__ void issue_pair(uint32_t st, uint32_t bar, SlabPtrs& s, int tile, int nt,
                                           int lane, const Cache& C, int b, int h) {
  using S = Stage<KB, KQ, KH, VB, VQ>;
  constexpr uint32_t KBL = S::VC, VBL = S::bytes - S::VC;
  if constexpr (!PAGED) {
    if (lane == 0) {
      mbar_arrive_expect_tx(bar, (uint32_t)nt * (KBL + VBL));
      bulk_g2s(st, s.kb + (unsigned long long)tile * KBL, (uint32_t)nt * KBL, bar);
      bulk_g2s(st + 2 * KBL, s.vb + (unsigned long long)tile * VBL, (uint32_t)nt * VBL, bar);
    }
  } else {
    int pg[2];
    pg[0] = s.page(C, b, tile, lane);
    pg[1] = nt > 1 ? s.page(C, b, tile + 1, lane) : pg[0];
    if (lane == 0) {
      mbar_arrive_expect_tx(bar, (uint32_t)nt * (KBL + VBL));
      for (int i = 0; i < nt; ++i) {
        bulk_g2s(st + i * KBL, C.page_block(0, pg[i], h), KBL, bar);
        bulk_g2s(st + 2 * KBL + i * VBL, C.page_block(1, pg[i], h), VBL, bar);
      }
    }
  }
}

__device__ __forceinline__ float lds_f32(const unsigned char* p) { return *reinterpret_cast<const float*>(p); }
__device__ __forceinline__ float lds_f16(const unsigned char* p) {
  return __half2float(*reinterpret_cast<const __half*>(p));
}
__device__ __forceinline__ uint32_t lds_u16(const unsigned char* p) {
  return *reinterpret_cast<const unsigned short*>(p);
}

// Read this thread's operands of one tile from a stage: the tile's K block at `st`, its V block
// at `vst` + S::VC (V field offsets of a 16-token stage are relative to `vst`).  For head dim D,
// the warp reads the 128-coordinate slice `sl` of every code and sign stream (sl = 0 for 128).
template <int KB, bool KQ, bool KH, int VB, bool VQ, int D = kDecD>
__device__ __forceinline__ void read_stage(TileData<KB, KQ, KH, VB, VQ>& d, const unsigned char* st,
                                           const unsigned char* vst, int lg, int lt, int sl = 0) {
  using S = Stage<KB, KQ, KH, VB, VQ, D>;
  constexpr int KR = KRec<KB, D>::value, VR = KRec<VB, D>::value;
  const int rA = tile_row_token(lg), rB = tile_row_token(lg + 8);
  // a 128-coordinate slice is 16 bytes per bit of a stream's width
  const unsigned char* ra = st + S::KC + rA * KR;  // token rows
  const unsigned char* rb = st + S::KC + rB * KR;
  const unsigned char* ka = ra + sl * (KB == 3 ? 32 : 16 * KB);
  const unsigned char* kb = rb + sl * (KB == 3 ? 32 : 16 * KB);
  if constexpr (KB == kSQ) {  // magnitudes (16 bytes) then signs (16 bytes), chunk lt = 4 bytes each
    d.kA.mg = *reinterpret_cast<const uint32_t*>(ra + 4 * lt);
    d.kB.mg = *reinterpret_cast<const uint32_t*>(rb + 4 * lt);
    d.kA.s = *reinterpret_cast<const uint32_t*>(ra + 16 + 4 * lt);
    d.kB.s = *reinterpret_cast<const uint32_t*>(rb + 16 + 4 * lt);
  } else if constexpr (KB == 4) {
    d.kA.c = *reinterpret_cast<const uint4*>(ka + 16 * lt);
    d.kB.c = *reinterpret_cast<const uint4*>(kb + 16 * lt);
  } else if constexpr (KB == 3 || KB == 2) {
    d.kA.k = *reinterpret_cast<const uint2*>(ka + 8 * lt);
    d.kB.k = *reinterpret_cast<const uint2*>(kb + 8 * lt);
    if constexpr (KB == 3) {  // the 1-bit stream follows the 2-bit stream (D / 4 bytes)
      d.kA.s = *reinterpret_cast<const uint32_t*>(ra + D / 4 + 16 * sl + 4 * lt);
      d.kB.s = *reinterpret_cast<const uint32_t*>(rb + D / 4 + 16 * sl + 4 * lt);
    }
  } else {
    d.kA.s = *reinterpret_cast<const uint32_t*>(ka + 4 * lt);
    d.kB.s = *reinterpret_cast<const uint32_t*>(kb + 4 * lt);
  }
  d.nuKA = lds_f32(st + S::KN + 4 * rA);
  d.nuKB = lds_f32(st + S::KN + 4 * rB);
  if constexpr (KQ) {
    d.sA.s = *reinterpret_cast<const uint32_t*>(st + S::KS + rA * (D / 8) + 16 * sl + 4 * lt);
    d.sB.s = *reinterpret_cast<const uint32_t*>(st + S::KS + rB * (D / 8) + 16 * sl + 4 * lt);
    d.rhoKA = lds_f16(st + S::KRH + 2 * rA);
    d.rhoKB = lds_f16(st + S::KRH + 2 * rB);
  }
  if constexpr (KH) {
    const uint2 za = *reinterpret_cast<const uint2*>(st + S::KZ + 8 * rA);
    const uint2 zb = *reinterpret_cast<const uint2*>(st + S::KZ + 8 * rB);
    d.zA = make_uint2((za.x >> (8 * lt)) & 0xffu, (za.y >> (8 * lt)) & 0xffu);
    d.zB = make_uint2((zb.x >> (8 * lt)) & 0xffu, (zb.y >> (8 * lt)) & 0xffu);
    d.zsA = lds_f16(st + S::KZS + 2 * rA);
    d.zsB = lds_f16(st + S::KZS + 2 * rB);
  }
  // value streams, stored by groups of 16 coordinates ([groups][16 tokens][2W bytes]): the four
  // tokens 4 lt .. 4 lt + 3 of this thread's group g are contiguous in every stream
  const int g = 8 * sl + lg;
  const unsigned char* vc = vst + S::VC;
  if constexpr (VB == kSQ) {  // magnitude stream, then sign stream (16 records each), 2 bytes per group
    const uint2 m2 = *reinterpret_cast<const uint2*>(vc + g * 32 + 8 * lt);
    const uint2 s2 = *reinterpret_cast<const uint2*>(vc + kTile * 16 + g * 32 + 8 * lt);
    d.v.m[0] = m2.x; d.v.m[1] = m2.y;
    d.v.s[0] = s2.x; d.v.s[1] = s2.y;
  } else if constexpr (VB == 4) {
    // 32 bytes; threads of odd groups load the two halves in the other order, so the eight
    // 16-byte loads of a quarter warp fall on distinct banks
    const unsigned char* a = vc + g * 128 + 32 * lt;
    const int o = 16 * (lg & 1);
    const uint4 h0 = *reinterpret_cast<const uint4*>(a + o);
    const uint4 h1 = *reinterpret_cast<const uint4*>(a + (16 ^ o));
    const uint4 lo = (lg & 1) ? h1 : h0, hi = (lg & 1) ? h0 : h1;
    d.v.w[0] = make_uint2(lo.x, lo.y);
    d.v.w[1] = make_uint2(lo.z, lo.w);
    d.v.w[2] = make_uint2(hi.x, hi.y);
    d.v.w[3] = make_uint2(hi.z, hi.w);
  } else if constexpr (VB == 3 || VB == 2) {
    const uint4 k4 = *reinterpret_cast<const uint4*>(vc + g * 64 + 16 * lt);
    d.v.k[0] = k4.x; d.v.k[1] = k4.y; d.v.k[2] = k4.z; d.v.k[3] = k4.w;
    if constexpr (VB == 3) {  // the 1-bit stream follows the 2-bit stream's 16 records
      const uint2 s2 = *reinterpret_cast<const uint2*>(vc + kTile * (D / 4) + g * 32 + 8 * lt);
      d.v.s[0] = s2.x; d.v.s[1] = s2.y;
    }
  } else {
    const uint2 s2 = *reinterpret_cast<const uint2*>(vc + g * 32 + 8 * lt);
    d.v.s[0] = s2.x; d.v.s[1] = s2.y;
  }
  if constexpr (VQ) {
    const uint2 s2 = *reinterpret_cast<const uint2*>(vst + S::VS + g * 32 + 8 * lt);
    d.vs.s[0] = s2.x; d.vs.s[1] = s2.y;
  }
  d.nuVA = lds_f32(vst + S::VN + 4 * rA);
  d.nuVB = lds_f32(vst + S::VN + 4 * rB);
  if constexpr (VQ) {
    d.rhoVA = lds_f16(vst + S::VRH + 2 * rA);
    d.rhoVB = lds_f16(vst + S::VRH + 2 * rB);
  }
}

// Direct (uncached) loads of a tile's key data from the K blocks, used by the logits kernel.
template <int KB, bool KQ, bool KH, int VB, bool VQ>
__device__ __forceinline__ void load_ktile(TileData<KB, KQ, KH, VB, VQ>& d, const SlabPtrs& s, int t0,
                                           int last, int lg, int lt) {
  using S = Stage<KB, KQ, KH, VB, VQ>;
  constexpr int KR = KRec<KB>::value;
  const int tA = min(t0 + tile_row_token(lg), last);
  const int tB = min(t0 + tile_row_token(lg + 8), last);
  const unsigned char* bA = s.kb + (unsigned long long)(tA / kTile) * s.kbytes;
  const unsigned char* bB = s.kb + (unsigned long long)(tB / kTile) * s.kbytes;
  const int jA = tA % kTile, jB = tB % kTile;
  if constexpr (KB == 4) {
    d.kA.c = ldg_stream16(bA + S::KC + jA * KR + 16 * lt);
    d.kB.c = ldg_stream16(bB + S::KC + jB * KR + 16 * lt);
  } else if constexpr (KB == 3 || KB == 2) {
    d.kA.k = ldg_stream8(bA + S::KC + jA * KR + 8 * lt);
    d.kB.k = ldg_stream8(bB + S::KC + jB * KR + 8 * lt);
    if constexpr (KB == 3) {
      d.kA.s = ldg_stream4(bA + S::KC + jA * KR + kDecD / 4 + 4 * lt);
      d.kB.s = ldg_stream4(bB + S::KC + jB * KR + kDecD / 4 + 4 * lt);
    }
  } else {
    d.kA.s = ldg_stream4(bA + S::KC + jA * KR + 4 * lt);
    d.kB.s = ldg_stream4(bB + S::KC + jB * KR + 4 * lt);
  }
  d.nuKA = __uint_as_float(ldg_stream4(bA + S::KN + 4 * jA));
  d.nuKB = __uint_as_float(ldg_stream4(bB + S::KN + 4 * jB));
  if constexpr (KQ) {
    d.sA.s = ldg_stream4(bA + S::KS + jA * (kDecD / 8) + 4 * lt);
    d.sB.s = ldg_stream4(bB + S::KS + jB * (kDecD / 8) + 4 * lt);
    d.rhoKA = half_of(ldg_stream4(bA + S::KRH + (jA & ~1) * 2), jA & 1);
    d.rhoKB = half_of(ldg_stream4(bB + S::KRH + (jB & ~1) * 2), jB & 1);
  }
  if constexpr (KH) {
    const uint2 za = ldg_stream8(bA + S::KZ + 8 * jA), zb = ldg_stream8(bB + S::KZ + 8 * jB);
    d.zA = make_uint2((za.x >> (8 * lt)) & 0xffu, (za.y >> (8 * lt)) & 0xffu);
    d.zB = make_uint2((zb.x >> (8 * lt)) & 0xffu, (zb.y >> (8 * lt)) & 0xffu);
    d.zsA = half_of(ldg_stream4(bA + S::KZS + (jA & ~1) * 2), jA & 1);
    d.zsB = half_of(ldg_stream4(bB + S::KZS + (jB & ~1) * 2), jB & 1);
  }
}

// Key scores of the thread's four accumulator slots (tokens pi(lg), pi(lg+8) x heads 2 lt,
// 2 lt + 1), times `sscale`: nu <q_rot, C[c]> (+ nu rho sqrt(pi/2)/m <S q_rot, 2 sigma - 1>)
// (+ scale <U^T q, zeta>).  sscale = 1/sqrt(d) gives the logit.
//
// The query's fp16 lo terms: with QLO in qfl / qsl (own MMAs on the same key fragments);
// otherwise, when lo_xor != 0, in other columns whose scores are added back at the end.
template <bool QLO = false, int KB, bool KQ, bool KH, int VB, bool VQ>
__device__ __forceinline__ void key_scores(TileData<KB, KQ, KH, VB, VQ>& d, float (&s)[4],
                                           const uint32_t (&qf)[16], const uint32_t (&qs)[16],
                                           const uint32_t (&qu)[2], uint32_t lxK, uint32_t k_m0,
                                           float qjl_scale, float sscale, const uint32_t (&qfl)[16],
                                           const uint32_t (&qsl)[16], int lo_xor) {
  d.kA.prepare();
  d.kB.prepare();
  // two independent accumulator chains (even / odd k-steps) halve the MMA dependency chain
  float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t a0 = d.kA.pair(lxK, k_m0, 2 * ks), a1 = d.kB.pair(lxK, k_m0, 2 * ks);
    const uint32_t a2 = d.kA.pair(lxK, k_m0, 2 * ks + 1), a3 = d.kB.pair(lxK, k_m0, 2 * ks + 1);
    mma16816(sc[ks & 1], a0, a1, a2, a3, qf[2 * ks], qf[2 * ks + 1]);
    if constexpr (QLO) mma16816(sc[ks & 1], a0, a1, a2, a3, qfl[2 * ks], qfl[2 * ks + 1]);
  }
  const float nA = d.nuKA * sscale, nB = d.nuKB * sscale;
  s[0] = (sc[0][0] + sc[1][0]) * nA;
  s[1] = (sc[0][1] + sc[1][1]) * nA;
  s[2] = (sc[0][2] + sc[1][2]) * nB;
  s[3] = (sc[0][3] + sc[1][3]) * nB;
  if constexpr (KQ) {
    d.sA.prepare();
    d.sB.prepare();
    float sq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t a0 = d.sA.pair(2 * ks), a1 = d.sB.pair(2 * ks);
      const uint32_t a2 = d.sA.pair(2 * ks + 1), a3 = d.sB.pair(2 * ks + 1);
      mma16816(sq, a0, a1, a2, a3, qs[2 * ks], qs[2 * ks + 1]);
      if constexpr (QLO) mma16816(sq, a0, a1, a2, a3, qsl[2 * ks], qsl[2 * ks + 1]);
    }
    const float fa = nA * d.rhoKA * qjl_scale, fb = nB * d.rhoKB * qjl_scale;
    s[0] = fmaf(sq[0], fa, s[0]);
    s[1] = fmaf(sq[1], fa, s[1]);
    s[2] = fmaf(sq[2], fb, s[2]);
    s[3] = fmaf(sq[3], fb, s[3]);
  }
  if constexpr (KH) {
    float sz[4] = {0.f, 0.f, 0.f, 0.f};
    mma16816(sz, side_pair(d.zA.x), side_pair(d.zB.x), side_pair(d.zA.y), side_pair(d.zB.y), qu[0], qu[1]);
    const float zA = d.zsA * sscale, zB = d.zsB * sscale;
    s[0] = fmaf(sz[0], zA, s[0]);
    s[1] = fmaf(sz[1], zA, s[1]);
    s[2] = fmaf(sz[2], zB, s[2]);
    s[3] = fmaf(sz[3], zB, s[3]);
  }
  if (lo_xor > 0) {  // lo columns (2 lt ^ 2 lo_xor, ...) belong to this thread's hi columns
#pragma unroll
    for (int k = 0; k < 4; ++k) s[k] += __shfl_xor_sync(kFull, s[k], lo_xor);
  } else if (lo_xor < 0) {  // one query column: its lo term is column 1 of the same thread
    s[0] += s[1];
    s[2] += s[3];
    if constexpr (VQ && !QLO) {  // column 1 becomes the value sketch's copy of column 0
      s[1] = s[0];
      s[3] = s[2];
    }
  }
}

constexpr float kMaxFloor = -1e30f;
// The running maximum is raised only when a score exceeds it by more than this (log2 units), so
// the weights 2^(s - m) stay below 2^3 between raises.  Most tiles then skip the column max
// reduction and the accumulator rescale (with eight query columns a warp otherwise raised some
// column's maximum on most tiles).  The value operands p nu stay fp16: value norms up to
// 65504 / 8.
constexpr float kRescaleSlack = 3.f;

// Per-warp running state.
template <bool VQ>
struct WarpState {
  // running max (log2 domain) of columns 2 lt, 2 lt + 1; it starts at kMaxFloor, not -inf, so
  // a column whose query has seen no token yet (all scores -inf) gets weights exp2(-inf) = 0
  // instead of exp2(-inf + inf)
  float m0, m1;
  float l0, l1;  // this thread's partial softmax denominators
  // weight sums of the masked sign operands per column 2 lt, 2 lt + 1 (Bits16::mask): [0] the
  // code readout of 1-bit value codes, [1] the value sketch; with the sketch readout packed into
  // the value MMA, [0] holds a sketch column's sum
  float w[2][2];
  float acc[8][4];
  float accs[VQ ? 8 : 1][4];
  __device__ __forceinline__ void reset() {
    m0 = m1 = kMaxFloor;
    l0 = l1 = 0.f;
    w[0][0] = w[0][1] = w[1][0] = w[1][1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[mt][j] = 0.f;
        if constexpr (VQ) accs[mt][j] = 0.f;
      }
  }
};

// The two fp16 halves of a packed pair as floats (low, high).
__device__ __forceinline__ float2 half2_floats(uint32_t h) {
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// 2^x on the special-function unit (inputs here are <= 0; -inf gives 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Online-softmax step over NT consecutive tiles (starting at token t0) whose scores are in s:
// mask rows at or past `end` (MASK = false when every token of the NT tiles is below it),
// rescale the running state, and accumulate the value readout.
// Rows (tokens) at or past `end` carry no data; a score of column c counts only for tokens
// below lmin + c / G, the causal end of that column's query (c = 2 lt, 2 lt + 1; lmin = end
// for plain decode).
// PK (a QJL value side, query columns Gc <= 4): columns c < Gc carry the code readout of query
// column c and columns Gc <= c < 2 Gc, whose scores are copies of column c - Gc's, its value
// sketch readout.  One MMA then takes the 8 tokens of a score-row half twice along k, codes
// then signs, against a B operand holding p nu in the code columns of the first half and
// p nu rho in the sketch columns of the second.  Both readouts share one accumulator.
// MV: the value sketch's sign bits (and 1-bit value codes) enter as masked operands
// (Bits16::mask), with their weight sums kept in st.w for the merge.
template <int NT, bool MASK, bool PK = false, bool MV = false, int KB, bool KQ, bool KH, int VB, bool VQ>
__device__ __forceinline__ void softmax_readout(TileData<KB, KQ, KH, VB, VQ> (&d)[2], float (&s)[NT][4],
                                                WarpState<VQ && !PK>& st, uint32_t lxV, uint32_t v_m0, int t0,
                                                int end, int lmin, int G, int Gc, int lg) {
  static_assert(!PK || VQ, "a packed sketch readout needs a QJL value side");
  const int lt2 = 2 * ((int)threadIdx.x & 3);
  // causal end of each column's query (a sketch column takes its code column's); masked tiles only
  const int e0 = lmin + (lt2 % Gc) / G, e1 = lmin + ((lt2 + 1) % Gc) / G;
  bool va[NT], vb[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int tA = t0 + kTile * j + tile_row_token(lg), tB = t0 + kTile * j + tile_row_token(lg + 8);
    va[j] = !MASK || tA < end;
    vb[j] = !MASK || tB < end;
    if constexpr (MASK) {
      s[j][0] = tA < e0 ? s[j][0] : -INFINITY;
      s[j][1] = tA < e1 ? s[j][1] : -INFINITY;
      s[j][2] = tB < e0 ? s[j][2] : -INFINITY;
      s[j][3] = tB < e1 ? s[j][3] : -INFINITY;
    }
  }

  // ---- online softmax (log2 domain).  A column's maximum over the tiles exceeds its running
  // maximum (plus the slack) exactly when some lane's own maximum does, so the max-reduction
  // across the lanes of a column (and the rescale) runs only on tiles that raise a maximum by
  // more than kRescaleSlack; elsewhere the running maximum stays the reference of the weights.
  float mx0 = fmaxf(s[0][0], s[0][2]), mx1 = fmaxf(s[0][1], s[0][3]);
#pragma unroll
  for (int j = 1; j < NT; ++j) {
    mx0 = fmaxf(mx0, fmaxf(s[j][0], s[j][2]));
    mx1 = fmaxf(mx1, fmaxf(s[j][1], s[j][3]));
  }
  float n0 = st.m0, n1 = st.m1;
  if (__any_sync(kFull, mx0 > st.m0 + kRescaleSlack || mx1 > st.m1 + kRescaleSlack)) {
#pragma unroll
    for (int m = 4; m <= 16; m <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, m));
      mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, m));
    }
    n0 = fmaxf(st.m0, mx0);
    n1 = fmaxf(st.m1, mx1);
    const float a0 = ex2(st.m0 - n0), a1 = ex2(st.m1 - n1);
    st.l0 *= a0;
    st.l1 *= a1;
    if constexpr (MV) {
      st.w[0][0] *= a0; st.w[1][0] *= a0;
      st.w[0][1] *= a1; st.w[1][1] *= a1;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      st.acc[mt][0] *= a0; st.acc[mt][1] *= a1; st.acc[mt][2] *= a0; st.acc[mt][3] *= a1;
      if constexpr (VQ && !PK) {
        st.accs[mt][0] *= a0; st.accs[mt][1] *= a1; st.accs[mt][2] *= a0; st.accs[mt][3] *= a1;
      }
    }
    st.m0 = n0;
    st.m1 = n1;
  }

  // ---- value readout
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const float p0 = ex2(s[j][0] - n0), p1 = ex2(s[j][1] - n1);
    const float p2 = ex2(s[j][2] - n0), p3 = ex2(s[j][3] - n1);
    st.l0 += p0 + p2;
    st.l1 += p1 + p3;
    // rows past the sequence end read whatever the cache holds there: select, don't multiply
    const float nA = va[j] ? d[j].nuVA : 0.f, nB = vb[j] ? d[j].nuVB : 0.f;
    if constexpr (PK) {
      const bool c0 = lt2 < Gc, c1 = lt2 + 1 < Gc;  // code columns (else sketch columns)
      const float fA = va[j] ? d[j].nuVA * d[j].rhoVA : 0.f, fB = vb[j] ? d[j].nuVB * d[j].rhoVB : 0.f;
      const uint32_t hcA = pack_half2(c0 ? p0 * nA : 0.f, c1 ? p1 * nA : 0.f);
      const uint32_t hsA = pack_half2(c0 ? 0.f : p0 * fA, c1 ? 0.f : p1 * fA);
      const uint32_t hcB = pack_half2(c0 ? p2 * nB : 0.f, c1 ? p3 * nB : 0.f);
      const uint32_t hsB = pack_half2(c0 ? 0.f : p2 * fB, c1 ? 0.f : p3 * fB);
      if constexpr (MV) {
        // one sum per column (the code readout's for 1-bit codes, or the sketch's), of the fp16
        // weights the MMA multiplies: a rounding common to all of a column's dims would
        // otherwise survive the 2 sum - W step and the inverse rotation gathers it into one
        // output coordinate
        const float2 a = half2_floats(VB == 1 ? (hcA | hsA) : hsA), bb = half2_floats(VB == 1 ? (hcB | hsB) : hsB);
        st.w[0][0] += a.x + bb.x;
        st.w[0][1] += a.y + bb.y;
      }
      const uint32_t cA = movmatrix_trans(hcA), sA = movmatrix_trans(hsA);
      const uint32_t cB = movmatrix_trans(hcB), sB = movmatrix_trans(hsB);
      d[j].v.prepare();
      d[j].vs.prepare();
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t a[4], g[4];
        if constexpr (MV && VB == 1) d[j].v.frag_mask(mt, a); else d[j].v.frag(lxV, v_m0, mt, a);
        if constexpr (MV) d[j].vs.frag_mask(mt, g); else d[j].vs.frag(mt, g);
        mma16816(st.acc[mt], a[0], a[1], g[0], g[1], cA, sA);
        mma16816(st.acc[mt], a[2], a[3], g[2], g[3], cB, sB);
      }
      continue;
    }
    const uint32_t hv0 = pack_half2(p0 * nA, p1 * nA), hv1 = pack_half2(p2 * nB, p3 * nB);
    if constexpr (MV && VB == 1) {  // sums of the fp16 weights the MMA multiplies
      const float2 a = half2_floats(hv0), bb = half2_floats(hv1);
      st.w[0][0] += a.x + bb.x;
      st.w[0][1] += a.y + bb.y;
    }
    const uint32_t bv0 = movmatrix_trans(hv0), bv1 = movmatrix_trans(hv1);
    d[j].v.prepare();
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      uint32_t a[4];
      if constexpr (MV && VB == 1) d[j].v.frag_mask(mt, a); else d[j].v.frag(lxV, v_m0, mt, a);
      mma16816(st.acc[mt], a[0], a[1], a[2], a[3], bv0, bv1);
    }
    if constexpr (VQ && !PK) {
      const float fa = va[j] ? d[j].nuVA * d[j].rhoVA : 0.f, fb = vb[j] ? d[j].nuVB * d[j].rhoVB : 0.f;
      const uint32_t hs0 = pack_half2(p0 * fa, p1 * fa), hs1 = pack_half2(p2 * fb, p3 * fb);
      if constexpr (MV) {
        const float2 a = half2_floats(hs0), bb = half2_floats(hs1);
        st.w[1][0] += a.x + bb.x;
        st.w[1][1] += a.y + bb.y;
      }
      const uint32_t bs0 = movmatrix_trans(hs0), bs1 = movmatrix_trans(hs1);
      d[j].vs.prepare();
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t a[4];
        if constexpr (MV) d[j].vs.frag_mask(mt, a); else d[j].vs.frag(mt, a);
        mma16816(st.accs[mt], a[0], a[1], a[2], a[3], bs0, bs1);
      }
    }
  }
}

// Value sides whose sign bits the head-dim-128 decode reads as masked operands: a QJL sketch, or
// 1-bit codes.
template <int VB, bool VQ> struct kMaskedValues { static constexpr bool value = VQ || VB == 1; };

// Scores and online-softmax step of NT consecutive tiles held by one warp (head dim 128).
template <int NT, bool MASK, bool QLO, int KB, bool KQ, bool KH, int VB, bool VQ>
__device__ __forceinline__ void compute_tiles(TileData<KB, KQ, KH, VB, VQ> (&d)[2], WarpState<VQ && QLO>& st,
                                              const uint32_t (&qf)[16], const uint32_t (&qs)[16],
                                              const uint32_t (&qu)[2], const uint32_t (&qfl)[16],
                                              const uint32_t (&qsl)[16], uint32_t lxK,
                                              uint32_t lxV, uint32_t k_m0,
                                              uint32_t v_m0, const DecodeParams& p, int t0, int end, int lmin,
                                              int lg) {
  float s[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j)
    key_scores<QLO>(d[j], s[j], qf, qs, qu, lxK, k_m0, p.qjl_scale, p.score_scale, qfl, qsl, p.lo_xor);
  softmax_readout<NT, MASK, VQ && !QLO, kMaskedValues<VB, VQ>::value>(d, s, st, lxV, v_m0, t0, end, lmin, p.G,
                                                                   p.Gc, lg);
}

// Placement of N equal regions of RS bytes around the code tables, in shared-window addresses:
// the key table (lutK bytes) sits at kLutAddrK, a separate value table (lutV bytes, 0 when the
// sides share one) at kLutAddrV.  Regions fill [kDynBaseMax, kLutAddrK), then the gap between
// the key table and the value table (when there is one), then the space after the last table;
// `bars` (8-byte aligned) follows the last region.  A dynamic allocation of `end(extra)` bytes
// covers the window from 0 to the end of `extra` bytes after `bars`, whatever the start of
// dynamic shared memory (at most kDynBaseMax, checked at run time).
template <uint32_t lutK, uint32_t lutV, uint32_t RS, int N>
struct RegionPlan {
  static constexpr bool sepV = lutV > 0;
  static constexpr uint32_t a0 = kDynBaseMax;
  static constexpr int nA = (kLutAddrK - a0) / RS < (uint32_t)N ? (int)((kLutAddrK - a0) / RS) : N;
  static constexpr uint32_t b0 = kLutAddrK + lutK;
  static constexpr int nBmax = sepV ? (int)((kLutAddrV - b0) / RS) : N;
  static constexpr int nB = nBmax < N - nA ? nBmax : N - nA;
  static constexpr uint32_t c0 = kLutAddrV + lutV;
  static constexpr int nC = N - nA - nB;
  static constexpr uint32_t bars = sepV ? c0 + nC * RS : b0 + nB * RS;
  static_assert(RS % 16 == 0, "regions must keep 16-byte alignment");
  static_assert(lutK <= kLutAddrV - kLutAddrK, "key table overlaps the value table");
  __host__ __device__ static constexpr uint32_t region(int w) {
    return w < nA ? a0 + w * RS : (w < nA + nB ? b0 + (w - nA) * RS : c0 + (w - nA - nB) * RS);
  }
};

constexpr uint32_t kSkA = 4096;  // byte offset of a column's merged acc_sk in its warp's region

// Shared-memory plan of a decode block: per-warp regions (the warp's bulk-copy ring, later its
// merge slot) placed by RegionPlan, then one mbarrier per pair stage and warp.
// A value codebook other than the key one gets its own table in the upper half (bytes 128 .. 255)
// of the key table's entries, so both share one 64 KiB-aligned range.
template <int KB, bool KQ, bool KH, int VB, bool VQ, bool QLO = false>
struct DecodeSmem {
  static constexpr int NK = LutEntries<KB>::value, NV = LutEntries<VB>::value;
  static constexpr bool sepV = KB != VB && NV > 0;  // same width, same codebook
  static constexpr uint32_t lutK = (NK > NV ? NK : NV) * kLutStride;
  static constexpr uint32_t kVHalf = 128;  // byte offset of the value table inside an entry
  static constexpr int PS = 4 + kDecD + (VQ ? kDecD : 0);  // per head: m, l, pad, pad, acc, (acc_sk)
  static constexpr int NW = DecWarps<KQ, VQ, QLO>::value;
  static constexpr uint32_t ring = kPairStages * 2 * Stage<KB, KQ, KH, VB, VQ>::bytes;
  static constexpr uint32_t mslot = kHeadsPad * PS * 4;
  static constexpr uint32_t RS = ring > mslot ? ring : mslot;
  using Plan = RegionPlan<lutK, 0, RS, NW>;
  static constexpr uint32_t bars = Plan::bars;
  // the slab merge of a QJL value side: per-column partial sketch products at the start of each
  // warp's region, the merged acc_sk of column h at kSkA in warp h's region
  static_assert(!VQ || (RS >= kSkA + 4 * kDecD && kHeadsPad * kDecD * 4 <= kSkA), "merge scratch");
  static constexpr uint32_t bytes = bars + NW * kPairStages * 8;
  __host__ __device__ static constexpr uint32_t region(int w) { return Plan::region(w); }
};

// Owner block of flattened tile x: the largest c with floor(c W / N) <= x.
__device__ __forceinline__ int owner_block(long long x, long long W, int N) {
  return (int)(((x + 1) * N - 1) / W);
}

// Paged pool: the stream-K split from the lengths in device memory, computed by every decode
// block into shared memory after its barriers (kPagedPlanBytes more dynamic shared memory):
// len[b] = the length clamped to [0, lmax], bs[b] = H_kv * sum over b' < b of ceil(len[b'] / 16),
// bs[TQ_MAX_BATCH] = W.  The lengths, like the cache and the block table, were complete before
// the query prep started, so nothing here waits for it.  Returns, block-uniformly, whether a
// length lay outside [0, lmax] (recorded after the first wait, once prep has cleared the word).
constexpr uint32_t kPlanLenOff = 8 * (TQ_MAX_BATCH + 2);       // after bs[TQ_MAX_BATCH + 1]
constexpr uint32_t kPlanSumOff = kPlanLenOff + 4 * TQ_MAX_BATCH;
constexpr uint32_t kPagedPlanBytes = kPlanSumOff + 8 * 32;    // + per-warp scan totals
template <int NW>
__device__ __forceinline__ bool paged_plan(const DecodeParams& p, unsigned char* area) {
  static_assert(NW * 64 >= TQ_MAX_BATCH && NW <= 32, "two batch entries per thread");
  long long* const bs = reinterpret_cast<long long*>(area);
  int* const len = reinterpret_cast<int*>(area + kPlanLenOff);
  long long* const wsum = reinterpret_cast<long long*>(area + kPlanSumOff);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long v[2];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int b = 2 * (int)threadIdx.x + i;
    int L = 0;
    if (b < p.B) {
      const int raw = __ldg(p.dev_seq_len + b);
      bad |= raw < 0 || raw > p.lmax;
      L = raw < 0 ? 0 : (raw > p.lmax ? p.lmax : raw);
    }
    if (b < TQ_MAX_BATCH) len[b] = L;
    v[i] = (long long)p.Hkv * ((L + kTile - 1) / kTile);
  }
  long long t = v[0] + v[1];  // inclusive scan over the block
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long n = __shfl_up_sync(kFull, t, o);
    if (lane >= o) t += n;
  }
  if (lane == 31) wsum[warp] = t;
  __syncthreads();
  long long before = 0;
  for (int w = 0; w < warp; ++w) before += wsum[w];
  const long long ex = before + t - v[0] - v[1];
  if (2 * (int)threadIdx.x < TQ_MAX_BATCH) bs[2 * threadIdx.x] = ex;
  if (2 * (int)threadIdx.x + 1 < TQ_MAX_BATCH) bs[2 * threadIdx.x + 1] = ex + v[0];
  if ((int)threadIdx.x == NW * 32 - 1) bs[TQ_MAX_BATCH] = before + t;
  return __syncthreads_or(bad) != 0;  // (also makes the plan visible to the whole block)
}

// Programmatic dependent launch: wait until the preceding kernel of the stream has completed and
// its memory is visible (returns at once when the launch had no programmatic dependency).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

constexpr uint32_t kWaitLimit = 1u << 20;  // polls of an mbarrier before giving up
constexpr int kErrWaitTimeout = TQ_DEVERR_WAIT_TIMEOUT;
constexpr int kErrSmemPlan = TQ_DEVERR_SMEM_PLAN;

template <int KB, bool KQ, bool KH, int VB, bool VQ, bool QLO, bool PAGED>
__global__ void __launch_bounds__(DecWarps<KQ, VQ, QLO>::value * 32, 1) decode_kernel(const DecodeParams p) {
  using SM = DecodeSmem<KB, KQ, KH, VB, VQ, QLO>;
  using SG = Stage<KB, KQ, KH, VB, VQ>;
  constexpr int PS = SM::PS;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_last;
  __shared__ float s_wscale[SM::NW][kHeadsPad];  // block merge: 2^(m_w - M) of warp w, column h
  __shared__ float s_wmax[kHeadsPad];            // block merge: M of column h
  __shared__ long long s_split[2];               // the split's P and virtual tile count
  __shared__ int s_page_err[SM::NW];  // paged: a bad table entry met before the first wait
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int lg = lane >> 2, lt = lane & 3;

  // generic pointer of shared-window address a
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(smem);
  if (sbase > kDynBaseMax) {  // the plan does not fit this launch: report, do nothing
    grid_dependency_wait();    // (after the prep kernel's reset of the error word)
    if (threadIdx.x == 0) atomicExch(p.err, kErrSmemPlan);
    return;
  }
  unsigned char* const win = smem - sbase;
  if constexpr (KB != 1) build_lut<KB>(win + kLutAddrK, p.tab.k_c);
  if constexpr (SM::sepV) build_lut<VB>(win + kLutAddrK + SM::kVHalf, p.tab.v_c);
  // the 1-bit magnitude: a 1-bit codebook's upper centroid, or a spectral side's floor centroid
  const float kc1 = KB == kSQ ? __ldg(p.tab.sq_c1) : __ldg(p.tab.k_c + 1);
  const float vc1 = VB == kSQ ? __ldg(p.tab.sq_c1 + 1) : __ldg(p.tab.v_c + 1);
  const uint32_t k_m0 = pack_half2(kc1, kc1);
  const uint32_t v_m0 = pack_half2(vc1, vc1);
  const uint32_t lxK = kLutAddrK | (4u * lane);
  const uint32_t lxV = kLutAddrK | (SM::sepV ? SM::kVHalf : 0u) | (4u * lane);
  const uint32_t my_bars = SM::bars + warp * kPairStages * 8;
  if (lane < kPairStages) mbar_init(my_bars + 8 * lane, 1);
  fence_mbar_init();
  __syncthreads();

  const uint32_t my_stages_s = SM::region(warp);
  unsigned char* my_stages = win + my_stages_s;
  const int G = p.G;          // query heads per KV head
  const int Gc = p.Gc;        // query columns per KV head (G nq)
  const int Hq = p.Hkv * G;
  unsigned char* const plan = win + SM::bytes;  // paged: the split (paged_plan)
  bool bad_len = false;
  if constexpr (PAGED) {
    if (lane == 0) s_page_err[warp] = 0;
    bad_len = paged_plan<SM::NW>(p, plan);
  }
  const long long* const pl_bs = reinterpret_cast<const long long*>(plan);
  const int* const pl_len = reinterpret_cast<const int*>(plan + kPlanLenOff);
  auto bstart = [&](int b) -> long long { return PAGED ? pl_bs[b] : p.batch_start[b]; };
  auto slen = [&](int b) -> int { return PAGED ? pl_len[b] : p.seq_len[b]; };
  const long long W = PAGED ? pl_bs[TQ_MAX_BATCH] : p.W;
  // with host lengths nblocks = min(W, #SMs); with device lengths (paged) the grid is #SMs and the
  // same min is taken here, so every working block has a non-empty range (the merge counts on it)
  const int N = PAGED ? (int)(W < p.nblocks ? W : p.nblocks) : p.nblocks;
  if ((int)blockIdx.x >= N) {
    if (PAGED && bad_len && blockIdx.x == 0) {  // no block works: block 0 records it
      grid_dependency_wait();
      if (threadIdx.x == 0) atomicExch(p.err, TQ_DEVERR_BAD_LENGTH);
    }
    return;
  }
  // The split runs over virtual tiles: every slab counts P tiles before its first real one, and
  // the virtual space is cut into N equal ranges.  A block whose range crosses into a slab so
  // gets P real tiles fewer for each crossing, which pays for what a segment boundary costs it
  // (the ring drained and refilled, a partial written, the per-warp split rounded once more).
  // With P = 0 the virtual and the real tiles coincide.  A range that lies inside a slab's P
  // virtual tiles holds no real tile; such a block owns no tile of any slab and does nothing.
  // (P and the virtual count go to shared memory for the merges, so no register holds them
  // through the streaming loop.)  The variants with separate query lo terms or a HeadQ side
  // keep the plain equal split (EQS): their register allocation is at its limit.
  constexpr bool EQS = QLO || KH;
  long long x, x_end;
  {
    const long long P = EQS ? 0 : W / N / 8;
    const long long Wv = W + P * p.Hkv * p.B;
    if (threadIdx.x == 0) { s_split[0] = P; s_split[1] = Wv; }
    auto real_tile = [&](long long v) -> long long {  // the first real tile at or after virtual v
      int lo = 0, hi = p.B - 1;  // largest b with its virtual start <= v
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (bstart(mid) + P * p.Hkv * mid <= v) lo = mid; else hi = mid - 1;
      }
      const long long nt = (slen(lo) + kTile - 1) / kTile;
      if (nt == 0) return bstart(lo);
      const long long off = v - (bstart(lo) + P * p.Hkv * lo), k = off / (nt + P), o = off % (nt + P);
      return bstart(lo) + k * nt + (o > P ? o - P : 0);
    };
    if constexpr (EQS) {
      x = (long long)blockIdx.x * W / N;
      x_end = (long long)(blockIdx.x + 1) * W / N;
    } else {
      x = real_tile((long long)blockIdx.x * Wv / N);
      x_end = real_tile((long long)(blockIdx.x + 1) * Wv / N);
    }
  }
  unsigned seq = 0;  // tile pairs this warp has streamed so far: stage seq % S, phase (seq / S) & 1
  bool timed_out = false;
  bool waited = false;  // grid_dependency_wait has returned

  while (x < x_end) {
    // ---- locate the slab segment that starts at tile x
    int lo = 0, hi = p.B - 1;  // largest b with batch_start[b] <= x
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (bstart(mid) <= x) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int L = slen(b);
    const int ntb = (L + kTile - 1) / kTile;  // tiles per slab of batch b
    const long long bs = bstart(b);
    const long long off = x - bs;
    const int kvh = (int)(off / ntb);
    const int ts = (int)(off % ntb);  // first tile of the segment
    const long long slab_start = bs + (long long)kvh * ntb;
    const long long seg_end = min(x_end, slab_start + ntb);
    const int te = ts + (int)(seg_end - x);
    const int pair = b * p.Hkv + kvh;

    // ---- this warp's tiles of the segment, streamed through its bulk-copy ring
    const int n = te - ts;
    const int per = (n + SM::NW - 1) / SM::NW;
    const int m0t = min(te, ts + warp * per);
    const int m1t = min(te, m0t + per);
    const int nt = m1t - m0t;
    SlabPtrs sp;
    if constexpr (!PAGED) sp.init(p.cache, b, kvh);
    else sp.init_pages(p.cache, b, m0t, m1t, lane, waited ? p.err : s_page_err + warp);
    WarpState<VQ && QLO> st;
    st.reset();
    // both pair stages in flight; a pair stage is refilled as soon as its operands are in
    // registers, before the pair is computed
    constexpr uint32_t KBL = SG::VC, VBL = SG::bytes - SG::VC, PB = 2 * SG::bytes;
    const int npairs = (nt + 1) >> 1;
    const int n_first = npairs < kPairStages ? npairs : kPairStages;
    // before the first wait, only pair stages whose tiles hold none of the step's new tokens
    int n_early = n_first;
    if (p.n_fresh > 0 && !waited) {
      const int fresh_tile = (L - p.n_fresh) / kTile;  // first tile with a new token
      for (int k = 0; k < n_first; ++k)
        if (m0t + 2 * k + min(2, nt - 2 * k) > fresh_tile) { n_early = k; break; }
    }
    for (int k = 0; k < n_early; ++k) {
      const unsigned sl = (seq + k) % kPairStages;
      issue_pair<KB, KQ, KH, VB, VQ, PAGED>(my_stages_s + sl * PB, my_bars + 8 * sl, sp, m0t + 2 * k,
                                     min(2, nt - 2 * k), lane, p.cache, b, kvh);
    }
    // the query prep kernel runs just before this one: its outputs (query fragments, tickets,
    // error word) are read only from here on, so the table build and the first bulk copies above
    // overlap it (programmatic dependent launch; a no-op without one).  In a decode step its
    // completion also covers the append's, so the deferred stages are issued after it.
    grid_dependency_wait();
    if constexpr (PAGED) {
      if (!waited) {  // prep has cleared the error word: record what the split and the early
        __syncwarp();  // table reads met, and record directly from here on
        if (lane == 0 && s_page_err[warp] != 0) atomicExch(p.err, s_page_err[warp]);
        if (threadIdx.x == 0 && bad_len) atomicExch(p.err, TQ_DEVERR_BAD_LENGTH);
        sp.err = p.err;
      }
    }
    waited = true;
    for (int k = n_early; k < n_first; ++k) {
      const unsigned sl = (seq + k) % kPairStages;
      issue_pair<KB, KQ, KH, VB, VQ, PAGED>(my_stages_s + sl * PB, my_bars + 8 * sl, sp, m0t + 2 * k,
                                     min(2, nt - 2 * k), lane, p.cache, b, kvh);
    }

    // ---- query fragments: column lg of KV head kvh, dims [32 lt, 32 lt + 32); columns Gc ..
    // 2 Gc - 1 hold the lo terms when they ride in the same MMA
    const bool hv = lg < (QLO ? Gc : 2 * Gc);
    const long long qrow = (long long)(b * p.Hkv + kvh) * kQCols + (hv ? lg : 0);
    const int Lmin = L - p.nq + 1;  // causal end of the chunk's first query
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
    uint32_t qfl[16], qsl[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) qfl[i] = qsl[i] = 0;
    if constexpr (QLO) {
      const bool hl = lg < Gc;
#pragma unroll
      for (int i = 0; i < 16; i += 4) {
        const uint4 v = hl ? *reinterpret_cast<const uint4*>(p.q_rot_lo + qrow * (kDecD / 2) + 16 * lt + i)
                           : make_uint4(0, 0, 0, 0);
        qfl[i] = v.x; qfl[i + 1] = v.y; qfl[i + 2] = v.z; qfl[i + 3] = v.w;
        if constexpr (KQ) {
          const uint4 w = hl ? *reinterpret_cast<const uint4*>(p.q_sk_lo + qrow * (kDecD / 2) + 16 * lt + i)
                             : make_uint4(0, 0, 0, 0);
          qsl[i] = w.x; qsl[i + 1] = w.y; qsl[i + 2] = w.z; qsl[i + 3] = w.w;
        }
      }
    }
    qu[0] = qu[1] = 0;
    if constexpr (KH) {
      if (lg < Gc) {  // hi columns only: a lo column must carry lo terms alone
        qu[0] = p.q_u[qrow * 8 + lt];
        qu[1] = p.q_u[qrow * 8 + lt + 4];
      }
    }

    for (int k = 0; k < npairs; ++k) {
      const unsigned cur = seq + k, sl = cur % kPairStages;
      const bool two = 2 * k + 1 < nt;
      if (!mbar_wait(my_bars + 8 * sl, (cur / kPairStages) & 1u, kWaitLimit)) timed_out = true;
      const unsigned char* stg = my_stages + sl * PB;
      TileData<KB, KQ, KH, VB, VQ> d[2];
      const int t0 = (m0t + 2 * k) * kTile;
      if constexpr (!(KH || ((KQ || VQ) && QLO))) {
        read_stage(d[0], stg, stg + 2 * KBL - SG::VC, lg, lt);
        if (two) read_stage(d[1], stg + KBL, stg + 2 * KBL + VBL - SG::VC, lg, lt);
        __syncwarp();  // every lane has read the stage
        fence_proxy_async_shared();
        if (k + kPairStages < npairs)
          issue_pair<KB, KQ, KH, VB, VQ, PAGED>(my_stages_s + sl * PB, my_bars + 8 * sl, sp, m0t + 2 * (k + kPairStages),
                                         min(2, nt - 2 * (k + kPairStages)), lane, p.cache, b, kvh);
        if (two) {
          if (t0 + 2 * kTile <= Lmin)
            compute_tiles<2, false, QLO>(d, st, qf, qs, qu, qfl, qsl, lxK, lxV, k_m0, v_m0, p, t0, L, Lmin, lg);
          else
            compute_tiles<2, true, QLO>(d, st, qf, qs, qu, qfl, qsl, lxK, lxV, k_m0, v_m0, p, t0, L, Lmin, lg);
        } else {
          compute_tiles<1, true, QLO>(d, st, qf, qs, qu, qfl, qsl, lxK, lxV, k_m0, v_m0, p, t0, L, Lmin, lg);
        }
      } else {
        // QJL and HeadQ variants keep one tile in registers at a time (their extra state leaves no
        // room for two); the stage is refilled once its last tile has been read
#pragma unroll 1
        for (int j = 0; j < 2; ++j) {
          if (j == 1 && !two) break;
          read_stage(d[0], stg + j * KBL, stg + 2 * KBL + j * VBL - SG::VC, lg, lt);
          if (j == 1 || !two) {
            __syncwarp();
            fence_proxy_async_shared();
            if (k + kPairStages < npairs)
              issue_pair<KB, KQ, KH, VB, VQ, PAGED>(my_stages_s + sl * PB, my_bars + 8 * sl, sp,
                                             m0t + 2 * (k + kPairStages), min(2, nt - 2 * (k + kPairStages)), lane, p.cache, b, kvh);
          }
          const int tj = t0 + j * kTile;
          if (tj + kTile <= Lmin)
            compute_tiles<1, false, QLO>(d, st, qf, qs, qu, qfl, qsl, lxK, lxV, k_m0, v_m0, p, tj, L, Lmin, lg);
          else
            compute_tiles<1, true, QLO>(d, st, qf, qs, qu, qfl, qsl, lxK, lxV, k_m0, v_m0, p, tj, L, Lmin, lg);
        }
      }
    }
    seq += npairs;

    // ---- merge the warps of this block for this segment
    constexpr bool MV = kMaskedValues<VB, VQ>::value;
    float l0 = st.l0, l1 = st.l1;
    constexpr bool PKD = VQ && !QLO;  // the sketch readout rides in the value MMA
    float w00 = st.w[0][0], w01 = st.w[0][1], w10 = st.w[1][0], w11 = st.w[1][1];
#pragma unroll
    for (int m = 4; m <= 16; m <<= 1) {
      l0 += __shfl_xor_sync(kFull, l0, m);
      l1 += __shfl_xor_sync(kFull, l1, m);
      if constexpr (MV) {
        w00 += __shfl_xor_sync(kFull, w00, m);
        w01 += __shfl_xor_sync(kFull, w01, m);
        if constexpr (!PKD) {
          w10 += __shfl_xor_sync(kFull, w10, m);
          w11 += __shfl_xor_sync(kFull, w11, m);
        }
      }
    }
    __syncthreads();  // every warp is done with its stages: reuse them for the merge
    float* mb = reinterpret_cast<float*>(my_stages);
    if (lg == 0) {
      mb[(2 * lt) * PS + 0] = st.m0;
      mb[(2 * lt) * PS + 1] = l0;
      mb[(2 * lt + 1) * PS + 0] = st.m1;
      mb[(2 * lt + 1) * PS + 1] = l1;
      if constexpr (MV) {
        // slot offsets 2 / 3: the code readout's and the value sketch's weight sums; with a
        // packed sketch readout a sketch column (Gc <= c < 2 Gc) files its sum under c - Gc
        const int cc[2] = {2 * lt, 2 * lt + 1};
        const float wc[2] = {w00, w01}, ws[2] = {w10, w11};
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int c = cc[k];
          if (PKD) {
            if (c < Gc) mb[c * PS + 2] = wc[k];
            else if (c < 2 * Gc) mb[(c - Gc) * PS + 3] = wc[k];
          } else {
            mb[c * PS + 2] = wc[k];
            mb[c * PS + 3] = ws[k];
          }
        }
      }
    }
    // accumulator of column c: the code readout of slot c, or with a packed sketch readout
    // (Gc <= c < 2 Gc) the sketch readout of slot c - Gc
    int o0 = (2 * lt) * PS + 4, o1 = (2 * lt + 1) * PS + 4;
    if constexpr (VQ && !QLO) {
      if (2 * lt >= Gc && 2 * lt < 2 * Gc) o0 = (2 * lt - Gc) * PS + 4 + kDecD;
      if (2 * lt + 1 >= Gc && 2 * lt + 1 < 2 * Gc) o1 = (2 * lt + 1 - Gc) * PS + 4 + kDecD;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int d0 = 16 * lg + 2 * mt;
      mb[o0 + d0] = st.acc[mt][0];
      mb[o1 + d0] = st.acc[mt][1];
      mb[o0 + d0 + 1] = st.acc[mt][2];
      mb[o1 + d0 + 1] = st.acc[mt][3];
      if constexpr (VQ && QLO) {
        mb[(2 * lt) * PS + 4 + kDecD + d0] = st.accs[mt][0];
        mb[(2 * lt + 1) * PS + 4 + kDecD + d0] = st.accs[mt][1];
        mb[(2 * lt) * PS + 4 + kDecD + d0 + 1] = st.accs[mt][2];
        mb[(2 * lt + 1) * PS + 4 + kDecD + d0 + 1] = st.accs[mt][3];
      }
    }
    __syncthreads();
    // each column's maximum over the warps and each warp's scale, once per column
    if (threadIdx.x < Gc) {
      const int h = threadIdx.x;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < SM::NW; ++w) M = fmaxf(M, reinterpret_cast<const float*>(win + SM::region(w))[h * PS]);
      s_wmax[h] = M;
#pragma unroll
      for (int w = 0; w < SM::NW; ++w)
        s_wscale[w][h] = M != -INFINITY ? exp2f(reinterpret_cast<const float*>(win + SM::region(w))[h * PS] - M) : 0.f;
    }
    __syncthreads();
    float* part_out = p.part + ((long long)(pair + blockIdx.x) * Gc) * PS;
    for (int idx = threadIdx.x; idx < Gc * PS; idx += blockDim.x) {
      const int h = idx / PS, e = idx % PS;
      float v = 0.f;
      if (e == 0) {
        v = s_wmax[h];
      } else if (MV || (e != 2 && e != 3)) {
#pragma unroll
        for (int w = 0; w < SM::NW; ++w)
          v = fmaf(s_wscale[w][h], reinterpret_cast<const float*>(win + SM::region(w))[h * PS + e], v);
      }
      part_out[h * PS + e] = v;
    }

    // ---- the last block of this slab merges all its partials
    int c_first, c_last;
    if constexpr (EQS) {
      c_first = owner_block(slab_start, W, N);
      c_last = owner_block(slab_start + ntb - 1, W, N);
    } else {
      const long long P = *reinterpret_cast<volatile long long*>(s_split);
      const long long Wv = *reinterpret_cast<volatile long long*>(s_split + 1);
      const long long vslab = slab_start + P * (pair + 1);  // its first real tile, slab pair
      c_first = owner_block(vslab, Wv, N);
      c_last = owner_block(vslab + ntb - 1, Wv, N);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const int prev = atomicAdd(p.tickets + pair, 1);
      s_last = prev == c_last - c_first;
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      // (2)'s rows of S_V, requested now so that their latency overlaps (1)
      constexpr int RPW = (kDecD + SM::NW - 1) / SM::NW;  // sketch rows per warp
      const int j0 = warp * RPW;
      float4 srow[VQ ? RPW : 1];
      if constexpr (VQ) {
#pragma unroll
        for (int r = 0; r < RPW; ++r)
          srow[r] = j0 + r < kDecD ? __ldg(reinterpret_cast<const float4*>(p.tab.S_V + (j0 + r) * kDecD + 4 * lane))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      // (1) warp h < Gc merges query column h's partials; with a QJL value side the merged
      // acc_sk goes to shared memory for (2)
      const int h = warp;  // query column
      float L2 = 0.f;
      float o[4] = {0.f, 0.f, 0.f, 0.f};
      if (warp < Gc) {
        const long long sstride = (long long)Gc * PS;
        const float* base = p.part + (long long)(pair + c_first) * sstride + h * PS;
        const int ns = c_last - c_first + 1;
        float M = -INFINITY;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f), accs = make_float4(0.f, 0.f, 0.f, 0.f);
        float Wc = 0.f, Ws = 0.f;  // weight sums of the masked operands (MV)
        if constexpr (MV) {
          // the partials' maxima, denominators and weight sums (a partial's first four floats)
          // are read lane-parallel as one float4 (lane s takes partial s, 32 at a time): a slab
          // spread over many blocks (long contexts, few slabs) would otherwise pay one dependent
          // L2 round trip per partial
          auto header = [&](int s) {
            return s < ns ? __ldcg(reinterpret_cast<const float4*>(base + (long long)s * sstride))
                          : make_float4(-INFINITY, 0.f, 0.f, 0.f);
          };
          float4 hd = header(lane);
          M = hd.x;
          for (int s0 = 32; s0 < ns; s0 += 32)
            if (s0 + lane < ns) M = fmaxf(M, __ldcg(base + (s0 + lane) * sstride));
          M = warp_max(M);
          if (M != -INFINITY) {
            for (int s0 = 0; s0 < ns; s0 += 32) {
              const int nn = min(32, ns - s0);
              if (s0 > 0) hd = header(s0 + lane);
              const float wl = lane < nn ? exp2f(hd.x - M) : 0.f;
              L2 = fmaf(wl, hd.y, L2);
              Wc = fmaf(wl, hd.z, Wc);
              Ws = fmaf(wl, hd.w, Ws);
#pragma unroll 8
              for (int i = 0; i < nn; ++i) {
                const float w = __shfl_sync(kFull, wl, i);
                const float* ps = base + (s0 + i) * sstride;
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
            L2 = warp_sum(L2);
            Wc = warp_sum(Wc);
            Ws = warp_sum(Ws);
          }
        } else {
          for (int s = 0; s < ns; ++s) M = fmaxf(M, __ldcg(base + s * sstride));
          if (M != -INFINITY) {
            for (int s = 0; s < ns; ++s) {
              const float* ps = base + s * sstride;
              const float w = exp2f(__ldcg(ps) - M);
              L2 = fmaf(w, __ldcg(ps + 1), L2);
              const float4 a = __ldcg(reinterpret_cast<const float4*>(ps + 4 + 4 * lane));
              acc.x = fmaf(w, a.x, acc.x); acc.y = fmaf(w, a.y, acc.y);
              acc.z = fmaf(w, a.z, acc.z); acc.w = fmaf(w, a.w, acc.w);
            }
          }
        }
        o[0] = acc.x; o[1] = acc.y; o[2] = acc.z; o[3] = acc.w;
        if constexpr (MV) {
          // masked operands: row k of a 16-dim group holds 2^e sum w sigma (the +-1 dims:
          // sum w (2 sigma - 1)); turn it into sum w (2 sigma - 1), times the 1-bit centroid for
          // value codes
          float sk[4] = {accs.x, accs.y, accs.z, accs.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int k = (4 * lane + e) & 15;
            const float f2 = 2.f * mask_unscale(k);
            const bool pm = mask_is_pm1(k);
            if constexpr (VB == 1) o[e] = vc1 * (pm ? o[e] : fmaf(f2, o[e], -Wc));
            if constexpr (VQ) sk[e] = pm ? sk[e] : fmaf(f2, sk[e], -Ws);
          }
          accs = make_float4(sk[0], sk[1], sk[2], sk[3]);
        }
        if constexpr (VQ)
          *reinterpret_cast<float4*>(win + SM::region(h) + kSkA + 16 * lane) = accs;
      }
      if constexpr (VQ) {
        // (2) o_rot += sqrt(pi/2)/m S_V^T acc_sk for every column: the warps split the m sketch
        // rows, so each loads its rows of S_V once (all in flight) and applies them to every
        // column; partial sums go to shared memory and (3) adds them up
        __syncthreads();
        float* part_sum = reinterpret_cast<float*>(win + SM::region(warp));
        for (int c = 0; c < Gc; ++c) {
          const float* a = reinterpret_cast<const float*>(win + SM::region(c) + kSkA);
          float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int r = 0; r < RPW; ++r) {
            const float ar = j0 + r < kDecD ? a[j0 + r] : 0.f;
            t.x = fmaf(srow[r].x, ar, t.x); t.y = fmaf(srow[r].y, ar, t.y);
            t.z = fmaf(srow[r].z, ar, t.z); t.w = fmaf(srow[r].w, ar, t.w);
          }
          *reinterpret_cast<float4*>(part_sum + c * kDecD + 4 * lane) = t;
        }
        __syncthreads();
        if (warp < Gc) {  // (3)
          float corr[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int w = 0; w < SM::NW; ++w) {
            const float4 t = *reinterpret_cast<const float4*>(win + SM::region(w) + (h * kDecD + 4 * lane) * 4);
            corr[0] += t.x; corr[1] += t.y; corr[2] += t.z; corr[3] += t.w;
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) o[i] = fmaf(p.qjl_scale, corr[i], o[i]);
        }
      }
      if (warp < Gc) {
        const float invL = L2 > 0.f ? 1.f / L2 : 0.f;
        if constexpr (VB == kSQ) {
          // SQU-KV values: o = E (s acc) / l with the basis and scales of KV head kvh
          const float4 s4 = __ldg(reinterpret_cast<const float4*>(p.tab.sq_s[1] + (long long)kvh * kDecD + 4 * lane));
          const float a[4] = {o[0] * s4.x, o[1] * s4.y, o[2] * s4.z, o[3] * s4.w};
          float r[4] = {0.f, 0.f, 0.f, 0.f};
          const float* ET = p.tab.sq_ET[1] + (long long)kvh * kDecD * kDecD + 4 * lane;
#pragma unroll 4
          for (int sl = 0; sl < 32; ++sl) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float ac = __shfl_sync(kFull, a[e], sl);
              const float4 er = __ldg(reinterpret_cast<const float4*>(ET + (4 * sl + e) * kDecD));
              r[0] = fmaf(er.x, ac, r[0]); r[1] = fmaf(er.y, ac, r[1]);
              r[2] = fmaf(er.z, ac, r[2]); r[3] = fmaf(er.w, ac, r[3]);
            }
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) o[i] = r[i] * invL;
        } else if (p.v_rotate) {
          wht_warp<4>(o);
          const float rs = 1.f / sqrtf((float)kDecD);
#pragma unroll
          for (int i = 0; i < 4; ++i) o[i] = o[i] * rs * __ldg(p.tab.v_sign + 4 * lane + i) * invL;
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) o[i] *= invL;
        }
        float* dst = p.out + (((long long)b * p.nq + h / G) * Hq + kvh * G + h % G) * kDecD + 4 * lane;
        *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
      }
      if (threadIdx.x == 0) p.tickets[pair] = 0;
    }
    __syncthreads();  // the merge area becomes the next segment's stages
    x = seg_end;
  }
  if (timed_out) atomicExch(p.err, kErrWaitTimeout);
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

// Query buffers at the start of dynamic shared memory; the key table at kLutAddrK.
template <int KB>
struct LogitsSmem {
  static constexpr uint32_t lut = LutEntries<KB>::value * kLutStride;
  static constexpr uint32_t qbytes = (kHeadsPad * (kDecD / 2) * 2 + kHeadsPad * 8) * 4;
  static constexpr uint32_t bytes = KB == 1 ? qbytes : kLutAddrK + lut;
  static_assert(kDynBaseMax + qbytes <= kLutAddrK, "query buffers overlap the key table");
};

template <int KB, bool KQ, bool KH>
__global__ void __launch_bounds__(kLogitsWarps * 32) logits_kernel(const LogitsParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int lg = lane >> 2, lt = lane & 3;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int T = p.seq_len[b];
  const int c0 = blockIdx.x * p.tokens_per_block;
  if (c0 >= T) return;  // the whole block leaves together
  const int G = p.G, Hq = p.Hkv * G;
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(smem);
  if (sbase > kDynBaseMax) {  // cannot happen with the documented limits; nothing is written
    return;
  }
  uint32_t* qrot = reinterpret_cast<uint32_t*>(smem);
  uint32_t* qsk = qrot + kHeadsPad * (kDecD / 2);
  uint32_t* qus = qsk + kHeadsPad * (kDecD / 2);
  if constexpr (KB != 1) build_lut<KB>(smem - sbase + kLutAddrK, p.tab.k_c);
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
      if (lane == 0) {
#pragma unroll
        for (int k = 0; k < 8; ++k) qus[warp * 8 + k] = pack_half2(z[2 * k], z[2 * k + 1]);
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
  const int per = ((c1 - c0 + kLogitsWarps - 1) / kLogitsWarps + kTile - 1) / kTile * kTile;
  const int w0 = c0 + warp * per;
  const int w1 = min(c1, w0 + per);
  SlabPtrs sp;
  sp.init(p.cache, b, kvh);
  for (int t0 = w0; t0 < w1; t0 += kTile) {
    TileData<KB, KQ, KH, 1, false> d;
    load_ktile(d, sp, t0, w1 - 1, lg, lt);
    float s[4];
    key_scores(d, s, qf, qs, qu, kLutAddrK | (4u * lane), k_m0, p.qjl_scale, p.inv_sqrt_d, qs, qs, 0);
    const int tA = t0 + tile_row_token(lg), tB = t0 + tile_row_token(lg + 8);
    const long long r0 = ((long long)b * Hq + kvh * G + 2 * lt) * p.stride;
    const long long r1 = r0 + p.stride;
    if (tA < w1) {
      if (2 * lt < G) p.logits[r0 + tA] = s[0];
      if (2 * lt + 1 < G) p.logits[r1 + tA] = s[1];
    }
    if (tB < w1) {
      if (2 * lt < G) p.logits[r0 + tB] = s[2];
      if (2 * lt + 1 < G) p.logits[r1 + tB] = s[3];
    }
  }
}

// Host check of the shared-memory plans: dynamic shared memory starts after the reserved and
// static shared memory, which must stay below kDynBaseMax.
template <typename K>
cudaError_t check_dyn_base(K kernel) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return e;
  int dev = 0, reserved = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) != cudaSuccess)
    return e;
  return (size_t)reserved + fa.sharedSizeBytes <= kDynBaseMax ? cudaSuccess : cudaErrorInvalidConfiguration;
}

// Launch helpers used by the per-bit-width instantiation units.
template <int KB, bool KQ, bool KH, int VB, bool VQ, bool QLO, bool PAGED>
cudaError_t launch_decode_t(const DecodeParams& p, dim3 grid, cudaStream_t s) {
  using SM = DecodeSmem<KB, KQ, KH, VB, VQ, QLO>;
  constexpr uint32_t bytes = SM::bytes + (PAGED ? kPagedPlanBytes : 0u);
  static_assert(SM::bytes % 8 == 0, "the paged plan area needs 8-byte alignment");
  static_assert(bytes <= 227 * 1024, "decode shared memory exceeds the per-block limit");
  auto kern = decode_kernel<KB, KQ, KH, VB, VQ, QLO, PAGED>;
  cudaError_t e = check_dyn_base(kern);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  // may start while the query prep kernel still runs (it waits in grid_dependency_wait)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(SM::NW * 32);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int KB, bool KQ, bool KH, int VB, bool VQ>
cudaError_t launch_decode_any(const DecodeParams& p, dim3 grid, cudaStream_t s) {
  const bool qlo = p.lo_xor == 0, paged = p.cache.block_table != nullptr;
  if (paged) return qlo ? launch_decode_t<KB, KQ, KH, VB, VQ, true, true>(p, grid, s)
                        : launch_decode_t<KB, KQ, KH, VB, VQ, false, true>(p, grid, s);
  return qlo ? launch_decode_t<KB, KQ, KH, VB, VQ, true, false>(p, grid, s)
             : launch_decode_t<KB, KQ, KH, VB, VQ, false, false>(p, grid, s);
}

template <int KB, bool KQ, bool KH>
cudaError_t launch_logits_t(const LogitsParams& p, dim3 grid, cudaStream_t s) {
  using SM = LogitsSmem<KB>;
  cudaError_t e = check_dyn_base(logits_kernel<KB, KQ, KH>);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(logits_kernel<KB, KQ, KH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)SM::bytes);
  if (e != cudaSuccess) return e;
  logits_kernel<KB, KQ, KH><<<grid, kLogitsWarps * 32, SM::bytes, s>>>(p);
  return cudaGetLastError();
}

// Per-bit-width dispatchers (one translation unit each).  Return false when the codec
// combination is not built.
bool dispatch_decode_k1(int kq, int kh, int vb, int vq, const DecodeParams& p, dim3 g, cudaStream_t s, cudaError_t* e);
bool dispatch_decode_k2(int kq, int kh, int vb, int vq, const DecodeParams& p, dim3 g, cudaStream_t s, cudaError_t* e);
bool dispatch_decode_k3(int kq, int kh, int vb, int vq, const DecodeParams& p, dim3 g, cudaStream_t s, cudaError_t* e);
bool dispatch_decode_k4(int kq, int kh, int vb, int vq, const DecodeParams& p, dim3 g, cudaStream_t s, cudaError_t* e);
bool dispatch_decode_ksq(int kq, int kh, int vb, int vq, const DecodeParams& p, dim3 g, cudaStream_t s, cudaError_t* e);
bool dispatch_logits_k1(int kq, int kh, const LogitsParams& p, dim3 g, cudaStream_t s, cudaError_t* e);
bool dispatch_logits_k2(int kq, int kh, const LogitsParams& p, dim3 g, cudaStream_t s, cudaError_t* e);
bool dispatch_logits_k3(int kq, int kh, const LogitsParams& p, dim3 g, cudaStream_t s, cudaError_t* e);
bool dispatch_logits_k4(int kq, int kh, const LogitsParams& p, dim3 g, cudaStream_t s, cudaError_t* e);

#define TQ_DECODE_CASE(KB_, KQ_, KH_, VB_, VQ_)                                           \
  if (kq == KQ_ && kh == KH_ && vb == VB_ && vq == VQ_) {                                 \
    if (e) *e = launch_decode_any<KB_, KQ_ != 0, KH_ != 0, VB_, VQ_ != 0>(p, g, s);                \
    return true;                                                                          \
  }
#define TQ_LOGITS_CASE(KB_, KQ_, KH_)                                                     \
  if (kq == KQ_ && kh == KH_) {                                                           \
    if (e) *e = launch_logits_t<KB_, KQ_ != 0, KH_ != 0>(p, g, s);                        \
    return true;                                                                          \
  }

}  // namespace tqd
