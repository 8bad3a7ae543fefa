// Write path: quantize-and-append, HeadQ basis rotation, and reconstruction for tests.
//
// [TQ-KV] "Esquemas de Cuantización": norm split, randomized Walsh-Hadamard rotation, Lloyd-Max
// scalar code, optional 1-bit QJL sketch of the residual.  [HEADQ] "Visão Geral do Algoritmo"
// 2 ("Escrita no Cache"): base key, residual, projection on the calibrated basis, side code.
//
// One warp owns one vector; lane l holds coordinates [l*E, l*E + E), E = d / 32.  The rotation
// runs in registers (local butterflies, then warp shuffles); codes are packed so that lane l's
// bits are contiguous in the stream and stored with one coalesced store per lane group.
#include <algorithm>
#include <cstdio>
#include <string>
#include <type_traits>

#include "tq_device.cuh"
#include "tq_tc05.cuh"

namespace tqd {

namespace {

constexpr int kWarpsPerBlock = 8;
// vectors per warp of append_kernel, their chains interleaved (one for the wide head dims,
// whose per-lane state is already large)
template <int D> struct AppendNV { static constexpr int value = D == 128 ? 2 : 1; };

struct AppendParams {
  Tables tab;
  Cache cache;
  const void* k;
  const void* v;
  int B, Hkv, n_new, m;
  int bits[2], rotate[2], qjl[2];
  int headq_rank;
  int qjl_mma;   // QJL sides go to append_qjl_mma_kernel (head dim 128)
  int side_base;     // append_kernel: side of blockIdx.y = 0 (the other, if any, is side_base + 1)
  int wait_primary;  // append_kernel runs as the dependent launch of append_qjl_mma_kernel
  int release_early; // append_kernel / append_quad_kernel let their dependents launch at once
  int start[TQ_MAX_BATCH];
  const int* dev_start;  // set: start positions from device memory (paged pool)
  // n / n_new and n / Hkv for 0 <= n < 2^31 as (umulhi(n, mul) + n) >> shift
  uint32_t div_n_mul, div_n_shift, div_h_mul, div_h_shift;
};

// Multiplier and shift of the division by d (1 <= d < 2^31) for dividends below 2^31: with
// l = ceil(log2 d) and mul = floor(2^32 (2^l - d) / d) + 1, n / d = (umulhi(n, mul) + n) >> l
// (the round-up reciprocal method; umulhi(n, mul) + n stays below 2^32).
inline void fast_div_magic(uint32_t d, uint32_t& mul, uint32_t& shift) {
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  mul = (uint32_t)((((1ull << 32) * ((1ull << l) - d)) / d + 1) & 0xffffffffull);
  shift = l;
}
__device__ __forceinline__ uint32_t fast_div(uint32_t n, uint32_t mul, uint32_t shift) {
  return (__umulhi(n, mul) + n) >> shift;
}

// Flat vector index (over [B][H_kv][n_new], below 2^31) -> batch, KV head, index in the chunk,
// position.
__device__ __forceinline__ void split_vec(const AppendParams& p, long long vec, int& b, int& h, int& j, int& t) {
  const uint32_t v = (uint32_t)vec;
  const uint32_t r = fast_div(v, p.div_n_mul, p.div_n_shift);
  j = (int)(v - r * (uint32_t)p.n_new);
  const uint32_t bq = fast_div(r, p.div_h_mul, p.div_h_shift);
  h = (int)(r - bq * (uint32_t)p.Hkv);
  b = (int)bq;
  t = (p.dev_start ? __ldg(p.dev_start + b) : p.start[b]) + j;
}

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// Sum of squares with a compensated (double-float) accumulation, then a corrected sqrt, so the
// fp32 norm is within about half an ulp of the exact one.
template <int E>
__device__ __forceinline__ float norm_compensated(const float (&x)[E]) {
  float S = 0.f, C = 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const float p = x[i] * x[i];
    const float pe = fmaf(x[i], x[i], -p);
    float s, e;
    two_sum(S, p, s, e);
    S = s;
    C += e + pe;
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    const float So = __shfl_xor_sync(kFull, S, m);
    const float Co = __shfl_xor_sync(kFull, C, m);
    float s, e;
    two_sum(S, So, s, e);
    S = s;
    C = (C + Co) + e;
  }
  S = __shfl_sync(kFull, S, 0);
  C = __shfl_sync(kFull, C, 0);
  if (S <= 0.f) return 0.f;
  const float r = sqrtf(S);
  const float res = fmaf(-r, r, S) + C;
  return r + res / (2.f * r);
}

// The norm split for any finite input.  The fast path is norm_compensated of x itself.  When
// that norm leaves [2^-30, 2^50) (a sum of squares that overflowed, underflowed, or lost bits
// to subnormal squares), x is first multiplied by the power of two 2^-e that brings max|x| to
// [1, 2) (clamped to e in [-126, 126]).  The scaling is exact and leaves the unit vector as it
// was, so the rotation, codes, residual and side code are computed from the scaled vector with
// no change; within the fast path's range it would give the same bits.  Returns the norm to
// store, nu_work * 2^e (which may round once more, or overflow to inf, only when it leaves the
// fp32 range); nu_work is the norm of the vector left in x, and pw = 2^e.
template <int E>
__device__ __forceinline__ float norm_split(float (&x)[E], float& nu_work, float& pw) {
  const float nu = norm_compensated<E>(x);  // the same value in every lane
  pw = 1.f;
  nu_work = nu;
  if (nu >= 0x1p-30f && nu < 0x1p50f) return nu;
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i) m = fmaxf(m, fabsf(x[i]));
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, s));
  if (!(m > 0.f)) {
    nu_work = 0.f;
    return 0.f;
  }
  const int e = max(-126, min(126, ((__float_as_int(m) >> 23) & 0xFF) - 127));
  const float down = __int_as_float((127 - e) << 23);
  pw = __int_as_float((127 + e) << 23);
#pragma unroll
  for (int i = 0; i < E; ++i) x[i] *= down;
  nu_work = norm_compensated<E>(x);
  return nu_work * pw;
}

// Store a w-bit stream: lane l's E values occupy bits [l*E*W, (l+1)*E*W) of the stream.
template <int E, int W>
__device__ __forceinline__ void store_stream(unsigned char* dst, const uint32_t (&v)[E]) {
  constexpr int BITS = E * W;
  const int lane = threadIdx.x & 31;
  if constexpr (BITS >= 32) {
    constexpr int WORDS = BITS / 32;
    uint32_t w[WORDS];
#pragma unroll
    for (int k = 0; k < WORDS; ++k) w[k] = 0;
#pragma unroll
    for (int i = 0; i < E; ++i) w[(i * W) / 32] |= v[i] << ((i * W) % 32);
    uint32_t* out = reinterpret_cast<uint32_t*>(dst) + lane * WORDS;
    if constexpr (WORDS % 4 == 0) {
#pragma unroll
      for (int k = 0; k < WORDS; k += 4)
        *reinterpret_cast<uint4*>(out + k) = make_uint4(w[k], w[k + 1], w[k + 2], w[k + 3]);
    } else if constexpr (WORDS % 2 == 0) {
#pragma unroll
      for (int k = 0; k < WORDS; k += 2) *reinterpret_cast<uint2*>(out + k) = make_uint2(w[k], w[k + 1]);
    } else {
      out[0] = w[0];
    }
  } else {
    uint32_t chunk = 0;
#pragma unroll
    for (int i = 0; i < E; ++i) chunk |= v[i] << (i * W);
    constexpr int LPW = 32 / BITS;
    uint32_t word = chunk << (BITS * (lane % LPW));
#pragma unroll
    for (int m = 1; m < LPW; m <<= 1) word |= __shfl_xor_sync(kFull, word, m);
    if (lane % LPW == 0) reinterpret_cast<uint32_t*>(dst)[lane / LPW] = word;
  }
}

// Store a W-bit value-side stream of one vector at block position pos: lane l's E values are
// coordinates [l*E, (l+1)*E); the group of coordinates [16 g, 16 g + 16) of this token is the
// 2W bytes at stream + g * 32W + pos * 2W (see grouped_byte).
template <int E, int W>
__device__ __forceinline__ void store_stream_grouped(unsigned char* stream, int pos, const uint32_t (&v)[E]) {
  static_assert(16 % E == 0 || E % 16 == 0, "a lane holds part of one group or whole groups");
  const int lane = threadIdx.x & 31;
  auto put = [&](int g, unsigned long long bits) {
    unsigned char* dst = stream + g * 32 * W + pos * 2 * W;
    if constexpr (W == 4) *reinterpret_cast<unsigned long long*>(dst) = bits;
    else if constexpr (W == 2) *reinterpret_cast<uint32_t*>(dst) = (uint32_t)bits;
    else *reinterpret_cast<unsigned short*>(dst) = (unsigned short)bits;
  };
  if constexpr (E >= 16) {
#pragma unroll
    for (int g = 0; g < E / 16; ++g) {
      unsigned long long bits = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) bits |= (unsigned long long)v[16 * g + i] << (i * W);
      put(lane * (E / 16) + g, bits);
    }
  } else {
    constexpr int LPG = 16 / E;  // lanes per group
    unsigned long long bits = 0;
#pragma unroll
    for (int i = 0; i < E; ++i) bits |= (unsigned long long)v[i] << (((lane % LPG) * E + i) * W);
#pragma unroll
    for (int m = 1; m < LPG; m <<= 1) bits |= __shfl_xor_sync(kFull, bits, m);
    if (lane % LPG == 0) put(lane / LPG, bits);
  }
}

// Read back element values of a w-bit stream for this lane's E coordinates: a whole record at
// src (pos < 0), or a value-side stream at src stored by coordinate groups (block position pos).
template <int E, int W>
__device__ __forceinline__ void load_stream(const unsigned char* src, uint32_t (&v)[E], int pos = -1) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int bit = (lane * E + i) * W;
    const unsigned j = (unsigned)bit >> 3;
    const unsigned char byte = pos < 0 ? src[j] : src[grouped_byte(j, (unsigned)pos, W)];
    v[i] = (byte >> (bit & 7)) & ((1u << W) - 1u);
  }
}

// NV vectors of one side through the write path ([TQ-KV] "Esquemas de Cuantización"), their
// dependency chains (loads, shuffle reductions, butterflies) interleaved: norm, rotation,
// scalar code, code and norm stores; on a QJL side the residual r = y - C[c] (left in res) and
// its fp16 norm; on a key with HeadQ the side code ([HEADQ] "Escrita no Cache").  Vectors with
// valid[v] false (the same in every lane) are neither loaded nor stored and leave res = 0.
template <int D, typename Tin, int NV>
__device__ __forceinline__ void encode_vectors(const AppendParams& p, int side, const int (&b)[NV],
                                               const int (&h)[NV], const int (&j)[NV], const int (&t)[NV],
                                               const bool (&valid)[NV], float (&res)[NV][D / 32]) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int bits = p.bits[side];
  const bool rotate = p.rotate[side] != 0;
  const float* sgn = side ? p.tab.v_sign : p.tab.k_sign;
  const float* cent = side ? p.tab.v_c : p.tab.k_c;
  const float* thr = side ? p.tab.v_t : p.tab.k_t;
  const Tin* base = reinterpret_cast<const Tin*>(side ? p.v : p.k);

  float x[NV][E];
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    if (valid[v]) {
      load_row<E>(base + ((long long)(b[v] * p.Hkv + h[v]) * p.n_new + j[v]) * D + lane * E, x[v]);
    } else {
#pragma unroll
      for (int i = 0; i < E; ++i) x[v][i] = 0.f;
    }
  }
  float nu[NV], nw[NV], pw[NV];  // stored norm, norm of the (possibly rescaled) x, rescale 2^e
#pragma unroll
  for (int v = 0; v < NV; ++v) nu[v] = norm_split<E>(x[v], nw[v], pw[v]);

  float dsg[E];
#pragma unroll
  for (int i = 0; i < E; ++i) dsg[i] = __ldg(sgn + lane * E + i);
  float hrot[NV][E];
#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int i = 0; i < E; ++i) hrot[v][i] = x[v][i] * dsg[i];
  if (rotate) {
#pragma unroll
    for (int v = 0; v < NV; ++v) wht_warp<E>(hrot[v]);
  }
  const float rs = rotate ? 1.f / sqrtf((float)D) : 1.f;
  const float scale = rotate ? sqrtf((float)D) : 1.f;

  // The code c = #{k : y > t_k} (ties to the lower cell) in sign-magnitude form.  The
  // thresholds are symmetric (t_{h-1} = 0 and t_{h-1+k} = -t_{h-1-k} exactly, h = 2^(b-1);
  // checked when the context is created), so s = [y > 0] and the magnitude counts only the
  // upper thresholds: #{k >= h : y > t_k} for y > 0, #{k >= h : -y >= t_k} otherwise; -y >= t
  // is tested as nextup(-y) > t.
  const uint32_t halfL = 1u << (bits - 1);
  float tu[7];  // t_h .. t_{h+6}; slots past the last threshold hold 3e38
#pragma unroll
  for (int k = 0; k < 7; ++k) tu[k] = __ldg(thr + halfL + k);
  float y[NV][E];
  uint32_t code[NV][E], sgnbit[NV][E], mag[NV][E];
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const float inv = nw[v] > 0.f ? 1.f / (nw[v] * scale) : 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      y[v][i] = hrot[v][i] * inv;
      const bool pos = y[v][i] > 0.f;
      const float a = pos ? y[v][i] : __int_as_float(__float_as_int(-y[v][i]) + 1);
      uint32_t m = 0;
#pragma unroll
      for (int k = 0; k < 7; ++k) m += a > tu[k] ? 1u : 0u;
      sgnbit[v][i] = pos ? 1u : 0u;
      mag[v][i] = m;
      code[v][i] = pos ? halfL + m : halfL - 1u - m;
    }
  }

  const Cache& C = p.cache;
  const int rc = side ? tqi::R_V_CODES : tqi::R_K_CODES;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    if (!valid[v]) continue;
    if (side == 0) {  // key records: whole records, token-major
      unsigned char* codes = C.ptr(rc, b[v], h[v], t[v]);
      if (bits == 4) {
        uint32_t w[E];
#pragma unroll
        for (int i = 0; i < E; ++i) w[i] = (sgnbit[v][i] << 3) | mag[v][i];
        store_stream<E, 4>(codes, w);
      } else if (bits == 3) {
        store_stream<E, 2>(codes, mag[v]);
        store_stream<E, 1>(codes + D / 4, sgnbit[v]);
      } else if (bits == 2) {
        uint32_t w[E];
#pragma unroll
        for (int i = 0; i < E; ++i) w[i] = (sgnbit[v][i] << 1) | mag[v][i];
        store_stream<E, 2>(codes, w);
      } else {
        store_stream<E, 1>(codes, sgnbit[v]);
      }
    } else {  // value streams: by groups of 16 coordinates
      unsigned char* f = C.fieldp(rc, b[v], h[v], t[v]);
      const int pos = t[v] & (tqi::kTileTokens - 1);
      if (bits == 4) {
        uint32_t w[E];
#pragma unroll
        for (int i = 0; i < E; ++i) w[i] = (sgnbit[v][i] << 3) | mag[v][i];
        store_stream_grouped<E, 4>(f, pos, w);
      } else if (bits == 3) {
        store_stream_grouped<E, 2>(f, pos, mag[v]);
        store_stream_grouped<E, 1>(f + tqi::kTileTokens * (D / 4), pos, sgnbit[v]);
      } else if (bits == 2) {
        uint32_t w[E];
#pragma unroll
        for (int i = 0; i < E; ++i) w[i] = (sgnbit[v][i] << 1) | mag[v][i];
        store_stream_grouped<E, 2>(f, pos, w);
      } else {
        store_stream_grouped<E, 1>(f, pos, sgnbit[v]);
      }
    }
    if (lane == 0) *reinterpret_cast<float*>(C.ptr(side ? tqi::R_V_NORM : tqi::R_K_NORM, b[v], h[v], t[v])) = nu[v];
  }

  if (p.qjl[side]) {
    float ss[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      ss[v] = 0.f;
#pragma unroll
      for (int i = 0; i < E; ++i) {
        res[v][i] = valid[v] ? y[v][i] - __ldg(cent + code[v][i]) : 0.f;
        ss[v] = fmaf(res[v][i], res[v][i], ss[v]);
      }
    }
#pragma unroll
    for (int v = 0; v < NV; ++v) ss[v] = warp_sum(ss[v]);
#pragma unroll
    for (int v = 0; v < NV; ++v)
      if (valid[v] && lane == 0)
        *reinterpret_cast<__half*>(C.ptr(side ? tqi::R_V_RHO : tqi::R_K_RHO, b[v], h[v], t[v])) =
            __float2half_rn(sqrtf(ss[v]));
  }

  if (side == 0 && p.headq_rank) {
    // e_rot = R k - nu C[c]; z = (R U)^T e_rot = U^T e   ([HEADQ] "Escrita no Cache")
    constexpr int RK = 16;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      if (!valid[v]) continue;
      const float* Ur = p.tab.U_rot + (long long)h[v] * D * RK;
      float z[RK];
#pragma unroll
      for (int k = 0; k < RK; ++k) z[k] = 0.f;
#pragma unroll
      for (int i = 0; i < E; ++i) {
        const float e = hrot[v][i] * rs - nw[v] * __ldg(cent + code[v][i]);
        const float* urow = Ur + (lane * E + i) * RK;
#pragma unroll
        for (int k = 0; k < RK; k += 4) {
          const float4 u4 = __ldg(reinterpret_cast<const float4*>(urow + k));
          z[k] = fmaf(u4.x, e, z[k]);
          z[k + 1] = fmaf(u4.y, e, z[k + 1]);
          z[k + 2] = fmaf(u4.z, e, z[k + 2]);
          z[k + 3] = fmaf(u4.w, e, z[k + 3]);
        }
      }
      float amax = 0.f;
#pragma unroll
      for (int k = 0; k < RK; ++k) {
        z[k] = warp_sum(z[k]) * pw[v];  // back to the key's units (exact)
        amax = fmaxf(amax, fabsf(z[k]));
      }
      const __half sh = __float2half_rn(amax / 7.0f);
      const float s32 = __half2float(sh);
      uint32_t w0 = 0, w1 = 0;
#pragma unroll
      for (int k = 0; k < RK; ++k) {
        int qz = 0;
        if (s32 > 0.f) {
          const float q = rintf(__fdiv_rn(z[k], s32));
          qz = (int)fminf(fmaxf(q, -7.f), 7.f);
        }
        const uint32_t nib = (uint32_t)qz & 0xFu;
        if (k < 8) w0 |= nib << (4 * k); else w1 |= nib << (4 * (k - 8));
      }
      if (lane == 0) {
        *reinterpret_cast<uint2*>(C.ptr(tqi::R_K_SIDE, b[v], h[v], t[v])) = make_uint2(w0, w1);
        *reinterpret_cast<__half*>(C.ptr(tqi::R_K_SIDE_SCALE, b[v], h[v], t[v])) = sh;
      }
    }
  }
}

// SQU-KV write path (head dim 128, rotate = 2): NV vectors of a spectral side.  The norm split
// as for the other codecs; the calibrated basis in place of the rotation, y = E^T x (E column c
// = stored coordinate c of head h), z = y / (nu s); a modeled coordinate takes the 4-bit code of
// z (sign-magnitude, the symmetric search of encode_vectors), a floor coordinate its sign.
// Stores the record: the modeled coordinates' 4-bit magnitudes, then all 128 signs (value side:
// both streams by 16-coordinate groups).  [ABL] "Configuração Experimental" (SpectralQuant),
// "Recomendações Práticas" 2 (uniform allocation).
template <typename Tin, int NV>
__device__ __forceinline__ void encode_vectors_sq(const AppendParams& p, int side, const int (&b)[NV],
                                                  const int (&h)[NV], const int (&j)[NV], const int (&t)[NV],
                                                  const bool (&valid)[NV]) {
  constexpr int D = 128, E = D / 32;
  const int lane = threadIdx.x & 31;
  const Tin* base = reinterpret_cast<const Tin*>(side ? p.v : p.k);
  float x[NV][E];
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    if (valid[v]) {
      load_row<E>(base + ((long long)(b[v] * p.Hkv + h[v]) * p.n_new + j[v]) * D + lane * E, x[v]);
    } else {
#pragma unroll
      for (int i = 0; i < E; ++i) x[v][i] = 0.f;
    }
  }
  float nu[NV], nw[NV], pw[NV];  // stored norm, norm of the (possibly rescaled) x, rescale 2^e
#pragma unroll
  for (int v = 0; v < NV; ++v) nu[v] = norm_split<E>(x[v], nw[v], pw[v]);
  // y_c = sum_i E[i][c] x_i for this lane's coordinates c = 4 lane + jj
  float y[NV][E];
#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int jj = 0; jj < E; ++jj) y[v][jj] = 0.f;
  const float* Eh[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) Eh[v] = p.tab.sq_E[side] + (long long)h[v] * D * D + lane * E;
#pragma unroll 4
  for (int sl = 0; sl < 32; ++sl) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const float xi = __shfl_sync(kFull, x[v][e], sl);
        const float4 er = __ldg(reinterpret_cast<const float4*>(Eh[v] + (E * sl + e) * D));
        y[v][0] = fmaf(er.x, xi, y[v][0]);
        y[v][1] = fmaf(er.y, xi, y[v][1]);
        y[v][2] = fmaf(er.z, xi, y[v][2]);
        y[v][3] = fmaf(er.w, xi, y[v][3]);
      }
    }
  }
  const float* thr = side ? p.tab.v_t : p.tab.k_t;  // the 4-bit thresholds on a spectral side
  float tu[7];
#pragma unroll
  for (int k = 0; k < 7; ++k) tu[k] = __ldg(thr + 8 + k);
  const bool modeled = sq_modeled(side, E * lane);  // the same for the lane's 4 coordinates
  const Cache& C = p.cache;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const float4 s4 = __ldg(reinterpret_cast<const float4*>(p.tab.sq_s[side] + (long long)h[v] * D + lane * E));
    const float sc[E] = {s4.x, s4.y, s4.z, s4.w};
    uint32_t sgnbit[E], nib = 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const float z = nw[v] > 0.f ? __fdiv_rn(y[v][i], nw[v] * sc[i]) : 0.f;
      const bool pos = z > 0.f;
      const float a = pos ? z : __int_as_float(__float_as_int(-z) + 1);
      uint32_t m = 0;
#pragma unroll
      for (int k = 0; k < 7; ++k) m += a > tu[k] ? 1u : 0u;
      sgnbit[i] = pos ? 1u : 0u;
      nib |= m << (4 * i);
    }
    if (!valid[v]) continue;
    const int pos = t[v] & (tqi::kTileTokens - 1);
    if (side == 0) {
      unsigned char* rec = C.ptr(tqi::R_K_CODES, b[v], h[v], t[v]);
      if (modeled)  // lanes 8 lt, 8 lt + 1 hold chunk lt's 8 modeled coordinates
        *reinterpret_cast<unsigned short*>(rec + 4 * (lane / 8) + 2 * (lane % 8)) = (unsigned short)nib;
      store_stream<E, 1>(rec + 16, sgnbit);
    } else {
      unsigned char* f = C.fieldp(tqi::R_V_CODES, b[v], h[v], t[v]);
      if (modeled)  // lane 4 g holds group g's 4 modeled coordinates
        *reinterpret_cast<unsigned short*>(f + grouped_byte(2 * (lane / 4), pos, 1)) = (unsigned short)nib;
      store_stream_grouped<E, 1>(f + tqi::kTileTokens * 16, pos, sgnbit);
    }
    if (lane == 0) *reinterpret_cast<float*>(C.ptr(side ? tqi::R_V_NORM : tqi::R_K_NORM, b[v], h[v], t[v])) = nu[v];
  }
}

// One vector (see encode_vectors).
template <int D, typename Tin>
__device__ __forceinline__ void encode_vector(const AppendParams& p, int side, int b, int h, int j, int t,
                                              float (&res)[D / 32]) {
  const int bb[1] = {b}, hh[1] = {h}, jj[1] = {j}, tt[1] = {t};
  const bool ok[1] = {true};
  float r[1][D / 32];
  encode_vectors<D, Tin, 1>(p, side, bb, hh, jj, tt, ok, r);
#pragma unroll
  for (int i = 0; i < D / 32; ++i) res[i] = r[0][i];
}

// Signs of S r for one vector by an FFMA product with ST = S^T ([d][m], m == d), read from
// shared memory when the block staged it, else from L2.
template <int D>
__device__ __forceinline__ void sketch_signs_ffma(const AppendParams& p, int side, int b, int h, int t,
                                                  const float (&res)[D / 32], const float* ST) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const Cache& C = p.cache;
  float acc[E];
#pragma unroll
  for (int q = 0; q < E; ++q) acc[q] = 0.f;
  // several rows in flight per lane: the loop is bound by the table's load latency
  constexpr int kUnroll = E <= 8 ? 4 : 1;
#pragma unroll kUnroll
  for (int jl = 0; jl < 32; ++jl) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float rj = __shfl_sync(kFull, res[e], jl);
      const float* row = ST + (long long)(jl * E + e) * D + lane * E;
#pragma unroll
      for (int q = 0; q < E; q += 4) {
        const float4 s4 = *reinterpret_cast<const float4*>(row + q);
        acc[q] = fmaf(s4.x, rj, acc[q]);
        acc[q + 1] = fmaf(s4.y, rj, acc[q + 1]);
        acc[q + 2] = fmaf(s4.z, rj, acc[q + 2]);
        acc[q + 3] = fmaf(s4.w, rj, acc[q + 3]);
      }
    }
  }
  uint32_t sbit[E];
#pragma unroll
  for (int q = 0; q < E; ++q) sbit[q] = acc[q] >= 0.f ? 1u : 0u;
  if (side == 0)
    store_stream<E, 1>(C.ptr(tqi::R_K_SIGNS, b, h, t), sbit);
  else
    store_stream_grouped<E, 1>(C.fieldp(tqi::R_V_SIGNS, b, h, t), t & (tqi::kTileTokens - 1), sbit);
}

// One block of append_kernel (below).
template <int D, typename Tin>
__device__ __forceinline__ void append_body(const AppendParams& p) {
  constexpr int E = D / 32;
  constexpr int NV = AppendNV<D>::value;
  const int side = p.side_base + (int)blockIdx.y;
  if (p.qjl[side] && p.qjl_mma) return;  // left to append_qjl_mma_kernel (whole block)
  const float* ST = side ? p.tab.S_V_T : p.tab.S_K_T;
  const long long w = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const long long per_side = (long long)p.B * p.Hkv * p.n_new;
  const long long W = (per_side + NV - 1) / NV;
  if (w >= W) return;
  const long long v0 = w * NV;
  int b[NV], h[NV], j[NV], t[NV];
  bool ok[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    ok[v] = v0 + v < per_side;
    split_vec(p, ok[v] ? v0 + v : v0, b[v], h[v], j[v], t[v]);
  }
  if constexpr (D == 128) {
    if (p.rotate[side] == 2) {
      encode_vectors_sq<Tin, NV>(p, side, b, h, j, t, ok);
      return;
    }
  }
  float res[NV][E];
  encode_vectors<D, Tin, NV>(p, side, b, h, j, t, ok, res);
  if (p.qjl[side]) {
#pragma unroll
    for (int v = 0; v < NV; ++v)
      if (ok[v]) sketch_signs_ffma<D>(p, side, b[v], h[v], t[v], res[v], ST);
  }
}

// AppendNV consecutive vectors of side side_base + blockIdx.y per warp (a QJL side at head dim
// above 128 takes its sketch on the FFMA path, S^T from L2).  Launched right after
// append_qjl_mma_kernel as its programmatic dependent (the other, non-QJL side), its blocks fill
// that kernel's last wave; each waits for it before exiting, so this grid's completion still
// implies the whole append's.  With release_early it lets its own dependent (a decode step's
// query preparation, which waits for it before exiting) launch at once.
template <int D, typename Tin>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) append_kernel(const AppendParams p) {
  if (p.release_early) asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  append_body<D, Tin>(p);
  if (p.wait_primary) asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

// ---- Large appends at head dim 128: four lanes per vector ----------------------------------
// A warp encodes eight vectors at once: lane l takes vector l / 4 and its coordinates
// [32 q, 32 q + 32), q = l % 4.  The rotation's first five butterfly stages run in registers and
// only the last two cross lanes (within the four lanes of a vector); the norm and residual sums
// reduce over those four lanes, and each lane's codes form whole words of the packed record.
// The stages run in the order and with the arithmetic of encode_vectors (butterflies over
// coordinate bits 0 .. 6), so the rotated values, and with them the codes, are the same.
constexpr int kQE = 32;        // coordinates per lane
constexpr int kQuadWarps = 4;  // warps per block of append_quad_kernel

__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(kFull, v, 1);
  return v + __shfl_xor_sync(kFull, v, 2);
}

// norm_compensated over the four lanes of a vector (their first lane's result in all four).
// EXACT_SQ: the squares are exact in fp32 (16-bit inputs: at most 22 significant bits), so the
// product error term, fma(x, x, -x x), is zero and is left out.
template <bool EXACT_SQ>
__device__ __forceinline__ float norm_compensated_quad(const float (&x)[kQE]) {
  float S = 0.f, C = 0.f;
#pragma unroll
  for (int i = 0; i < kQE; ++i) {
    const float pr = x[i] * x[i];
    const float pe = EXACT_SQ ? 0.f : fmaf(x[i], x[i], -pr);
    float s, e;
    two_sum(S, pr, s, e);
    S = s;
    C += e + pe;
  }
#pragma unroll
  for (int m = 2; m >= 1; m >>= 1) {
    const float So = __shfl_xor_sync(kFull, S, m);
    const float Co = __shfl_xor_sync(kFull, C, m);
    float s, e;
    two_sum(S, So, s, e);
    S = s;
    C = (C + Co) + e;
  }
  const int q0 = (threadIdx.x & 31) & ~3;
  S = __shfl_sync(kFull, S, q0);
  C = __shfl_sync(kFull, C, q0);
  if (S <= 0.f) return 0.f;
  const float r = sqrtf(S);
  const float res = fmaf(-r, r, S) + C;
  return r + res / (2.f * r);
}

// norm_split for a vector held by four lanes (see norm_split).  The shuffles run in every lane
// of the warp: a vector that needs the rescale makes the whole warp take that branch.
template <bool EXACT_SQ>
__device__ __forceinline__ float norm_split_quad(float (&x)[kQE], float& nu_work, float& pw) {
  const float nu = norm_compensated_quad<EXACT_SQ>(x);  // the same value in the vector's four lanes
  pw = 1.f;
  nu_work = nu;
  const bool fast = nu >= 0x1p-30f && nu < 0x1p50f;
  if (__all_sync(kFull, fast)) return nu;
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < kQE; ++i) m = fmaxf(m, fabsf(x[i]));
  m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
  m = fmaxf(m, __shfl_xor_sync(kFull, m, 2));
  const bool rescale = !fast && m > 0.f;
  const int e = rescale ? max(-126, min(126, ((__float_as_int(m) >> 23) & 0xFF) - 127)) : 0;
  if (rescale) {
    const float down = __int_as_float((127 - e) << 23);
#pragma unroll
    for (int i = 0; i < kQE; ++i) x[i] *= down;
  }
  const float nu2 = norm_compensated_quad<EXACT_SQ>(x);
  if (fast) return nu;
  if (!rescale) {
    nu_work = 0.f;
    return 0.f;
  }
  pw = __int_as_float((127 + e) << 23);
  nu_work = nu2;
  return nu2 * pw;
}

// Walsh-Hadamard butterflies of a vector held as 32 consecutive coordinates per lane by four
// lanes: stages over coordinate bits 0 .. 4 in registers, bits 5 and 6 by lane shuffles.
__device__ __forceinline__ void wht_quad(float (&x)[kQE]) {
#pragma unroll
  for (int hb = 1; hb < kQE; hb <<= 1) {
#pragma unroll
    for (int i = 0; i < kQE; ++i) {
      if ((i & hb) == 0) {
        const float a = x[i], b = x[i + hb];
        x[i] = a + b;
        x[i + hb] = a - b;
      }
    }
  }
  const int q = threadIdx.x & 3;
#pragma unroll
  for (int m = 1; m < 4; m <<= 1) {
    // the upper lane of the butterfly takes other - x, the lower x + other: one fma with a
    // factor of -1 or 1 gives the same rounded sum
    const float f = (q & m) ? -1.f : 1.f;
#pragma unroll
    for (int i = 0; i < kQE; ++i) {
      const float other = __shfl_xor_sync(kFull, x[i], m);
      x[i] = fmaf(f, x[i], other);
    }
  }
}

// One vector per four lanes through the write path ([TQ-KV] "Esquemas de Cuantización"):
// norm, rotation, scalar code, code and norm stores, and on a QJL side the residual (left in
// res) and its fp16 norm.  Sides without a HeadQ side code and not spectral.  An invalid vector
// (the same in its four lanes) is neither loaded nor stored and leaves res = 0.
template <typename Tin, int BITS>
__device__ __forceinline__ void encode_quad(const AppendParams& p, int side, int b, int h, int j, int t,
                                            bool valid, float (&res)[kQE]) {
  constexpr int D = 128;
  const int q = threadIdx.x & 3;
  constexpr int bits = BITS;
  const bool rotate = p.rotate[side] != 0;
  const float* sgn = side ? p.tab.v_sign : p.tab.k_sign;
  const float* cent = side ? p.tab.v_c : p.tab.k_c;
  const float* thr = side ? p.tab.v_t : p.tab.k_t;
  const Tin* base = reinterpret_cast<const Tin*>(side ? p.v : p.k);
  float x[kQE];
  if (valid) {
    load_row<kQE>(base + ((long long)(b * p.Hkv + h) * p.n_new + j) * D + kQE * q, x);
  } else {
#pragma unroll
    for (int i = 0; i < kQE; ++i) x[i] = 0.f;
  }
  float nw, pw;
  const float nu = norm_split_quad<!std::is_same<Tin, float>::value>(x, nw, pw);
#pragma unroll
  for (int i = 0; i < kQE; i += 4) {
    const float4 s4 = __ldg(reinterpret_cast<const float4*>(sgn + kQE * q + i));
    x[i] *= s4.x; x[i + 1] *= s4.y; x[i + 2] *= s4.z; x[i + 3] *= s4.w;
  }
  if (rotate) wht_quad(x);
  const float scale = rotate ? sqrtf((float)D) : 1.f;
  const float inv = nw > 0.f ? 1.f / (nw * scale) : 0.f;
  // the sign-magnitude code of encode_vectors: s = [y > 0], the magnitude from the upper
  // thresholds (-y >= t tested as nextup(-y) > t)
  const uint32_t halfL = 1u << (bits - 1);
  float tu[7];
#pragma unroll
  for (int k = 0; k < 7; ++k) tu[k] = __ldg(thr + halfL + k);
  uint32_t w4[4] = {0u, 0u, 0u, 0u}, w2[2] = {0u, 0u}, w1 = 0u;  // packed streams
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kQE; ++i) {
    const float y = x[i] * inv;
    const bool pos = y > 0.f;
    const float a = pos ? y : __int_as_float(__float_as_int(-y) + 1);
    // m = #{k : a > tu[k]} over the ascending tu[0..6] (unused slots 3e38), by binary search
    const bool c4 = a > tu[3];
    const bool c2 = a > (c4 ? tu[5] : tu[1]);
    const bool c1 = a > (c4 ? (c2 ? tu[6] : tu[4]) : (c2 ? tu[2] : tu[0]));
    const uint32_t m = (c4 ? 4u : 0u) | (c2 ? 2u : 0u) | (c1 ? 1u : 0u);
    const uint32_t sb = pos ? 1u : 0u;
    if constexpr (BITS == 4) w4[i >> 3] |= ((sb << 3) | m) << (4 * (i & 7));
    if constexpr (BITS == 2) w2[i >> 4] |= ((sb << 1) | m) << (2 * (i & 15));
    if constexpr (BITS == 3) w2[i >> 4] |= m << (2 * (i & 15));  // magnitudes; signs below
    if constexpr (BITS == 3 || BITS == 1) w1 |= sb << i;
    if (p.qjl[side]) {
      const uint32_t code = pos ? halfL + m : halfL - 1u - m;
      res[i] = valid ? y - __ldg(cent + code) : 0.f;
      ss = fmaf(res[i], res[i], ss);
    }
  }
  if (p.qjl[side]) ss = quad_sum(ss);  // (every lane: the shuffles take the whole warp)
  if (!valid) return;
  const Cache& C = p.cache;
  if (side == 0) {  // key records, token-major: this lane's coordinates are bytes [4 q W, ..)
    unsigned char* codes = C.ptr(tqi::R_K_CODES, b, h, t);
    if (bits == 4) {
      *reinterpret_cast<uint4*>(codes + 16 * q) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
    } else if (bits == 3) {
      *reinterpret_cast<uint2*>(codes + 8 * q) = make_uint2(w2[0], w2[1]);
      *reinterpret_cast<uint32_t*>(codes + D / 4 + 4 * q) = w1;
    } else if (bits == 2) {
      *reinterpret_cast<uint2*>(codes + 8 * q) = make_uint2(w2[0], w2[1]);
    } else {
      *reinterpret_cast<uint32_t*>(codes + 4 * q) = w1;
    }
  } else {  // value streams by 16-coordinate groups 2 q and 2 q + 1 at block position pos
    unsigned char* f = C.fieldp(tqi::R_V_CODES, b, h, t);
    const int pos = t & (tqi::kTileTokens - 1);
    const int g0 = 2 * q, g1 = 2 * q + 1;
    if (bits == 4) {
      *reinterpret_cast<uint2*>(f + g0 * 128 + pos * 8) = make_uint2(w4[0], w4[1]);
      *reinterpret_cast<uint2*>(f + g1 * 128 + pos * 8) = make_uint2(w4[2], w4[3]);
    } else if (bits == 3 || bits == 2) {
      *reinterpret_cast<uint32_t*>(f + g0 * 64 + pos * 4) = w2[0];
      *reinterpret_cast<uint32_t*>(f + g1 * 64 + pos * 4) = w2[1];
      if (bits == 3) {
        unsigned char* s1 = f + tqi::kTileTokens * (D / 4);
        *reinterpret_cast<unsigned short*>(s1 + g0 * 32 + pos * 2) = (unsigned short)w1;
        *reinterpret_cast<unsigned short*>(s1 + g1 * 32 + pos * 2) = (unsigned short)(w1 >> 16);
      }
    } else {
      *reinterpret_cast<unsigned short*>(f + g0 * 32 + pos * 2) = (unsigned short)w1;
      *reinterpret_cast<unsigned short*>(f + g1 * 32 + pos * 2) = (unsigned short)(w1 >> 16);
    }
  }
  if (q == 0) *reinterpret_cast<float*>(C.ptr(side ? tqi::R_V_NORM : tqi::R_K_NORM, b, h, t)) = nu;
  if (p.qjl[side] && q == 0)
    *reinterpret_cast<__half*>(C.ptr(side ? tqi::R_V_RHO : tqi::R_K_RHO, b, h, t)) = __float2half_rn(sqrtf(ss));
}

template <typename Tin>
__device__ __forceinline__ void encode_quad_bits(const AppendParams& p, int side, int b, int h, int j, int t,
                                                 bool valid, float (&res)[kQE]) {
  switch (p.bits[side]) {
    case 4: encode_quad<Tin, 4>(p, side, b, h, j, t, valid, res); break;
    case 3: encode_quad<Tin, 3>(p, side, b, h, j, t, valid, res); break;
    case 2: encode_quad<Tin, 2>(p, side, b, h, j, t, valid, res); break;
    default: encode_quad<Tin, 1>(p, side, b, h, j, t, valid, res); break;
  }
}

// Sides of a large append at head dim 128 that carry no QJL sketch (a QJL side goes to
// append_qjl_mma_kernel): 32 vectors per block of 4 warps, four lanes per vector; seven blocks
// per SM (at most 73 registers) put a 4096-token chunk of eight heads in one wave.  As the
// programmatic dependent of append_qjl_mma_kernel (wait_primary) it waits for that kernel
// before exiting, as append_kernel does, and release_early has the same meaning.
template <typename Tin>
__global__ void __launch_bounds__(kQuadWarps * 32, 7) append_quad_kernel(const AppendParams p) {
  if (p.release_early) asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int side = p.side_base + (int)blockIdx.y;
  if (!(p.qjl[side] && p.qjl_mma)) {
    const long long per_side = (long long)p.B * p.Hkv * p.n_new;
    const long long v = (long long)blockIdx.x * (kQuadWarps * 8) + (threadIdx.x >> 2);
    const bool ok = v < per_side;
    int b, h, j, t;
    split_vec(p, ok ? v : 0, b, h, j, t);
    float res[kQE];
    encode_quad_bits<Tin>(p, side, b, h, j, t, ok, res);
  }
  if (p.wait_primary) asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

constexpr uint32_t kStageWaitLimit = 1u << 20;  // polls of a table copy's mbarrier

// QJL sides at head dim 128: a block of kQjlWarps warps takes VEC vectors of one side (64 for
// large appends, 16 for small ones).  (1) The vectors go through the codec -- four lanes per
// vector for VEC = 64, a warp per vector (two at a time) for VEC = 16, where the latency of one
// vector matters more than the throughput -- and r, scaled by 256, is kept in shared memory as
// two fp16 terms (hi, lo = fp16(256 r - hi)).  (2) S r for the block is a [VEC x 128] x
// [128 x 128] product on the tensor cores, S split the same way and bulk-copied from the table
// blob once per block.  VEC = 64: tcgen05, D[128 sketch rows x 64 vectors] = S R^T accumulated
// in tensor memory from hi*hi, hi*lo and lo*hi (24 MMAs of K = 16), one ballot per vector column
// for 32 of its sign bits.  VEC = 16: mma.sync m16n8k16 with ldmatrix fragments, hi*hi in one
// fp32 chain and hi*lo + lo*hi in another, warp ballots for the sign bytes.
// (3) Every product with |S r| below kSignRecheck is listed and taken again as an fp32 FFMA dot
// product of the row of S with hi + lo (a warp per listed product), so decisions near zero have
// fp32 accuracy; the sign bits are patched.  (If more than kRecheckMax products of a block are
// listed, a vector whose product did not fit gets all its signs from the FFMA path instead.)
// (4) The sign records are stored.
constexpr int kQjlWarps = 8;
constexpr int kQjlBlockVec = 64;        // vectors per block of a large append: 4 MMA row tiles of 16
constexpr int kQjlSmallVec = 16;        // vectors per block of a small append: one row tile
constexpr float kQjlUp = 256.f;         // residual scale before the fp16 split
constexpr float kSignRecheck = 2e-5f;   // in units of S r
constexpr long long kQjlMmaMin = 256;   // vectors per side from which 64-vector blocks are used
constexpr int kRecheckMax = 256;        // listed near-zero products per block

// Operands in 8 x 8 fp16 core matrices (the tensor cores' no-swizzle K-major layout): element
// (row r, coordinate k) of a 128-coordinate operand at byte cm_off(r, k).
__host__ __device__ constexpr int cm_off(int r, int k) { return (r >> 3) * 2048 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2; }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// bits 0..3 of n to bits 0, 2, 4, 6
__device__ __forceinline__ uint32_t spread4(uint32_t n) {
  n = (n | (n << 2)) & 0x33u;
  return (n | (n << 1)) & 0x55u;
}

template <int VEC>
struct QjlSmem {
  static constexpr int table = 128 * 128 * 2;               // one fp16 table (hi or lo): S, 128 rows
  static constexpr int resid = VEC * 128 * 2;               // one fp16 residual array (hi or lo): VEC rows
  static constexpr int signs = VEC * 16;                    // sign records of the block
  static constexpr int flags = VEC * 4;
  static constexpr int list = kRecheckMax * 4 + 16;         // listed products + their count
  static constexpr int bytes = 2 * table + 2 * resid + signs + flags + list;
};

// BITS: the code width of the QJL side(s) as a compile-time constant (one encode variant in the
// kernel's code), or 0 when two QJL sides differ (chosen at run time).  HQ: the key side carries
// a HeadQ side code (its vectors take encode_vectors); only that variant holds that code.
template <typename Tin, int BITS, bool HQ, int VEC = kQjlBlockVec>
__global__ void __launch_bounds__(kQjlWarps * 32) append_qjl_mma_kernel(const AppendParams p) {
  constexpr int D = 128, E = 4;
  using QjlSmem = tqd::QjlSmem<VEC>;
  static_assert(VEC == kQjlBlockVec || VEC == kQjlSmallVec, "block sizes");
  constexpr uint32_t kCols = VEC < 32 ? 32 : VEC;  // tensor-memory columns: one per vector
  extern __shared__ __align__(16) unsigned char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int side = (p.qjl[0] && p.qjl[1]) ? (int)blockIdx.y : (p.qjl[0] ? 0 : 1);
  __half* Shi = reinterpret_cast<__half*>(smem);
  __half* Slo = reinterpret_cast<__half*>(smem + QjlSmem::table);
  __half* Rhi = reinterpret_cast<__half*>(smem + 2 * QjlSmem::table);
  __half* Rlo = reinterpret_cast<__half*>(smem + 2 * QjlSmem::table + QjlSmem::resid);
  unsigned char* sg = smem + 2 * QjlSmem::table + 2 * QjlSmem::resid;  // [VEC][16] sign bytes
  uint32_t* unc = reinterpret_cast<uint32_t*>(sg + QjlSmem::signs);    // [VEC] whole-vector recheck flags
  uint32_t* re_list = unc + VEC;                                       // [kRecheckMax] (v << 7) | row
  uint32_t* re_cnt = re_list + kRecheckMax;
  // the other side's append_kernel, launched next as a programmatic dependent, may start as soon
  // as every block of this grid is running (it fills the last wave)
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const long long per_side = (long long)p.B * p.Hkv * p.n_new;
  const long long v0 = (long long)blockIdx.x * VEC;

  // ---- (0) S as fp16 hi / lo rows: the table blob holds them in this layout, so bulk copies
  // bring them in while the vectors are encoded; cleared flags
  static_assert(2 * QjlSmem::table == (int)tqi::kSketchH16Bytes, "table layout");
  __shared__ __align__(8) unsigned long long s_bar, s_mma;
  __shared__ uint32_t s_tmem;
  const uint32_t sbar = (uint32_t)__cvta_generic_to_shared(&s_bar), smma = (uint32_t)__cvta_generic_to_shared(&s_mma);
  // S r: [128 sketch rows][VEC] in tensor memory (64-vector blocks)
  if (VEC == kQjlBlockVec && warp == 0) tc_alloc((uint32_t)__cvta_generic_to_shared(&s_tmem), kCols);
  if (threadIdx.x == 0) {
    constexpr uint32_t kPiece = (uint32_t)tqi::kSketchH16Bytes / 4;
    mbar_init(sbar, 1);
    mbar_init(smma, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(sbar, (uint32_t)tqi::kSketchH16Bytes);
    const uint32_t dst = (uint32_t)__cvta_generic_to_shared(smem);
#pragma unroll
    for (uint32_t k = 0; k < 4; ++k) bulk_g2s(dst + k * kPiece, p.tab.S_h16[side] + k * kPiece, kPiece, sbar);
  }
  for (int i = threadIdx.x; i < VEC; i += blockDim.x) unc[i] = 0u;
  if (threadIdx.x == 0) *re_cnt = 0u;

  // ---- (1) the block's vectors through the codec; residuals to shared memory.  Four lanes per
  // vector (encode_quad), eight vectors per warp; a key side with a HeadQ side code, and every
  // side of a small append, takes encode_vectors, two vectors at a time per warp.
  static_assert(kQjlBlockVec == kQjlWarps * 8, "eight vectors per warp");
  if (VEC == kQjlBlockVec && !(HQ && side == 0)) {
    const int vl = warp * 8 + (lane >> 2), q = lane & 3;
    const bool okq = v0 + vl < per_side;
    int bq, hq, jq, tq;
    split_vec(p, okq ? v0 + vl : v0, bq, hq, jq, tq);
    float rq[kQE];
    if constexpr (BITS == 0) encode_quad_bits<Tin>(p, side, bq, hq, jq, tq, okq, rq);
    else encode_quad<Tin, BITS>(p, side, bq, hq, jq, tq, okq, rq);
#pragma unroll
    for (int i = 0; i < kQE; i += 8) {
      __half hi[8], lo[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float x = rq[i + e] * kQjlUp;
        hi[e] = __float2half_rn(x);
        lo[e] = __float2half_rn(x - __half2float(hi[e]));
      }
      *reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(Rhi) + cm_off(vl, kQE * q + i)) =
          *reinterpret_cast<const uint4*>(hi);
      *reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(Rlo) + cm_off(vl, kQE * q + i)) =
          *reinterpret_cast<const uint4*>(lo);
    }
  } else {
  constexpr int NV = 2;
  for (int vb = warp * (VEC / kQjlWarps); vb < (warp + 1) * (VEC / kQjlWarps); vb += NV) {
    int b[NV], h[NV], j[NV], t[NV];
    bool ok[NV];
#pragma unroll
    for (int u = 0; u < NV; ++u) {
      ok[u] = v0 + vb + u < per_side;
      split_vec(p, ok[u] ? v0 + vb + u : v0, b[u], h[u], j[u], t[u]);
    }
    float res[NV][E];
    encode_vectors<D, Tin, NV>(p, side, b, h, j, t, ok, res);
#pragma unroll
    for (int u = 0; u < NV; ++u) {
      __half hi[E], lo[E];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float x = res[u][e] * kQjlUp;
        hi[e] = __float2half_rn(x);
        lo[e] = __float2half_rn(x - __half2float(hi[e]));
      }
      *reinterpret_cast<uint2*>(reinterpret_cast<unsigned char*>(Rhi) + cm_off(vb + u, lane * E)) =
          *reinterpret_cast<const uint2*>(hi);
      *reinterpret_cast<uint2*>(reinterpret_cast<unsigned char*>(Rlo) + cm_off(vb + u, lane * E)) =
          *reinterpret_cast<const uint2*>(lo);
    }
  }
  }
  __syncthreads();  // residuals in place; the barrier's initialization is visible
  if (!mbar_wait(sbar, 0, kStageWaitLimit)) {
    // the copy did not arrive within the poll limit: convert the fp32 table here (the same values)
    const float* S = side ? p.tab.S_V : p.tab.S_K;  // [m][d], S[i][j]
    for (int idx = threadIdx.x * 4; idx < D * D; idx += blockDim.x * 4) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(S + idx));
      const int i = idx / D, jj = idx % D;
      const float xs[4] = {x.x, x.y, x.z, x.w};
      __half hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        hi[e] = __float2half_rn(xs[e]);
        lo[e] = __float2half_rn(xs[e] - __half2float(hi[e]));
      }
      *reinterpret_cast<uint2*>(reinterpret_cast<unsigned char*>(Shi) + cm_off(i, jj)) = *reinterpret_cast<const uint2*>(hi);
      *reinterpret_cast<uint2*>(reinterpret_cast<unsigned char*>(Slo) + cm_off(i, jj)) = *reinterpret_cast<const uint2*>(lo);
    }
  }
  __syncthreads();

  // ---- (2) S r on the tensor cores, transposed: D[128 sketch rows x VEC vectors] = S R^T, with
  // D in tensor memory (row i in lane i, vector v in column v).  A = S (hi, lo) and B = the
  // residuals (hi, lo) are K-major core-matrix operands in shared memory: 8 k-steps of 16
  // coordinates, passes hi.hi, hi.lo, lo.hi into one fp32 accumulator.
  const float thr = kSignRecheck * kQjlUp;
  // a product too close to zero goes on the block's list (or, past its end, flags the vector)
  auto near_zero = [&](float sv, int v, int row) {
    if (fabsf(sv) < thr && v0 + v < per_side) {
      const uint32_t k = atomicAdd(re_cnt, 1u);
      if (k < (uint32_t)kRecheckMax) re_list[k] = ((uint32_t)v << 7) | (uint32_t)row;
      else atomicOr(unc + v, 1u);
    }
  };
  if constexpr (VEC == kQjlBlockVec) {
    tc_fence_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    if (threadIdx.x == 0) {
      const uint32_t sh = (uint32_t)__cvta_generic_to_shared(Shi), sl = (uint32_t)__cvta_generic_to_shared(Slo);
      const uint32_t rh = (uint32_t)__cvta_generic_to_shared(Rhi), rl = (uint32_t)__cvta_generic_to_shared(Rlo);
      constexpr uint32_t id = tc_idesc_f16(128, VEC);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        tc_mma_f16(tmem, tc_sdesc(sh + 256 * kk, 128, 2048), tc_sdesc(rh + 256 * kk, 128, 2048), id, kk > 0 ? 1u : 0u);
        tc_mma_f16(tmem, tc_sdesc(sh + 256 * kk, 128, 2048), tc_sdesc(rl + 256 * kk, 128, 2048), id, 1u);
        tc_mma_f16(tmem, tc_sdesc(sl + 256 * kk, 128, 2048), tc_sdesc(rh + 256 * kk, 128, 2048), id, 1u);
      }
      tc_commit(smma);
    }
    // signs: warp w reads lanes 32 (w % 4) .. + 31 (sketch rows) of the columns of vectors
    // 32 (w / 4) .. + 31; a ballot per vector gives 32 sign bits of its record (bit k of word q =
    // sketch row 32 q + k)
    // warp-uniform: the tensor-memory load below is a warp-collective instruction
    const bool mma_ok = __all_sync(kFull, mbar_wait(smma, 0, kStageWaitLimit));
    tc_fence_after();
    const int q = warp & 3, vh = warp >> 2;
    uint32_t* sgw = reinterpret_cast<uint32_t*>(sg);
    if (mma_ok) {
      float val[32];
      tc_ld32(tmem + ((uint32_t)(32 * q) << 16) + 32 * vh, val);
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const int v = 32 * vh + c;
        const uint32_t word = __ballot_sync(kFull, val[c] >= 0.f);
        if (lane == c) sgw[v * 4 + q] = word;
        if (__any_sync(kFull, fabsf(val[c]) < thr)) near_zero(val[c], v, 32 * q + lane);
      }
    } else {
      // the product did not complete within the poll limit: every vector takes the FFMA path
      for (int v = threadIdx.x; v < VEC; v += blockDim.x) unc[v] = 1u;
    }
  } else {
  // 16-vector blocks (small appends): warp-level MMAs, whose latency is lower than a tensor-memory
  // round trip at this size.  Warp w takes sketch rows 16 w .. 16 w + 15 (two n-tiles of 8) for
  // the block's 16 vectors (one row tile); fragments by ldmatrix from the core matrices, hi*hi in
  // one fp32 chain and hi*lo + lo*hi in another
  const uint32_t rhi_s = (uint32_t)__cvta_generic_to_shared(Rhi), rlo_s = (uint32_t)__cvta_generic_to_shared(Rlo);
  const uint32_t shi_s = (uint32_t)__cvta_generic_to_shared(Shi), slo_s = (uint32_t)__cvta_generic_to_shared(Slo);
  const int mi = lane >> 3, mr = lane & 7;
  uint32_t ah[8][4], al[8][4];
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t off = (uint32_t)cm_off(mr + 8 * (mi & 1), 16 * ks + 8 * (mi >> 1));
    ldsm_x4(rhi_s + off, ah[ks][0], ah[ks][1], ah[ks][2], ah[ks][3]);
    ldsm_x4(rlo_s + off, al[ks][0], al[ks][1], al[ks][2], al[ks][3]);
  }
#pragma unroll 1
  for (int nt = 2 * warp; nt < 2 * warp + 2; ++nt) {
    float c[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kp = 0; kp < 4; ++kp) {
      const uint32_t off = (uint32_t)cm_off(8 * nt + mr, 16 * (2 * kp + (mi >> 1)) + 8 * (mi & 1));
      uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
      ldsm_x4(shi_s + off, h0, h1, h2, h3);
      ldsm_x4(slo_s + off, l0, l1, l2, l3);
      const int k0 = 2 * kp, k1 = 2 * kp + 1;
      mma16816(c, ah[k0][0], ah[k0][1], ah[k0][2], ah[k0][3], h0, h1);
      mma16816(e, ah[k0][0], ah[k0][1], ah[k0][2], ah[k0][3], l0, l1);
      mma16816(e, al[k0][0], al[k0][1], al[k0][2], al[k0][3], h0, h1);
      mma16816(c, ah[k1][0], ah[k1][1], ah[k1][2], ah[k1][3], h2, h3);
      mma16816(e, ah[k1][0], ah[k1][1], ah[k1][2], ah[k1][3], l2, l3);
      mma16816(e, al[k1][0], al[k1][1], al[k1][2], al[k1][3], h2, h3);
    }
    // accumulator (row g, columns 2t, 2t + 1) = vector g, sketch rows 8 nt + 2t (+1); rows g + 8
    const float s0 = c[0] + e[0], s1 = c[1] + e[1], s2 = c[2] + e[2], s3 = c[3] + e[3];
    const uint32_t b0 = __ballot_sync(kFull, s0 >= 0.f), b1 = __ballot_sync(kFull, s1 >= 0.f);
    const uint32_t b2 = __ballot_sync(kFull, s2 >= 0.f), b3 = __ballot_sync(kFull, s3 >= 0.f);
    if (__any_sync(kFull, fminf(fminf(fabsf(s0), fabsf(s1)), fminf(fabsf(s2), fabsf(s3))) < thr)) {
      const int vg = lane >> 2, rw = 8 * nt + 2 * (lane & 3);
      near_zero(s0, vg, rw);
      near_zero(s1, vg, rw + 1);
      near_zero(s2, vg + 8, rw);
      near_zero(s3, vg + 8, rw + 1);
    }
    if (lane < 16) {  // byte nt of vector lane: bit 2t from b0 / b2, bit 2t + 1 from b1 / b3
      const int sh = 4 * (lane & 7);
      const uint32_t lo = ((lane < 8 ? b0 : b2) >> sh) & 0xFu, hi = ((lane < 8 ? b1 : b3) >> sh) & 0xFu;
      sg[lane * 16 + nt] = (unsigned char)(spread4(lo) | (spread4(hi) << 1));
    }
  }
  }
  __syncthreads();

  // ---- (3) listed products again in fp32: row `row` of S (fp32, L2) against hi + lo of the
  // vector's scaled residual, a warp per product; the sign bit is patched in place
  {
    const uint32_t nre = min(*re_cnt, (uint32_t)kRecheckMax);
    const float* S = side ? p.tab.S_V : p.tab.S_K;  // [m][d], S[i][j]
    for (uint32_t k = warp; k < nre; k += kQjlWarps) {
      const uint32_t e = re_list[k];
      const int v = (int)(e >> 7), row = (int)(e & 127u);
      if (unc[v]) continue;  // the whole vector is taken again below
      const float4 s4 = __ldg(reinterpret_cast<const float4*>(S + row * D + 4 * lane));
      const uint2 h4 = *reinterpret_cast<const uint2*>(reinterpret_cast<const unsigned char*>(Rhi) + cm_off(v, 4 * lane));
      const uint2 l4 = *reinterpret_cast<const uint2*>(reinterpret_cast<const unsigned char*>(Rlo) + cm_off(v, 4 * lane));
      const float2 h01 = __half22float2(*reinterpret_cast<const __half2*>(&h4.x));
      const float2 h23 = __half22float2(*reinterpret_cast<const __half2*>(&h4.y));
      const float2 l01 = __half22float2(*reinterpret_cast<const __half2*>(&l4.x));
      const float2 l23 = __half22float2(*reinterpret_cast<const __half2*>(&l4.y));
      float acc = s4.x * (h01.x + l01.x);
      acc = fmaf(s4.y, h01.y + l01.y, acc);
      acc = fmaf(s4.z, h23.x + l23.x, acc);
      acc = fmaf(s4.w, h23.y + l23.y, acc);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
      if (lane == 0) {
        const int byte = v * 16 + (row >> 3);
        const uint32_t bit = 1u << (8 * (byte & 3) + (row & 7));
        uint32_t* word = reinterpret_cast<uint32_t*>(sg) + (byte >> 2);
        if (acc >= 0.f) atomicOr(word, bit);
        else atomicAnd(word, ~bit);
      }
    }
  }
  __syncthreads();

  // ---- (4) sign records of the valid vectors, one 32-bit word per thread
  const Cache& C = p.cache;
  for (int w = threadIdx.x; w < VEC * 4; w += blockDim.x) {
    const int v = w >> 2;
    const long long vec = v0 + v;
    if (vec < per_side) {
      int b, h, j, t;
      split_vec(p, vec, b, h, j, t);
      const uint32_t word = reinterpret_cast<const uint32_t*>(sg)[w];  // signs of rows 32 (w & 3) ..
      if (side == 0) {
        reinterpret_cast<uint32_t*>(C.ptr(tqi::R_K_SIGNS, b, h, t))[w & 3] = word;
      } else {  // two 16-row groups of the value side's sign stream
        unsigned char* f = C.fieldp(tqi::R_V_SIGNS, b, h, t);
        const int pos = t & (tqi::kTileTokens - 1);
        *reinterpret_cast<unsigned short*>(f + grouped_byte(4 * (w & 3), pos, 1)) = (unsigned short)word;
        *reinterpret_cast<unsigned short*>(f + grouped_byte(4 * (w & 3) + 2, pos, 1)) = (unsigned short)(word >> 16);
      }
    }
  }
  __syncthreads();

  // ---- (5) vectors whose near-zero products overflowed the list: every sign again from the
  // FFMA path (only when a block has more than kRecheckMax of them)
  for (int v = warp * (VEC / kQjlWarps); v < (warp + 1) * (VEC / kQjlWarps); ++v) {
    const long long vec = v0 + v;
    if (vec >= per_side || !unc[v]) continue;
    int b, h, j, t;
    split_vec(p, vec, b, h, j, t);
    float res[E];
    encode_vector<D, Tin>(p, side, b, h, j, t, res);
    sketch_signs_ffma<D>(p, side, b, h, t, res, side ? p.tab.S_V_T : p.tab.S_K_T);
  }
  if constexpr (VEC == kQjlBlockVec) {
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
      // a product still in flight after the poll limit gets one more bounded wait before its
      // accumulator is freed (returns at once when it has completed)
      mbar_wait(smma, 0, kStageWaitLimit);
      tc_fence_after();
      tc_dealloc(s_tmem, kCols);
    }
  }
}

// SQU-KV tables in storage order: E_st[h][i][c] = E[h][i][rank(c)], its transpose, and
// s_st[h][c] = s[h][rank(c)] (a permutation: no value changes).
__global__ void __launch_bounds__(256) spectral_basis_kernel(const float* E, const float* sv, float* E_st,
                                                             float* ET_st, float* s_st, int side, int H, int D) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)H * D * D) return;
  const int c = (int)(idx % D), i = (int)((idx / D) % D), h = (int)(idx / ((long long)D * D));
  const int r = sq_rank_of_coord(side, c);
  const float e = E[((long long)h * D + i) * D + r];
  E_st[((long long)h * D + i) * D + c] = e;
  ET_st[((long long)h * D + c) * D + i] = e;
  if (i == 0) s_st[(long long)h * D + c] = sv[(long long)h * D + r];
}

// R_K U for every column of every KV head's basis: U [H][d][r] -> U_rot [H][d][r].
template <int D>
__global__ void __launch_bounds__(256) rotate_basis_kernel(const float* U, float* U_rot,
                                                           const float* sign, int H, int rank) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int col = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (col >= H * rank) return;
  const int h = col / rank, k = col % rank;
  float x[E];
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int j = lane * E + i;
    x[i] = U[((long long)h * D + j) * rank + k] * __ldg(sign + j);
  }
  wht_warp<E>(x);
  const float rs = 1.f / sqrtf((float)D);
#pragma unroll
  for (int i = 0; i < E; ++i) U_rot[((long long)h * D + lane * E + i) * rank + k] = x[i] * rs;
}

struct DequantParams {
  Tables tab;
  Cache cache;
  float* out[2];
  int b, kvh, t0, n, m;
  int bits[2], rotate[2], qjl[2];
  int headq_rank;
  float qjl_scale;
};

// x_hat = R^T (nu * (C[c] + sqrt(pi/2)/m * rho * S^T (2 sigma - 1)) + U_rot z_hat)
template <int D>
__global__ void __launch_bounds__(256) dequantize_kernel(const DequantParams p) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int w = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (w >= 2 * p.n) return;
  const int side = w >= p.n ? 1 : 0;
  const int t = p.t0 + (side ? w - p.n : w);
  const Cache& C = p.cache;
  const int bits = p.bits[side];
  // key records are whole; value streams are stored by coordinate groups at block position pos
  const int pos = side ? (t & (tqi::kTileTokens - 1)) : -1;
  const unsigned char* codes = side ? C.fieldp(tqi::R_V_CODES, p.b, p.kvh, t) : C.ptr(tqi::R_K_CODES, p.b, p.kvh, t);
  const int second = side ? tqi::kTileTokens * (D / 4) : D / 4;  // start of a 3-bit code's 1-bit stream
  const float* cent = side ? p.tab.v_c : p.tab.k_c;
  if (p.rotate[side] == 2) {
    if constexpr (D == 128) {
      // SQU-KV: z_hat_c = +-M[m] (modeled) or +-c1 (floor), x_hat = nu E (s z_hat)
      const bool modeled = sq_modeled(side, E * lane);
      uint32_t sg[E];
      load_stream<E, 1>(codes + (side ? tqi::kTileTokens * 16 : 16), sg, pos);
      uint32_t mag = 0;
      if (modeled) {
        const int byte = side ? 2 * (lane / 4) : 4 * (lane / 8) + 2 * (lane % 8);
        const unsigned char* mp = side ? codes + grouped_byte((unsigned)byte, (unsigned)pos, 1) : codes + byte;
        mag = mp[0] | ((uint32_t)mp[side ? 1 : 1] << 8);
      }
      const float c1 = __ldg(p.tab.sq_c1 + side);
      const float nu = *reinterpret_cast<const float*>(C.ptr(side ? tqi::R_V_NORM : tqi::R_K_NORM, p.b, p.kvh, t));
      const float4 s4 = __ldg(reinterpret_cast<const float4*>(p.tab.sq_s[side] + (long long)p.kvh * D + lane * E));
      const float sc[E] = {s4.x, s4.y, s4.z, s4.w};
      float a[E];
#pragma unroll
      for (int i = 0; i < E; ++i) {
        const float mg = modeled ? __ldg(cent + 8 + ((mag >> (4 * i)) & 7u)) : c1;
        a[i] = nu * sc[i] * (sg[i] ? mg : -mg);
      }
      float o[E] = {0.f, 0.f, 0.f, 0.f};
      const float* ET = p.tab.sq_ET[side] + (long long)p.kvh * D * D + lane * E;
      for (int sl = 0; sl < 32; ++sl) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float ac = __shfl_sync(kFull, a[e], sl);
          const float4 er = __ldg(reinterpret_cast<const float4*>(ET + (E * sl + e) * D));
          o[0] = fmaf(er.x, ac, o[0]); o[1] = fmaf(er.y, ac, o[1]);
          o[2] = fmaf(er.z, ac, o[2]); o[3] = fmaf(er.w, ac, o[3]);
        }
      }
      float* out = p.out[side] + (long long)(t - p.t0) * D + lane * E;
#pragma unroll
      for (int e = 0; e < E; ++e) out[e] = o[e];
    }
    return;
  }
  const uint32_t halfL = 1u << (bits - 1);
  uint32_t sym[E], sgn[E];
  if (bits == 4) {
    load_stream<E, 4>(codes, sym, pos);
#pragma unroll
    for (int i = 0; i < E; ++i) { sgn[i] = sym[i] >> 3; sym[i] &= 7u; }
  } else if (bits == 3) {
    load_stream<E, 2>(codes, sym, pos);
    load_stream<E, 1>(codes + second, sgn, pos);
  } else if (bits == 2) {
    load_stream<E, 2>(codes, sym, pos);
#pragma unroll
    for (int i = 0; i < E; ++i) { sgn[i] = sym[i] >> 1; sym[i] &= 1u; }
  } else {
    load_stream<E, 1>(codes, sgn, pos);
#pragma unroll
    for (int i = 0; i < E; ++i) sym[i] = 0;
  }
  float yh[E];
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const uint32_t c = sgn[i] ? halfL + sym[i] : halfL - 1u - sym[i];
    yh[i] = __ldg(cent + c);
  }
  const float nu = *reinterpret_cast<const float*>(C.ptr(side ? tqi::R_V_NORM : tqi::R_K_NORM, p.b, p.kvh, t));
  if (p.qjl[side]) {
    const unsigned char* sg = side ? C.fieldp(tqi::R_V_SIGNS, p.b, p.kvh, t) : C.ptr(tqi::R_K_SIGNS, p.b, p.kvh, t);
    const float rho = __half2float(*reinterpret_cast<const __half*>(C.ptr(side ? tqi::R_V_RHO : tqi::R_K_RHO, p.b, p.kvh, t)));
    const float* S = side ? p.tab.S_V : p.tab.S_K;  // [m][d]
    float acc[E];
#pragma unroll
    for (int i = 0; i < E; ++i) acc[i] = 0.f;
    for (int i = 0; i < p.m; ++i) {
      const unsigned char byte = side ? sg[grouped_byte((unsigned)i >> 3, (unsigned)pos, 1)] : sg[i >> 3];
      const float pm = ((byte >> (i & 7)) & 1u) ? 1.f : -1.f;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(__ldg(S + (long long)i * D + lane * E + e), pm, acc[e]);
    }
#pragma unroll
    for (int e = 0; e < E; ++e) yh[e] = fmaf(p.qjl_scale * rho, acc[e], yh[e]);
  }
  float wv[E];
#pragma unroll
  for (int e = 0; e < E; ++e) wv[e] = nu * yh[e];
  if (side == 0 && p.headq_rank) {
    const uint2 sw = *reinterpret_cast<const uint2*>(C.ptr(tqi::R_K_SIDE, p.b, p.kvh, t));
    const float sc = __half2float(*reinterpret_cast<const __half*>(C.ptr(tqi::R_K_SIDE_SCALE, p.b, p.kvh, t)));
    const float* Ur = p.tab.U_rot + (long long)p.kvh * D * 16;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint32_t word = k < 8 ? sw.x : sw.y;
      int zk = (int)((word >> (4 * (k & 7))) & 0xFu);
      zk = zk >= 8 ? zk - 16 : zk;
      const float zh = sc * (float)zk;
#pragma unroll
      for (int e = 0; e < E; ++e) wv[e] = fmaf(__ldg(Ur + (lane * E + e) * 16 + k), zh, wv[e]);
    }
  }
  if (p.rotate[side]) {
    wht_warp<E>(wv);
    const float* sg = side ? p.tab.v_sign : p.tab.k_sign;
    const float rs = 1.f / sqrtf((float)D);
#pragma unroll
    for (int e = 0; e < E; ++e) wv[e] = wv[e] * rs * __ldg(sg + lane * E + e);
  }
  float* o = p.out[side] + (long long)(t - p.t0) * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = wv[e];
}

template <typename F>
tq_status dispatch_d(int d, F&& f) {
  switch (d) {
    case 128: f(std::integral_constant<int, 128>{}); return TQ_OK;
    case 256: f(std::integral_constant<int, 256>{}); return TQ_OK;
    case 512: f(std::integral_constant<int, 512>{}); return TQ_OK;
    case 1024: f(std::integral_constant<int, 1024>{}); return TQ_OK;
  }
  return TQ_ERR_UNSUPPORTED;
}

tq_status launch_status(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    tqi::set_error(std::string(what) + ": " + cudaGetErrorString(e));
    return TQ_ERR_CUDA;
  }
  return TQ_OK;
}

}  // namespace
}  // namespace tqd

namespace tqi {

// Paged pool (tq_quantize_append_paged): block table, device start positions, error word.
struct PagedAppend {
  const tq_page_table* pt;
  const int32_t* dev_start;
  int32_t* dev_error;
};

static tq_status append_impl(const tq_context* ctx, void* cache, const void* k, const void* v,
                             tq_dtype dtype, int n_new, const int32_t* start, const PagedAppend* pg,
                             Stream stream, bool release_early = false) {
  using namespace tqd;
  AppendParams p;
  p.tab = make_tables(ctx);
  p.cache = pg ? make_paged_cache(ctx, cache, *pg->pt, pg->dev_error) : make_cache(ctx, cache);
  p.dev_start = pg ? pg->dev_start : nullptr;
  p.k = k;
  p.v = v;
  p.B = ctx->cfg.batch;
  p.Hkv = ctx->cfg.num_kv_heads;
  p.n_new = n_new;
  p.m = ctx->m;
  p.bits[0] = ctx->cfg.k.bits; p.rotate[0] = ctx->cfg.k.rotate; p.qjl[0] = ctx->cfg.k.qjl;
  p.bits[1] = ctx->cfg.v.bits; p.rotate[1] = ctx->cfg.v.rotate; p.qjl[1] = ctx->cfg.v.qjl;
  p.headq_rank = ctx->cfg.headq_rank;
  p.release_early = release_early ? 1 : 0;  // (append_qjl_mma_kernel always releases at its start)
  for (int b = 0; b < TQ_MAX_BATCH; ++b) p.start[b] = (!pg && b < ctx->cfg.batch) ? start[b] : 0;
  const int nv = ctx->cfg.head_dim == 128 ? AppendNV<128>::value : 1;
  const long long per_side = (long long)p.B * p.Hkv * n_new;
  const long long blocks = ((per_side + nv - 1) / nv + kWarpsPerBlock - 1) / kWarpsPerBlock;  // per side
  if (per_side >= 0x7fffffffLL) { set_error("append too large"); return TQ_ERR_INVALID_ARG; }
  fast_div_magic((uint32_t)std::max(n_new, 1), p.div_n_mul, p.div_n_shift);
  fast_div_magic((uint32_t)p.Hkv, p.div_h_mul, p.div_h_shift);
  const int nq = (p.qjl[0] ? 1 : 0) + (p.qjl[1] ? 1 : 0);
  p.qjl_mma = (ctx->cfg.head_dim == 128 && nq > 0) ? 1 : 0;
  const cudaStream_t cs = (cudaStream_t)stream;
  // An append with a QJL side at head dim 128: the tensor-core sketch kernel takes the QJL
  // side(s) first (64-vector blocks for large appends, 16-vector blocks for small ones), and the
  // other side (if any) follows as its programmatic dependent launch.
  if (p.qjl_mma) {
    const bool small = per_side < kQjlMmaMin;
    const int vec = small ? kQjlSmallVec : kQjlBlockVec;
    const int qbytes = small ? QjlSmem<kQjlSmallVec>::bytes : QjlSmem<kQjlBlockVec>::bytes;
    const dim3 qgrid((unsigned)((per_side + vec - 1) / vec), (unsigned)nq), qblock(kQjlWarps * 32);
    auto goq = [&](auto kern) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, qbytes);
      if (e == cudaSuccess) kern<<<qgrid, qblock, qbytes, cs>>>(p);
      return e;
    };
    // the QJL sides' code width as a template constant (0: two QJL sides of different widths)
    const int qb = (p.qjl[0] && p.qjl[1] && p.bits[0] != p.bits[1]) ? 0 : p.bits[p.qjl[0] ? 0 : 1];
    const bool hq = p.headq_rank && p.qjl[0];
    auto by_bits = [&](auto tin) {
      using T = decltype(tin);
      if (small) return goq(append_qjl_mma_kernel<T, 0, true, kQjlSmallVec>);
      if (hq) return goq(append_qjl_mma_kernel<T, 0, true>);
      switch (qb) {
        case 4: return goq(append_qjl_mma_kernel<T, 4, false>);
        case 3: return goq(append_qjl_mma_kernel<T, 3, false>);
        case 2: return goq(append_qjl_mma_kernel<T, 2, false>);
        case 1: return goq(append_qjl_mma_kernel<T, 1, false>);
        default: return goq(append_qjl_mma_kernel<T, 0, false>);
      }
    };
    const cudaError_t e = dtype == TQ_F32 ? by_bits(float())
                          : dtype == TQ_BF16 ? by_bits(__nv_bfloat16())
                                             : by_bits(__half());
    if (e != cudaSuccess) {
      set_error(std::string("append sketch: ") + cudaGetErrorString(e));
      return TQ_ERR_CUDA;
    }
    tq_status s = launch_status("append sketch");
    if (s != TQ_OK || nq == 2) return s;  // both sides done by the sketch kernel
    p.side_base = p.qjl[0] ? 1 : 0;
    p.wait_primary = 1;
  } else {
    p.side_base = 0;
    p.wait_primary = 0;
  }
  const unsigned nsides = p.qjl_mma ? 1u : 2u;
  cudaError_t ae = cudaSuccess;
  // large appends at head dim 128 (no HeadQ side code, no spectral side): four lanes per vector
  const bool quad = ctx->cfg.head_dim == 128 && per_side >= kQjlMmaMin && !ctx->cfg.headq_rank &&
                    ctx->cfg.k.rotate != 2 && ctx->cfg.v.rotate != 2;
  if (quad) {
    auto go = [&](auto kern) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)((per_side + kQuadWarps * 8 - 1) / (kQuadWarps * 8)), nsides);
      cfg.blockDim = dim3(kQuadWarps * 32);
      cfg.dynamicSmemBytes = 0;
      cfg.stream = cs;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = p.wait_primary ? 1 : 0;
      ae = cudaLaunchKernelEx(&cfg, kern, p);
    };
    if (dtype == TQ_F32) go(append_quad_kernel<float>);
    else if (dtype == TQ_BF16) go(append_quad_kernel<__nv_bfloat16>);
    else go(append_quad_kernel<__half>);
    if (ae != cudaSuccess) {
      set_error(std::string("append: ") + cudaGetErrorString(ae));
      return TQ_ERR_CUDA;
    }
    return launch_status("append");
  }
  tq_status s = dispatch_d(ctx->cfg.head_dim, [&](auto dc) {
    constexpr int D = decltype(dc)::value;
    auto go = [&](auto kern) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)blocks, nsides);
      cfg.blockDim = dim3(kWarpsPerBlock * 32);
      cfg.dynamicSmemBytes = 0;
      cfg.stream = cs;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = p.wait_primary ? 1 : 0;
      ae = cudaLaunchKernelEx(&cfg, kern, p);
    };
    if (dtype == TQ_F32) go(append_kernel<D, float>);
    else if (dtype == TQ_BF16) go(append_kernel<D, __nv_bfloat16>);
    else go(append_kernel<D, __half>);
  });
  if (ae != cudaSuccess) {
    set_error(std::string("append: ") + cudaGetErrorString(ae));
    return TQ_ERR_CUDA;
  }
  if (s != TQ_OK) return s;
  return launch_status("append");
}

tq_status launch_append(const tq_context* ctx, void* cache, const void* k, const void* v,
                        tq_dtype dtype, int n_new, const int32_t* start, Stream stream) {
  return append_impl(ctx, cache, k, v, dtype, n_new, start, nullptr, stream);
}

tq_status launch_append_early(const tq_context* ctx, void* cache, const void* k, const void* v,
                              tq_dtype dtype, int n_new, const int32_t* start, Stream stream) {
  return append_impl(ctx, cache, k, v, dtype, n_new, start, nullptr, stream, true);
}

tq_status launch_append_paged(const tq_context* ctx, void* pool, const tq_page_table* pt, const void* k,
                              const void* v, tq_dtype dtype, int n_new, const int32_t* dev_start,
                              int32_t* dev_error, Stream stream) {
  const PagedAppend pg{pt, dev_start, dev_error};
  return append_impl(ctx, pool, k, v, dtype, n_new, nullptr, &pg, stream);
}

tq_status launch_spectral_basis(const tq_context* ctx, int side, const float* E, const float* sv, Stream stream) {
  using namespace tqd;
  const Tables t = make_tables(ctx);
  const int H = ctx->cfg.num_kv_heads, D = ctx->cfg.head_dim;
  const long long n = (long long)H * D * D;
  spectral_basis_kernel<<<(unsigned)((n + 255) / 256), 256, 0, (cudaStream_t)stream>>>(
      E, sv, const_cast<float*>(t.sq_E[side]), const_cast<float*>(t.sq_ET[side]), const_cast<float*>(t.sq_s[side]),
      side, H, D);
  return launch_status("spectral_basis");
}

tq_status launch_rotate_basis(const tq_context* ctx, const float* U, Stream stream) {
  using namespace tqd;
  const Tables t = make_tables(ctx);
  const int H = ctx->cfg.num_kv_heads, r = ctx->cfg.headq_rank;
  float* U_rot = const_cast<float*>(t.U_rot);
  tq_status s = dispatch_d(ctx->cfg.head_dim, [&](auto dc) {
    constexpr int D = decltype(dc)::value;
    rotate_basis_kernel<D><<<(H * r + 7) / 8, 256, 0, (cudaStream_t)stream>>>(U, U_rot, t.k_sign, H, r);
  });
  if (s != TQ_OK) return s;
  return launch_status("rotate_basis");
}

tq_status launch_dequantize(const tq_context* ctx, const void* cache, int b, int kvh, int t0, int t1,
                            float* k_out, float* v_out, Stream stream) {
  using namespace tqd;
  DequantParams p;
  p.tab = make_tables(ctx);
  p.cache = make_cache(ctx, cache);
  p.out[0] = k_out;
  p.out[1] = v_out;
  p.b = b; p.kvh = kvh; p.t0 = t0; p.n = t1 - t0; p.m = ctx->m;
  p.bits[0] = ctx->cfg.k.bits; p.rotate[0] = ctx->cfg.k.rotate; p.qjl[0] = ctx->cfg.k.qjl;
  p.bits[1] = ctx->cfg.v.bits; p.rotate[1] = ctx->cfg.v.rotate; p.qjl[1] = ctx->cfg.v.qjl;
  p.headq_rank = ctx->cfg.headq_rank;
  p.qjl_scale = (float)(1.2533141373155003 / ctx->m);  // sqrt(pi/2) / m
  tq_status s = dispatch_d(ctx->cfg.head_dim, [&](auto dc) {
    constexpr int D = decltype(dc)::value;
    dequantize_kernel<D><<<(2 * p.n + 7) / 8, 256, 0, (cudaStream_t)stream>>>(p);
  });
  if (s != TQ_OK) return s;
  return launch_status("dequantize");
}

}  // namespace tqi
