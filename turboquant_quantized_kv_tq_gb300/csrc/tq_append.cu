// Write path: quantize-and-append, HeadQ basis rotation, and reconstruction for tests.
//
// [TQ-KV] "Esquemas de Cuantización": norm split, randomized Walsh-Hadamard rotation, Lloyd-Max
// scalar code, optional 1-bit QJL sketch of the residual.  [HEADQ] "Visão Geral do Algoritmo"
// 2 ("Escrita no Cache"): base key, residual, projection on the calibrated basis, side code.
//
// One warp owns one vector; lane l holds coordinates [l*E, l*E + E), E = d / 32.  The rotation
// runs in registers (local butterflies, then warp shuffles); codes are packed so that lane l's
// bits are contiguous in the stream and stored with one coalesced store per lane group.
#include <cstdio>
#include <string>
#include <type_traits>

#include "tq_device.cuh"

namespace tqd {

namespace {

constexpr int kWarpsPerBlock = 8;

struct AppendParams {
  Tables tab;
  Cache cache;
  const void* k;
  const void* v;
  int B, Hkv, n_new, m;
  int bits[2], rotate[2], qjl[2];
  int headq_rank;
  int start[TQ_MAX_BATCH];
};

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

// Read back element values of a w-bit stream for this lane's E coordinates.
template <int E, int W>
__device__ __forceinline__ void load_stream(const unsigned char* src, uint32_t (&v)[E]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int bit = (lane * E + i) * W;
    v[i] = (src[bit >> 3] >> (bit & 7)) & ((1u << W) - 1u);
  }
}

template <int D, typename Tin>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) append_kernel(const AppendParams p) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const long long vec = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const long long per_side = (long long)p.B * p.Hkv * p.n_new;
  if (vec >= 2 * per_side) return;
  const int side = vec >= per_side ? 1 : 0;
  long long r = side ? vec - per_side : vec;
  const int j = (int)(r % p.n_new);
  r /= p.n_new;
  const int h = (int)(r % p.Hkv);
  const int b = (int)(r / p.Hkv);
  const int t = p.start[b] + j;

  const Tin* src = reinterpret_cast<const Tin*>(side ? p.v : p.k) +
                   ((long long)(b * p.Hkv + h) * p.n_new + j) * D;
  float x[E];
  load_row<E>(src + lane * E, x);

  const float nu = norm_compensated<E>(x);
  const int bits = p.bits[side];
  const bool rotate = p.rotate[side] != 0;
  const float* sgn = side ? p.tab.v_sign : p.tab.k_sign;
  const float* cent = side ? p.tab.v_c : p.tab.k_c;
  const float* thr = side ? p.tab.v_t : p.tab.k_t;

  float hrot[E];
#pragma unroll
  for (int i = 0; i < E; ++i) hrot[i] = x[i] * __ldg(sgn + lane * E + i);
  if (rotate) wht_warp<E>(hrot);
  const float rs = rotate ? 1.f / sqrtf((float)D) : 1.f;
  const float scale = rotate ? sqrtf((float)D) : 1.f;
  const float inv = nu > 0.f ? 1.f / (nu * scale) : 0.f;

  float y[E];
#pragma unroll
  for (int i = 0; i < E; ++i) y[i] = hrot[i] * inv;

  float tr[15];
#pragma unroll
  for (int k = 0; k < 15; ++k) tr[k] = __ldg(thr + k);
  uint32_t code[E];
#pragma unroll
  for (int i = 0; i < E; ++i) {
    uint32_t c = 0;
#pragma unroll
    for (int k = 0; k < 15; ++k) c += y[i] > tr[k] ? 1u : 0u;
    code[i] = c;
  }

  // sign-magnitude symbols
  const uint32_t halfL = 1u << (bits - 1);
  uint32_t sgnbit[E], mag[E];
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const bool s = code[i] >= halfL;
    sgnbit[i] = s ? 1u : 0u;
    mag[i] = s ? code[i] - halfL : halfL - 1u - code[i];
  }

  const Cache& C = p.cache;
  const int rc = side ? tqi::R_V_CODES : tqi::R_K_CODES;
  unsigned char* codes = C.ptr(rc, b, h, t);
  if (bits == 4) {
    uint32_t v[E];
#pragma unroll
    for (int i = 0; i < E; ++i) v[i] = (sgnbit[i] << 3) | mag[i];
    store_stream<E, 4>(codes, v);
  } else if (bits == 3) {
    store_stream<E, 2>(codes, mag);
    store_stream<E, 1>(codes + D / 4, sgnbit);
  } else if (bits == 2) {
    uint32_t v[E];
#pragma unroll
    for (int i = 0; i < E; ++i) v[i] = (sgnbit[i] << 1) | mag[i];
    store_stream<E, 2>(codes, v);
  } else {
    store_stream<E, 1>(codes, sgnbit);
  }
  if (lane == 0) *reinterpret_cast<float*>(C.ptr(side ? tqi::R_V_NORM : tqi::R_K_NORM, b, h, t)) = nu;

  if (p.qjl[side]) {
    // residual of the rotated unit vector, its norm, and the signs of S r
    float res[E];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      res[i] = y[i] - __ldg(cent + code[i]);
      ss = fmaf(res[i], res[i], ss);
    }
    ss = warp_sum(ss);
    const float* ST = side ? p.tab.S_V_T : p.tab.S_K_T;  // [d][m], m == d
    float acc[E];
#pragma unroll
    for (int q = 0; q < E; ++q) acc[q] = 0.f;
    // several rows in flight per lane: the table is read from L2 and the loop is latency-bound
    constexpr int kUnroll = E <= 8 ? 4 : 1;
#pragma unroll kUnroll
    for (int jl = 0; jl < 32; ++jl) {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float rj = __shfl_sync(kFull, res[e], jl);
        const float* row = ST + (long long)(jl * E + e) * D + lane * E;
#pragma unroll
        for (int q = 0; q < E; q += 4) {
          const float4 s4 = __ldg(reinterpret_cast<const float4*>(row + q));
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
    store_stream<E, 1>(C.ptr(side ? tqi::R_V_SIGNS : tqi::R_K_SIGNS, b, h, t), sbit);
    if (lane == 0)
      *reinterpret_cast<__half*>(C.ptr(side ? tqi::R_V_RHO : tqi::R_K_RHO, b, h, t)) =
          __float2half_rn(sqrtf(ss));
  }

  if (side == 0 && p.headq_rank) {
    // e_rot = R k - nu C[c]; z = (R U)^T e_rot = U^T e   ([HEADQ] "Escrita no Cache")
    constexpr int RK = 16;
    const float* Ur = p.tab.U_rot + (long long)h * D * RK;
    float z[RK];
#pragma unroll
    for (int k = 0; k < RK; ++k) z[k] = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const float e = hrot[i] * rs - nu * __ldg(cent + code[i]);
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
      z[k] = warp_sum(z[k]);
      amax = fmaxf(amax, fabsf(z[k]));
    }
    const __half sh = __float2half_rn(amax / 7.0f);
    const float s32 = __half2float(sh);
    uint32_t w0 = 0, w1 = 0;
#pragma unroll
    for (int k = 0; k < RK; ++k) {
      int qz = 0;
      if (s32 > 0.f) {
        const float v = rintf(__fdiv_rn(z[k], s32));
        qz = (int)fminf(fmaxf(v, -7.f), 7.f);
      }
      const uint32_t nib = (uint32_t)qz & 0xFu;
      if (k < 8) w0 |= nib << (4 * k); else w1 |= nib << (4 * (k - 8));
    }
    if (lane == 0) {
      *reinterpret_cast<uint2*>(C.ptr(tqi::R_K_SIDE, b, h, t)) = make_uint2(w0, w1);
      *reinterpret_cast<__half*>(C.ptr(tqi::R_K_SIDE_SCALE, b, h, t)) = sh;
    }
  }
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
  const unsigned char* codes = C.ptr(side ? tqi::R_V_CODES : tqi::R_K_CODES, p.b, p.kvh, t);
  const float* cent = side ? p.tab.v_c : p.tab.k_c;
  const uint32_t halfL = 1u << (bits - 1);
  uint32_t sym[E], sgn[E];
  if (bits == 4) {
    load_stream<E, 4>(codes, sym);
#pragma unroll
    for (int i = 0; i < E; ++i) { sgn[i] = sym[i] >> 3; sym[i] &= 7u; }
  } else if (bits == 3) {
    load_stream<E, 2>(codes, sym);
    load_stream<E, 1>(codes + D / 4, sgn);
  } else if (bits == 2) {
    load_stream<E, 2>(codes, sym);
#pragma unroll
    for (int i = 0; i < E; ++i) { sgn[i] = sym[i] >> 1; sym[i] &= 1u; }
  } else {
    load_stream<E, 1>(codes, sgn);
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
    const unsigned char* sg = C.ptr(side ? tqi::R_V_SIGNS : tqi::R_K_SIGNS, p.b, p.kvh, t);
    const float rho = __half2float(*reinterpret_cast<const __half*>(C.ptr(side ? tqi::R_V_RHO : tqi::R_K_RHO, p.b, p.kvh, t)));
    const float* S = side ? p.tab.S_V : p.tab.S_K;  // [m][d]
    float acc[E];
#pragma unroll
    for (int i = 0; i < E; ++i) acc[i] = 0.f;
    for (int i = 0; i < p.m; ++i) {
      const float pm = ((sg[i >> 3] >> (i & 7)) & 1u) ? 1.f : -1.f;
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

tq_status launch_append(const tq_context* ctx, void* cache, const void* k, const void* v,
                        tq_dtype dtype, int n_new, const int32_t* start, Stream stream) {
  using namespace tqd;
  AppendParams p;
  p.tab = make_tables(ctx);
  p.cache = make_cache(ctx, cache);
  p.k = k;
  p.v = v;
  p.B = ctx->cfg.batch;
  p.Hkv = ctx->cfg.num_kv_heads;
  p.n_new = n_new;
  p.m = ctx->m;
  p.bits[0] = ctx->cfg.k.bits; p.rotate[0] = ctx->cfg.k.rotate; p.qjl[0] = ctx->cfg.k.qjl;
  p.bits[1] = ctx->cfg.v.bits; p.rotate[1] = ctx->cfg.v.rotate; p.qjl[1] = ctx->cfg.v.qjl;
  p.headq_rank = ctx->cfg.headq_rank;
  for (int b = 0; b < TQ_MAX_BATCH; ++b) p.start[b] = b < ctx->cfg.batch ? start[b] : 0;
  const long long vectors = 2LL * p.B * p.Hkv * n_new;
  const long long blocks = (vectors + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (blocks > 0x7fffffffLL) { set_error("append too large"); return TQ_ERR_INVALID_ARG; }
  tq_status s = dispatch_d(ctx->cfg.head_dim, [&](auto dc) {
    constexpr int D = decltype(dc)::value;
    const dim3 grid((unsigned)blocks), block(kWarpsPerBlock * 32);
    if (dtype == TQ_F32) append_kernel<D, float><<<grid, block, 0, (cudaStream_t)stream>>>(p);
    else if (dtype == TQ_BF16) append_kernel<D, __nv_bfloat16><<<grid, block, 0, (cudaStream_t)stream>>>(p);
    else append_kernel<D, __half><<<grid, block, 0, (cudaStream_t)stream>>>(p);
  });
  if (s != TQ_OK) return s;
  return launch_status("append");
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
