// Device-side views and helpers shared by the write-path and read-path kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "tq_internal.h"

namespace tqd {

constexpr unsigned kFull = 0xffffffffu;

// Device pointers into the table blob.
struct Tables {
  const float* k_c;   // centroids, ascending, 16 slots
  const float* k_t;   // thresholds, 16 slots (unused = 3e38)
  const float* v_c;
  const float* v_t;
  const float* k_sign;  // D_K as +-1 (all +1 when K is not rotated)
  const float* v_sign;
  const float* S_K;   // [m][d]
  const float* S_K_T; // [d][m]
  const float* S_V;
  const float* S_V_T;
  const float* U_rot; // [H_kv][d][r], R_K U
  const float* S_V_R; // [m][d], S_V R_V (head dim > 128 with a QJL value side)
  const unsigned char* S_h16[2];  // fp16 hi / lo rows of S_K, S_V (head dim 128; tqi::kSketchH16Bytes)
  const float* sq_c1;     // [2]: 1-bit centroid of each side (spectral sides' floor)
  const float* sq_E[2];   // spectral side: [H_kv][d][d] basis, column c = stored coordinate c
  const float* sq_ET[2];  // its transpose
  const float* sq_s[2];   // [H_kv][d] coordinate scales, storage order
};

// The packed cache in 16-token blocks: field r of token t of slab s = b * H + h at
// base + side_off[side] + (s * tiles_per_slab + t / 16) * block[side] + off[r] + (t % 16) * rec[r].
// Paged (block_table set): block t / 16 of (b, h) is block page * H + h of its side's array, page
// = block_table[b * max_blocks + t / 16]; a block index past max_blocks or a page outside
// [0, num_pages) goes to page num_pages (the pool's redirect page) and records
// TQ_DEVERR_BAD_PAGE in *err (when err is set).
struct Cache {
  unsigned char* base;
  unsigned long long side_off[2];
  unsigned int block[2];
  unsigned int off[tqi::R_COUNT];
  unsigned int rec[tqi::R_COUNT];
  int num_kv_heads;
  int tiles_per_slab;
  const int* block_table;
  int max_blocks;
  int num_pages;
  int* err;

  // (e: where a bad entry is recorded, when not null)
  __device__ __forceinline__ int page_of(int b, int tile, int* e) const {
    int page = -1;
    if ((unsigned)tile < (unsigned)max_blocks) page = __ldg(block_table + (long long)b * max_blocks + tile);
    if ((unsigned)page >= (unsigned)num_pages) {
      if (e) atomicExch(e, TQ_DEVERR_BAD_PAGE);
      page = num_pages;
    }
    return page;
  }
  __device__ __forceinline__ int page_of(int b, int tile) const { return page_of(b, tile, err); }
  // block `tile` of slab (b, h) on side 0 (K) or 1 (V)
  __device__ __forceinline__ unsigned char* blockp(int side, int b, int h, int tile) const {
    const unsigned long long blk =
        block_table ? (unsigned long long)page_of(b, tile) * num_kv_heads + h
                    : (unsigned long long)(b * num_kv_heads + h) * tiles_per_slab + tile;
    return base + side_off[side] + blk * block[side];
  }
  // block of KV head h in page `page` of a paged pool, side 0 (K) or 1 (V)
  __device__ __forceinline__ const unsigned char* page_block(int side, int page, int h) const {
    return base + side_off[side] + ((unsigned long long)page * num_kv_heads + h) * block[side];
  }
  // (t >> 4, t & 15: a negative position of a paged append lands in the redirect page)
  __device__ __forceinline__ unsigned char* ptr(int r, int b, int h, int t) const {
    const int side = r >= tqi::R_V_CODES ? 1 : 0;
    return blockp(side, b, h, t >> 4) + off[r] + (t & (tqi::kTileTokens - 1)) * rec[r];
  }
  // start of field r in the block of token t (for the value streams, stored by coordinate group)
  __device__ __forceinline__ unsigned char* fieldp(int r, int b, int h, int t) const {
    const int side = r >= tqi::R_V_CODES ? 1 : 0;
    return blockp(side, b, h, t >> 4) + off[r];
  }
};

// SQU-KV storage order (head dim 128): the eigen-rank held by stored coordinate c of a side.
// Keys: the first 8 coordinates of each 32-coordinate chunk hold ranks 0..31 (rank 4 r + chunk);
// values: the first 4 of each 16-coordinate group (rank 8 r + group); the others hold ranks
// 32.. in increasing coordinate order.
__host__ __device__ __forceinline__ int sq_rank_of_coord(int side, int c) {
  if (side == 0) {
    const int lt = c / 32, r = c % 32;
    return r < 8 ? 4 * r + lt : 32 + 24 * lt + (r - 8);
  }
  const int g = c / 16, r = c % 16;
  return r < 4 ? 8 * r + g : 32 + 12 * g + (r - 4);
}
// whether stored coordinate c of a side is modeled (4 bits) rather than floor (1 bit)
__host__ __device__ __forceinline__ bool sq_modeled(int side, int c) {
  return side == 0 ? (c % 32) < 8 : (c % 16) < 4;
}

// Value-side streams (V codes, each stream of a 3-bit code on its own, V QJL signs) are stored
// by groups of 16 coordinates: [groups][16 tokens][2W bytes] for a W-bit stream, so byte j of
// the record of block position pos is at grouped_byte(j, pos, W) from the stream's start.
__device__ __forceinline__ unsigned grouped_byte(unsigned j, unsigned pos, unsigned W) {
  return (j / (2 * W)) * 32 * W + pos * 2 * W + j % (2 * W);
}
static_assert(tqi::kTileTokens == 16, "ptr() splits positions with shifts by 4");

inline Tables make_tables(const tq_context* ctx) {
  const unsigned char* b = (const unsigned char*)ctx->dev_tables;
  Tables t;
  t.k_c = (const float*)(b + ctx->tab.k_centroids);
  t.k_t = (const float*)(b + ctx->tab.k_thresholds);
  t.v_c = (const float*)(b + ctx->tab.v_centroids);
  t.v_t = (const float*)(b + ctx->tab.v_thresholds);
  t.k_sign = (const float*)(b + ctx->tab.k_signs);
  t.v_sign = (const float*)(b + ctx->tab.v_signs);
  t.S_K = ctx->cfg.k.qjl ? (const float*)(b + ctx->tab.s_k) : nullptr;
  t.S_K_T = ctx->cfg.k.qjl ? (const float*)(b + ctx->tab.s_k_t) : nullptr;
  t.S_V = ctx->cfg.v.qjl ? (const float*)(b + ctx->tab.s_v) : nullptr;
  t.S_V_T = ctx->cfg.v.qjl ? (const float*)(b + ctx->tab.s_v_t) : nullptr;
  t.U_rot = ctx->cfg.headq_rank ? (const float*)(b + ctx->tab.headq_u) : nullptr;
  t.S_V_R = ctx->tab.s_v_r ? (const float*)(b + ctx->tab.s_v_r) : nullptr;
  for (int side = 0; side < 2; ++side) t.S_h16[side] = ctx->tab.s_h16[side] ? b + ctx->tab.s_h16[side] : nullptr;
  t.sq_c1 = (const float*)(b + ctx->tab.sq_c1);
  for (int side = 0; side < 2; ++side) {
    const bool sq = ctx->tab.sq_e[side] != 0;
    t.sq_E[side] = sq ? (const float*)(b + ctx->tab.sq_e[side]) : nullptr;
    t.sq_ET[side] = sq ? (const float*)(b + ctx->tab.sq_et[side]) : nullptr;
    t.sq_s[side] = sq ? (const float*)(b + ctx->tab.sq_s[side]) : nullptr;
  }
  return t;
}

inline Cache make_cache(const tq_context* ctx, const void* cache) {
  Cache c;
  c.base = (unsigned char*)cache;
  for (int r = 0; r < tqi::R_COUNT; ++r) {
    c.off[r] = (unsigned)ctx->layout.off[r];
    c.rec[r] = (unsigned)ctx->layout.rec[r];
  }
  for (int s = 0; s < 2; ++s) {
    c.side_off[s] = ctx->layout.side_off[s];
    c.block[s] = (unsigned)ctx->layout.block[s];
  }
  c.num_kv_heads = ctx->cfg.num_kv_heads;
  c.tiles_per_slab = (int)ctx->layout.tiles_per_slab;
  c.block_table = nullptr;
  c.max_blocks = 0;
  c.num_pages = 0;
  c.err = nullptr;
  return c;
}

// The paged pool's view: the same block format, arrays of (num_pages + 1) * H_kv blocks.
inline Cache make_paged_cache(const tq_context* ctx, const void* pool, const tq_page_table& pt, int* err) {
  Cache c = make_cache(ctx, pool);
  const tqi::Layout L = tqi::make_layout(ctx->cfg, ctx->m, pt.num_pages);
  c.side_off[0] = L.side_off[0];
  c.side_off[1] = L.side_off[1];
  c.tiles_per_slab = 0;
  c.block_table = pt.block_table;
  c.max_blocks = pt.max_blocks_per_seq;
  c.num_pages = pt.num_pages;
  c.err = err;
  return c;
}

// Walsh-Hadamard butterflies over a warp holding E consecutive elements per lane
// (element index lane * E + i): computes H x with H_ij = (-1)^popcount(i & j), natural order.
template <int E>
__device__ __forceinline__ void wht_warp(float (&x)[E]) {
#pragma unroll
  for (int h = 1; h < E; h <<= 1) {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      if ((i & h) == 0) {
        const float a = x[i], b = x[i + h];
        x[i] = a + b;
        x[i + h] = a - b;
      }
    }
  }
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const float other = __shfl_xor_sync(kFull, x[i], m);
      x[i] = (lane & m) ? (other - x[i]) : (x[i] + other);
    }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(kFull, v, m);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, m));
  return v;
}

// Load E consecutive input elements as fp32.
template <int E, typename T>
__device__ __forceinline__ void load_row(const T* p, float (&x)[E]);

template <int E>
__device__ __forceinline__ void load_row(const float* p, float (&x)[E]) {
#pragma unroll
  for (int i = 0; i < E; i += 4) {
    const float4 v = *reinterpret_cast<const float4*>(p + i);
    x[i] = v.x; x[i + 1] = v.y; x[i + 2] = v.z; x[i + 3] = v.w;
  }
}

template <int E>
__device__ __forceinline__ void load_row(const __nv_bfloat16* p, float (&x)[E]) {
#pragma unroll
  for (int i = 0; i < E; i += 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(p + i);
    x[i] = __uint_as_float(v.x << 16);
    x[i + 1] = __uint_as_float(v.x & 0xffff0000u);
    x[i + 2] = __uint_as_float(v.y << 16);
    x[i + 3] = __uint_as_float(v.y & 0xffff0000u);
  }
}

template <int E>
__device__ __forceinline__ void load_row(const __half* p, float (&x)[E]) {
#pragma unroll
  for (int i = 0; i < E; i += 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(p + i);
    const __half2 a = *reinterpret_cast<const __half2*>(&v.x);
    const __half2 b = *reinterpret_cast<const __half2*>(&v.y);
    const float2 fa = __half22float2(a), fb = __half22float2(b);
    x[i] = fa.x; x[i + 1] = fa.y; x[i + 2] = fb.x; x[i + 3] = fb.y;
  }
}

// ---- tensor-core fragments (mma.sync m16n8k16, fp16 inputs, fp32 accumulators) ----

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose an 8x8 matrix of 16-bit elements held as one register per lane in the mma
// accumulator layout (lane (g, t) holds row g, columns 2t, 2t+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Streaming 128/64/32/16-bit loads that do not allocate in L1.
__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ldg_stream8(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_stream4(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_stream2(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// ---- mbarrier + bulk (TMA) copies global -> shared ----

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
               : "memory");
}
// Wait for the phase with the given parity to complete; gives up after `limit` polls and
// returns false (the caller records an error instead of spinning forever).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}
// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) completing on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Copies n floats (n a multiple of 32 NT) from global to shared memory with the NT threads of a
// block, eight 16-byte loads in flight per thread.  Used for the 64 KiB sketch tables that a
// block stages once: they are often evicted from L2 between calls, and one load in flight per
// thread would pay a DRAM latency per 4 KiB of table.
template <int NT>
__device__ __forceinline__ void stage_table(float* dst, const float* __restrict__ src, int n) {
  for (int base = (int)threadIdx.x * 4; base < n; base += NT * 32) {
    float4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = __ldg(reinterpret_cast<const float4*>(src + base + k * NT * 4));
#pragma unroll
    for (int k = 0; k < 8; ++k) *reinterpret_cast<float4*>(dst + base + k * NT * 4) = v[k];
  }
}

}  // namespace tqd
