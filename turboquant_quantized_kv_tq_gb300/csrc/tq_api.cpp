// C ABI entry points: validation, context and table management, layout, dispatch.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>

#include <cuda_runtime.h>

#include <cuda_fp16.h>

#include "tq_internal.h"

namespace tqi {
namespace {
thread_local std::string g_last_error;
}
void set_error(const std::string& msg) { g_last_error = msg; }
}  // namespace tqi

using namespace tqi;

namespace {

tq_status fail(tq_status s, const std::string& msg) {
  set_error(msg);
  return s;
}

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

tq_status validate_codec(const tq_codec& c, const char* side) {
  if (c.bits < 1 || c.bits > 4) return fail(TQ_ERR_INVALID_ARG, std::string(side) + ": bits must be 1..4");
  if ((c.rotate < 0 || c.rotate > 2) || (c.qjl != 0 && c.qjl != 1))
    return fail(TQ_ERR_INVALID_ARG, std::string(side) + ": rotate must be 0, 1 or 2 and qjl 0 or 1");
  if (c.rotate == 2 && (c.bits != 2 || c.qjl))
    return fail(TQ_ERR_UNSUPPORTED, std::string(side) + ": the spectral codec is built at 2 bits without QJL");
  return TQ_OK;
}

tq_status validate_config(const tq_config& c) {
  if (!pow2(c.head_dim) || c.head_dim < 8 || c.head_dim > 1024)
    return fail(TQ_ERR_INVALID_ARG, "head_dim must be a power of two in [8, 1024]");
  if (c.head_dim != 128 && c.head_dim != 256 && c.head_dim != 512 && c.head_dim != 1024)
    return fail(TQ_ERR_UNSUPPORTED, "head_dim: the GPU path is built for 128, 256, 512, 1024");
  if (c.num_kv_heads <= 0 || c.num_q_heads <= 0 || c.num_q_heads % c.num_kv_heads)
    return fail(TQ_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of num_kv_heads");
  const int G = c.num_q_heads / c.num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return fail(TQ_ERR_UNSUPPORTED, "G = num_q_heads / num_kv_heads must be 1, 2, 4 or 8");
  if (c.batch <= 0 || c.batch > TQ_MAX_BATCH) return fail(TQ_ERR_INVALID_ARG, "batch must be in [1, TQ_MAX_BATCH]");
  if (c.capacity <= 0 || c.capacity % 64) return fail(TQ_ERR_INVALID_ARG, "capacity must be a positive multiple of 64");
  if ((uint64_t)c.batch * c.num_kv_heads * c.capacity > (1ull << 40))
    return fail(TQ_ERR_INVALID_ARG, "cache too large");
  tq_status s = validate_codec(c.k, "k");
  if (s != TQ_OK) return s;
  s = validate_codec(c.v, "v");
  if (s != TQ_OK) return s;
  if (c.qjl_m != 0 && c.qjl_m != c.head_dim) return fail(TQ_ERR_UNSUPPORTED, "qjl_m must be 0 or head_dim");
  if (c.headq_rank < 0) return fail(TQ_ERR_INVALID_ARG, "headq_rank must be >= 0");
  if (c.headq_rank) {
    if (c.headq_rank != 16 || c.headq_bits != 4)
      return fail(TQ_ERR_UNSUPPORTED, "HeadQ is built for rank 16 with 4-bit side codes");
    if (c.k.qjl) return fail(TQ_ERR_UNSUPPORTED, "HeadQ with a QJL key side is not built");
  }
  if (c.head_dim > 128 && (c.k.qjl || c.headq_rank))
    return fail(TQ_ERR_UNSUPPORTED, "key-side QJL and HeadQ are built for head_dim 128");
  if ((c.k.rotate == 2) != (c.v.rotate == 2))
    return fail(TQ_ERR_UNSUPPORTED, "the spectral codec is built for both sides together (SQU-KV)");
  if (c.k.rotate == 2 && (c.head_dim != 128 || c.headq_rank))
    return fail(TQ_ERR_UNSUPPORTED, "the spectral codec is built for head_dim 128 without HeadQ");
  return TQ_OK;
}

}  // namespace

extern "C" {

const char* tq_status_string(tq_status s) {
  switch (s) {
    case TQ_OK: return "ok";
    case TQ_ERR_INVALID_ARG: return "invalid argument";
    case TQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case TQ_ERR_CAPACITY: return "cache capacity exceeded";
    case TQ_ERR_WORKSPACE: return "workspace too small";
    case TQ_ERR_CUDA: return "CUDA error";
    case TQ_ERR_DEVICE: return "device-side error";
    case TQ_ERR_STATE: return "context not ready";
  }
  return "unknown status";
}

const char* tq_last_error(void) { return g_last_error.c_str(); }

tq_status tq_config_from_scheme(tq_scheme scheme, int32_t n, tq_config* c) {
  if (!c) return fail(TQ_ERR_INVALID_ARG, "null config");
  if (n < 1 || n > 4) return fail(TQ_ERR_INVALID_ARG, "n must be 1..4");
  switch (scheme) {
    case TQ_PLAIN_KV: c->k = {n, 0, 0}; c->v = {n, 0, 0}; break;
    case TQ_TQ_KV: c->k = {n, 1, 0}; c->v = {n, 1, 0}; break;
    case TQ_KQV:
      if (n < 2) return fail(TQ_ERR_INVALID_ARG, "KQV needs n >= 2");
      c->k = {n, 1, 0}; c->v = {n - 1, 1, 1}; break;
    case TQ_QKQV:
      if (n < 2) return fail(TQ_ERR_INVALID_ARG, "QKQV needs n >= 2");
      c->k = {n - 1, 1, 1}; c->v = {n - 1, 1, 1}; break;
    case TQ_SQU_KV:
      if (n != 2) return fail(TQ_ERR_UNSUPPORTED, "SQU-KV is built at n = 2");
      c->k = {2, 2, 0}; c->v = {2, 2, 0}; break;
    default: return fail(TQ_ERR_INVALID_ARG, "unknown scheme");
  }
  return TQ_OK;
}

tq_status tq_context_create(const tq_config* cfg, tq_context** out) {
  if (!cfg || !out) return fail(TQ_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  tq_status s = validate_config(*cfg);
  if (s != TQ_OK) return s;
  tq_context* ctx = new (std::nothrow) tq_context();
  if (!ctx) return fail(TQ_ERR_INVALID_ARG, "out of host memory");
  ctx->cfg = *cfg;
  const int d = cfg->head_dim;
  ctx->m = cfg->qjl_m ? cfg->qjl_m : d;
  ctx->tab = make_table_offsets(*cfg, ctx->m);
  ctx->layout = make_layout(*cfg, ctx->m);
  ctx->host_tables.assign(ctx->tab.total, 0);
  unsigned char* base = ctx->host_tables.data();
  double c[kMaxLevels], t[kMaxLevels];
  auto put_codebook = [&](int bits, size_t off_c, size_t off_t) {
    lloyd_max_beta(d, bits, c, t);
    float* fc = (float*)(base + off_c);
    float* ft = (float*)(base + off_t);
    const int L = 1 << bits;
    for (int i = 0; i < kMaxLevels; ++i) fc[i] = i < L ? (float)c[i] : 0.0f;
    for (int i = 0; i < kMaxLevels; ++i) ft[i] = i < L - 1 ? (float)t[i] : 3.0e38f;
  };
  // a spectral side's modeled coordinates use the 4-bit codebook, its floor the 1-bit centroid
  const int kcb = cfg->k.rotate == 2 ? 4 : cfg->k.bits, vcb = cfg->v.rotate == 2 ? 4 : cfg->v.bits;
  put_codebook(kcb, ctx->tab.k_centroids, ctx->tab.k_thresholds);
  put_codebook(vcb, ctx->tab.v_centroids, ctx->tab.v_thresholds);
  {
    lloyd_max_beta(d, 1, c, t);
    float* c1 = (float*)(base + ctx->tab.sq_c1);
    c1[0] = c1[1] = (float)c[1];
  }
  // the write path's sign-magnitude code search relies on exactly symmetric thresholds
  for (int side = 0; side < 2; ++side) {
    const int bits = side ? vcb : kcb;
    const float* ft = (const float*)(base + (side ? ctx->tab.v_thresholds : ctx->tab.k_thresholds));
    const int h = 1 << (bits - 1);
    bool ok = ft[h - 1] == 0.0f;
    for (int k = 1; k < h; ++k) ok = ok && ft[h - 1 + k] == -ft[h - 1 - k];
    if (!ok) {
      delete ctx;
      return fail(TQ_ERR_INVALID_ARG, "codebook thresholds are not symmetric");
    }
  }
  float* ks = (float*)(base + ctx->tab.k_signs);
  float* vs = (float*)(base + ctx->tab.v_signs);
  if (cfg->k.rotate) rotation_signs(cfg->seed, 1, d, ks); else for (int i = 0; i < d; ++i) ks[i] = 1.0f;
  if (cfg->v.rotate) rotation_signs(cfg->seed, 2, d, vs); else for (int i = 0; i < d; ++i) vs[i] = 1.0f;
  auto put_sketch = [&](uint64_t stream, size_t off, size_t off_t) {
    float* S = (float*)(base + off);
    float* St = (float*)(base + off_t);
    sketch_matrix(cfg->seed, stream, ctx->m, d, S);
    for (int i = 0; i < ctx->m; ++i)
      for (int j = 0; j < d; ++j) St[(size_t)j * ctx->m + i] = S[(size_t)i * d + j];
  };
  if (cfg->k.qjl) put_sketch(3, ctx->tab.s_k, ctx->tab.s_k_t);
  if (cfg->v.qjl) put_sketch(4, ctx->tab.s_v, ctx->tab.s_v_t);
  for (int side = 0; side < 2; ++side) {  // fp16 hi / lo terms of S for the tensor-core sketch
    if (!ctx->tab.s_h16[side]) continue;
    const float* S = (const float*)(base + (side ? ctx->tab.s_v : ctx->tab.s_k));
    unsigned char* hi = base + ctx->tab.s_h16[side];
    unsigned char* lo = hi + kSketchH16Bytes / 2;
    for (int i = 0; i < 128; ++i)
      for (int j = 0; j < 128; ++j) {
        const float x = S[i * 128 + j];
        const __half h = __float2half_rn(x);
        *(__half*)(hi + sketch_cm_offset(i, j)) = h;
        *(__half*)(lo + sketch_cm_offset(i, j)) = __float2half_rn(x - __half2float(h));
      }
  }
  if (ctx->tab.s_v_r) {
    // rows of S_V R_V = S_V H D_V / sqrt(d): a float64 Walsh-Hadamard transform of each row of
    // S_V, then the D_V signs and the 1/sqrt(d) scale, rounded once to fp32 (R_V = I when the
    // value side is not rotated)
    const float* S = (const float*)(base + ctx->tab.s_v);
    float* T = (float*)(base + ctx->tab.s_v_r);
    std::vector<double> row(d);
    const bool rot = cfg->v.rotate != 0;
    const double rs = rot ? 1.0 / std::sqrt((double)d) : 1.0;
    for (int i = 0; i < ctx->m; ++i) {
      for (int j = 0; j < d; ++j) row[j] = S[(size_t)i * d + j];
      for (int h = 1; rot && h < d; h <<= 1)
        for (int j = 0; j < d; j += 2 * h)
          for (int k = j; k < j + h; ++k) {
            const double a = row[k], b = row[k + h];
            row[k] = a + b;
            row[k + h] = a - b;
          }
      for (int j = 0; j < d; ++j) T[(size_t)i * d + j] = (float)(row[j] * vs[j] * rs);
    }
  }
  *out = ctx;
  return TQ_OK;
}

void tq_context_destroy(tq_context* ctx) { delete ctx; }

size_t tq_tables_bytes(const tq_context* ctx) { return ctx ? ctx->tab.total : 0; }

tq_status tq_tables_host(const tq_context* ctx, void* dst, size_t bytes) {
  if (!ctx || !dst) return fail(TQ_ERR_INVALID_ARG, "null argument");
  if (bytes < ctx->tab.total) return fail(TQ_ERR_INVALID_ARG, "destination smaller than tq_tables_bytes");
  std::memcpy(dst, ctx->host_tables.data(), ctx->tab.total);
  return TQ_OK;
}

tq_status tq_tables_upload(tq_context* ctx, void* dev_tables, tq_stream stream) {
  if (!ctx || !dev_tables) return fail(TQ_ERR_INVALID_ARG, "null argument");
  if (!aligned(dev_tables, 256)) return fail(TQ_ERR_INVALID_ARG, "dev_tables must be 256-byte aligned");
  cudaError_t e = cudaMemcpyAsync(dev_tables, ctx->host_tables.data(), ctx->tab.total,
                                  cudaMemcpyHostToDevice, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(TQ_ERR_CUDA, std::string("table upload: ") + cudaGetErrorString(e));
  ctx->dev_tables = dev_tables;
  ctx->basis_set = false;
  ctx->sq_set[0] = ctx->sq_set[1] = false;
  return TQ_OK;
}

tq_status tq_headq_set_basis(tq_context* ctx, const float* dev_U, tq_stream stream) {
  if (!ctx || !dev_U) return fail(TQ_ERR_INVALID_ARG, "null argument");
  if (!ctx->cfg.headq_rank) return fail(TQ_ERR_STATE, "HeadQ is off in this context");
  if (!ctx->dev_tables) return fail(TQ_ERR_STATE, "tables not uploaded");
  if (!aligned(dev_U, 16)) return fail(TQ_ERR_INVALID_ARG, "dev_U must be 16-byte aligned");
  tq_status s = launch_rotate_basis(ctx, dev_U, stream);
  if (s == TQ_OK) ctx->basis_set = true;
  return s;
}

tq_status tq_spectral_set_basis(tq_context* ctx, int32_t side, const float* dev_E, const float* dev_s,
                                tq_stream stream) {
  if (!ctx || !dev_E || !dev_s) return fail(TQ_ERR_INVALID_ARG, "null argument");
  if (side != 0 && side != 1) return fail(TQ_ERR_INVALID_ARG, "side must be 0 (K) or 1 (V)");
  if ((side ? ctx->cfg.v.rotate : ctx->cfg.k.rotate) != 2) return fail(TQ_ERR_STATE, "not a spectral side");
  if (!ctx->dev_tables) return fail(TQ_ERR_STATE, "tables not uploaded");
  if (!aligned(dev_E, 16) || !aligned(dev_s, 4)) return fail(TQ_ERR_INVALID_ARG, "misaligned pointer");
  tq_status s = launch_spectral_basis(ctx, side, dev_E, dev_s, stream);
  if (s == TQ_OK) ctx->sq_set[side] = true;
  return s;
}

tq_status tq_get_cache_layout(const tq_context* ctx, tq_cache_layout* out) {
  if (!ctx || !out) return fail(TQ_ERR_INVALID_ARG, "null argument");
  std::memset(out, 0, sizeof(*out));
  out->layout_version = TQ_LAYOUT_VERSION;
  out->tile_tokens = TQ_TILE_TOKENS;
  out->total_bytes = ctx->layout.total;
  out->k_offset = ctx->layout.side_off[0];
  out->k_block_bytes = ctx->layout.block[0];
  out->v_offset = ctx->layout.side_off[1];
  out->v_block_bytes = ctx->layout.block[1];
  tq_region* r[R_COUNT] = {&out->k_codes, &out->k_norm, &out->k_signs, &out->k_rho, &out->k_side,
                           &out->k_side_scale, &out->v_codes, &out->v_norm, &out->v_signs, &out->v_rho};
  for (int i = 0; i < R_COUNT; ++i) {
    r[i]->offset = ctx->layout.off[i];
    r[i]->record_bytes = ctx->layout.rec[i];
  }
  return TQ_OK;
}

static tq_status check_pages(const tq_context* ctx, const tq_page_table* pt) {
  if (!pt || !pt->block_table) return fail(TQ_ERR_INVALID_ARG, "null page table");
  if (pt->max_blocks_per_seq < 1 || pt->num_pages < 1) return fail(TQ_ERR_INVALID_ARG, "empty page table");
  if ((int64_t)pt->max_blocks_per_seq * TQ_TILE_TOKENS > INT32_MAX / 2)
    return fail(TQ_ERR_INVALID_ARG, "max_blocks_per_seq too large");
  if (!aligned(pt->block_table, 4)) return fail(TQ_ERR_INVALID_ARG, "block_table must be 4-byte aligned");
  if (ctx->cfg.head_dim != 128) return fail(TQ_ERR_UNSUPPORTED, "the paged pool is built for head_dim 128");
  return TQ_OK;
}

tq_status tq_get_paged_cache_layout(const tq_context* ctx, int32_t num_pages, tq_cache_layout* out) {
  tq_status s = tq_get_cache_layout(ctx, out);
  if (s != TQ_OK) return s;
  if (num_pages < 1) return fail(TQ_ERR_INVALID_ARG, "num_pages must be >= 1");
  const Layout L = make_layout(ctx->cfg, ctx->m, num_pages);
  out->total_bytes = L.total;
  out->k_offset = L.side_off[0];
  out->v_offset = L.side_off[1];
  return TQ_OK;
}

static tq_status ready(const tq_context* ctx) {
  if (!ctx) return fail(TQ_ERR_INVALID_ARG, "null context");
  if (!ctx->dev_tables) return fail(TQ_ERR_STATE, "tables not uploaded");
  if (ctx->cfg.headq_rank && !ctx->basis_set) return fail(TQ_ERR_STATE, "HeadQ basis not set");
  for (int side = 0; side < 2; ++side)
    if ((side ? ctx->cfg.v.rotate : ctx->cfg.k.rotate) == 2 && !ctx->sq_set[side])
      return fail(TQ_ERR_STATE, "spectral basis not set");
  return TQ_OK;
}

tq_status tq_quantize_append(const tq_context* ctx, void* dev_cache, const void* k, const void* v,
                             tq_dtype dtype, int32_t n_new, const int32_t* host_start,
                             tq_stream stream) {
  tq_status s = ready(ctx);
  if (s != TQ_OK) return s;
  if (n_new < 0) return fail(TQ_ERR_INVALID_ARG, "n_new must be >= 0");
  if (n_new == 0) return TQ_OK;
  if (!dev_cache || !k || !v || !host_start) return fail(TQ_ERR_INVALID_ARG, "null argument");
  if (dtype != TQ_F32 && dtype != TQ_BF16 && dtype != TQ_F16) return fail(TQ_ERR_INVALID_ARG, "bad dtype");
  if (!aligned(dev_cache, 256)) return fail(TQ_ERR_INVALID_ARG, "cache must be 256-byte aligned");
  if (!aligned(k, 16) || !aligned(v, 16)) return fail(TQ_ERR_INVALID_ARG, "k, v must be 16-byte aligned");
  for (int b = 0; b < ctx->cfg.batch; ++b) {
    if (host_start[b] < 0) return fail(TQ_ERR_INVALID_ARG, "start must be >= 0");
    if ((int64_t)host_start[b] + n_new > ctx->cfg.capacity) return fail(TQ_ERR_CAPACITY, "start + n_new > capacity");
  }
  return launch_append(ctx, dev_cache, k, v, dtype, n_new, host_start, stream);
}

tq_status tq_quantize_append_paged(const tq_context* ctx, void* dev_pool, const tq_page_table* pages,
                                   const void* k, const void* v, tq_dtype dtype, int32_t n_new,
                                   const int32_t* dev_start, int32_t* dev_error, tq_stream stream) {
  tq_status s = ready(ctx);
  if (s != TQ_OK) return s;
  if (n_new < 0) return fail(TQ_ERR_INVALID_ARG, "n_new must be >= 0");
  if (n_new == 0) return TQ_OK;
  if (!dev_pool || !k || !v || !dev_start) return fail(TQ_ERR_INVALID_ARG, "null argument");
  s = check_pages(ctx, pages);
  if (s != TQ_OK) return s;
  if (dtype != TQ_F32 && dtype != TQ_BF16 && dtype != TQ_F16) return fail(TQ_ERR_INVALID_ARG, "bad dtype");
  if (!aligned(dev_pool, 256)) return fail(TQ_ERR_INVALID_ARG, "pool must be 256-byte aligned");
  if (!aligned(k, 16) || !aligned(v, 16)) return fail(TQ_ERR_INVALID_ARG, "k, v must be 16-byte aligned");
  if (!aligned(dev_start, 4) || !aligned(dev_error, 4)) return fail(TQ_ERR_INVALID_ARG, "misaligned pointer");
  return launch_append_paged(ctx, dev_pool, pages, k, v, dtype, n_new, dev_start, dev_error, stream);
}

tq_status tq_decode_attention_paged(const tq_context* ctx, const void* dev_pool, const tq_page_table* pages,
                                    const float* q, int32_t nq, const int32_t* dev_seq_len, float* out,
                                    void* ws, size_t ws_bytes, tq_stream stream) {
  tq_status s = ready(ctx);
  if (s != TQ_OK) return s;
  if (!dev_pool || !q || !dev_seq_len || !out || !ws) return fail(TQ_ERR_INVALID_ARG, "null argument");
  s = check_pages(ctx, pages);
  if (s != TQ_OK) return s;
  if (nq < 1) return fail(TQ_ERR_INVALID_ARG, "nq must be >= 1");
  const int G = ctx->cfg.num_q_heads / ctx->cfg.num_kv_heads;
  if ((int64_t)G * nq > 8) return fail(TQ_ERR_UNSUPPORTED, "several queries per sequence are built for G * nq <= 8");
  if (!aligned(dev_pool, 256) || !aligned(q, 16) || !aligned(out, 16) || !aligned(ws, 256) ||
      !aligned(dev_seq_len, 4))
    return fail(TQ_ERR_INVALID_ARG, "misaligned pointer (pool/ws 256 B, q/out 16 B, lengths 4 B)");
  if (ws_bytes < decode_workspace_bytes(ctx, TQ_TILE_TOKENS * pages->max_blocks_per_seq))
    return fail(TQ_ERR_WORKSPACE, "workspace too small");
  return launch_decode_paged(ctx, dev_pool, pages, q, nq, dev_seq_len, out, ws, ws_bytes, stream);
}

size_t tq_decode_workspace_bytes(const tq_context* ctx, int32_t max_seq) {
  if (!ctx || max_seq < 0) return 0;
  return decode_workspace_bytes(ctx, max_seq);
}

static tq_status check_lengths(const tq_context* ctx, const int32_t* seq_len, int* max_seq) {
  *max_seq = 0;
  for (int b = 0; b < ctx->cfg.batch; ++b) {
    if (seq_len[b] < 0) return fail(TQ_ERR_INVALID_ARG, "seq_len must be >= 0");
    if (seq_len[b] > ctx->cfg.capacity) return fail(TQ_ERR_CAPACITY, "seq_len > capacity");
    if (seq_len[b] > *max_seq) *max_seq = seq_len[b];
  }
  return TQ_OK;
}

tq_status tq_decode_attention(const tq_context* ctx, const void* dev_cache, const float* q,
                              const int32_t* host_seq_len, float* out, void* ws, size_t ws_bytes,
                              tq_stream stream) {
  tq_status s = ready(ctx);
  if (s != TQ_OK) return s;
  if (!dev_cache || !q || !host_seq_len || !out || !ws) return fail(TQ_ERR_INVALID_ARG, "null argument");
  if (!aligned(dev_cache, 256) || !aligned(q, 16) || !aligned(out, 16) || !aligned(ws, 256))
    return fail(TQ_ERR_INVALID_ARG, "misaligned pointer (cache/ws 256 B, q/out 16 B)");
  int max_seq;
  s = check_lengths(ctx, host_seq_len, &max_seq);
  if (s != TQ_OK) return s;
  if (ws_bytes < decode_workspace_bytes(ctx, max_seq)) return fail(TQ_ERR_WORKSPACE, "workspace too small");
  return launch_decode(ctx, dev_cache, q, host_seq_len, out, ws, ws_bytes, stream);
}

tq_status tq_append_decode_attention(const tq_context* ctx, void* dev_cache, const void* k, const void* v,
                                     tq_dtype dtype, int32_t n_new, const float* q,
                                     const int32_t* host_seq_len, float* out, void* ws, size_t ws_bytes,
                                     tq_stream stream) {
  tq_status s = ready(ctx);
  if (s != TQ_OK) return s;
  if (n_new < 0) return fail(TQ_ERR_INVALID_ARG, "n_new must be >= 0");
  if (!dev_cache || !q || !host_seq_len || !out || !ws) return fail(TQ_ERR_INVALID_ARG, "null argument");
  if (n_new > 0) {
    if (!k || !v) return fail(TQ_ERR_INVALID_ARG, "null argument");
    if (dtype != TQ_F32 && dtype != TQ_BF16 && dtype != TQ_F16) return fail(TQ_ERR_INVALID_ARG, "bad dtype");
    if (!aligned(k, 16) || !aligned(v, 16)) return fail(TQ_ERR_INVALID_ARG, "k, v must be 16-byte aligned");
  }
  if (!aligned(dev_cache, 256) || !aligned(q, 16) || !aligned(out, 16) || !aligned(ws, 256))
    return fail(TQ_ERR_INVALID_ARG, "misaligned pointer (cache/ws 256 B, q/out 16 B)");
  int max_seq;
  s = check_lengths(ctx, host_seq_len, &max_seq);
  if (s != TQ_OK) return s;
  if (ws_bytes < decode_workspace_bytes(ctx, max_seq)) return fail(TQ_ERR_WORKSPACE, "workspace too small");
  if (n_new == 0) return launch_decode(ctx, dev_cache, q, host_seq_len, out, ws, ws_bytes, stream);
  std::vector<int32_t> start((size_t)ctx->cfg.batch);
  for (int b = 0; b < ctx->cfg.batch; ++b) {
    if (host_seq_len[b] < n_new) return fail(TQ_ERR_INVALID_ARG, "seq_len must be >= n_new");
    start[(size_t)b] = host_seq_len[b] - n_new;
  }
  if (ctx->cfg.head_dim != 128) {  // the two calls in stream order
    s = launch_append(ctx, dev_cache, k, v, dtype, n_new, start.data(), stream);
    if (s != TQ_OK) return s;
    return launch_decode(ctx, dev_cache, q, host_seq_len, out, ws, ws_bytes, stream);
  }
  s = launch_append_early(ctx, dev_cache, k, v, dtype, n_new, start.data(), stream);
  if (s != TQ_OK) return s;
  return launch_decode_after_append(ctx, dev_cache, q, host_seq_len, n_new, out, ws, stream);
}

tq_status tq_decode_attention_multi(const tq_context* ctx, const void* dev_cache, const float* q,
                                    int32_t nq, const int32_t* host_seq_len, float* out, void* ws,
                                    size_t ws_bytes, tq_stream stream) {
  tq_status s = ready(ctx);
  if (s != TQ_OK) return s;
  if (!dev_cache || !q || !host_seq_len || !out || !ws) return fail(TQ_ERR_INVALID_ARG, "null argument");
  if (nq < 1) return fail(TQ_ERR_INVALID_ARG, "nq must be >= 1");
  const int G = ctx->cfg.num_q_heads / ctx->cfg.num_kv_heads;
  if (nq > 1 && (ctx->cfg.head_dim != 128 || (int64_t)G * nq > 8))
    return fail(TQ_ERR_UNSUPPORTED, "several queries per sequence are built for head_dim 128 with G * nq <= 8");
  if (!aligned(dev_cache, 256) || !aligned(q, 16) || !aligned(out, 16) || !aligned(ws, 256))
    return fail(TQ_ERR_INVALID_ARG, "misaligned pointer (cache/ws 256 B, q/out 16 B)");
  int max_seq;
  s = check_lengths(ctx, host_seq_len, &max_seq);
  if (s != TQ_OK) return s;
  if (ws_bytes < decode_workspace_bytes(ctx, max_seq)) return fail(TQ_ERR_WORKSPACE, "workspace too small");
  return launch_decode_multi(ctx, dev_cache, q, nq, host_seq_len, out, ws, ws_bytes, stream);
}

size_t tq_prefill_workspace_bytes(const tq_context* ctx, int32_t nq) {
  if (!ctx || nq < 1) return 0;
  return prefill_workspace_bytes(ctx, nq);
}

tq_status tq_prefill_attention(const tq_context* ctx, const void* dev_cache, const float* q, int32_t nq,
                               const int32_t* host_seq_len, float* out, void* ws, size_t ws_bytes,
                               tq_stream stream) {
  tq_status s = ready(ctx);
  if (s != TQ_OK) return s;
  if (!dev_cache || !q || !host_seq_len || !out || !ws) return fail(TQ_ERR_INVALID_ARG, "null argument");
  if (nq < 1) return fail(TQ_ERR_INVALID_ARG, "nq must be >= 1");
  if (ctx->cfg.head_dim != 128 || ctx->m != 128)
    return fail(TQ_ERR_UNSUPPORTED, "prefill attention is built for head_dim 128 (m = 128)");
  if (ctx->cfg.headq_rank || ctx->cfg.k.rotate == 2 || ctx->cfg.v.rotate == 2)
    return fail(TQ_ERR_UNSUPPORTED, "prefill attention is not built for HeadQ or spectral codecs");
  if ((int64_t)ctx->cfg.batch * ctx->cfg.num_kv_heads > 65535)
    return fail(TQ_ERR_UNSUPPORTED, "prefill attention takes at most 65535 (batch, KV head) slabs");
  if ((int64_t)nq * (ctx->cfg.num_q_heads / ctx->cfg.num_kv_heads) > (int64_t)1 << 24)
    return fail(TQ_ERR_INVALID_ARG, "nq too large");
  if (!aligned(dev_cache, 256) || !aligned(q, 16) || !aligned(out, 16) || !aligned(ws, 256))
    return fail(TQ_ERR_INVALID_ARG, "misaligned pointer (cache/ws 256 B, q/out 16 B)");
  int max_seq;
  s = check_lengths(ctx, host_seq_len, &max_seq);
  if (s != TQ_OK) return s;
  if (ws_bytes < prefill_workspace_bytes(ctx, nq)) return fail(TQ_ERR_WORKSPACE, "workspace too small");
  return launch_prefill(ctx, dev_cache, q, nq, host_seq_len, out, ws, stream);
}

tq_status tq_decode_attention_static(const tq_context* ctx, const void* dev_cache, const float* q,
                                     const int32_t* host_seq_len, float* out, tq_stream stream) {
  tq_status s = ready(ctx);
  if (s != TQ_OK) return s;
  if (!dev_cache || !q || !host_seq_len || !out) return fail(TQ_ERR_INVALID_ARG, "null argument");
  if (!aligned(dev_cache, 256) || !aligned(q, 16) || !aligned(out, 16))
    return fail(TQ_ERR_INVALID_ARG, "misaligned pointer (cache 256 B, q/out 16 B)");
  int max_seq;
  s = check_lengths(ctx, host_seq_len, &max_seq);
  if (s != TQ_OK) return s;
  const size_t need = decode_workspace_bytes(ctx, max_seq);
  if (need > TQ_STATIC_SCRATCH_BYTES)
    return fail(TQ_ERR_WORKSPACE, "this configuration needs " + std::to_string(need) +
                                      " bytes of decode scratch; the built-in scratch holds " +
                                      std::to_string((size_t)TQ_STATIC_SCRATCH_BYTES) +
                                      " (use tq_decode_attention with a caller workspace)");
  void* ws = nullptr;
  s = static_scratch(&ws);
  if (s != TQ_OK) return s;
  return launch_decode(ctx, dev_cache, q, host_seq_len, out, ws, TQ_STATIC_SCRATCH_BYTES, stream);
}

tq_status tq_headq_correct(const tq_context* ctx, const void* dev_cache, const float* q,
                           const int32_t* host_seq_len, float* logits, int32_t logits_stride,
                           tq_stream stream) {
  tq_status s = ready(ctx);
  if (s == TQ_OK && ctx->cfg.k.rotate == 2)
    return fail(TQ_ERR_UNSUPPORTED, "corrected logits are not built for the spectral codec");
  if (s != TQ_OK) return s;
  if (!dev_cache || !q || !host_seq_len || !logits) return fail(TQ_ERR_INVALID_ARG, "null argument");
  if (!aligned(dev_cache, 256) || !aligned(q, 16) || !aligned(logits, 4))
    return fail(TQ_ERR_INVALID_ARG, "misaligned pointer");
  int max_seq;
  s = check_lengths(ctx, host_seq_len, &max_seq);
  if (s != TQ_OK) return s;
  if (logits_stride < max_seq) return fail(TQ_ERR_INVALID_ARG, "logits_stride < max(seq_len)");
  return launch_logits(ctx, dev_cache, q, host_seq_len, logits, logits_stride, stream);
}

tq_status tq_dequantize(const tq_context* ctx, const void* dev_cache, int32_t b, int32_t kvh,
                        int32_t t0, int32_t t1, float* k_out, float* v_out, tq_stream stream) {
  tq_status s = ready(ctx);
  if (s != TQ_OK) return s;
  if (!dev_cache || !k_out || !v_out) return fail(TQ_ERR_INVALID_ARG, "null argument");
  if (b < 0 || b >= ctx->cfg.batch || kvh < 0 || kvh >= ctx->cfg.num_kv_heads)
    return fail(TQ_ERR_INVALID_ARG, "slab index out of range");
  if (t0 < 0 || t1 < t0 || t1 > ctx->cfg.capacity) return fail(TQ_ERR_INVALID_ARG, "token range out of range");
  if (t1 == t0) return TQ_OK;
  if (!aligned(dev_cache, 256) || !aligned(k_out, 16) || !aligned(v_out, 16))
    return fail(TQ_ERR_INVALID_ARG, "misaligned pointer");
  return launch_dequantize(ctx, dev_cache, b, kvh, t0, t1, k_out, v_out, stream);
}

tq_status tq_get_device_error(const void* ws, int32_t* code, tq_stream stream) {
  if (!ws || !code) return fail(TQ_ERR_INVALID_ARG, "null argument");
  return read_device_error(ws, code, stream);
}

tq_status tq_get_static_device_error(int32_t* code, tq_stream stream) {
  if (!code) return fail(TQ_ERR_INVALID_ARG, "null argument");
  return read_static_device_error(code, stream);
}

}  // extern "C"
