// Read path launchers: query preparation, fused split-K decode, corrected logits.
#include <mutex>
#include <string>

#include "tq_decode_kernel.cuh"
#include "tq_decode_wide.cuh"

namespace tqd {
namespace {

constexpr int kLogitsTokensPerBlock = 2048;
constexpr float kLog2e = 1.4426950408889634f;

struct WsLayout {
  size_t err, tickets, q_rot, q_sk, q_u, q_rot_lo, q_sk_lo, part, sk_final, sk_part, total;
  int ps;
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// The workspace does not depend on the sequence lengths: partial slots are reserved for every
// slab plus one per possible block.
WsLayout ws_layout(const tq_context* ctx) {
  WsLayout w;
  const int B = ctx->cfg.batch, Hkv = ctx->cfg.num_kv_heads, Hq = ctx->cfg.num_q_heads;
  const int D = ctx->cfg.head_dim;
  const int pairs = B * Hkv;
  w.ps = 4 + D + (ctx->cfg.v.qjl ? ctx->m : 0);
  size_t off = 0;
  w.err = off; off = align256(off + 64 * sizeof(int));
  w.tickets = off; off = align256(off + (size_t)pairs * sizeof(int));
  // eight query columns per KV head (queries of the chunk x heads of the group, then the lo
  // terms of the queries when they fit); partial slots for up to 8 columns at head dim 128
  const size_t cols = (size_t)Hkv * kQCols;
  w.q_rot = off; off = align256(off + (size_t)B * cols * D * 2);
  w.q_sk = off; off = align256(off + (ctx->cfg.k.qjl ? (size_t)B * cols * ctx->m * 2 : 0));
  w.q_u = off; off = align256(off + (ctx->cfg.headq_rank ? (size_t)B * cols * 16 * 2 : 0));
  w.q_rot_lo = off; off = align256(off + (D == kDecD ? (size_t)B * cols * D * 2 : 0));
  w.q_sk_lo = off; off = align256(off + (D == kDecD && ctx->cfg.k.qjl ? (size_t)B * cols * ctx->m * 2 : 0));
  const size_t pcols = D == kDecD ? kHeadsPad : Hq / Hkv;
  w.part = off; off = align256(off + (size_t)(pairs + kMaxBlocks) * pcols * w.ps * sizeof(float));
  const bool wide_vq = D > kDecD && ctx->cfg.v.qjl;  // acc_sk / l per head for the sketch pass
  w.sk_final = off; off = align256(off + (wide_vq ? (size_t)B * Hq * ctx->m * sizeof(float) : 0));
  w.sk_part = off; off = align256(off + (wide_vq ? (size_t)(ctx->m / kSkRows) * B * Hq * D * sizeof(float) : 0));
  w.total = off;
  return w;
}

// Number of SMs of the current device (the decode runs one block per SM).
int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return kMaxBlocks;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return kMaxBlocks;
  return n < kMaxBlocks ? n : kMaxBlocks;
}

struct PrepParams {
  Tables tab;
  const float* q;
  uint32_t* q_rot;
  uint32_t* q_sk;
  uint32_t* q_u;
  uint32_t* q_rot_lo;  // lo terms when they do not fit the spare columns (else nullptr)
  uint32_t* q_sk_lo;
  int* tickets;
  int* err;
  float* out;
  float* sk_final;  // zeroed for empty sequences (head dim > 128 with a QJL value side)
  int n_tickets, n_heads, Hq, Hkv, G, Gc, nq, k_rotate, kq, kh, m, B;
  int after_append;  // launched as the programmatic dependent of a decode step's append
  int seq_len[TQ_MAX_BATCH];
  const int* dev_seq_len;  // set: lengths from device memory, clamped to [0, lmax] (the decode
  int lmax;                // blocks compute the work split from them)
  __device__ __forceinline__ int len(int b) const {
    if (!dev_seq_len) return seq_len[b];
    const int L = __ldg(dev_seq_len + b);
    return L < 0 ? 0 : (L > lmax ? lmax : L);
  }
};

// E values as fp16 pairs at hi and their fp16 remainders (x - hi) at lo.
template <int E>
__device__ __forceinline__ void store_hi_lo(uint32_t* hi, uint32_t* lo, const float (&x)[E]) {
  uint32_t h[E / 2], l[E / 2];
#pragma unroll
  for (int i = 0; i < E; i += 2) {
    const __half2 hh = __floats2half2_rn(x[i], x[i + 1]);
    const float2 hf = __half22float2(hh);
    h[i / 2] = *reinterpret_cast<const uint32_t*>(&hh);
    l[i / 2] = pack_half2(x[i] - hf.x, x[i + 1] - hf.y);
  }
#pragma unroll
  for (int i = 0; i < E / 2; i += 2) {
    *reinterpret_cast<uint2*>(hi + i) = make_uint2(h[i], h[i + 1]);
    *reinterpret_cast<uint2*>(lo + i) = make_uint2(l[i], l[i + 1]);
  }
}

// Per query column (one warp, E = D / 32 coordinates per lane; columns [B][Hkv][Gc], column c
// = query c / G of the sequence, head c % G of the KV head's group): q_rot = R_K q; for head
// dim 128 also S_K q_rot for a QJL key side and U_rot^T q_rot = U^T q for HeadQ; stored as fp16
// pairs.  Block 0 also clears the split tickets and the error word; queries of empty sequences
// get a zero output (no decode block writes them).
template <int D>
__device__ __forceinline__ void prep_body(const PrepParams& p) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  extern __shared__ __align__(16) float skt_smem[];
  const float* SKT = p.tab.S_K_T;
  if (D == kDecD && p.kq) {  // S_K^T (64 KiB) into shared memory: 128 dependent rows per head
    stage_table<256>(skt_smem, SKT, D * D);
    __syncthreads();
    SKT = skt_smem;
  }
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < p.n_tickets; i += blockDim.x) p.tickets[i] = 0;
    if (threadIdx.x == 0) p.err[0] = 0;
  }
  const int head = blockIdx.x * 8 + (threadIdx.x >> 5);  // flat column index
  if (head >= p.n_heads) return;
  const int b = head / (p.Hkv * p.Gc), r = head % (p.Hkv * p.Gc);
  const int kvh = r / p.Gc, c = r % p.Gc;
  const long long qrow = ((long long)b * p.nq + c / p.G) * p.Hq + kvh * p.G + c % p.G;  // [B][nq][Hq]
  if (p.len(b) == 0) {
#pragma unroll
    for (int e = 0; e < E; e += 4)
      *reinterpret_cast<float4*>(p.out + qrow * D + lane * E + e) = make_float4(0.f, 0.f, 0.f, 0.f);
    if (p.sk_final)
      for (int i = lane; i < p.m; i += 32) p.sk_final[qrow * p.m + i] = 0.f;
  }
  float x[E];
  load_row<E>(p.q + qrow * D + lane * E, x);
  if (p.k_rotate == 2) {
    // SQU-KV keys: q_c = s_c sum_i E[i][c] q_i (the basis and scales of KV head kvh), so that
    // <q_c, z_hat_c> summed over stored coordinates is q^T E (s z_hat)
    float y[E];
#pragma unroll
    for (int i = 0; i < E; ++i) y[i] = 0.f;
    const float* Eh = p.tab.sq_E[0] + (long long)kvh * D * D + lane * E;
    for (int sl = 0; sl < 32; ++sl) {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float qi = __shfl_sync(kFull, x[e], sl);
#pragma unroll
        for (int i = 0; i < E; ++i) y[i] = fmaf(__ldg(Eh + (E * sl + e) * D + i), qi, y[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < E; ++i) x[i] = y[i] * __ldg(p.tab.sq_s[0] + (long long)kvh * D + lane * E + i);
  } else {
#pragma unroll
    for (int i = 0; i < E; ++i) x[i] *= __ldg(p.tab.k_sign + lane * E + i);
    if (p.k_rotate) {
      wht_warp<E>(x);
      const float rs = 1.f / sqrtf((float)D);
#pragma unroll
      for (int i = 0; i < E; ++i) x[i] *= rs;
    }
  }
  // hi term to column c, lo term (x - hi) to column Gc + c or to the separate lo array
  const long long col = ((long long)b * p.Hkv + kvh) * kQCols + c;
  const long long col_lo = p.q_rot_lo ? col : col + p.Gc;
  uint32_t* lo_base = p.q_rot_lo ? p.q_rot_lo : p.q_rot;
  store_hi_lo<E>(p.q_rot + col * (D / 2) + lane * (E / 2), lo_base + col_lo * (D / 2) + lane * (E / 2), x);
  if constexpr (D == kDecD) {
    if (p.kq) {
      float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
      for (int jl = 0; jl < 32; ++jl) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float xj = __shfl_sync(kFull, x[e], jl);
          const float4 s4 = *reinterpret_cast<const float4*>(SKT + (4 * jl + e) * D + 4 * lane);
          a[0] = fmaf(s4.x, xj, a[0]); a[1] = fmaf(s4.y, xj, a[1]);
          a[2] = fmaf(s4.z, xj, a[2]); a[3] = fmaf(s4.w, xj, a[3]);
        }
      }
      uint32_t* sk_lo = p.q_sk_lo ? p.q_sk_lo : p.q_sk;
      store_hi_lo<4>(p.q_sk + col * (D / 2) + 2 * lane, sk_lo + col_lo * (D / 2) + 2 * lane, a);
    }
    if (p.kh) {
      const float* Ur = p.tab.U_rot + (long long)kvh * D * 16;
      float z[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) z[k] = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
#pragma unroll
        for (int k = 0; k < 16; k += 4) {
          const float4 u4 = __ldg(reinterpret_cast<const float4*>(Ur + (4 * lane + e) * 16 + k));
          z[k] = fmaf(u4.x, x[e], z[k]); z[k + 1] = fmaf(u4.y, x[e], z[k + 1]);
          z[k + 2] = fmaf(u4.z, x[e], z[k + 2]); z[k + 3] = fmaf(u4.w, x[e], z[k + 3]);
        }
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) z[k] = warp_sum(z[k]);
      if (lane == 0) {
        uint32_t* dst = p.q_u + col * 8;
#pragma unroll
        for (int k = 0; k < 8; ++k) dst[k] = pack_half2(z[2 * k], z[2 * k + 1]);
      }
    }
  }
}

// The decode launched after this kernel may start its own setup at once: it waits for this
// kernel's results before reading them.  In a decode step (after_append) this kernel is itself
// the programmatic dependent of the step's append, whose output it never reads: it waits for the
// append only before exiting, so its completion -- what the decode waits for -- implies the
// append's.
template <int D>
__global__ void __launch_bounds__(256) prep_kernel(const PrepParams p) {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  prep_body<D>(p);
  if (p.after_append) asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

tq_status cuda_fail(const char* what, cudaError_t e) {
  tqi::set_error(std::string(what) + ": " + cudaGetErrorString(e));
  return TQ_ERR_CUDA;
}

}  // namespace
}  // namespace tqd

namespace tqi {

size_t decode_workspace_bytes(const tq_context* ctx, int max_seq) {
  (void)max_seq;
  return tqd::ws_layout(ctx).total;
}

static bool dispatch_decode(const tq_context* ctx, const tqd::DecodeParams& p, dim3 grid,
                            cudaStream_t s, cudaError_t* e) {
  using namespace tqd;
  // code-width tag of the decode templates: kSQ for a spectral (SQU-KV) side
  const int kb = ctx->cfg.k.rotate == 2 ? kSQ : ctx->cfg.k.bits, kq = ctx->cfg.k.qjl;
  const int kh = ctx->cfg.headq_rank ? 1 : 0;
  const int vb = ctx->cfg.v.rotate == 2 ? kSQ : ctx->cfg.v.bits, vq = ctx->cfg.v.qjl;
  if (ctx->cfg.head_dim != kDecD) {
    if (kq || kh) return false;
    switch (ctx->cfg.head_dim) {
      case 256: return dispatch_decode_wide_d256(kb, vb, vq, p, grid, s, e);
      case 512: return dispatch_decode_wide_d512(kb, vb, vq, p, grid, s, e);
      case 1024: return dispatch_decode_wide_d1024(kb, vb, vq, p, grid, s, e);
    }
    return false;
  }
  switch (kb) {
    case 1: return dispatch_decode_k1(kq, kh, vb, vq, p, grid, s, e);
    case 2: return dispatch_decode_k2(kq, kh, vb, vq, p, grid, s, e);
    case 3: return dispatch_decode_k3(kq, kh, vb, vq, p, grid, s, e);
    case 4: return dispatch_decode_k4(kq, kh, vb, vq, p, grid, s, e);
    case kSQ: return dispatch_decode_ksq(kq, kh, vb, vq, p, grid, s, e);
  }
  return false;
}

tq_status launch_decode(const tq_context* ctx, const void* cache, const float* q,
                        const int32_t* seq_len, float* out, void* ws, size_t ws_bytes,
                        Stream stream) {
  return launch_decode_multi(ctx, cache, q, 1, seq_len, out, ws, ws_bytes, stream);
}

// Paged pool and device lengths (tq_decode_attention_paged), or none (host lengths).
struct PagedDecode {
  const tq_page_table* pt;
  const int32_t* dev_seq_len;
};

// n_fresh > 0: a decode step right after launch_append_early on the same stream (head dim 128,
// contiguous cache), whose tokens are each sequence's last n_fresh.
static tq_status decode_impl(const tq_context* ctx, const void* cache, const float* q, int nq,
                             const int32_t* seq_len, const PagedDecode* pg, float* out, void* ws,
                             Stream stream, int n_fresh = 0) {
  using namespace tqd;
  const int D = ctx->cfg.head_dim;
  const WsLayout w = ws_layout(ctx);
  unsigned char* base = (unsigned char*)ws;
  const cudaStream_t s = (cudaStream_t)stream;
  const Tables tab = make_tables(ctx);
  const int B = ctx->cfg.batch, Hkv = ctx->cfg.num_kv_heads, Hq = ctx->cfg.num_q_heads;

  DecodeParams p;
  if (!dispatch_decode(ctx, p, dim3(1), s, nullptr)) {  // probe only: nothing launches
    set_error("decode attention is not built for this combination of key and value codecs");
    return TQ_ERR_UNSUPPORTED;
  }

  PrepParams pp;
  pp.tab = tab;
  pp.q = q;
  pp.q_rot = (uint32_t*)(base + w.q_rot);
  pp.q_sk = (uint32_t*)(base + w.q_sk);
  pp.q_u = (uint32_t*)(base + w.q_u);
  const int Gc = (Hq / Hkv) * nq;
  // the lo terms go to a separate array when they do not fit the spare columns, or when Gc is odd
  // and above 1: the shuffle that adds them back pairs lanes, which takes an even Gc
  const bool lo_sep = 2 * Gc > kQCols || (Gc > 1 && Gc % 2);
  if (lo_sep && D != kDecD) {
    set_error("head dims above 128 are built for H_q / H_kv <= 4");
    return TQ_ERR_UNSUPPORTED;
  }
  pp.q_rot_lo = lo_sep ? (uint32_t*)(base + w.q_rot_lo) : nullptr;
  pp.q_sk_lo = lo_sep ? (uint32_t*)(base + w.q_sk_lo) : nullptr;
  pp.tickets = (int*)(base + w.tickets);
  pp.err = (int*)(base + w.err);
  pp.n_tickets = B * Hkv;
  pp.n_heads = B * Hq * nq;
  pp.Hq = Hq;
  pp.Hkv = Hkv;
  pp.G = Hq / Hkv;
  pp.nq = nq;
  pp.Gc = pp.G * nq;
  pp.k_rotate = ctx->cfg.k.rotate;
  pp.kq = ctx->cfg.k.qjl;
  pp.kh = ctx->cfg.headq_rank ? 1 : 0;
  pp.out = out;
  const bool wide_vq = D > kDecD && ctx->cfg.v.qjl;
  pp.sk_final = wide_vq ? (float*)(base + w.sk_final) : nullptr;
  pp.m = ctx->m;
  pp.B = B;
  for (int b = 0; b < TQ_MAX_BATCH; ++b) pp.seq_len[b] = (!pg && b < B) ? seq_len[b] : 0;
  pp.dev_seq_len = pg ? pg->dev_seq_len : nullptr;
  pp.lmax = pg ? kTile * pg->pt->max_blocks_per_seq : 0;
  pp.after_append = n_fresh > 0 ? 1 : 0;
  if (n_fresh > 0 && (pg || D != kDecD)) {
    set_error("the overlapped decode step is built for a contiguous cache at head dim 128");
    return TQ_ERR_UNSUPPORTED;
  }
  if (pg && D != kDecD) {
    set_error("the paged decode is built for head dim 128");
    return TQ_ERR_UNSUPPORTED;
  }
  const dim3 pgrid((B * Hq * nq + 7) / 8);
  const int psmem = (D == kDecD && pp.kq) ? kDecD * kDecD * 4 : 0;
  if (psmem) {
    cudaError_t ae = cudaFuncSetAttribute(prep_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, psmem);
    if (ae != cudaSuccess) return cuda_fail("decode prep", ae);
  }
  if (pp.after_append) {  // the programmatic dependent of the step's append (head dim 128)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = pgrid;
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = (size_t)psmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t le = cudaLaunchKernelEx(&cfg, prep_kernel<128>, pp);
    if (le != cudaSuccess) return cuda_fail("decode prep", le);
  } else switch (D) {
    case 128: prep_kernel<128><<<pgrid, 256, psmem, s>>>(pp); break;
    case 256: prep_kernel<256><<<pgrid, 256, 0, s>>>(pp); break;
    case 512: prep_kernel<512><<<pgrid, 256, 0, s>>>(pp); break;
    default: prep_kernel<1024><<<pgrid, 256, 0, s>>>(pp); break;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail("decode prep", e);

  p.tab = tab;
  p.cache = pg ? make_paged_cache(ctx, cache, *pg->pt, pp.err) : make_cache(ctx, cache);
  p.dev_seq_len = pp.dev_seq_len;
  p.lmax = pp.lmax;
  p.q_rot = pp.q_rot;
  p.q_sk = pp.q_sk;
  p.q_u = pp.q_u;
  p.q_rot_lo = pp.q_rot_lo;
  p.q_sk_lo = pp.q_sk_lo;
  p.lo_xor = lo_sep ? 0 : (Gc == 1 ? -1 : Gc / 2);
  p.part = (float*)(base + w.part);
  p.tickets = pp.tickets;
  p.out = out;
  p.B = B;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.nq = nq;
  p.Gc = p.G * nq;
  p.v_rotate = ctx->cfg.v.rotate;
  p.sk_final = pp.sk_final;
  p.score_scale = kLog2e / sqrtf((float)D);
  p.qjl_scale = (float)(1.2533141373155003 / ctx->m);
  p.err = pp.err;
  p.n_fresh = n_fresh;
  long long W = 0;  // 16-token tiles over all slabs
  for (int b = 0; b < TQ_MAX_BATCH; ++b) {
    p.seq_len[b] = pp.seq_len[b];
    p.batch_start[b] = W;
    W += (long long)Hkv * ((p.seq_len[b] + kTile - 1) / kTile);
  }
  p.batch_start[TQ_MAX_BATCH] = W;
  p.W = W;
  const int nsm = sm_count();
  if (pg) {
    p.nblocks = nsm;  // the split is computed on the device; blocks with an empty range exit
  } else {
    if (W == 0) return TQ_OK;  // every sequence is empty: prep wrote the zero outputs
    p.nblocks = W < nsm ? (int)W : nsm;  // every block gets a non-empty range
  }
  e = cudaSuccess;
  dispatch_decode(ctx, p, dim3(p.nblocks), s, &e);
  if (e != cudaSuccess) return cuda_fail("decode", e);
  if (wide_vq) {  // out += sqrt(pi/2)/m (S_V R_V)^T acc_sk / l, all heads in one pass
    e = launch_finalize_sketch(D, tab.S_V_R, pp.sk_final, (float*)(base + w.sk_part), out, B * Hq, ctx->m,
                               p.qjl_scale, s);
    if (e != cudaSuccess) return cuda_fail("decode sketch finalize", e);
  }
  return TQ_OK;
}

tq_status launch_decode_multi(const tq_context* ctx, const void* cache, const float* q, int nq,
                              const int32_t* seq_len, float* out, void* ws, size_t ws_bytes,
                              Stream stream) {
  (void)ws_bytes;
  return decode_impl(ctx, cache, q, nq, seq_len, nullptr, out, ws, stream);
}

tq_status launch_decode_after_append(const tq_context* ctx, const void* cache, const float* q,
                                     const int32_t* seq_len, int n_fresh, float* out, void* ws,
                                     Stream stream) {
  return decode_impl(ctx, cache, q, 1, seq_len, nullptr, out, ws, stream, n_fresh);
}

tq_status launch_decode_paged(const tq_context* ctx, const void* pool, const tq_page_table* pt,
                              const float* q, int nq, const int32_t* dev_seq_len, float* out, void* ws,
                              size_t ws_bytes, Stream stream) {
  (void)ws_bytes;
  const PagedDecode pg{pt, dev_seq_len};
  return decode_impl(ctx, pool, q, nq, nullptr, &pg, out, ws, stream);
}

tq_status launch_logits(const tq_context* ctx, const void* cache, const float* q,
                        const int32_t* seq_len, float* logits, int stride, Stream stream) {
  using namespace tqd;
  if (ctx->cfg.head_dim != kDecD) {
    set_error("corrected logits are built for head_dim 128");
    return TQ_ERR_UNSUPPORTED;
  }
  const int B = ctx->cfg.batch, Hkv = ctx->cfg.num_kv_heads, Hq = ctx->cfg.num_q_heads;
  int max_seq = 0;
  for (int b = 0; b < B; ++b) max_seq = seq_len[b] > max_seq ? seq_len[b] : max_seq;
  if (max_seq == 0) return TQ_OK;
  LogitsParams p;
  p.tab = make_tables(ctx);
  p.cache = make_cache(ctx, cache);
  p.q = q;
  p.logits = logits;
  p.B = B;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.stride = stride;
  p.tokens_per_block = kLogitsTokensPerBlock;
  p.k_rotate = ctx->cfg.k.rotate;
  p.qjl_scale = (float)(1.2533141373155003 / ctx->m);
  p.inv_sqrt_d = 1.f / sqrtf((float)kDecD);
  for (int b = 0; b < TQ_MAX_BATCH; ++b) p.seq_len[b] = b < B ? seq_len[b] : 0;
  const dim3 grid((max_seq + kLogitsTokensPerBlock - 1) / kLogitsTokensPerBlock, Hkv, B);
  const int kq = ctx->cfg.k.qjl, kh = ctx->cfg.headq_rank ? 1 : 0;
  cudaError_t e = cudaSuccess;
  bool built = false;
  switch (ctx->cfg.k.bits) {
    case 1: built = dispatch_logits_k1(kq, kh, p, grid, (cudaStream_t)stream, &e); break;
    case 2: built = dispatch_logits_k2(kq, kh, p, grid, (cudaStream_t)stream, &e); break;
    case 3: built = dispatch_logits_k3(kq, kh, p, grid, (cudaStream_t)stream, &e); break;
    case 4: built = dispatch_logits_k4(kq, kh, p, grid, (cudaStream_t)stream, &e); break;
  }
  if (!built) {
    set_error("corrected logits are not built for this key codec");
    return TQ_ERR_UNSUPPORTED;
  }
  if (e != cudaSuccess) return cuda_fail("logits", e);
  return TQ_OK;
}

// Built-in scratch of tq_decode_attention_static.  In host code the array's name is only a
// stand-in, so its device address is looked up once per device and cached.
static __device__ __align__(256) unsigned char g_tq_static_scratch[TQ_STATIC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {nullptr};
}  // namespace

tq_status static_scratch(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return tqd::cuda_fail("cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("device ordinal out of range for the static scratch");
    return TQ_ERR_INVALID_ARG;
  }
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_tq_static_scratch);
    if (e != cudaSuccess) return tqd::cuda_fail("cudaGetSymbolAddress(static scratch)", e);
    g_static_ptr[dev] = p;
  }
  *ptr = g_static_ptr[dev];
  return TQ_OK;
}

tq_status read_static_device_error(int32_t* code, Stream stream) {
  void* ws = nullptr;
  tq_status s = static_scratch(&ws);
  if (s != TQ_OK) return s;
  return read_device_error(ws, code, stream);
}

tq_status read_device_error(const void* ws, int32_t* code, Stream stream) {
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return tqd::cuda_fail("stream synchronize", e);
  e = cudaMemcpy(code, ws, sizeof(int32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return tqd::cuda_fail("read error word", e);
  return *code ? TQ_ERR_DEVICE : TQ_OK;
}

}  // namespace tqi
