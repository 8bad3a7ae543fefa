/*
 * tq.h -- C ABI of the rotated-codebook quantized KV cache for NVIDIA GB300 (sm_103a).
 *
 * The method (three technical summaries of papers, cited by page title and section):
 *   [TQ-KV] "Resumen Técnico: Inferencia Estadística y Medidas de Calidad de Cuantizaciones
 *           de Cache KV Inspiradas en TurboQuant" (gist.science/es/paper/2605.08114)
 *   [ABL]   "Resumo Técnico: Ablação, Inferência Estatística e Validação para Compressão de
 *           KV-Cache" (gist.science/pt/paper/2607.09683)
 *   [HEADQ] "Resumo Técnico: HeadQ: Distorção Visível ao Modelo e Correção no Espaço de
 *           Pontuação para Quantização de KV-Cache" (gist.science/pt/paper/2605.03562)
 *
 * Write path (tq_quantize_append): per K/V vector, split off the norm, rotate the unit vector
 * with a seeded randomized Walsh-Hadamard transform y = H D u / sqrt(d), quantize each
 * coordinate with a Lloyd-Max codebook for the Beta((d-1)/2,(d-1)/2) sphere marginal, pack the
 * codes; optionally store a 1-bit QJL sketch sign(S r) of the residual r plus ||r||, and for
 * HeadQ keys a 4-bit side code of the residual projected on a calibrated basis.
 * Read path (tq_decode_attention): one fused split-K kernel reads the packed cache, forms
 * scores (with the QJL or HeadQ logit corrections), runs an online softmax and accumulates the
 * value readout (with the QJL value correction); a last-arriving block per (batch, KV head)
 * merges the splits and applies the inverse rotation.
 *
 * Conventions shared by every entry point:
 *   - The caller owns all device memory and all streams.  The library allocates no device
 *     memory and never synchronizes, except tq_get_device_error, which waits on its stream.
 *   - Calls are asynchronous and ordered on the given stream (a cudaStream_t; 0 = default).
 *   - Arguments, capacity and workspace sizes are checked on the host before any launch; a
 *     failed check launches nothing and returns the error.  Launch failures return
 *     TQ_ERR_CUDA.  tq_last_error() gives a message for the calling thread's last error.
 *   - A context is host memory.  It is read-only after tq_tables_upload (and
 *     tq_headq_set_basis), and may then be shared by threads.
 *   - Device pointers must be 16-byte aligned; the cache and table buffers 256-byte aligned.
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, spelled without the CUDA headers. */
typedef struct CUstream_st* tq_stream;

typedef enum {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer, bad enum        */
  TQ_ERR_UNSUPPORTED = 2,  /* valid but not built: head_dim, G, bit width combination      */
  TQ_ERR_CAPACITY = 3,     /* start + n_new or a sequence length beyond the cache capacity */
  TQ_ERR_WORKSPACE = 4,    /* workspace smaller than tq_decode_workspace_bytes             */
  TQ_ERR_CUDA = 5,         /* a CUDA runtime call or kernel launch failed                  */
  TQ_ERR_DEVICE = 6,       /* a kernel recorded an error word (see tq_get_device_error)    */
  TQ_ERR_STATE = 7         /* tables not uploaded / HeadQ basis not set                    */
} tq_status;

/* Schemes at n bits per coordinate ([TQ-KV] "Esquemas de Cuantización"; [ABL]
 * "Contribuições Principais" 1):
 *   TQ_PLAIN_KV  K, V: n-bit scalar code, no rotation, no sketch.
 *   TQ_TQ_KV     K, V: rotation + n-bit code.
 *   TQ_KQV       K: rotation + n-bit code; V: rotation + (n-1)-bit code + 1-bit QJL.
 *   TQ_QKQV      K, V: rotation + (n-1)-bit code + 1-bit QJL (also named TQ-QKV). */
typedef enum { TQ_PLAIN_KV = 0, TQ_TQ_KV = 1, TQ_KQV = 2, TQ_QKQV = 3, TQ_SQU_KV = 4 } tq_scheme;

typedef enum { TQ_F32 = 0, TQ_BF16 = 1, TQ_F16 = 2 } tq_dtype;

/* One side's codec: scalar code bits (1..4), rotation (0 none, 1 seeded Walsh-Hadamard, 2 the
 * calibrated per-head eigenbasis of SQU-KV), QJL residual sketch on/off.
 *
 * rotate = 2 (SQU-KV, SpectralQuant with uniform allocation; [ABL] "Configuração Experimental",
 * "Armazenamento vs. Qualidade", "Recomendações Práticas" 2-3): bits must be 2 (the budget: 256
 * bits per vector), qjl 0, head_dim 128.  Per head, the 32 highest-variance directions of the
 * calibrated basis are coded at 4 bits (the 4-bit Beta Lloyd-Max codebook) and the other 96 at
 * 1 bit.  Coordinate c of the stored vector is (E^T u)_c / s_c, with E and s set by
 * tq_spectral_set_basis.  Storage order: with eigen-rank i, key coordinate 32 (i % 4) + i / 4
 * and value coordinate 16 (i % 8) + i / 8 hold the 32 modeled ranks; the other coordinates
 * hold ranks 32.. in increasing order.  A code record (32 bytes) is the 4-bit stream of the
 * modeled coordinates' magnitudes (sign-magnitude form, in increasing coordinate order), then
 * the 1-bit stream of all 128 signs (1 = positive); on the value side each of the two streams
 * is stored by 16-coordinate groups (2 bytes per group and token, see tq_cache_layout). */
typedef struct {
  int32_t bits;
  int32_t rotate;
  int32_t qjl;
} tq_codec;

typedef struct {
  int32_t head_dim;      /* d: 128, 256, 512 or 1024 on the GPU path                       */
  int32_t num_q_heads;   /* H_q; query head h reads KV head h / (H_q / H_kv)               */
  int32_t num_kv_heads;  /* H_kv; G = H_q / H_kv must be 1, 2, 4 or 8                      */
  int32_t batch;         /* B <= TQ_MAX_BATCH                                              */
  int32_t capacity;      /* tokens per (batch, KV head) slab; a multiple of 64             */
  tq_codec k, v;
  int32_t qjl_m;         /* QJL sketch rows m; 0 means m = d (the only value built)        */
  int32_t headq_rank;    /* HeadQ rank r on the K side; 0 = off; 16 is the value built      */
  int32_t headq_bits;    /* HeadQ side-code bits; 4 is the value built                     */
  uint64_t seed;         /* drives the rotation signs D_K, D_V and sketches S_K, S_V        */
} tq_config;

#define TQ_MAX_BATCH 512
#define TQ_LAYOUT_VERSION 3u
#define TQ_TILE_TOKENS 16

/* One field of a side's 16-token block: `offset` within the block, `record_bytes` per token
 * (0 when the field is absent).  Token j of the block has its record at offset +
 * j * record_bytes. */
typedef struct {
  uint64_t offset;
  uint64_t record_bytes;
} tq_region;

/* The packed cache layout (version TQ_LAYOUT_VERSION).  The buffer holds two arrays of
 * 16-token blocks, K at k_offset and V at v_offset (256-byte aligned), each
 * [B][H_kv][capacity / 16] blocks of k_block_bytes / v_block_bytes.  Token t of (b, h) lives in
 * block (b * H_kv + h) * capacity / 16 + t / 16 at position t % 16.  A K block holds, one after
 * another, 16 records of each present field: codes, norm, [signs, rho], [side, side_scale]; a V
 * block: codes, norm, [signs, rho].  So one contiguous copy brings all of a tile's data of a side.
 * Record p of a field sits at offset + p * record_bytes, except the V block's streams (its codes,
 * each stream of a 3-bit code on its own, and its QJL signs): a w-bit stream there is stored by
 * groups of 16 coordinates, [coordinates / 16][16 tokens][2w bytes], so byte j of token p's record
 * is at (j / 2w) * 32w + p * 2w + j % 2w from the stream's start (the 1-bit stream of a 3-bit code
 * starts 16 * d / 4 bytes after the 2-bit one).  One coordinate group of several tokens is then
 * one contiguous read.
 * (A spectral side's 32-byte code record is described with tq_codec.)
 * Codes are stored in sign-magnitude form (s = [c >= 2^(b-1)], k = magnitude rank) as streams of
 * power-of-two widths, coordinate i of a w-bit stream in bits [w*i, w*i + w), least significant
 * bit first:
 *   b = 4: (s << 3) | k;  b = 3: 2-bit stream of k then 1-bit stream of s;
 *   b = 2: (s << 1) | k;  b = 1: s.
 * QJL signs: bit i = 1 iff (S r)_i >= 0.  HeadQ side code: 4-bit two's complement, zeta_0 in
 * the low nibble.  Norms are fp32; rho and side scales fp16. */
typedef struct {
  uint32_t layout_version;
  uint32_t tile_tokens;
  uint64_t total_bytes;
  uint64_t k_offset, k_block_bytes, v_offset, v_block_bytes;
  tq_region k_codes, k_norm, k_signs, k_rho, k_side, k_side_scale;
  tq_region v_codes, v_norm, v_signs, v_rho;
} tq_cache_layout;

typedef struct tq_context tq_context;

/* Fill cfg->k and cfg->v for a scheme at n bits per coordinate (n in 1..4; KQV and QKQV need
 * n >= 2).  Other fields are left as they are.  [TQ-KV] "Esquemas de Cuantización". */
tq_status tq_config_from_scheme(tq_scheme scheme, int32_t n, tq_config* inout);

/* Validate cfg and build the host tables: the Beta Lloyd-Max codebooks of both sides
 * ([ABL] "Configuração Experimental": data-oblivious Beta Lloyd-Max codebook; [TQ-KV]
 * "Marco Teórico": the Beta sphere marginal), the rotation signs and the sketch matrices
 * (SplitMix64 counter streams D_K=1, D_V=2, S_K=3, S_V=4 of cfg->seed).  Host only; no CUDA
 * call.  *out receives a new context on TQ_OK. */
tq_status tq_context_create(const tq_config* cfg, tq_context** out);
void tq_context_destroy(tq_context* ctx);

/* Bytes of the device table buffer the caller must provide to tq_tables_upload. */
size_t tq_tables_bytes(const tq_context* ctx);

/* Copy the host-built table blob (the same bytes tq_tables_upload sends) into host memory.
 * Host only.  Blob layout: fp32 k_centroids[16], k_thresholds[16], v_centroids[16],
 * v_thresholds[16]; fp32 k_signs[d], v_signs[d] (+1/-1); fp32 S_K[m][d] and its transpose
 * [d][m] (if K has QJL); fp32 S_V[m][d] and its transpose (if V has QJL); the HeadQ basis area
 * [H_kv][d][r] (zeros until tq_headq_set_basis); when d > 128 and V has QJL, fp32
 * S_V R_V [m][d] (R_V = H D_V / sqrt(d), each row rounded once from a float64 transform), which
 * maps the value sketch accumulator straight to the output domain; when d = m = 128, for each
 * side with QJL (K, then V), S as fp16 -- the terms fp16(S), then fp16(S - fp16(S)), 32 KiB each, element
 * (i, j) at byte (i / 8) * 2048 + (j / 8) * 128 + (i % 8) * 16 + (j % 8) * 2 (8 x 8 core matrices:
 * the tensor-core residual sketch's operand layout); fp32 c1[2], the 1-bit
 * codebook's upper centroid (a spectral side's floor); and for each spectral side (K, then V)
 * its basis E and E^T [H_kv][d][d] and scales s [H_kv][d] in storage order (zeros until
 * tq_spectral_set_basis).  A spectral side's centroid / threshold slots hold the 4-bit codebook.
 * Each array starts on a 256-byte boundary. */
tq_status tq_tables_host(const tq_context* ctx, void* host_dst, size_t bytes);

/* Copy the tables into dev_tables (tq_tables_bytes bytes, caller-owned, 256-byte aligned) on
 * stream and bind that buffer to the context.  The buffer must outlive every later call. */
tq_status tq_tables_upload(tq_context* ctx, void* dev_tables, tq_stream stream);

/* SQU-KV: store a spectral side's calibrated basis (side 0 = K, 1 = V).  dev_E is fp32
 * [H_kv][d][d] on the device with column j of head h = eigenvector j (component i at
 * dev_E[(h d + i) d + j]), ordered by descending eigenvalue.  dev_s is fp32 [H_kv][d], the
 * coordinate scales in the same eigen-rank order: s_j = sqrt(d lambda_j) for an eigenvalue
 * lambda_j of the mean of u u^T over the side's calibration unit vectors u (a caller may floor
 * it; every s_j must be > 0).  The library permutes both into the storage order (see tq_codec)
 * in the bound table buffer, with a kernel on stream; no value is rounded again.  Needs a
 * spectral side and uploaded tables; every spectral side must be set before append or decode. */
tq_status tq_spectral_set_basis(tq_context* ctx, int32_t side, const float* dev_E, const float* dev_s,
                                tq_stream stream);

/* HeadQ ([HEADQ] "Visão Geral do Algoritmo" 1): store the calibrated key-side basis.
 * dev_U is fp32 [H_kv][d][r] on the device (column k of head h is U_h e_k).  The library keeps
 * R_K U_h in the bound table buffer (a kernel on stream), so later calls see the basis in the
 * rotated domain.  Needs headq_rank > 0 and tables uploaded. */
tq_status tq_headq_set_basis(tq_context* ctx, const float* dev_U, tq_stream stream);

tq_status tq_get_cache_layout(const tq_context* ctx, tq_cache_layout* out);

/* Write path ([TQ-KV] "Esquemas de Cuantización"; [HEADQ] "Escrita no Cache").
 * k, v: device [B][H_kv][n_new][d] of dtype.  Token j of (b, h) is stored at position
 * host_start[b] + j.  host_start: host array of B entries with host_start[b] + n_new <=
 * capacity.  n_new = 0 is a no-op.  dev_cache: total_bytes of tq_get_cache_layout. */
tq_status tq_quantize_append(const tq_context* ctx, void* dev_cache, const void* k, const void* v,
                             tq_dtype dtype, int32_t n_new, const int32_t* host_start,
                             tq_stream stream);

/* Workspace bytes for tq_decode_attention with sequences up to max_seq tokens. */
size_t tq_decode_workspace_bytes(const tq_context* ctx, int32_t max_seq);

/* Read path: o[b][h] = sum_j softmax_j(q^T k_hat_j / sqrt(d)) v_hat_j over the first
 * host_seq_len[b] tokens of slab (b, h / G) ([HEADQ] "Espaço de Pontuação da Chave",
 * "Geometria de Leitura de Valores"; [TQ-KV] "Marco Teórico", K-V asymmetry).
 * q, out: device fp32 [B][H_q][d].  host_seq_len: host array of B entries in [0, capacity];
 * a length of 0 gives an output of zeros.  ws: device workspace of at least
 * tq_decode_workspace_bytes(ctx, max(host_seq_len)) bytes; its contents need no
 * initialization and are owned by the call until it completes on stream. */
tq_status tq_decode_attention(const tq_context* ctx, const void* dev_cache, const float* q,
                              const int32_t* host_seq_len, float* out, void* ws, size_t ws_bytes,
                              tq_stream stream);

/* One decode step: tq_quantize_append of the step's n_new tokens at positions
 * host_seq_len[b] - n_new .. host_seq_len[b] - 1 of each sequence, then tq_decode_attention of q
 * over the first host_seq_len[b] tokens (the new ones included).  The cache and out hold exactly
 * what those two calls give.  Arguments as there (k, v: device [B][H_kv][n_new][d] of dtype; q,
 * out: device fp32 [B][H_q][d]); every host_seq_len[b] must be >= n_new (else
 * TQ_ERR_INVALID_ARG, nothing launched).  At head dim 128 the query preparation runs while the
 * append's kernels do, and the decode starts on the tokens the append does not write; the
 * decode reads the new tokens only after the append has completed.  n_new = 0 is
 * tq_decode_attention. */
tq_status tq_append_decode_attention(const tq_context* ctx, void* dev_cache, const void* k, const void* v,
                                     tq_dtype dtype, int32_t n_new, const float* q,
                                     const int32_t* host_seq_len, float* out, void* ws, size_t ws_bytes,
                                     tq_stream stream);

/* Several queries per sequence in one pass over the cache (speculative-decode drafts, prefill
 * chunks; [ABL] "Recomendações Práticas" names prefill workloads): the nq queries of sequence b
 * are the chunk's last nq positions, and query i attends causally to the first
 * host_seq_len[b] - nq + 1 + i tokens (none when that is <= 0: output zeros).  Each query's
 * result is what tq_decode_attention gives for that query alone over that prefix; the packed
 * tiles are read and unpacked once for all nq queries (they become extra MMA columns).
 * q, out: device fp32 [B][nq][H_q][d].  Built for head dim 128 with G * nq <= 8 (G =
 * H_q / H_kv); otherwise TQ_ERR_UNSUPPORTED.  ws as for tq_decode_attention (the same size
 * serves every nq).  nq = 1 is tq_decode_attention. */
tq_status tq_decode_attention_multi(const tq_context* ctx, const void* dev_cache, const float* q,
                                    int32_t nq, const int32_t* host_seq_len, float* out, void* ws,
                                    size_t ws_bytes, tq_stream stream);

/* Chunked-prefill attention ([ABL] "Recomendações Práticas" 2 names prefill workloads): the
 * same result as tq_decode_attention_multi -- the nq queries of sequence b are the chunk's last
 * nq positions, already appended, and query i attends causally to the first
 * host_seq_len[b] - nq + 1 + i tokens (none when that is <= 0: output zeros) -- for chunks of any
 * size.  The (query, head) rows of a KV head are taken 128 at a time; each 32-token tile of the
 * packed cache is unpacked once per 128 rows into shared memory and both products (scores and
 * value readout) run as dense fp16 tensor-core MMAs with fp32 accumulation, the queries split
 * into fp16 hi + lo terms.  q, out: device fp32 [B][nq][H_q][d] (16-byte aligned).  ws: device
 * workspace of at least tq_prefill_workspace_bytes(ctx, nq) bytes (an error word, then the
 * rotated queries as fp16 terms), 256-byte aligned, owned by the call until it completes on
 * stream; tq_get_device_error(ws, ...) reads the error word (a bounded copy wait that gave up).  Built for head dim
 * 128 (m = 128), every Plain / TQ-KV / KQV / QKQV codec pair and any G = H_q / H_kv; HeadQ and
 * spectral codecs, or more than 65535 (batch, KV head) slabs, give TQ_ERR_UNSUPPORTED.  Errors
 * are detected on the host before any launch. */
size_t tq_prefill_workspace_bytes(const tq_context* ctx, int32_t nq);
tq_status tq_prefill_attention(const tq_context* ctx, const void* dev_cache, const float* q, int32_t nq,
                               const int32_t* host_seq_len, float* out, void* ws, size_t ws_bytes,
                               tq_stream stream);

/* Size of the library's built-in decode scratch (see tq_decode_attention_static). */
#define TQ_STATIC_SCRATCH_BYTES (8u << 20)

/* tq_decode_attention without a workspace argument: the pages have no counterpart for this
 * entry point; it exists for callers that cannot allocate device memory at the call site --
 * code running inside another framework's stream with no access to its allocator, real-time
 * decode loops whose memory is planned up front and where a cudaMalloc (which may synchronize
 * the device) is not allowed, or plugins that are handed only input and output pointers.
 * The scratch is a file-scope device array of TQ_STATIC_SCRATCH_BYTES (8 MiB) that every GPU
 * which loads the library holds until the process exits.  The first call on a device looks up
 * that array's device address (with the device current) and caches it; make that first call
 * before any stream capture.  Every call shares the one array, so calls that overlap on the GPU
 * (other streams, other threads) race: serialize them.  A configuration whose workspace
 * (tq_decode_workspace_bytes) exceeds TQ_STATIC_SCRATCH_BYTES returns TQ_ERR_WORKSPACE without
 * launching.  No device memory is allocated.  Arguments otherwise as tq_decode_attention.
 * The cached address belongs to the device's current primary context: it does not survive a
 * cudaDeviceReset (or any teardown of that context), after which this entry point must not be
 * called again in the process.  The kernels report a device-side failure (a bounded wait that
 * gave up, a shared-memory plan that did not fit) in the scratch's error word, and then leave
 * `out` unwritten; read it with tq_get_static_device_error. */
tq_status tq_decode_attention_static(const tq_context* ctx, const void* dev_cache, const float* q,
                                     const int32_t* host_seq_len, float* out, tq_stream stream);

/* Wait for stream, then read the error word of the built-in scratch on the current device (the
 * one tq_decode_attention_static used): 0 = the last static decode completed, else a
 * TQ_DEVERR_* code (and TQ_ERR_DEVICE is returned).  Each static decode clears the word before
 * its kernels run.  Like tq_get_device_error, it synchronizes the stream. */
tq_status tq_get_static_device_error(int32_t* code, tq_stream stream);

/* HeadQ read path, unfused ([HEADQ] "Leitura do Cache"): corrected logits
 * s_hat_j = q^T k_base_j / sqrt(d) + q^T U z_hat_j / sqrt(d) for every stored token, written to
 * logits[b][h][j] (fp32, row stride logits_stride >= max(host_seq_len)); entries at j >=
 * host_seq_len[b] are not written.  For a K side without HeadQ the scores of the K codec
 * (with the QJL correction on a QJL side) are written. */
tq_status tq_headq_correct(const tq_context* ctx, const void* dev_cache, const float* q,
                           const int32_t* host_seq_len, float* logits, int32_t logits_stride,
                           tq_stream stream);

/* Reconstruct k_hat, v_hat (fp32 [t1 - t0][d], device) of tokens [t0, t1) of slab (b, kvh),
 * including QJL and HeadQ terms.  For tests and debugging. */
tq_status tq_dequantize(const tq_context* ctx, const void* dev_cache, int32_t b, int32_t kvh,
                        int32_t t0, int32_t t1, float* k_out, float* v_out, tq_stream stream);

/* ---- Paged cache (serving layout) ---------------------------------------------------------
 * The pages speak of KV-cache traffic in serving terms ([ABL] "Declaração do Problema") but give
 * no cache organisation; this one is the library's own.  A pool of pages replaces the
 * [B][H_kv][capacity] slabs: a page holds one 16-token block per KV head on each side, so page p's
 * K block of head h is K block p * H_kv + h (and likewise for V), each block laid out exactly as
 * in tq_cache_layout.  A block table maps logical block j of sequence b (tokens 16 j .. 16 j + 15)
 * to a page.  Sequence lengths and append positions come from device memory, so a serving step
 * (append + decode) can be captured once in a CUDA graph and replayed while they change.
 * Entries are not checked on the host.  On the device, a position at or past
 * 16 * max_blocks_per_seq, or a page outside [0, num_pages), is redirected to an extra page at
 * the end of the pool that belongs to no sequence, and an error code is recorded.  Memory
 * outside the pool is never touched.  Built for head dim 128. */
typedef struct {
  const int32_t* block_table;   /* device [B][max_blocks_per_seq] page indices */
  int32_t max_blocks_per_seq;
  int32_t num_pages;            /* pages the caller owns in the pool */
} tq_page_table;

/* Device error codes (tq_get_device_error, or the append's dev_error word). */
#define TQ_DEVERR_WAIT_TIMEOUT 1  /* a bulk-copy wait gave up (the output is not valid)        */
#define TQ_DEVERR_SMEM_PLAN 2     /* the shared-memory plan did not fit the launch             */
#define TQ_DEVERR_BAD_PAGE 3      /* a block-table entry or position outside the pool/table    */
#define TQ_DEVERR_BAD_LENGTH 4    /* a device sequence length outside [0, 16 * max_blocks]     */

/* Layout of a pool of num_pages pages (plus the one redirect page): total_bytes and the block
 * offsets/sizes of the K and V arrays, each [(num_pages + 1) * H_kv] blocks. */
tq_status tq_get_paged_cache_layout(const tq_context* ctx, int32_t num_pages, tq_cache_layout* out);

/* tq_quantize_append into a paged pool: token j of (b, h) goes to position dev_start[b] + j
 * (dev_start: device int32 [B]).  k, v as for tq_quantize_append.  dev_error: device int32 or
 * NULL; on a bad position or page the kernel stores a TQ_DEVERR_* code there (the caller zeroes
 * it beforehand). */
tq_status tq_quantize_append_paged(const tq_context* ctx, void* dev_pool, const tq_page_table* pages,
                                   const void* k, const void* v, tq_dtype dtype, int32_t n_new,
                                   const int32_t* dev_start, int32_t* dev_error, tq_stream stream);

/* tq_decode_attention_multi over a paged pool with device sequence lengths (dev_seq_len: device
 * int32 [B], each in [0, 16 * max_blocks_per_seq]; a length outside is clamped and recorded as
 * TQ_DEVERR_BAD_LENGTH).  ws: tq_decode_workspace_bytes(ctx, 16 * max_blocks_per_seq) bytes.
 * nq = 1 is plain decode.  The work split over the GPU is computed on the device from the
 * lengths. */
tq_status tq_decode_attention_paged(const tq_context* ctx, const void* dev_pool, const tq_page_table* pages,
                                    const float* q, int32_t nq, const int32_t* dev_seq_len, float* out,
                                    void* ws, size_t ws_bytes, tq_stream stream);

/* Wait for stream, then read the device error word of a decode workspace: 0 = none, else a
 * TQ_DEVERR_* code. */
tq_status tq_get_device_error(const void* ws, int32_t* code, tq_stream stream);

const char* tq_status_string(tq_status status);

/* Message of the calling thread's last failed call ("" if none). */
const char* tq_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* TQ_H */
