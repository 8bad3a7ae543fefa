// Internal declarations shared by the host API and the CUDA launchers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include "tq.h"

namespace tqi {

constexpr int kMaxLevels = 16;     // 4-bit codebooks
constexpr int kTableAlign = 256;
constexpr int kRegionAlign = 256;

enum RegionId {
  R_K_CODES = 0, R_K_NORM, R_K_SIGNS, R_K_RHO, R_K_SIDE, R_K_SIDE_SCALE,
  R_V_CODES, R_V_NORM, R_V_SIGNS, R_V_RHO, R_COUNT
};

// Byte offsets of the arrays inside the table blob (see tq_tables_host in tq.h).
struct TableOffsets {
  size_t k_centroids, k_thresholds, v_centroids, v_thresholds;
  size_t k_signs, v_signs, s_k, s_k_t, s_v, s_v_t, headq_u, s_v_r;
  size_t s_h16[2];                       // head dim 128, QJL side: S as fp16 hi then lo rows (sketch_h16_bytes)
  size_t sq_c1;                          // fp32 [2]: 1-bit centroid of each spectral side
  size_t sq_e[2], sq_et[2], sq_s[2];     // spectral side: E, E^T [H_kv][d][d], s [H_kv][d] (storage order)
  size_t total;
};
// 16-token block layout: field r of token t of slab s at
// side_off[side(r)] + (s * tiles_per_slab + t / 16) * block[side(r)] + off[r] + (t % 16) * rec[r].
struct Layout {
  uint64_t off[R_COUNT];  // offset of the field inside its side's block
  uint64_t rec[R_COUNT];  // bytes per token (0 = absent)
  uint64_t side_off[2];   // K array, V array
  uint64_t block[2];      // bytes per block
  uint64_t tiles_per_slab;
  uint64_t total;
};
constexpr int kTileTokens = TQ_TILE_TOKENS;
// fp16 copies of a 128 x 128 sketch matrix for the tensor-core residual sketch, the hi terms
// fp16(S) then the lo terms fp16(S - hi), each in 8 x 8 core matrices (the operand layout of the
// tensor cores): element (i, j) at byte sketch_cm_offset(i, j) of its 32 KiB table
constexpr size_t kSketchH16Bytes = 2 * 128 * 128 * 2;
inline size_t sketch_cm_offset(int i, int j) {
  return (size_t)(i >> 3) * 2048 + (size_t)(j >> 3) * 128 + (size_t)(i & 7) * 16 + (size_t)(j & 7) * 2;
}
inline int region_side(int r) { return r >= R_V_CODES ? 1 : 0; }

// Host tables: Beta Lloyd-Max codebook (float64) and SplitMix64-driven D and S.
void lloyd_max_beta(int d, int bits, double* centroids, double* thresholds);
uint64_t splitmix_mix64(uint64_t z);
void rotation_signs(uint64_t seed, uint64_t stream, int d, float* out);
void sketch_matrix(uint64_t seed, uint64_t stream, int m, int d, float* out);

// pages >= 0: a paged pool of pages + 1 pages (the last one takes redirected accesses)
Layout make_layout(const tq_config& cfg, int m, long long pages = -1);
TableOffsets make_table_offsets(const tq_config& cfg, int m);

void set_error(const std::string& msg);

}  // namespace tqi

struct tq_context {
  tq_config cfg;
  int m;
  tqi::TableOffsets tab;
  tqi::Layout layout;
  std::vector<unsigned char> host_tables;
  void* dev_tables = nullptr;
  bool basis_set = false;
  bool sq_set[2] = {false, false};  // spectral sides: basis stored
};

// Launchers (tq_append.cu, tq_decode.cu, tq_prefill.cu).  They assume validated arguments.
namespace tqi {
typedef struct CUstream_st* Stream;
tq_status launch_append(const tq_context* ctx, void* cache, const void* k, const void* v,
                        tq_dtype dtype, int n_new, const int32_t* start, Stream stream);
// The same append with its last kernel releasing its programmatic dependents at its start, so
// that a decode step's query preparation (launch_decode_after_append) runs beside it.
tq_status launch_append_early(const tq_context* ctx, void* cache, const void* k, const void* v,
                              tq_dtype dtype, int n_new, const int32_t* start, Stream stream);
tq_status launch_append_paged(const tq_context* ctx, void* pool, const tq_page_table* pt, const void* k,
                              const void* v, tq_dtype dtype, int n_new, const int32_t* dev_start,
                              int32_t* dev_error, Stream stream);
tq_status launch_rotate_basis(const tq_context* ctx, const float* U, Stream stream);
tq_status launch_spectral_basis(const tq_context* ctx, int side, const float* E, const float* s, Stream stream);
tq_status launch_dequantize(const tq_context* ctx, const void* cache, int b, int kvh, int t0,
                            int t1, float* k_out, float* v_out, Stream stream);
size_t decode_workspace_bytes(const tq_context* ctx, int max_seq);
tq_status launch_decode_multi(const tq_context* ctx, const void* cache, const float* q, int nq,
                              const int32_t* seq_len, float* out, void* ws, size_t ws_bytes,
                              Stream stream);
tq_status launch_decode_paged(const tq_context* ctx, const void* pool, const tq_page_table* pt,
                              const float* q, int nq, const int32_t* dev_seq_len, float* out, void* ws,
                              size_t ws_bytes, Stream stream);
tq_status launch_decode(const tq_context* ctx, const void* cache, const float* q,
                        const int32_t* seq_len, float* out, void* ws, size_t ws_bytes,
                        Stream stream);
// The decode right after launch_append_early on the same stream (head dim 128): the query
// preparation is the append's programmatic dependent and waits for it before it exits; the decode
// reads each sequence's last n_fresh tokens only after its own wait for the preparation.
tq_status launch_decode_after_append(const tq_context* ctx, const void* cache, const float* q,
                                     const int32_t* seq_len, int n_fresh, float* out, void* ws,
                                     Stream stream);
size_t prefill_workspace_bytes(const tq_context* ctx, int nq);
tq_status launch_prefill(const tq_context* ctx, const void* cache, const float* q, int nq,
                         const int32_t* seq_len, float* out, void* ws, Stream stream);
tq_status launch_logits(const tq_context* ctx, const void* cache, const float* q,
                        const int32_t* seq_len, float* logits, int stride, Stream stream);
tq_status read_device_error(const void* ws, int32_t* code, Stream stream);
// Device address of the built-in decode scratch on the current device (looked up once per device).
tq_status static_scratch(void** ptr);
tq_status read_static_device_error(int32_t* code, Stream stream);
}  // namespace tqi
