// Host tables of the codec: the Beta Lloyd-Max codebook and the seeded rotation / sketch tables.
//
// Codebook: [TQ-KV] "Marco Teórico" (a coordinate of a uniform unit vector on S^{d-1} has
// (x + 1) / 2 ~ Beta((d-1)/2, (d-1)/2)) and [ABL] "Configuração Experimental" (data-oblivious
// Beta Lloyd-Max codebook).  The density of x on [-1, 1] is f(x) = (1 - x^2)^((d-3)/2) /
// B(1/2, (d-1)/2).  Cell masses come from the regularized incomplete beta function, evaluated
// here by its continued fraction (Abramowitz & Stegun 26.5.8, modified Lentz evaluation), and
// cell first moments from the closed form of the integral of x f(x).
//
// Tables: SplitMix64 (Steele, Lea & Flood, OOPSLA 2014) counter streams; D_i = +1 when the top
// bit of draw i is 0; S entries are the cosine branch of Box-Muller on two consecutive draws.
#include <cmath>
#include <cstring>

#include "tq_internal.h"

namespace tqi {

namespace {

// I_x(a, a) for x <= 1/2 by the continued fraction of the incomplete beta function.
double ibeta_sym_lower(double a, double x) {
  if (x <= 0.0) return 0.0;
  if (x >= 0.5 && x <= 0.5) {
    // exact by symmetry
    return 0.5;
  }
  const double b = a;
  const double log_front = a * std::log(x) + b * std::log1p(-x) - std::log(a) -
                           (std::lgamma(a) + std::lgamma(b) - std::lgamma(a + b));
  const double tiny = 1e-300;
  // modified Lentz on 1 / (1 + d1 / (1 + d2 / (1 + ...)))
  double f = 1.0, C = 1.0, D = 0.0;
  for (int i = 1; i <= 20000; ++i) {
    const int k = i / 2;
    double num;
    if (i % 2 == 1) {
      num = -(a + k) * (a + b + k) * x / ((a + 2.0 * k) * (a + 2.0 * k + 1.0));
    } else {
      num = k * (b - k) * x / ((a + 2.0 * k - 1.0) * (a + 2.0 * k));
    }
    D = 1.0 + num * D;
    if (std::fabs(D) < tiny) D = tiny;
    D = 1.0 / D;
    C = 1.0 + num / C;
    if (std::fabs(C) < tiny) C = tiny;
    const double delta = C * D;
    f *= delta;
    if (std::fabs(delta - 1.0) < 4e-16) break;
  }
  // f currently holds the product of the convergents of 1 + d1/(1 + ...): the fraction value
  // is 1 / f.
  return std::exp(log_front) / f;
}

// P(x_coord > t) for t >= 0 and P(x_coord <= t) for t <= 0 (both tails without cancellation).
double tail(double a, double t) {  // mass beyond |t| on one side
  return ibeta_sym_lower(a, (1.0 - std::fabs(t)) / 2.0);
}

double cell_mass(double a, double lo, double hi) {
  if (lo >= 0.0) return tail(a, lo) - tail(a, hi);
  if (hi <= 0.0) return tail(a, hi) - tail(a, lo);
  return 1.0 - tail(a, lo) - tail(a, hi);
}

double cell_first_moment(int d, double lo, double hi) {
  const double p = (d - 1) / 2.0;
  const double la = std::log1p(-lo * lo), lb = std::log1p(-hi * hi);
  double num;
  if (std::fabs(lo) <= std::fabs(hi)) {
    num = -std::exp(p * la) * std::expm1(p * (lb - la));
  } else {
    num = std::exp(p * lb) * std::expm1(p * (la - lb));
  }
  if (!std::isfinite(num)) num = std::exp(p * la) - std::exp(p * lb);
  const double log_b = std::lgamma(0.5) + std::lgamma(p) - std::lgamma(p + 0.5);
  return num / ((d - 1) * std::exp(log_b));
}

double cdf(double a, double t) {
  return t <= 0.0 ? tail(a, t) : 1.0 - tail(a, t);
}

// Inverse CDF by bisection (used only for the starting point).
double quantile(double a, double p) {
  double lo = -1.0, hi = 1.0;
  for (int it = 0; it < 200; ++it) {
    const double mid = 0.5 * (lo + hi);
    if (cdf(a, mid) < p) lo = mid; else hi = mid;
  }
  return 0.5 * (lo + hi);
}

}  // namespace

void lloyd_max_beta(int d, int bits, double* c, double* t) {
  const int L = 1 << bits;
  const double a = (d - 1) / 2.0;
  for (int k = 0; k < L; ++k) c[k] = quantile(a, (k + 0.5) / L);
  double next[kMaxLevels];
  for (int it = 0; it < 100000; ++it) {
    double moved = 0.0;
    for (int k = 0; k < L; ++k) {
      const double lo = k == 0 ? -1.0 : 0.5 * (c[k - 1] + c[k]);
      const double hi = k == L - 1 ? 1.0 : 0.5 * (c[k] + c[k + 1]);
      next[k] = cell_first_moment(d, lo, hi) / cell_mass(a, lo, hi);
    }
    for (int k = 0; k < L; ++k) {
      moved = std::fmax(moved, std::fabs(next[k] - c[k]));
      c[k] = next[k];
    }
    if (moved < 1e-13) break;
  }
  for (int k = 0; k < L / 2; ++k) {  // exact odd symmetry
    const double v = 0.5 * (c[L - 1 - k] - c[k]);
    c[k] = -v;
    c[L - 1 - k] = v;
  }
  for (int k = 0; k + 1 < L; ++k) t[k] = 0.5 * (c[k] + c[k + 1]);
}

uint64_t splitmix_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

namespace {
const uint64_t kGamma = 0x9E3779B97F4A7C15ULL;
inline uint64_t draw(uint64_t key, uint64_t i) { return splitmix_mix64(key + (i + 1) * kGamma); }
}  // namespace

void rotation_signs(uint64_t seed, uint64_t stream, int d, float* out) {
  const uint64_t key = seed ^ splitmix_mix64(stream);
  for (int i = 0; i < d; ++i) out[i] = (draw(key, i) >> 63) ? -1.0f : 1.0f;
}

void sketch_matrix(uint64_t seed, uint64_t stream, int m, int d, float* out) {
  const uint64_t key = seed ^ splitmix_mix64(stream);
  const double two_pi = 6.283185307179586;
  const uint64_t n_total = (uint64_t)m * (uint64_t)d;
  for (uint64_t n = 0; n < n_total; ++n) {
    const uint64_t h1 = draw(key, 2 * n), h2 = draw(key, 2 * n + 1);
    const double u1 = (double)((h1 >> 11) + 1) * 0x1.0p-53;
    const double u2 = (double)(h2 >> 11) * 0x1.0p-53;
    const double g = std::sqrt(-2.0 * std::log(u1)) * std::cos(two_pi * u2);
    out[n] = (float)g;
  }
}

static uint64_t align_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

Layout make_layout(const tq_config& cfg, int m, long long pages) {
  Layout L;
  L.tiles_per_slab = pages < 0 ? (uint64_t)cfg.capacity / kTileTokens : 0;
  const uint64_t blocks = pages < 0 ? (uint64_t)cfg.batch * cfg.num_kv_heads * L.tiles_per_slab
                                    : (uint64_t)(pages + 1) * cfg.num_kv_heads;
  const uint64_t d = cfg.head_dim;
  uint64_t rec[R_COUNT] = {0};
  rec[R_K_CODES] = d * cfg.k.bits / 8;
  rec[R_K_NORM] = 4;
  if (cfg.k.qjl) { rec[R_K_SIGNS] = m / 8; rec[R_K_RHO] = 2; }
  if (cfg.headq_rank) { rec[R_K_SIDE] = (uint64_t)cfg.headq_rank * cfg.headq_bits / 8; rec[R_K_SIDE_SCALE] = 2; }
  rec[R_V_CODES] = d * cfg.v.bits / 8;
  rec[R_V_NORM] = 4;
  if (cfg.v.qjl) { rec[R_V_SIGNS] = m / 8; rec[R_V_RHO] = 2; }
  uint64_t in_block[2] = {0, 0};
  for (int r = 0; r < R_COUNT; ++r) {
    L.rec[r] = rec[r];
    const int side = region_side(r);
    L.off[r] = rec[r] ? in_block[side] : 0;
    in_block[side] += kTileTokens * rec[r];
  }
  uint64_t off = 0;
  for (int side = 0; side < 2; ++side) {
    off = align_up(off, kRegionAlign);
    L.side_off[side] = off;
    L.block[side] = in_block[side];
    off += blocks * in_block[side];
  }
  L.total = off;
  return L;
}

TableOffsets make_table_offsets(const tq_config& cfg, int m) {
  TableOffsets T;
  uint64_t off = 0;
  auto take = [&](uint64_t bytes) { off = align_up(off, kTableAlign); uint64_t o = off; off += bytes; return (size_t)o; };
  const uint64_t d = cfg.head_dim;
  T.k_centroids = take(kMaxLevels * 4);
  T.k_thresholds = take(kMaxLevels * 4);
  T.v_centroids = take(kMaxLevels * 4);
  T.v_thresholds = take(kMaxLevels * 4);
  T.k_signs = take(d * 4);
  T.v_signs = take(d * 4);
  T.s_k = cfg.k.qjl ? take((uint64_t)m * d * 4) : 0;
  T.s_k_t = cfg.k.qjl ? take((uint64_t)m * d * 4) : 0;
  T.s_v = cfg.v.qjl ? take((uint64_t)m * d * 4) : 0;
  T.s_v_t = cfg.v.qjl ? take((uint64_t)m * d * 4) : 0;
  T.headq_u = cfg.headq_rank ? take((uint64_t)cfg.num_kv_heads * d * cfg.headq_rank * 4) : 0;
  T.s_v_r = (cfg.v.qjl && d > 128) ? take((uint64_t)m * d * 4) : 0;
  T.s_h16[0] = (cfg.k.qjl && d == 128 && m == 128) ? take(kSketchH16Bytes) : 0;
  T.s_h16[1] = (cfg.v.qjl && d == 128 && m == 128) ? take(kSketchH16Bytes) : 0;
  T.sq_c1 = take(2 * 4);
  const uint64_t hdd = (uint64_t)cfg.num_kv_heads * d * d * 4;
  for (int side = 0; side < 2; ++side) {
    const bool sq = (side ? cfg.v.rotate : cfg.k.rotate) == 2;
    T.sq_e[side] = sq ? take(hdd) : 0;
    T.sq_et[side] = sq ? take(hdd) : 0;
    T.sq_s[side] = sq ? take((uint64_t)cfg.num_kv_heads * d * 4) : 0;
  }
  T.total = align_up(off, kTableAlign);
  return T;
}

}  // namespace tqi
