// Host-side set-up math of libtq: SplitMix64 streams, Hadamard signs, the
// dense Haar rotation (Householder QR), the QJL projection, the Lloyd-Max
// codebook, descriptor validation and error reporting.
//
// Everything here runs once per process on the CPU in fp64; the results are
// uploaded by the caller.  The specification these follow is include/tq.h
// (random streams, rotation kinds, codebook density and emission rule).
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "tq_internal.h"

namespace tq {

static thread_local std::string g_last_error;

tq_status fail(tq_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

void clear_error() { g_last_error.clear(); }

// ---------------------------------------------------------------- streams
// SplitMix64 (Vigna), keyed per (seed, kind, layer) as include/tq.h states.
struct SplitMix64 {
  uint64_t s;
  explicit SplitMix64(uint64_t seed, int kind, int layer)
      : s(seed ^ ((((uint64_t)(uint32_t)kind << 32) + (uint64_t)(uint32_t)layer) * 0x9E3779B97F4A7C15ull)) {}
  uint64_t next() {
    s += 0x9E3779B97F4A7C15ull;
    uint64_t z = s;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  }
  double uniform() { return (double)(next() >> 11) * 0x1.0p-53; }
};

// Box-Muller on consecutive uniform pairs, cos branch first.
static void gaussian_fill(uint64_t seed, int kind, int layer, double* out, size_t n) {
  SplitMix64 g(seed, kind, layer);
  const double two_pi = 6.283185307179586476925286766559;
  for (size_t i = 0; i < n; i += 2) {
    double u1 = 1.0 - g.uniform();
    double u2 = g.uniform();
    double r = std::sqrt(-2.0 * std::log(u1));
    out[i] = r * std::cos(two_pi * u2);
    if (i + 1 < n) out[i + 1] = r * std::sin(two_pi * u2);
  }
}

// Householder QR of the row-major n x n matrix; writes Pi = Q diag(sign(diag R))
// row-major into `pi`.
static void haar_q(const std::vector<double>& a_rowmajor, int n, float* pi) {
  // column-major working copy: A(i, j) = a[j * n + i]
  std::vector<double> a((size_t)n * n);
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j) a[(size_t)j * n + i] = a_rowmajor[(size_t)i * n + j];
  std::vector<double> vs((size_t)n * n, 0.0);  // Householder vectors
  std::vector<double> rdiag(n);
  for (int k = 0; k < n; ++k) {
    double* col = &a[(size_t)k * n];
    double norm = 0.0;
    for (int i = k; i < n; ++i) norm += col[i] * col[i];
    norm = std::sqrt(norm);
    double alpha = col[k] > 0 ? -norm : norm;  // R(k,k) = alpha
    double* v = &vs[(size_t)k * n];
    for (int i = k; i < n; ++i) v[i] = col[i];
    v[k] -= alpha;
    double vn = 0.0;
    for (int i = k; i < n; ++i) vn += v[i] * v[i];
    rdiag[k] = alpha;
    if (vn == 0.0) continue;
    for (int j = k; j < n; ++j) {  // H = I - 2 v v^T / (v^T v) on the trailing columns
      double* cj = &a[(size_t)j * n];
      double dot = 0.0;
      for (int i = k; i < n; ++i) dot += v[i] * cj[i];
      double f = 2.0 * dot / vn;
      for (int i = k; i < n; ++i) cj[i] -= f * v[i];
    }
  }
  // Q = H_0 H_1 ... H_{n-1}: column j is Q e_j.
  std::vector<double> q((size_t)n * n, 0.0);
  for (int j = 0; j < n; ++j) {
    double* e = &q[(size_t)j * n];
    e[j] = 1.0;
    for (int k = n - 1; k >= 0; --k) {
      const double* v = &vs[(size_t)k * n];
      double vn = 0.0, dot = 0.0;
      for (int i = k; i < n; ++i) { vn += v[i] * v[i]; dot += v[i] * e[i]; }
      if (vn == 0.0) continue;
      double f = 2.0 * dot / vn;
      for (int i = k; i < n; ++i) e[i] -= f * v[i];
    }
  }
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j) {
      double s = rdiag[j] < 0 ? -1.0 : 1.0;
      pi[(size_t)i * n + j] = (float)(q[(size_t)j * n + i] * s);
    }
}

// ---------------------------------------------------------------- codebook
// Gauss-Legendre nodes/weights on [-1, 1] by Newton iteration on P_n.
static void gauss_legendre(int n, std::vector<double>& x, std::vector<double>& w) {
  x.assign(n, 0.0);
  w.assign(n, 0.0);
  const double pi = 3.14159265358979323846264338327950288;
  for (int i = 0; i < (n + 1) / 2; ++i) {
    double z = std::cos(pi * (i + 0.75) / (n + 0.5));
    double pp = 0.0;
    for (int it = 0; it < 100; ++it) {
      double p0 = 1.0, p1 = z;
      for (int k = 2; k <= n; ++k) {
        double p2 = ((2.0 * k - 1.0) * z * p1 - (k - 1.0) * p0) / k;
        p0 = p1;
        p1 = p2;
      }
      pp = n * (z * p1 - p0) / (z * z - 1.0);
      double dz = p1 / pp;
      z -= dz;
      if (std::fabs(dz) < 1e-16) break;
    }
    x[i] = -z;
    x[n - 1 - i] = z;
    w[i] = w[n - 1 - i] = 2.0 / ((1.0 - z * z) * pp * pp);
  }
}

// Density of one coordinate of a uniform unit vector in R^d,
// f(t) = Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2)) (1 - t^2)^((d-3)/2).
struct CoordDensity {
  int d;
  double log_k, expo;
  std::vector<double> gx, gw;
  explicit CoordDensity(int dim) : d(dim) {
    log_k = std::lgamma(d / 2.0) - std::lgamma((d - 1) / 2.0) - 0.5 * std::log(3.14159265358979323846264338327950288);
    expo = (d - 3) / 2.0;
    gauss_legendre(24, gx, gw);
  }
  double f(double t) const {
    if (1.0 - t * t <= 0.0) return 0.0;
    return std::exp(log_k + expo * std::log1p(-t * t));
  }
  // integral over [a, b] of t^p f(t), p in {0, 1}, composite Gauss-Legendre.
  double integrate(double a, double b, int p) const {
    const int panels = 32;
    double h = (b - a) / panels, sum = 0.0;
    for (int k = 0; k < panels; ++k) {
      double mid = a + (k + 0.5) * h, part = 0.0;
      for (size_t i = 0; i < gx.size(); ++i) {
        double t = mid + 0.5 * h * gx[i];
        part += gw[i] * (p ? t : 1.0) * f(t);
      }
      sum += 0.5 * h * part;
    }
    return sum;
  }
};

// Inverse of the standard normal CDF by bisection on erfc (starting point only).
static double normal_quantile(double p) {
  double lo = -40.0, hi = 40.0;
  for (int it = 0; it < 200; ++it) {
    double mid = 0.5 * (lo + hi);
    double cdf = 0.5 * std::erfc(-mid / std::sqrt(2.0));
    if (cdf < p) lo = mid; else hi = mid;
  }
  return 0.5 * (lo + hi);
}

// Lloyd iteration: boundaries at midpoints, centroids at cell conditional means.
static bool lloyd_max(int d, int bits, std::vector<double>& c) {
  const int k = 1 << bits;
  CoordDensity dens(d);
  c.resize(k);
  for (int i = 0; i < k; ++i) {
    double g = normal_quantile((i + 0.5) / k) / std::sqrt((double)d);
    c[i] = std::fmax(-0.999, std::fmin(0.999, g));
  }
  std::vector<double> edges(k + 1), nc(k);
  for (int it = 0; it < 200000; ++it) {
    edges[0] = -1.0;
    edges[k] = 1.0;
    for (int i = 1; i < k; ++i) edges[i] = 0.5 * (c[i - 1] + c[i]);
    double delta = 0.0;
    for (int i = 0; i < k; ++i) {
      double mass = dens.integrate(edges[i], edges[i + 1], 0);
      double mom = dens.integrate(edges[i], edges[i + 1], 1);
      nc[i] = mom / mass;
      delta = std::fmax(delta, std::fabs(nc[i] - c[i]));
    }
    c = nc;
    if (delta < 1e-15) return true;
  }
  return false;
}

namespace {
std::atomic<uint64_t> g_launches{0};
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

}  // namespace tq

using namespace tq;

extern "C" {

const char* tq_last_error(void) { return g_last_error.c_str(); }

uint32_t tq_format_version(void) { return TQ_FORMAT_VERSION; }

uint64_t tq_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

tq_status tq_make_codebook(int head_dim, int bits, float* centroids, float* boundaries) {
  clear_error();
  if (!centroids || !boundaries) return fail(TQ_ERR_INVALID_ARG, "tq_make_codebook: null output");
  if (bits < 1 || bits > 4) return fail(TQ_ERR_INVALID_ARG, "tq_make_codebook: bits %d not in 1..4", bits);
  if (head_dim < 3 || head_dim > 65536)
    return fail(TQ_ERR_INVALID_ARG, "tq_make_codebook: head_dim %d not in 3..65536", head_dim);
  static std::mutex mu;
  static std::map<std::pair<int, int>, std::vector<float>> cache;
  std::vector<float> tab;
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find({head_dim, bits});
    if (it != cache.end()) tab = it->second;
  }
  const int k = 1 << bits;
  if (tab.empty()) {
    std::vector<double> c;
    if (!lloyd_max(head_dim, bits, c))
      return fail(TQ_ERR_UNSUPPORTED, "tq_make_codebook: Lloyd iteration did not converge");
    tab.resize(2 * k - 1);
    for (int i = k / 2; i < k; ++i) tab[i] = (float)c[i];
    for (int i = 0; i < k / 2; ++i) tab[i] = -tab[k - 1 - i];
    for (int i = 0; i + 1 < k; ++i) {
      volatile float s = tab[i] + tab[i + 1];  // fp32 sum, then exact halving
      tab[k + i] = s * 0.5f;
    }
    std::lock_guard<std::mutex> lock(mu);
    cache[{head_dim, bits}] = tab;
  }
  std::memcpy(centroids, tab.data(), sizeof(float) * k);
  std::memcpy(boundaries, tab.data() + k, sizeof(float) * (k - 1));
  return TQ_OK;
}

tq_status tq_make_rotation(int kind, int head_dim, uint64_t seed, int layer, float* out) {
  clear_error();
  if (!out) return fail(TQ_ERR_INVALID_ARG, "tq_make_rotation: null output");
  if (head_dim < 1 || head_dim > 1024)
    return fail(TQ_ERR_INVALID_ARG, "tq_make_rotation: head_dim %d not in 1..1024", head_dim);
  if (layer < 0) return fail(TQ_ERR_INVALID_ARG, "tq_make_rotation: negative layer");
  const int n = head_dim;
  if (kind == TQ_ROT_HADAMARD) {
    if (n & (n - 1)) return fail(TQ_ERR_INVALID_ARG, "tq_make_rotation: Hadamard needs a power-of-two head_dim");
    SplitMix64 g(seed, kind, layer);
    for (int i = 0; i < n; ++i) out[i] = (g.next() >> 63) ? -1.0f : 1.0f;
    return TQ_OK;
  }
  if (kind == TQ_ROT_DENSE) {
    std::vector<double> a((size_t)n * n);
    gaussian_fill(seed, kind, layer, a.data(), a.size());
    haar_q(a, n, out);
    return TQ_OK;
  }
  if (kind == TQ_RNG_QJL) {
    std::vector<double> a((size_t)n * n);
    gaussian_fill(seed, kind, 0, a.data(), a.size());
    for (size_t i = 0; i < a.size(); ++i) out[i] = (float)a[i];
    return TQ_OK;
  }
  return fail(TQ_ERR_INVALID_ARG, "tq_make_rotation: unknown kind %d", kind);
}

size_t tq_page_bytes(const tq_cache_desc* desc, int which) {
  if (check_desc(desc, false) != TQ_OK || (which != 0 && which != 1)) return 0;
  return page_bytes_of(*desc, which);
}

}  // extern "C"

namespace tq {

size_t page_bytes_of(const tq_cache_desc& d, int which) {
  const size_t blk = (size_t)d.block_size;
  if (d.fmt.kv_format == TQ_KV_BF16) return blk * (size_t)d.head_dim * 2;
  if (d.fmt.kv_format == TQ_KV_K8V4 && which == 0) return blk * (size_t)d.head_dim;  // FP8 E4M3 keys
  if (d.fmt.kv_format == TQ_KV_POLAR)  // angle-code records + fp16 radii
    return blk * (size_t)(d.head_dim * (which == 0 ? d.fmt.bits_k : d.fmt.bits_v) / 8) + blk * 2;
  const int bits = which == 0 ? d.fmt.bits_k : d.fmt.bits_v;
  size_t n = blk * (size_t)(d.head_dim * bits / 8) + blk * 4;
  if (which == 0 && d.fmt.qjl_k) n += blk * (size_t)(d.head_dim / 8) + blk * 4;
  return n;
}

static bool table_ok(const float* c, const float* b, int bits) {
  const int k = 1 << bits;
  for (int i = 0; i + 1 < k; ++i)
    if (!(c[i] < c[i + 1])) return false;
  for (int i = 0; i < k; ++i)
    if (c[i] != -c[k - 1 - i]) return false;
  for (int i = 0; i + 1 < k - 1; ++i)
    if (!(b[i] < b[i + 1])) return false;
  for (int i = 0; i < k - 1; ++i)
    if (b[i] != -b[k - 2 - i]) return false;
  for (int i = 0; i < k - 1; ++i)
    if (!(c[i] <= b[i] && b[i] <= c[i + 1])) return false;
  return b[k / 2 - 1] == 0.0f;
}

tq_status check_desc(const tq_cache_desc* d, bool need_data) {
  if (!d) return fail(TQ_ERR_INVALID_ARG, "null descriptor");
  if (d->format_version != TQ_FORMAT_VERSION)
    return fail(TQ_ERR_VERSION, "descriptor format_version %u, library %u", d->format_version, TQ_FORMAT_VERSION);
  if (d->head_dim != TQ_HEAD_DIM) return fail(TQ_ERR_UNSUPPORTED, "head_dim %d: only 128 is implemented", d->head_dim);
  if (d->block_size != TQ_BLOCK_SIZE)
    return fail(TQ_ERR_UNSUPPORTED, "block_size %d: only 16 is implemented", d->block_size);
  if (d->num_kv_heads < 1 || d->num_kv_heads > 1024) return fail(TQ_ERR_INVALID_ARG, "num_kv_heads %d", d->num_kv_heads);
  if (d->num_blocks < 1) return fail(TQ_ERR_INVALID_ARG, "num_blocks %lld", (long long)d->num_blocks);
  if (need_data && (!d->k_cache || !d->v_cache)) return fail(TQ_ERR_INVALID_ARG, "null cache pool");
  if (((uintptr_t)d->k_cache | (uintptr_t)d->v_cache) & 15)
    return fail(TQ_ERR_INVALID_ARG, "cache pools must be 16-byte aligned");
  const tq_layer_format& f = d->fmt;
  if (f.norm_mode != TQ_NORM_CORRECTED && f.norm_mode != TQ_NORM_RAW)
    return fail(TQ_ERR_INVALID_ARG, "norm_mode %d", f.norm_mode);
  if (f.kv_format == TQ_KV_BF16) return TQ_OK;
  if (f.kv_format == TQ_KV_K8V4) {  // FP8 E4M3 keys, packed values
    if (f.bits_k != 8) return fail(TQ_ERR_INVALID_ARG, "k8v4: bits_k %d must be 8", f.bits_k);
    if (f.bits_v < 2 || f.bits_v > 4) return fail(TQ_ERR_INVALID_ARG, "k8v4: bits_v %d not in 2..4", f.bits_v);
    if (f.qjl_k != 0) return fail(TQ_ERR_INVALID_ARG, "k8v4: keys carry no QJL residual");
    if (f.rot_kind != TQ_ROT_HADAMARD && f.rot_kind != TQ_ROT_DENSE)
      return fail(TQ_ERR_INVALID_ARG, "rot_kind %d", f.rot_kind);
    if (need_data && !d->rotation) return fail(TQ_ERR_INVALID_ARG, "null rotation");
    if (!table_ok(d->centroids_v, d->boundaries_v, f.bits_v))
      return fail(TQ_ERR_INVALID_ARG, "value codebook is not increasing/antisymmetric with its midpoints");
    return TQ_OK;
  }
  if (f.kv_format == TQ_KV_POLAR) {  // PolarQuant angle codes, Hadamard rotation only
    if (f.bits_k < 2 || f.bits_k > 4 || f.bits_v < 2 || f.bits_v > 4)
      return fail(TQ_ERR_INVALID_ARG, "polar: bits_k %d / bits_v %d not in 2..4", f.bits_k, f.bits_v);
    if (f.qjl_k != 0) return fail(TQ_ERR_INVALID_ARG, "polar: keys carry no QJL residual");
    if (f.rot_kind != TQ_ROT_HADAMARD) return fail(TQ_ERR_UNSUPPORTED, "polar: rot_kind %d (Hadamard only)", f.rot_kind);
    if (need_data && !d->rotation) return fail(TQ_ERR_INVALID_ARG, "null rotation");
    return TQ_OK;
  }
  if (f.kv_format != TQ_KV_PACKED) return fail(TQ_ERR_INVALID_ARG, "kv_format %d", f.kv_format);
  if (f.bits_k < 2 || f.bits_k > 4 || f.bits_v < 2 || f.bits_v > 4)
    return fail(TQ_ERR_INVALID_ARG, "bits_k %d / bits_v %d not in 2..4", f.bits_k, f.bits_v);
  if (f.qjl_k != 0 && f.qjl_k != 1) return fail(TQ_ERR_INVALID_ARG, "qjl_k %d", f.qjl_k);
  if (f.rot_kind != TQ_ROT_HADAMARD && f.rot_kind != TQ_ROT_DENSE)
    return fail(TQ_ERR_INVALID_ARG, "rot_kind %d", f.rot_kind);
  if (need_data && !d->rotation) return fail(TQ_ERR_INVALID_ARG, "null rotation");
  if (need_data && f.qjl_k && !d->qjl_proj) return fail(TQ_ERR_INVALID_ARG, "qjl_k set but qjl_proj is null");
  if (!table_ok(d->centroids_k, d->boundaries_k, f.bits_k))
    return fail(TQ_ERR_INVALID_ARG, "key codebook is not increasing/antisymmetric with its midpoints");
  if (!table_ok(d->centroids_v, d->boundaries_v, f.bits_v))
    return fail(TQ_ERR_INVALID_ARG, "value codebook is not increasing/antisymmetric with its midpoints");
  return TQ_OK;
}

int auto_splits(int num_sms, int warps, int batch, int num_kv_heads, int max_blocks_per_seq) {
  // One wave: at most one chunk per decode warp of the GPU over (sequence, kv head
  // group, split) -- rounded down, since one chunk over makes a second wave of a
  // few CTAs -- each split keeping at least 4 blocks of the table (two stages of the
  // decode's ring), and at most 128 splits (the most the decode kernel merges itself).
  const long units = (long)batch * num_kv_heads;
  if (units <= 0 || max_blocks_per_seq <= 0) return 1;
  long target = (long)num_sms * warps;
  long s = target / units;
  long cap = (max_blocks_per_seq + 3) / 4;
  if (s > cap) s = cap;
  if (s < 1) s = 1;
  if (s > 128) s = 128;
  return (int)s;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

DecodeWorkspace decode_workspace(int batch, int num_q_heads, int splits, int head_dim, bool qjl) {
  DecodeWorkspace w;
  const size_t bh = (size_t)batch * num_q_heads;
  // the chunk counters come first, in a region of fixed size for every shape that fits
  // it, so a workspace reused across shapes keeps its zeroed counters where they were
  w.cnt_off = 0;
  const size_t cnt_bytes = align256(bh * sizeof(int32_t));
  w.qrot_off = cnt_bytes > kCounterRegionBytes ? cnt_bytes : kCounterRegionBytes;
  size_t qbytes = bh * head_dim * sizeof(float) * (qjl ? 2 : 1);
  w.part_off = align256(w.qrot_off + qbytes);
  w.ml_off = align256(w.part_off + bh * splits * head_dim * sizeof(float));
  w.total = align256(w.ml_off + bh * splits * 2 * sizeof(float));
  return w;
}

}  // namespace tq
