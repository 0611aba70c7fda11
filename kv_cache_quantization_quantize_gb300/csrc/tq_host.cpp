// Host side of libtq: argument validation, tables (codebook, rotation signs, QJL matrix), cache
// layout, canonical record conversion and the C ABI entry points.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>

#include "tq_internal.h"

namespace {

thread_local std::string g_last_error;

tq_status fail(tq_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

tq_status ok() {
  g_last_error.clear();
  return TQ_OK;
}

tq_status cuda_fail(cudaError_t e, const char* what) {
  return fail(TQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

float bf16_to_float(uint16_t b) {
  const uint32_t x = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &x, 4);
  return f;
}

// bf16 bits -> f16 bits, round to nearest even (overflow to inf; values below 2^-14 become subnormal).
uint16_t bf16_to_f16_rne(uint16_t b) {
  const uint32_t x = (uint32_t)b << 16;
  const uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
  const uint32_t ax = x & 0x7fffffffu;
  if (ax >= 0x7f800000u) return sign | (ax > 0x7f800000u ? 0x7e00u : 0x7c00u);
  if (ax >= 0x477ff000u) return sign | 0x7c00u;  // >= 65520 rounds to inf
  if (ax <= 0x33000000u) return sign;            // <= 2^-25 rounds to zero (ties to even)
  const int e = (int)(ax >> 23) - 127;
  const uint32_t mant = (ax & 0x7fffffu) | 0x800000u;
  if (e >= -14) {
    uint32_t h = ((uint32_t)(e + 15) << 10) | ((mant >> 13) & 0x3ffu);
    const uint32_t rem = mant & 0x1fffu;
    if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) ++h;  // a carry moves into the exponent
    return sign | (uint16_t)h;
  }
  const int sh = -(e + 1);  // units of 2^-24: mant * 2^(e + 1)
  uint32_t m = mant >> sh;
  const uint32_t rem = mant & ((1u << sh) - 1u), half = 1u << (sh - 1);
  if (rem > half || (rem == half && (m & 1u))) ++m;
  return sign | (uint16_t)m;
}

tq_status validate(const tq_config* c) {
  if (!c) return fail(TQ_ERR_INVALID_ARG, "cfg is NULL");
  if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256)
    return fail(TQ_ERR_UNSUPPORTED, "head_dim %d: supported 64, 128, 256", c->head_dim);
  if (c->key_bits != 3 && c->key_bits != 4)
    return fail(TQ_ERR_UNSUPPORTED, "key_bits %d: supported 3 and 4 ((key_bits-1)-bit Lloyd-Max + 1-bit QJL)",
                c->key_bits);
  if (c->value_bits != 2 && c->value_bits != 4)
    return fail(TQ_ERR_UNSUPPORTED, "value_bits %d: supported 2, 4", c->value_bits);
  if (c->value_group != 32) return fail(TQ_ERR_UNSUPPORTED, "value_group %d: supported 32", c->value_group);
  if (c->ring_size != tq::kPage && c->ring_size != 0)
    return fail(TQ_ERR_UNSUPPORTED, "ring_size %d: supported 128 (hybrid) and 0 (full_tq)", c->ring_size);
  if (c->n_layers < 1 || c->n_kv_heads < 1 || c->n_q_heads < 1 || c->max_seqs < 1 || c->max_ctx < 1)
    return fail(TQ_ERR_INVALID_ARG, "n_layers, n_kv_heads, n_q_heads, max_seqs, max_ctx must be >= 1");
  if (c->n_q_heads % c->n_kv_heads != 0)
    return fail(TQ_ERR_INVALID_ARG, "n_q_heads %d not a multiple of n_kv_heads %d", c->n_q_heads, c->n_kv_heads);
  const int G = c->n_q_heads / c->n_kv_heads;
  if (G != 1 && G != 2 && G != 4) return fail(TQ_ERR_UNSUPPORTED, "GQA group %d: supported 1, 2, 4", G);
  if (c->max_ctx > (1 << 24)) return fail(TQ_ERR_UNSUPPORTED, "max_ctx %d above 2^24", c->max_ctx);
  if (c->n_blocks < 0) return fail(TQ_ERR_INVALID_ARG, "n_blocks %d < 0", c->n_blocks);
  if (c->key_bits == 4 && c->value_bits != 4)
    return fail(TQ_ERR_UNSUPPORTED, "key_bits 4 is served with value_bits 4 (the 4-bit configuration)");
  return TQ_OK;
}

// ---- SplitMix64 (Steele, Lea & Flood 2014), written from its published definition ----
inline uint64_t splitmix64(uint64_t seed, uint64_t counter) {
  uint64_t z = seed + counter * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
inline double uniform_open(uint64_t x) { return (double(x >> 11) + 0.5) * 0x1p-53; }

// Nearest-even rounding of a double to bf16 (8 significant bits); returns the bf16 bit pattern.
uint16_t bf16_rne_bits(double v) {
  int e = 0;
  const double m = std::frexp(v, &e);              // v = m * 2^e, 0.5 <= |m| < 1
  const double r = std::ldexp(std::nearbyint(m * 256.0), e - 8);  // default rounding: to nearest even
  const float f = static_cast<float>(r);           // exact: r has <= 8 significant bits
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return static_cast<uint16_t>(u >> 16);
}

// ---- Lloyd-Max codebook of f_d(x) ~ (1-x^2)^((d-3)/2) on [-1, 1] ([Guide] §二 step 2) ----
// Cell integrals by composite 16-point Gauss-Legendre quadrature (nodes from Newton iteration on
// the Legendre polynomial), independent of any closed form.
struct GaussLegendre {
  double x[16], w[16];
  GaussLegendre() {
    const int n = 16;
    for (int i = 0; i < n; ++i) {
      double z = std::cos(M_PI * (i + 0.75) / (n + 0.5));
      for (int it = 0; it < 100; ++it) {
        double p0 = 1.0, p1 = z;
        for (int k = 2; k <= n; ++k) {
          const double p2 = ((2.0 * k - 1.0) * z * p1 - (k - 1.0) * p0) / k;
          p0 = p1;
          p1 = p2;
        }
        const double dp = n * (z * p1 - p0) / (z * z - 1.0);
        const double dz = p1 / dp;
        z -= dz;
        if (std::fabs(dz) < 1e-16) break;
      }
      double p0 = 1.0, p1 = z;
      for (int k = 2; k <= n; ++k) {
        const double p2 = ((2.0 * k - 1.0) * z * p1 - (k - 1.0) * p0) / k;
        p0 = p1;
        p1 = p2;
      }
      const double dp = n * (z * p1 - p0) / (z * z - 1.0);
      x[i] = z;
      w[i] = 2.0 / ((1.0 - z * z) * dp * dp);
    }
  }
};

struct BetaMarginal {
  int d;
  double log_c;
  explicit BetaMarginal(int dd) : d(dd) {
    log_c = std::lgamma(d / 2.0) - 0.5 * std::log(M_PI) - std::lgamma((d - 1) / 2.0);
  }
  double pdf(double x) const {
    if (std::fabs(x) >= 1.0) return 0.0;
    return std::exp(log_c + 0.5 * (d - 3) * std::log1p(-x * x));
  }
  // integrals of f and x f over [a, b]
  void integrate(double a, double b, double& m0, double& m1) const {
    static const GaussLegendre gl;
    const int panels = 256;
    m0 = m1 = 0.0;
    const double h = (b - a) / panels;
    for (int p = 0; p < panels; ++p) {
      const double lo = a + p * h, mid = lo + 0.5 * h;
      for (int i = 0; i < 16; ++i) {
        const double x = mid + 0.5 * h * gl.x[i];
        const double f = pdf(x) * gl.w[i] * 0.5 * h;
        m0 += f;
        m1 += x * f;
      }
    }
  }
};

void lloyd_max(int d, int bits, double* cent, double* bnd) {
  const int L = 1 << bits;
  const BetaMarginal f(d);
  // initial boundaries: uniform over +-3 standard deviations of the N(0, 1/d) approximation
  std::vector<double> t(L - 1), c(L);
  for (int i = 0; i < L - 1; ++i) t[i] = (-3.0 + 6.0 * (i + 1) / L) / std::sqrt((double)d);
  // integrate only where the density is non-negligible
  const double span = std::min(1.0, 40.0 / std::sqrt((double)d));
  for (int it = 0; it < 100000; ++it) {
    for (int i = 0; i < L; ++i) {
      const double a = i == 0 ? -span : t[i - 1];
      const double b = i == L - 1 ? span : t[i];
      double m0, m1;
      f.integrate(a, b, m0, m1);
      c[i] = m1 / m0;
    }
    double delta = 0.0;
    for (int i = 0; i < L - 1; ++i) {
      const double nt = 0.5 * (c[i] + c[i + 1]);
      delta = std::max(delta, std::fabs(nt - t[i]));
      t[i] = nt;
    }
    if (delta < 1e-16) break;
  }
  // the density is even: make the codebook exactly odd-symmetric (middle boundary exactly 0)
  for (int i = 0; i < L; ++i) cent[i] = 0.5 * (c[i] - c[L - 1 - i]);
  for (int i = 0; i < L - 1; ++i) bnd[i] = 0.5 * (t[i] - t[L - 2 - i]);
}

size_t ring_elems(const tq_config& c) { return (size_t)2 * tq::kPage * c.head_dim; }

void compute_offsets(tq_ctx* ctx) {
  const tq_config& c = ctx->cfg;
  ctx->pl = tq::page_layout(c.head_dim, c.value_bits, c.key_bits);
  ctx->to = tq::table_offsets(c.head_dim);
  ctx->max_pages = (c.max_ctx + tq::kPage - 1) / tq::kPage;
  const size_t units = (size_t)c.n_layers * c.max_seqs * c.n_kv_heads;
  const size_t page_units = c.n_blocks > 0 ? (size_t)c.n_layers * c.n_blocks * c.n_kv_heads : units * ctx->max_pages;
  ctx->pages_off = 0;
  ctx->ring_off = align_up(page_units * ctx->pl.bytes, 256);
  ctx->state_off = align_up(ctx->ring_off + units * ring_elems(c) * 2, 256);
  ctx->acnt_off = align_up(ctx->state_off + (size_t)c.n_layers * c.max_seqs * 8, 256);
  ctx->btab_off = align_up(ctx->acnt_off + (size_t)c.n_layers * c.max_seqs * 4, 256);
  const size_t btab_bytes = c.n_blocks > 0 ? (size_t)c.max_seqs * ctx->max_pages * 4 : 0;
  ctx->status_off = align_up(ctx->btab_off + btab_bytes, 256);
  ctx->total_bytes = ctx->status_off + 256;
}

}  // namespace

namespace tq {

TableOffsets table_offsets(int d) {
  TableOffsets o;
  o.D = 0;
  o.S = align_up(o.D + sizeof(float) * d, 256);
  o.St = align_up(o.S + 2ull * d * d, 256);
  o.cb = align_up(o.St + 2ull * d * d, 256);
  o.S_sw = align_up(o.cb + sizeof(float) * kCbFloats, 1024);
  o.HD_sw = align_up(o.S_sw + 2ull * d * d, 1024);
  // head_dim 256: H diag(D) for each 128-coordinate half of D (2 x 128 x 128)
  o.S_frag = align_up(o.HD_sw + (d <= 128 ? 2ull * d * d : 2ull * 2 * 128 * 128), 256);
  o.bytes = align_up(o.S_frag + 2ull * d * d, 256);
  return o;
}

LayerView layer_view(const tq_ctx* ctx, int layer) {
  const tq_config& c = ctx->cfg;
  LayerView v;
  v.d = c.head_dim;
  v.vb = c.value_bits;
  v.kb = c.key_bits;
  v.G = c.n_q_heads / c.n_kv_heads;
  v.Hkv = c.n_kv_heads;
  v.Hq = c.n_q_heads;
  v.max_seqs = c.max_seqs;
  v.max_ctx = c.max_ctx;
  v.max_pages = ctx->max_pages;
  v.page_bytes = ctx->pl.bytes;
  uint8_t* tb = static_cast<uint8_t*>(ctx->d_tables);
  v.D = reinterpret_cast<const float*>(tb + ctx->to.D);
  v.S = reinterpret_cast<const uint16_t*>(tb + ctx->to.S);
  v.St = reinterpret_cast<const uint16_t*>(tb + ctx->to.St);
  v.cb = reinterpret_cast<const float*>(tb + ctx->to.cb);
  v.S_sw = reinterpret_cast<const uint16_t*>(tb + ctx->to.S_sw);
  v.S_frag = reinterpret_cast<const uint4*>(tb + ctx->to.S_frag);
  v.HD_sw = reinterpret_cast<const uint16_t*>(tb + ctx->to.HD_sw);
  uint8_t* cb = static_cast<uint8_t*>(ctx->d_cache);
  const size_t units_per_layer = (size_t)c.max_seqs * c.n_kv_heads;
  if (c.n_blocks > 0) {
    v.pages = cb + ctx->pages_off + (size_t)layer * c.n_blocks * c.n_kv_heads * ctx->pl.bytes;
    v.btab = reinterpret_cast<const int32_t*>(cb + ctx->btab_off);
  } else {
    v.pages = cb + ctx->pages_off + (size_t)layer * units_per_layer * ctx->max_pages * ctx->pl.bytes;
    v.btab = nullptr;
  }
  v.n_blocks = c.n_blocks;
  v.ring = reinterpret_cast<uint16_t*>(cb + ctx->ring_off) + (size_t)layer * units_per_layer * ring_elems(c);
  v.state = reinterpret_cast<int32_t*>(cb + ctx->state_off) + (size_t)layer * c.max_seqs * 2;
  v.acnt = reinterpret_cast<int32_t*>(cb + ctx->acnt_off) + (size_t)layer * c.max_seqs;
  v.status = reinterpret_cast<uint32_t*>(cb + ctx->status_off);
  return v;
}

DecodePlan decode_plan(const tq_ctx* ctx, int batch, int max_ctx_hint, int cnt_rows, int ncol) {
  const tq_config& c = ctx->cfg;
  const int hint = (max_ctx_hint <= 0 || max_ctx_hint > c.max_ctx) ? c.max_ctx : max_ctx_hint;
  const int max_pages = std::max(1, (hint + kPage - 1) / kPage);
  const int units = batch * c.n_kv_heads;
  const int sms = ctx->sm_count > 0 ? ctx->sm_count : 152;
  // The wide variant (head_dim 128, K3/V2, contiguous cache, decode rows) when there are at least 128
  // packed pages per CTA slot of two per SM: at batch 32 x 128K it ran 1145 against 1205 us per launch;
  // at batch 1 x 32K (8 pages per slot) and batch 16 x 8K (27) its extra splits made it slower.
  const bool wide = !ctx->host_only && c.head_dim == 128 && c.value_bits == 2 && c.key_bits == 3 &&
                    c.n_blocks == 0 && cnt_rows == 0 && ncol == kMaxG &&
                    (double)units * max_pages >= 128.0 * 2 * sms;
  const int per_sm = ctx->host_only ? 2 : decode_resident_ctas(ctx, wide);
  const int target = per_sm * sms;  // split-K CTAs that fit in one wave
  // Splits per (row, KV head): the fewest whose estimated time is within 3 % of the least, with every
  // row taken at the hint's length. Time = waves x (page rounds of a split + the fixed cost of a split
  // CTA: query prep, merge of its streams, arrival). A split CTA runs 3 page streams at head_dim <= 128
  // and one at 256; its fixed cost is about 2.5 page rounds (batch-1 trace: 2.5 us query prep and
  // 2.7 us merge and arrival against 2.1 us per page round). The ring CTA of a (row, KV head) is short:
  // it counts as that fixed cost's share of a wave slot.
  const int ns = c.head_dim <= 128 ? (wide ? 2 : 3) : 1;
  const double fixed_rounds = 2.5;
  const int max_splits = std::min(max_pages, 1024);  // the combine keeps 4 weights per split in shared memory
  auto cost_of = [&](int pps) {
    const int n = (max_pages + pps - 1) / pps;
    const double rounds = (double)((pps + ns - 1) / ns);
    const double slots = (double)units * (n + fixed_rounds / (rounds + fixed_rounds));
    return std::ceil(slots / target - 1e-9) * (rounds + fixed_rounds);
  };
  double best_cost = cost_of(max_pages);
  for (int s = 2; s <= max_splits; ++s) best_cost = std::min(best_cost, cost_of((max_pages + s - 1) / s));
  int best_pps = max_pages;
  for (int s = 1; s <= max_splits; ++s) {
    const int pps = (max_pages + s - 1) / s;
    if (cost_of(pps) <= 1.03 * best_cost) {
      best_pps = pps;
      break;
    }
  }
  DecodePlan p;
  p.px_off = 0;
  p.px_pages = 0;
  p.wide = wide ? 1 : 0;
  p.pages_per_split = best_pps;
  p.n_splits = (max_pages + p.pages_per_split - 1) / p.pages_per_split;
  const int d = c.head_dim;
  // The arrival counters sit at a fixed place (offset 0, sized for max_seqs rows), so that calls with
  // other batch sizes or hints on the same workspace find them where the last call left them (zero).
  const size_t rows = (size_t)std::max(c.max_seqs, cnt_rows);
  p.cnt_off = 0;
  p.row_cnt_off = sizeof(int32_t) * rows * c.n_kv_heads;  // then one counter per row (decode step)
  p.part_off = align_up(p.row_cnt_off + sizeof(int32_t) * rows, 256);
  p.part_stride = align_up((size_t)(2 * ncol + ncol * d) * sizeof(float), 16);  // m, l [ncol], o [ncol][d]
  p.bytes = align_up(p.part_off + p.part_stride * (size_t)units * (p.n_splits + 1), 256);
  return p;
}

tq_status set_error(tq_status st, const char* msg) {
  g_last_error = msg ? msg : "";
  return st;
}

bool step_follows(tq_ctx* ctx, int layer, cudaStream_t s) {
  const bool follows = ctx->step_layer >= 0 && ctx->step_layer == layer && ctx->step_stream == (void*)s;
  ctx->step_layer = -1;
  return follows;
}

void record_step(tq_ctx* ctx, int layer, cudaStream_t s) {
  ctx->step_layer = layer;
  ctx->step_stream = (void*)s;
}

tq_status check_layer_ready(const tq_ctx* ctx, int layer) {
  if (!ctx) return fail(TQ_ERR_INVALID_ARG, "ctx is NULL");
  if (ctx->host_only || !ctx->d_cache) return fail(TQ_ERR_INVALID_ARG, "no cache bound (tq_cache_bind)");
  if (layer < 0 || layer >= ctx->cfg.n_layers) return fail(TQ_ERR_INVALID_ARG, "layer %d out of range", layer);
  return TQ_OK;
}

}  // namespace tq

// =============================================================================================
// C ABI
// =============================================================================================
extern "C" {

const char* tq_last_error(void) { return g_last_error.c_str(); }

size_t tq_tables_bytes(const tq_config* cfg) {
  if (validate(cfg) != TQ_OK) return 0;
  return tq::table_offsets(cfg->head_dim).bytes;
}

size_t tq_page_bytes(const tq_config* cfg) {
  if (validate(cfg) != TQ_OK) return 0;
  return tq::page_layout(cfg->head_dim, cfg->value_bits, cfg->key_bits).bytes;
}

size_t tq_cache_bytes(const tq_config* cfg) {
  if (validate(cfg) != TQ_OK) return 0;
  tq_ctx tmp;
  tmp.cfg = *cfg;
  compute_offsets(&tmp);
  return tmp.total_bytes;
}

tq_status tq_init_codebooks(const tq_config* cfg, void* d_tables, size_t tables_bytes, tq_stream_t stream,
                            tq_ctx** out) {
  const tq::NvtxRange nvtx_range("tq_init_codebooks");
  if (!out) return fail(TQ_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  tq_status st = validate(cfg);
  if (st != TQ_OK) return st;
  const size_t need = tq::table_offsets(cfg->head_dim).bytes;
  if (d_tables) {
    if (tables_bytes < need) return fail(TQ_ERR_INVALID_ARG, "tables_bytes %zu < %zu", tables_bytes, need);
    if (reinterpret_cast<uintptr_t>(d_tables) % 256) return fail(TQ_ERR_INVALID_ARG, "d_tables not 256-byte aligned");
  }
  tq_ctx* ctx = new (std::nothrow) tq_ctx();
  if (!ctx) return fail(TQ_ERR_INVALID_ARG, "host allocation failed");
  ctx->cfg = *cfg;
  compute_offsets(ctx);
  const int d = cfg->head_dim;
  // rotation signs D and QJL matrix S (bf16), from SplitMix64 streams 1 and 2 of the seed
  const uint64_t seed_D = splitmix64(cfg->seed, 1), seed_S = splitmix64(cfg->seed, 2);
  ctx->D.resize(d);
  for (int i = 0; i < d; ++i) ctx->D[i] = (splitmix64(seed_D, (uint64_t)i + 1) >> 63) ? -1.0f : 1.0f;
  ctx->S.resize((size_t)d * d);
  for (uint64_t k = 0; k < (uint64_t)d * d; ++k) {
    const double u1 = uniform_open(splitmix64(seed_S, 2 * k + 1));
    const double u2 = uniform_open(splitmix64(seed_S, 2 * k + 2));
    const double g = std::sqrt(-2.0 * std::log(u1)) * std::cos(6.283185307179586476925286766559 * u2);
    ctx->S[k] = bf16_rne_bits(g);
  }
  lloyd_max(d, cfg->key_bits - 1, ctx->cent, ctx->bnd);
  if (!d_tables) {  // host-only context: inspection helpers only
    ctx->host_only = true;
    *out = ctx;
    return ok();
  }
  cudaError_t e = cudaGetDevice(&ctx->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&ctx->sm_count, cudaDevAttrMultiProcessorCount, ctx->device);
  if (e != cudaSuccess) {
    delete ctx;
    return cuda_fail(e, "cudaGetDevice");
  }
  // Stage the tables in a host buffer and upload it with one copy. The pageable source is copied
  // before cudaMemcpyAsync returns, so the buffer can be freed right after.
  std::vector<uint8_t> host(need, 0);
  std::memcpy(host.data() + ctx->to.D, ctx->D.data(), sizeof(float) * d);
  std::memcpy(host.data() + ctx->to.S, ctx->S.data(), 2ull * d * d);
  uint16_t* st_h = reinterpret_cast<uint16_t*>(host.data() + ctx->to.St);
  for (int i = 0; i < d; ++i)
    for (int j = 0; j < d; ++j) st_h[(size_t)j * d + i] = ctx->S[(size_t)i * d + j];
  float cb[tq::kCbFloats] = {0};
  const int nlev = 1 << (cfg->key_bits - 1);
  for (int i = 0; i < nlev; ++i) cb[tq::kCbCent + i] = (float)ctx->cent[i];
  for (int i = 0; i < nlev - 1; ++i) cb[tq::kCbBnd + i] = (float)ctx->bnd[i];
  const double* c = ctx->cent;
  if (nlev == 4) {  // c[idx] = w0 (2 b1 - 1) + w1 (2 b0 - 1)
    cb[tq::kCbW + 0] = (float)(0.5 * (c[2] + c[3]));
    cb[tq::kCbW + 1] = (float)(0.5 * (c[3] - c[2]));
  } else {  // c[idx] = A s2 + B t1 + C t0 + E s2 t1 t0 (s, t = 2 bit - 1), fitted to c4..c7 exactly
    cb[tq::kCbW + 0] = (float)(0.25 * (c[4] + c[5] + c[6] + c[7]));
    cb[tq::kCbW + 1] = (float)(0.25 * (-c[4] - c[5] + c[6] + c[7]));
    cb[tq::kCbW + 2] = (float)(0.25 * (-c[4] + c[5] - c[6] + c[7]));
    cb[tq::kCbW + 3] = (float)(0.25 * (c[4] - c[5] - c[6] + c[7]));
  }
  {  // cb[kCbSmax]: max_i sum_j |S_ij| (rounded up), a bound on |(S x)_i| / max|x|
    double m = 0.0;
    for (int i = 0; i < d; ++i) {
      double r = 0.0;
      for (int j = 0; j < d; ++j) r += std::fabs((double)bf16_to_float(ctx->S[(size_t)i * d + j]));
      m = std::max(m, r);
    }
    cb[tq::kCbSmax] = (float)(m * (1.0 + 1e-6));
  }
  std::memcpy(host.data() + ctx->to.cb, cb, sizeof(cb));
  if (d == 256) {
    // S (256 rows) K-major in the 128-byte swizzle: four 32 KB atoms, atom c = columns [64c, 64c + 64)
    uint8_t* sw = host.data() + ctx->to.S_sw;
    for (int n = 0; n < d; ++n)
      for (int k = 0; k < d; ++k)
        std::memcpy(sw + tq::sw128_offset_rows(n, k, 256), &ctx->S[(size_t)n * d + k], 2);
    // H diag(D1) and H diag(D2) for the halves D1 = D[0, 128), D2 = D[128, 256) of the sign vector, with H
    // the 128-point Hadamard: H_256 = [[H, H], [H, -H]] makes the 256-point rotation two of them
    uint8_t* hd = host.data() + ctx->to.HD_sw;
    for (int half = 0; half < 2; ++half)
      for (int i = 0; i < 128; ++i)
        for (int j = 0; j < 128; ++j) {
          const bool neg = (__builtin_popcount((unsigned)(i & j)) & 1) != (ctx->D[128 * half + j] < 0.f);
          const uint16_t v = neg ? 0xBF80u : 0x3F80u;
          std::memcpy(hd + (size_t)half * 32768 + tq::sw128_offset(i, j), &v, 2);
        }
  }
  if (d <= 128) {  // head_dim 64 and 128: one tile of d rows (one or two 64-column atoms)
    uint8_t* sw = host.data() + ctx->to.S_sw;
    for (int n = 0; n < d; ++n)
      for (int k = 0; k < d; ++k) std::memcpy(sw + tq::sw128_offset(n, k), &ctx->S[(size_t)n * d + k], 2);
    // (H diag(D))[i][j] = (-1)^popcount(i & j) * D[j], exact in bf16 (+-1)
    uint8_t* hd = host.data() + ctx->to.HD_sw;
    for (int i = 0; i < d; ++i)
      for (int j = 0; j < d; ++j) {
        const bool neg = (__builtin_popcount((unsigned)(i & j)) & 1) != (ctx->D[j] < 0.f);
        const uint16_t v = neg ? 0xBF80u : 0x3F80u;
        std::memcpy(hd + tq::sw128_offset(i, j), &v, 2);
      }
  }
  {  // S as f16 m16n8k16 A fragments (bf16 -> f16 is exact except below 2^-14, rounded to nearest even)
    uint16_t* fr = reinterpret_cast<uint16_t*>(host.data() + ctx->to.S_frag);
    for (int mt = 0; mt < d / 16; ++mt)
      for (int ks = 0; ks < d / 16; ++ks)
        for (int lane = 0; lane < 32; ++lane) {
          const int g = lane >> 2, c = lane & 3;
          uint16_t* w = fr + (size_t)tq::sfrag_idx(d, mt, ks, lane) * 8;
          for (int r = 0; r < 4; ++r)
            for (int e2 = 0; e2 < 2; ++e2) {
              const int row = 16 * mt + g + 8 * (r & 1), col = 16 * ks + 2 * c + 8 * (r >> 1) + e2;
              w[2 * r + e2] = bf16_to_f16_rne(ctx->S[(size_t)row * d + col]);
            }
        }
  }
  e = cudaMemcpyAsync(d_tables, host.data(), need, cudaMemcpyHostToDevice, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) {
    delete ctx;
    return cuda_fail(e, "upload tables");
  }
  ctx->d_tables = d_tables;
  *out = ctx;
  return ok();
}

tq_status tq_cache_bind(tq_ctx* ctx, void* d_cache, size_t cache_bytes, tq_stream_t stream) {
  const tq::NvtxRange nvtx_range("tq_cache_bind");
  if (!ctx || !d_cache) return fail(TQ_ERR_INVALID_ARG, "ctx or d_cache is NULL");
  if (ctx->host_only) return fail(TQ_ERR_INVALID_ARG, "host-only context (created without d_tables)");
  if (cache_bytes < ctx->total_bytes)
    return fail(TQ_ERR_INVALID_ARG, "cache_bytes %zu < %zu", cache_bytes, ctx->total_bytes);
  if (reinterpret_cast<uintptr_t>(d_cache) % 256) return fail(TQ_ERR_INVALID_ARG, "d_cache not 256-byte aligned");
  uint8_t* base = static_cast<uint8_t*>(d_cache);
  cudaError_t e = cudaMemsetAsync(base + ctx->state_off, 0, ctx->total_bytes - ctx->state_off, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(state)");
  if (ctx->cfg.n_blocks > 0) {  // block table: every entry -1 ("no block")
    e = cudaMemsetAsync(base + ctx->btab_off, 0xFF, (size_t)ctx->cfg.max_seqs * ctx->max_pages * 4, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(block table)");
  }
  ctx->d_cache = d_cache;
  ctx->cache_bytes = cache_bytes;
  return ok();
}

static tq_status check_ready(const tq_ctx* ctx, int layer) {
  if (!ctx) return fail(TQ_ERR_INVALID_ARG, "ctx is NULL");
  if (ctx->host_only || !ctx->d_cache) return fail(TQ_ERR_INVALID_ARG, "no cache bound (tq_cache_bind)");
  if (layer < 0 || layer >= ctx->cfg.n_layers) return fail(TQ_ERR_INVALID_ARG, "layer %d out of range", layer);
  return TQ_OK;
}

tq_status tq_reset_seqs(tq_ctx* ctx, int layer, const int32_t* d_seq_ids, int batch, tq_stream_t stream) {
  const tq::NvtxRange nvtx_range("tq_reset_seqs");
  if (!ctx) return fail(TQ_ERR_INVALID_ARG, "ctx is NULL");
  if (layer != -1) {
    tq_status st = check_ready(ctx, layer);
    if (st != TQ_OK) return st;
  } else if (ctx->host_only || !ctx->d_cache) {
    return fail(TQ_ERR_INVALID_ARG, "no cache bound");
  }
  if (batch < 0 || (batch > 0 && !d_seq_ids)) return fail(TQ_ERR_INVALID_ARG, "bad batch / d_seq_ids");
  if (batch == 0) return ok();
  tq::step_follows(ctx, layer, (cudaStream_t)stream);  // a plain launch: it waits for the whole step
  cudaError_t e = tq::launch_reset(ctx, layer, d_seq_ids, batch, (cudaStream_t)stream);
  return e == cudaSuccess ? ok() : cuda_fail(e, "reset kernel");
}

tq_status tq_quantize_append(tq_ctx* ctx, int layer, const void* k, const void* v, tq_dtype dt,
                             const int32_t* d_seq_ids, const int32_t* d_n_new, int batch, int max_new,
                             tq_stream_t stream) {
  const tq::NvtxRange nvtx_range("tq_quantize_append");
  tq_status st = check_ready(ctx, layer);
  if (st != TQ_OK) return st;
  if (dt != TQ_BF16 && dt != TQ_F32) return fail(TQ_ERR_INVALID_ARG, "dtype %d", (int)dt);
  if (batch < 0 || max_new < 0) return fail(TQ_ERR_INVALID_ARG, "batch %d / max_new %d negative", batch, max_new);
  if (batch == 0 || max_new == 0) return ok();
  if (!k || !v || !d_seq_ids || !d_n_new) return fail(TQ_ERR_INVALID_ARG, "NULL k/v/d_seq_ids/d_n_new");
  if (batch > ctx->cfg.max_seqs) return fail(TQ_ERR_CAPACITY, "batch %d > max_seqs %d", batch, ctx->cfg.max_seqs);
  if (max_new > ctx->cfg.max_ctx) return fail(TQ_ERR_CAPACITY, "max_new %d > max_ctx %d", max_new, ctx->cfg.max_ctx);
  const size_t esz = dt == TQ_BF16 ? 2 : 4;
  if (reinterpret_cast<uintptr_t>(k) % (esz * 4) || reinterpret_cast<uintptr_t>(v) % (esz * 4))
    return fail(TQ_ERR_INVALID_ARG, "k/v must be %zu-byte aligned", esz * 4);
  tq::step_follows(ctx, layer, (cudaStream_t)stream);  // the append kernels read the state after their wait
  cudaError_t e = tq::launch_append(ctx, layer, k, v, (int)dt, d_seq_ids, d_n_new, batch, max_new, (cudaStream_t)stream);
  return e == cudaSuccess ? ok() : cuda_fail(e, "append kernels");
}

tq_status tq_ring_flush(tq_ctx* ctx, int layer, const int32_t* d_seq_ids, int batch, tq_stream_t stream) {
  const tq::NvtxRange nvtx_range("tq_ring_flush");
  tq_status st = check_ready(ctx, layer);
  if (st != TQ_OK) return st;
  if (batch < 0) return fail(TQ_ERR_INVALID_ARG, "batch %d negative", batch);
  if (batch == 0) return ok();
  if (!d_seq_ids) return fail(TQ_ERR_INVALID_ARG, "d_seq_ids is NULL");
  if (batch > ctx->cfg.max_seqs) return fail(TQ_ERR_CAPACITY, "batch %d > max_seqs %d", batch, ctx->cfg.max_seqs);
  tq::step_follows(ctx, layer, (cudaStream_t)stream);  // the flush kernels read the state after their wait
  cudaError_t e = tq::launch_flush(ctx, layer, d_seq_ids, batch, (cudaStream_t)stream);
  return e == cudaSuccess ? ok() : cuda_fail(e, "flush kernel");
}

tq_status tq_dequantize_tokens(tq_ctx* ctx, int layer, int seq_slot, int kv_head, int t0, int count, int with_qjl,
                               float* d_k_out, float* d_v_out, tq_stream_t stream) {
  const tq::NvtxRange nvtx_range("tq_dequantize_tokens");
  tq_status st = check_ready(ctx, layer);
  if (st != TQ_OK) return st;
  const tq_config& c = ctx->cfg;
  if (seq_slot < 0 || seq_slot >= c.max_seqs) return fail(TQ_ERR_INVALID_ARG, "seq_slot %d out of range", seq_slot);
  if (kv_head < 0 || kv_head >= c.n_kv_heads) return fail(TQ_ERR_INVALID_ARG, "kv_head %d out of range", kv_head);
  if (t0 < 0 || count < 0) return fail(TQ_ERR_INVALID_ARG, "t0 %d / count %d negative", t0, count);
  if ((long long)t0 + count > (long long)ctx->max_pages * tq::kPage)
    return fail(TQ_ERR_CAPACITY, "tokens [%d, %lld) beyond the %d pages of a sequence", t0, (long long)t0 + count,
                ctx->max_pages);
  if (with_qjl != 0 && with_qjl != 1) return fail(TQ_ERR_INVALID_ARG, "with_qjl must be 0 or 1");
  if (count == 0) return ok();
  if (!d_k_out || !d_v_out) return fail(TQ_ERR_INVALID_ARG, "NULL output");
  cudaError_t e = tq::launch_dequantize(ctx, layer, seq_slot, kv_head, t0, count, with_qjl, d_k_out, d_v_out,
                                        (cudaStream_t)stream);
  return e == cudaSuccess ? ok() : cuda_fail(e, "dequantize kernel");
}

size_t tq_workspace_bytes(const tq_ctx* ctx, int batch, int max_ctx_hint) {
  if (!ctx || batch < 1) return 0;
  return tq::decode_plan(ctx, batch, max_ctx_hint).bytes;
}

static tq_status decode_common(tq_ctx* ctx, int phase, int layer, const void* q, float* out, const int32_t* d_seq_ids,
                               int batch, float softmax_scale, void* d_workspace, size_t workspace_bytes,
                               int max_ctx_hint, tq_stream_t stream);

// Query rows per prefill CTA: two (that share the key operands of their sequence) when a row's chunk
// has an even number of query slots, the cache is contiguous and the pair kernel's shared memory fits
// (it does for every supported shape, with one page stage fewer at head_dim 128 and key_bits 4), else
// one.
static int prefill_qp(const tq_ctx* ctx, int q_per_row) {
  return q_per_row % 2 == 0 && ctx->cfg.n_blocks == 0 && tq::decode_pairs_fit(ctx) ? 2 : 1;
}

static std::atomic<int> g_prefill_path{0};  // tq_debug_prefill_path: 1 forces the CUDA-core path

// The tcgen05 path fills 128-row tiles with 32 queries; chunks of fewer queries per row take the decode
// kernel, whose CTAs hold one or two query rows.
static bool prefill_tc(const tq_ctx* ctx, int q_per_row) {
  return g_prefill_path.load() == 0 && q_per_row >= 32 && tq::prefill_tc_eligible(ctx);
}

// Workspace plan of the tcgen05 prefill: one query per row (4 columns), n_splits history partials from the
// tensor-core kernel (the ring split runs inside the combine kernel and keeps its part in registers).
// After the partials: every page of every (row, KV head), expanded once for all query tiles (kPxBytes each,
// for the pages of a `max_ctx_hint`-token sequence).
static tq::DecodePlan prefill_tc_plan(const tq_ctx* ctx, int batch, int q_per_row, int max_ctx_hint) {
  const int rows = batch * q_per_row;
  tq::DecodePlan p = tq::decode_plan(ctx, rows, max_ctx_hint, rows, tq::kMaxG);
  p.n_splits = tq::prefill_tc_splits(ctx, batch, q_per_row, max_ctx_hint);
  const int hint = (max_ctx_hint <= 0 || max_ctx_hint > ctx->cfg.max_ctx) ? ctx->cfg.max_ctx : max_ctx_hint;
  p.px_pages = std::max(1, (hint + tq::kPage - 1) / tq::kPage);
  p.px_off = align_up(p.part_off + p.part_stride * (size_t)rows * ctx->cfg.n_kv_heads * p.n_splits, 1024);
  p.bytes = align_up(p.px_off + tq::kPxBytes * (size_t)batch * ctx->cfg.n_kv_heads * p.px_pages, 256);
  return p;
}

size_t tq_prefill_workspace_bytes(const tq_ctx* ctx, int batch, int q_per_row, int max_ctx_hint) {
  if (!ctx || batch < 1 || q_per_row < 1 || (long long)batch * q_per_row > 65535) return 0;
  if (prefill_tc(ctx, q_per_row)) return prefill_tc_plan(ctx, batch, q_per_row, max_ctx_hint).bytes;
  const int qp = prefill_qp(ctx, q_per_row), cta_rows = batch * q_per_row / qp;
  return tq::decode_plan(ctx, cta_rows, max_ctx_hint, cta_rows, tq::kMaxG * qp).bytes;
}

tq_status tq_debug_prefill_path(int mode) {
  if (mode != 0 && mode != 1) return fail(TQ_ERR_INVALID_ARG, "prefill path mode %d not in {0, 1}", mode);
  g_prefill_path.store(mode);
  return ok();
}

tq_status tq_prefill_attention(tq_ctx* ctx, int layer, const void* q, float* out, const int32_t* d_seq_ids,
                               const int32_t* d_n_q, int batch, int q_per_row, float softmax_scale,
                               void* d_workspace, size_t workspace_bytes, int max_ctx_hint, tq_stream_t stream) {
  const tq::NvtxRange nvtx_range("tq_prefill_attention");
  tq_status st = check_ready(ctx, layer);
  if (st != TQ_OK) return st;
  if (batch < 0 || q_per_row < 1) return fail(TQ_ERR_INVALID_ARG, "batch %d / q_per_row %d", batch, q_per_row);
  if (batch == 0) return ok();
  if ((long long)batch * q_per_row > 65535) return fail(TQ_ERR_CAPACITY, "batch * q_per_row above 65535");
  if (!q || !out || !d_seq_ids || !d_n_q || !d_workspace)
    return fail(TQ_ERR_INVALID_ARG, "NULL q/out/d_seq_ids/d_n_q/d_workspace");
  if (batch > ctx->cfg.max_seqs) return fail(TQ_ERR_CAPACITY, "batch %d > max_seqs %d", batch, ctx->cfg.max_seqs);
  if (reinterpret_cast<uintptr_t>(q) % 16 || reinterpret_cast<uintptr_t>(out) % 16)
    return fail(TQ_ERR_INVALID_ARG, "q/out must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(d_workspace) % 256) return fail(TQ_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  if (!(softmax_scale == softmax_scale)) return fail(TQ_ERR_INVALID_ARG, "softmax_scale is NaN");
  if (prefill_tc(ctx, q_per_row)) {
    const tq::DecodePlan plan = prefill_tc_plan(ctx, batch, q_per_row, max_ctx_hint);
    if (workspace_bytes < plan.bytes)
      return fail(TQ_ERR_INVALID_ARG, "workspace_bytes %zu < %zu", workspace_bytes, plan.bytes);
    const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt((float)ctx->cfg.head_dim);
    const cudaStream_t s = (cudaStream_t)stream;
    // The expansion and combine kernels read the sequence state after their stream wait, the tile kernel
    // before it (what it reads was complete when the expansion passed its wait). None uses arrival counters.
    tq::step_follows(ctx, layer, s);
    const cudaError_t e =
        tq::launch_prefill_tc(ctx, layer, q, d_seq_ids, d_n_q, batch, q_per_row, scale, d_workspace, plan, out, s);
    return e == cudaSuccess ? ok() : cuda_fail(e, "prefill attention kernels");
  }
  const int qp = prefill_qp(ctx, q_per_row), cta_rows = batch * q_per_row / qp;
  const tq::DecodePlan plan = tq::decode_plan(ctx, cta_rows, max_ctx_hint, cta_rows, tq::kMaxG * qp);
  if (workspace_bytes < plan.bytes)
    return fail(TQ_ERR_INVALID_ARG, "workspace_bytes %zu < %zu", workspace_bytes, plan.bytes);
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt((float)ctx->cfg.head_dim);
  // Phase 0 zeroes the arrival counters with a memset. It also keeps the prefill kernel from
  // overlapping a preceding append (a memset waits for the whole kernel before it), which the kernel
  // relies on: it reads the sequence lengths, which fix every query's causal extent, before its wait.
  tq::step_follows(ctx, layer, (cudaStream_t)stream);  // the counter memset waits for the whole step
  cudaError_t e = tq::launch_decode(ctx, layer, q, out, d_seq_ids, cta_rows, scale, d_workspace, plan, 0,
                                    (cudaStream_t)stream, q_per_row, d_n_q, qp);  // zero the counters
  if (e == cudaSuccess)
    e = tq::launch_decode(ctx, layer, q, out, d_seq_ids, cta_rows, scale, d_workspace, plan, 1, (cudaStream_t)stream,
                          q_per_row, d_n_q, qp);
  return e == cudaSuccess ? ok() : cuda_fail(e, "prefill attention kernels");
}

tq_status tq_decode_attention(tq_ctx* ctx, int layer, const void* q, float* out, const int32_t* d_seq_ids,
                              int batch, float softmax_scale, void* d_workspace, size_t workspace_bytes,
                              int max_ctx_hint, tq_stream_t stream) {
  const tq::NvtxRange nvtx_range("tq_decode_attention");
  return decode_common(ctx, -1, layer, q, out, d_seq_ids, batch, softmax_scale, d_workspace, workspace_bytes,
                       max_ctx_hint, stream);
}

tq_status tq_decode_phase(tq_ctx* ctx, int phase, int layer, const void* q, float* out, const int32_t* d_seq_ids,
                          int batch, float softmax_scale, void* d_workspace, size_t workspace_bytes,
                          int max_ctx_hint, tq_stream_t stream) {
  const tq::NvtxRange nvtx_range("tq_decode_phase");
  if (phase < 0 || phase > 1) return fail(TQ_ERR_INVALID_ARG, "phase %d not in {0, 1}", phase);
  return decode_common(ctx, phase, layer, q, out, d_seq_ids, batch, softmax_scale, d_workspace, workspace_bytes,
                       max_ctx_hint, stream);
}

tq_status tq_decode_step(tq_ctx* ctx, int layer, const void* k_new, const void* v_new, tq_dtype dt, const void* q,
                         float* out, const int32_t* d_seq_ids, int batch, float softmax_scale, void* d_workspace,
                         size_t workspace_bytes, int max_ctx_hint, tq_stream_t stream) {
  const tq::NvtxRange nvtx_range("tq_decode_step");
  tq_status st = check_ready(ctx, layer);
  if (st != TQ_OK) return st;
  if (dt != TQ_BF16 && dt != TQ_F32) return fail(TQ_ERR_INVALID_ARG, "dtype %d", (int)dt);
  if (batch < 0) return fail(TQ_ERR_INVALID_ARG, "batch %d negative", batch);
  if (batch == 0) return ok();
  if (!k_new || !v_new || !q || !out || !d_seq_ids || !d_workspace)
    return fail(TQ_ERR_INVALID_ARG, "NULL k_new/v_new/q/out/d_seq_ids/d_workspace");
  if (batch > ctx->cfg.max_seqs) return fail(TQ_ERR_CAPACITY, "batch %d > max_seqs %d", batch, ctx->cfg.max_seqs);
  const size_t esz = dt == TQ_BF16 ? 2 : 4;
  if (reinterpret_cast<uintptr_t>(k_new) % (esz * 4) || reinterpret_cast<uintptr_t>(v_new) % (esz * 4))
    return fail(TQ_ERR_INVALID_ARG, "k_new/v_new must be %zu-byte aligned", esz * 4);
  if (reinterpret_cast<uintptr_t>(q) % 16 || reinterpret_cast<uintptr_t>(out) % 16)
    return fail(TQ_ERR_INVALID_ARG, "q/out must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(d_workspace) % 256) return fail(TQ_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  if (!(softmax_scale == softmax_scale)) return fail(TQ_ERR_INVALID_ARG, "softmax_scale is NaN");
  const tq::DecodePlan plan = tq::decode_plan(ctx, batch, max_ctx_hint);
  if (workspace_bytes < plan.bytes)
    return fail(TQ_ERR_INVALID_ARG, "workspace_bytes %zu < %zu", workspace_bytes, plan.bytes);
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt((float)ctx->cfg.head_dim);
  const cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  if (ctx->cfg.ring_size == 0) {  // full_tq: the append codes the token into its page, then the decode
    tq::step_follows(ctx, layer, s);
    e = tq::launch_append(ctx, layer, k_new, v_new, (int)dt, d_seq_ids, nullptr, batch, 1, s);
    if (e == cudaSuccess) e = tq::launch_decode(ctx, layer, q, out, d_seq_ids, batch, scale, d_workspace, plan, -1, s);
  } else {
    const int late = tq::step_follows(ctx, layer, s) ? 1 : 0;
    e = tq::launch_decode(ctx, layer, q, out, d_seq_ids, batch, scale, d_workspace, plan, -1, s, 1, nullptr, 1, k_new,
                          v_new, (int)dt, late);
    if (e == cudaSuccess) tq::record_step(ctx, layer, s);
  }
  return e == cudaSuccess ? ok() : cuda_fail(e, "decode step kernels");
}

static tq_status decode_common(tq_ctx* ctx, int phase, int layer, const void* q, float* out, const int32_t* d_seq_ids,
                               int batch, float softmax_scale, void* d_workspace, size_t workspace_bytes,
                               int max_ctx_hint, tq_stream_t stream) {
  tq_status st = check_ready(ctx, layer);
  if (st != TQ_OK) return st;
  if (batch < 0) return fail(TQ_ERR_INVALID_ARG, "batch %d negative", batch);
  if (batch == 0) return ok();
  if (!q || !out || !d_seq_ids || !d_workspace) return fail(TQ_ERR_INVALID_ARG, "NULL q/out/d_seq_ids/d_workspace");
  if (batch > ctx->cfg.max_seqs) return fail(TQ_ERR_CAPACITY, "batch %d > max_seqs %d", batch, ctx->cfg.max_seqs);
  if (reinterpret_cast<uintptr_t>(q) % 16 || reinterpret_cast<uintptr_t>(out) % 16)
    return fail(TQ_ERR_INVALID_ARG, "q/out must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(d_workspace) % 256) return fail(TQ_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  if (!(softmax_scale == softmax_scale)) return fail(TQ_ERR_INVALID_ARG, "softmax_scale is NaN");
  const tq::DecodePlan plan = tq::decode_plan(ctx, batch, max_ctx_hint);
  if (workspace_bytes < plan.bytes)
    return fail(TQ_ERR_INVALID_ARG, "workspace_bytes %zu < %zu", workspace_bytes, plan.bytes);
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt((float)ctx->cfg.head_dim);
  cudaError_t e =
      tq::launch_decode(ctx, layer, q, out, d_seq_ids, batch, scale, d_workspace, plan, phase, (cudaStream_t)stream, 1,
                        nullptr, 1, nullptr, nullptr, 0, tq::step_follows(ctx, layer, (cudaStream_t)stream) ? 1 : 0);
  return e == cudaSuccess ? ok() : cuda_fail(e, "decode kernels");
}

tq_status tq_check_status(tq_ctx* ctx, tq_stream_t stream, uint32_t* word, int clear) {
  if (!ctx || ctx->host_only || !ctx->d_cache) return fail(TQ_ERR_INVALID_ARG, "no cache bound");
  uint32_t w = 0;
  uint8_t* p = static_cast<uint8_t*>(ctx->d_cache) + ctx->status_off;
  cudaError_t e = cudaMemcpyAsync(&w, p, 4, cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "read status");
  if (word) *word = w;
  if (clear && w) {
    e = cudaMemsetAsync(p, 0, 4, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "clear status");
  }
  if (w) return fail(TQ_ERR_DEVICE, "device status word 0x%x", w);
  return ok();
}

void tq_destroy(tq_ctx* ctx) { delete ctx; }

size_t tq_page_offset(const tq_ctx* ctx, int layer, int slot, int kv_head, int page) {
  const tq_config& c = ctx->cfg;
  if (c.n_blocks > 0) return (size_t)-1;
  return ctx->pages_off +
         ((((size_t)layer * c.max_seqs + slot) * c.n_kv_heads + kv_head) * ctx->max_pages + page) * ctx->pl.bytes;
}

size_t tq_block_page_offset(const tq_ctx* ctx, int layer, int block, int kv_head) {
  const tq_config& c = ctx->cfg;
  if (c.n_blocks <= 0) return (size_t)-1;
  return ctx->pages_off + ((((size_t)layer * c.n_blocks + block) * c.n_kv_heads) + kv_head) * ctx->pl.bytes;
}

size_t tq_block_table_offset(const tq_ctx* ctx) { return ctx->cfg.n_blocks > 0 ? ctx->btab_off : (size_t)-1; }

size_t tq_ring_offset(const tq_ctx* ctx, int layer, int slot, int kv_head, int which) {
  const tq_config& c = ctx->cfg;
  return ctx->ring_off +
         ((((size_t)layer * c.max_seqs + slot) * c.n_kv_heads + kv_head) * 2 + which) * tq::kPage * c.head_dim * 2;
}

size_t tq_state_offset(const tq_ctx* ctx, int layer, int slot) {
  return ctx->state_off + ((size_t)layer * ctx->cfg.max_seqs + slot) * 8;
}

size_t tq_status_offset(const tq_ctx* ctx) { return ctx->status_off; }

tq_status tq_page_to_records(const tq_ctx* ctx, const void* h_page, int n_tokens, uint8_t* out_keys,
                             uint8_t* out_values) {
  if (!ctx || !h_page || !out_keys || !out_values) return fail(TQ_ERR_INVALID_ARG, "NULL argument");
  if (n_tokens < 0 || n_tokens > tq::kPage) return fail(TQ_ERR_INVALID_ARG, "n_tokens %d", n_tokens);
  const int d = ctx->cfg.head_dim, vb = ctx->cfg.value_bits;
  const tq::PageLayout& pl = ctx->pl;
  const uint8_t* pg = static_cast<const uint8_t*>(h_page);
  const uint32_t* kw = reinterpret_cast<const uint32_t*>(pg + pl.kbits_off);
  const uint32_t* vw = reinterpret_cast<const uint32_t*>(pg + pl.vbits_off);
  const int kb = ctx->cfg.key_bits, mb = kb - 1;  // planes; index bits
  const size_t kidx = (size_t)d * mb / 8, krec = kidx + d / 8 + 4, vrec = (size_t)d * vb / 8 + d / 16;
  for (int t = 0; t < n_tokens; ++t) {
    uint8_t* kr = out_keys + t * krec;
    uint8_t* vr = out_values + t * vrec;
    std::memset(kr, 0, krec);
    std::memset(vr, 0, vrec);
    for (int j = 0; j < d; ++j) {
      int w, b, idx = 0;
      for (int pi = 0; pi < mb; ++pi) {  // index bits, highest first
        tq::kbit_loc(d, kb, t, j, pi, w, b);
        idx = 2 * idx + (int)((kw[w] >> b) & 1);
      }
      tq::kbit_loc(d, kb, t, j, mb, w, b);
      const int sg = (kw[w] >> b) & 1;
      for (int i = 0; i < mb; ++i) {  // little-endian bit stream: index bit i of element j at stream bit mb j + i
        const int sb = mb * j + i;
        kr[sb / 8] |= (uint8_t)(((idx >> i) & 1) << (sb % 8));
      }
      kr[kidx + j / 8] |= (uint8_t)(sg << (j % 8));
      tq::vcode_loc(d, vb, t, j, w, b);
      const int code = (vw[w] >> b) & ((1 << vb) - 1);
      const int per = 8 / vb;
      vr[j / per] |= (uint8_t)(code << (vb * (j % per)));
    }
    std::memcpy(kr + kidx + d / 8, pg + pl.norms_off + 4 * t, 4);
    for (int q = 0; q < d / 32; ++q)
      std::memcpy(vr + (size_t)d * vb / 8 + 2 * q, pg + pl.vscale_off + 2 * (size_t)tq::vscale_idx(d, t, q), 2);
  }
  return ok();
}

tq_status tq_records_to_page(const tq_ctx* ctx, const uint8_t* keys, const uint8_t* values, int n_tokens,
                             void* h_page) {
  if (!ctx || !keys || !values || !h_page) return fail(TQ_ERR_INVALID_ARG, "NULL argument");
  if (n_tokens < 0 || n_tokens > tq::kPage) return fail(TQ_ERR_INVALID_ARG, "n_tokens %d", n_tokens);
  const int d = ctx->cfg.head_dim, vb = ctx->cfg.value_bits;
  const tq::PageLayout& pl = ctx->pl;
  uint8_t* pg = static_cast<uint8_t*>(h_page);
  std::memset(pg, 0, pl.bytes);
  uint32_t* kw = reinterpret_cast<uint32_t*>(pg + pl.kbits_off);
  uint32_t* vw = reinterpret_cast<uint32_t*>(pg + pl.vbits_off);
  const int kb = ctx->cfg.key_bits, mb = kb - 1;
  const size_t kidx = (size_t)d * mb / 8, krec = kidx + d / 8 + 4, vrec = (size_t)d * vb / 8 + d / 16;
  for (int t = 0; t < n_tokens; ++t) {
    const uint8_t* kr = keys + t * krec;
    const uint8_t* vr = values + t * vrec;
    for (int j = 0; j < d; ++j) {
      int idx = 0;
      for (int i = 0; i < mb; ++i) {
        const int sb = mb * j + i;
        idx |= ((kr[sb / 8] >> (sb % 8)) & 1) << i;
      }
      const int sg = (kr[kidx + j / 8] >> (j % 8)) & 1;
      int w, b;
      for (int pi = 0; pi < mb; ++pi) {
        tq::kbit_loc(d, kb, t, j, pi, w, b);
        kw[w] |= (uint32_t)((idx >> (mb - 1 - pi)) & 1) << b;
      }
      tq::kbit_loc(d, kb, t, j, mb, w, b);
      kw[w] |= (uint32_t)sg << b;
      const int per = 8 / vb;
      const int code = (vr[j / per] >> (vb * (j % per))) & ((1 << vb) - 1);
      tq::vcode_loc(d, vb, t, j, w, b);
      vw[w] |= (uint32_t)code << b;
    }
    std::memcpy(pg + pl.norms_off + 4 * t, kr + kidx + d / 8, 4);
    for (int q = 0; q < d / 32; ++q)
      std::memcpy(pg + pl.vscale_off + 2 * (size_t)tq::vscale_idx(d, t, q), vr + (size_t)d * vb / 8 + 2 * q, 2);
  }
  return ok();
}

tq_status tq_get_tables(const tq_ctx* ctx, float* D, uint16_t* S_bf16, double* centroids, double* boundaries) {
  if (!ctx) return fail(TQ_ERR_INVALID_ARG, "ctx is NULL");
  const int d = ctx->cfg.head_dim;
  if (D) std::memcpy(D, ctx->D.data(), sizeof(float) * d);
  if (S_bf16) std::memcpy(S_bf16, ctx->S.data(), 2ull * d * d);
  const int nlev = 1 << (ctx->cfg.key_bits - 1);
  if (centroids) std::memcpy(centroids, ctx->cent, sizeof(double) * nlev);
  if (boundaries) std::memcpy(boundaries, ctx->bnd, sizeof(double) * (nlev - 1));
  return ok();
}

}  // extern "C"
