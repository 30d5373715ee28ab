// Seeded synthetic parameters and pixels; the recipe is documented in synth.h.
#include "synth.h"

#include <cmath>
#include <cstdio>
#include <cstring>
#include <thread>
#include <vector>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;   // SplitMix64 increment
constexpr uint64_t kTagMul = 0xD1B54A32D192ED03ull;  // spreads tags over key space

// SplitMix64 output finaliser (Steele, Lea & Flood 2014).
inline uint64_t mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

inline uint64_t stream_key(uint64_t seed, uint64_t tag) { return mix(seed ^ (kTagMul * (tag + 1))); }
inline uint64_t draw(uint64_t key, uint64_t i) { return mix(key + (i + 1) * kGamma); }
inline double uniform01(uint64_t key, uint64_t i) {
  return (static_cast<double>(draw(key, i) >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}
inline double normal(uint64_t key, uint64_t i) {
  const double u1 = uniform01(key, 2 * i), u2 = uniform01(key, 2 * i + 1);
  return std::sqrt(-2.0 * std::log(u1)) * std::cos(6.283185307179586476925286766559 * u2);
}

// Runs f(begin, end) over [0, n) on all hardware threads for large n.
template <class F>
void parallel_for(size_t n, F f, size_t work_per_item = 1) {
  unsigned nt = std::thread::hardware_concurrency();
  if (nt == 0) nt = 1;
  if (n * work_per_item < (size_t(1) << 20) || nt == 1 || n < nt) {
    f(size_t(0), n);
    return;
  }
  std::vector<std::thread> th;
  const size_t chunk = (n + nt - 1) / nt;
  for (unsigned t = 0; t < nt; ++t) {
    const size_t b = t * chunk, e = b + chunk < n ? b + chunk : n;
    if (b >= e) break;
    th.emplace_back([=] { f(b, e); });
  }
  for (auto& x : th) x.join();
}

}  // namespace

extern "C" {

uint16_t synth_f16_from_double(double x) {
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  if (std::isnan(x)) return 0x7E00;
  const double a = std::fabs(x);
  if (a >= 65520.0) return sign | 0x7C00;  // at or past the midpoint above 65504
  if (a < 6.103515625e-05) {               // below 2^-14: subnormal quantum 2^-24
    const double q = std::nearbyint(a * 16777216.0);  // RNE in the default mode
    return sign | static_cast<uint16_t>(q);           // q == 1024 encodes 2^-14 exactly
  }
  int ex;
  const double m = std::frexp(a, &ex);  // a = m * 2^ex, m in [0.5, 1)
  int e = ex - 1;                       // a = (2m) * 2^e, 2m in [1, 2)
  double q = std::nearbyint((2.0 * m - 1.0) * 1024.0);
  if (q >= 1024.0) {
    q = 0.0;
    ++e;
  }
  return sign | static_cast<uint16_t>(((e + 15) << 10) | static_cast<int>(q));
}

synth_dims synth_so400m(int layers) {
  synth_dims d;
  d.tokens = 729;
  d.patch_dim = 588;
  d.width = 1152;
  d.heads = 16;
  d.mlp = 4304;
  d.layers = layers;
  return d;
}

int synth_tensor_count(const synth_dims* d) { return 3 + 12 * d->layers + 15; }

static void set(synth_tensor* t, const char* name, int layer, int rows, int cols, int kind, double mean,
                double std) {
  std::snprintf(t->name, sizeof(t->name), "%s", name);
  t->layer = layer;
  t->rows = rows;
  t->cols = cols;
  t->kind = kind;
  t->mean = mean;
  t->std = std;
}

int synth_tensor_info(const synth_dims* d, int id, synth_tensor* t) {
  const int D = d->width, P = d->patch_dim, T = d->tokens, F = d->mlp, L = d->layers;
  auto xavier = [](int k, int n) { return std::sqrt(2.0 / (double(k) + double(n))); };
  const double bias_std = 0.01, emb_std = 1.0 / std::sqrt(double(D));
  if (id < 0 || id >= synth_tensor_count(d)) return -1;
  if (id == 0) return set(t, "patch_w", -1, P, D, SYNTH_NORMAL, 0, xavier(P, D)), 0;
  if (id == 1) return set(t, "patch_b", -1, 1, D, SYNTH_NORMAL, 0, bias_std), 0;
  if (id == 2) return set(t, "pos", -1, T, D, SYNTH_NORMAL, 0, emb_std), 0;
  if (id < 3 + 12 * L) {
    const int l = (id - 3) / 12, j = (id - 3) % 12;
    switch (j) {
      case 0: set(t, "ln1_g", l, 1, D, SYNTH_CONST, 1, 0); break;
      case 1: set(t, "ln1_b", l, 1, D, SYNTH_CONST, 0, 0); break;
      case 2: set(t, "qkv_w", l, D, 3 * D, SYNTH_NORMAL, 0, xavier(D, D)); break;
      case 3: set(t, "qkv_b", l, 1, 3 * D, SYNTH_NORMAL, 0, bias_std); break;
      case 4: set(t, "out_w", l, D, D, SYNTH_NORMAL, 0, xavier(D, D)); break;
      case 5: set(t, "out_b", l, 1, D, SYNTH_NORMAL, 0, bias_std); break;
      case 6: set(t, "ln2_g", l, 1, D, SYNTH_CONST, 1, 0); break;
      case 7: set(t, "ln2_b", l, 1, D, SYNTH_CONST, 0, 0); break;
      case 8: set(t, "fc1_w", l, D, F, SYNTH_NORMAL, 0, xavier(D, F)); break;
      case 9: set(t, "fc1_b", l, 1, F, SYNTH_NORMAL, 0, bias_std); break;
      case 10: set(t, "fc2_w", l, F, D, SYNTH_NORMAL, 0, xavier(F, D)); break;
      default: set(t, "fc2_b", l, 1, D, SYNTH_NORMAL, 0, bias_std); break;
    }
    return 0;
  }
  switch (id - 3 - 12 * L) {
    case 0: set(t, "enc_ln_g", -1, 1, D, SYNTH_CONST, 1, 0); break;
    case 1: set(t, "enc_ln_b", -1, 1, D, SYNTH_CONST, 0, 0); break;
    case 2: set(t, "probe", -1, 1, D, SYNTH_NORMAL, 0, emb_std); break;
    case 3: set(t, "map_q_w", -1, D, D, SYNTH_NORMAL, 0, xavier(D, D)); break;
    case 4: set(t, "map_q_b", -1, 1, D, SYNTH_NORMAL, 0, bias_std); break;
    case 5: set(t, "map_kv_w", -1, D, 2 * D, SYNTH_NORMAL, 0, xavier(D, D)); break;
    case 6: set(t, "map_kv_b", -1, 1, 2 * D, SYNTH_NORMAL, 0, bias_std); break;
    case 7: set(t, "map_out_w", -1, D, D, SYNTH_NORMAL, 0, xavier(D, D)); break;
    case 8: set(t, "map_out_b", -1, 1, D, SYNTH_NORMAL, 0, bias_std); break;
    case 9: set(t, "map_ln_g", -1, 1, D, SYNTH_CONST, 1, 0); break;
    case 10: set(t, "map_ln_b", -1, 1, D, SYNTH_CONST, 0, 0); break;
    case 11: set(t, "map_fc1_w", -1, D, F, SYNTH_NORMAL, 0, xavier(D, F)); break;
    case 12: set(t, "map_fc1_b", -1, 1, F, SYNTH_NORMAL, 0, bias_std); break;
    case 13: set(t, "map_fc2_w", -1, F, D, SYNTH_NORMAL, 0, xavier(F, D)); break;
    default: set(t, "map_fc2_b", -1, 1, D, SYNTH_NORMAL, 0, bias_std); break;
  }
  return 0;
}

void synth_normal_f16(uint64_t seed, uint64_t tag, double mean, double std, uint16_t* out, size_t n) {
  const uint64_t key = stream_key(seed, tag);
  parallel_for(n, [&](size_t b, size_t e) {
    for (size_t i = b; i < e; ++i) out[i] = synth_f16_from_double(mean + std * normal(key, i));
  });
}

void synth_uniform_f16(uint64_t seed, uint64_t tag, double lo, double hi, uint16_t* out, size_t n) {
  const uint64_t key = stream_key(seed, tag);
  parallel_for(n, [&](size_t b, size_t e) {
    for (size_t i = b; i < e; ++i) out[i] = synth_f16_from_double(lo + (hi - lo) * uniform01(key, i));
  });
}

uint64_t synth_draw_u64(uint64_t seed, uint64_t tag, uint64_t i) { return draw(stream_key(seed, tag), i); }
double synth_draw_normal(uint64_t seed, uint64_t tag, uint64_t i) { return normal(stream_key(seed, tag), i); }

int synth_fill_tensor_f16(uint64_t seed, const synth_dims* d, int id, uint16_t* out) {
  synth_tensor t;
  if (synth_tensor_info(d, id, &t) != 0) return -1;
  const size_t n = size_t(t.rows) * size_t(t.cols);
  if (t.kind == SYNTH_CONST) {
    const uint16_t v = synth_f16_from_double(t.mean);
    for (size_t i = 0; i < n; ++i) out[i] = v;
    return 0;
  }
  synth_normal_f16(seed, uint64_t(id), t.mean, t.std, out, n);
  return 0;
}

int synth_fill_tensor_f16_t(uint64_t seed, const synth_dims* d, int id, uint16_t* out, int k_stride) {
  synth_tensor t;
  if (synth_tensor_info(d, id, &t) != 0 || k_stride < t.rows) return -1;
  const int K = t.rows, N = t.cols;
  const uint64_t key = stream_key(seed, uint64_t(id));
  const uint16_t cval = synth_f16_from_double(t.mean);
  parallel_for(size_t(N), [&](size_t b, size_t e) {
    for (size_t n = b; n < e; ++n) {
      uint16_t* row = out + n * size_t(k_stride);
      for (int k = 0; k < K; ++k) {
        const size_t i = size_t(k) * size_t(N) + n;  // index in the logical [K][N] order
        row[k] = t.kind == SYNTH_CONST ? cval : synth_f16_from_double(t.mean + t.std * normal(key, i));
      }
      for (int k = K; k < k_stride; ++k) row[k] = 0;
    }
  }, size_t(K));
  return 0;
}

void synth_pixels_f16(uint64_t seed, int batch, int tokens, int patch_dim, uint16_t* out) {
  synth_uniform_f16(seed, SYNTH_PIXEL_TAG, -1.0, 1.0, out, size_t(batch) * tokens * patch_dim);
}

}  // extern "C"
