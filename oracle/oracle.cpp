/*
 * ORACLE — test infrastructure only. Plain, slow, obviously correct CPU
 * implementation of the So400m/14 SigLIP image encoder forward pass, used to
 * check the CUDA library. Only tests, the smoke check and the benchmark's CPU
 * baseline may load it; the product never does. It shares no code with the
 * CUDA path: its inputs are parameters and pixels drawn by the seeded
 * generator (synth/) and converted to float by the caller.
 *
 * Precision: tensors are FP32 (the pages validate against an "unquantised FP32
 * reference": "SigLIP optimized execution and PV padding" page, "Full-model
 * results"); every dot product and reduction accumulates in double, so the
 * oracle's own rounding sits far below the F16 path's.
 *
 * What it computes (all from the "SigLIP ViT benchmark" page unless noted):
 *   - patch embedding: the 588->1152 GEMM + bias, then the learned positional
 *     embedding (network paragraph, flowchart, pixel-binding paragraph);
 *   - per layer, pre-norm: Y = LN1(X); [Q K V] = Y [Wq|Wk|Wv] + b ("fused QKV"
 *     section: one 1152->3456 GEMM, then last-axis slices); per head h the
 *     channels h*72 .. h*72+71; S = Q_h K_h^T / sqrt(72); P = softmax(S) (row
 *     max subtracted); O_h = P V_h; X += O Wo + bo; Y = LN2(X);
 *     X += gelu(Y W1 + b1) W2 + b2 (flowchart);
 *   - final encoder LayerNorm, then MAP pooling: a learned probe is projected
 *     by its own Q projection, the fused 1152->2304 KV projection of the
 *     encoder output gives K and V, one query per head attends over the 729
 *     tokens, the output projection gives A, and out = A + MLP(LN(A))
 *     (network paragraph, flowchart, "fused QKV" section);
 *   - LayerNorm: epsilon 1e-6, affine, mean then centred (biased) variance
 *     (LayerNorm paragraph);
 *   - GELU: the tanh form 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)));
 *   - optional FP8 mode: every dense-GEMM operand is rounded to OCP E4M3
 *     (saturating, round-to-nearest-even) at scale 2^-4, i.e.
 *     x_hat = E4M3(16 x) / 16 (FP8 example and paragraph after it).
 *
 * Readings of points the pages leave open: scores scaled by 1/sqrt(72); the
 * GELU is the tanh form; LN variance is biased with eps inside the square
 * root; the MAP residual wraps only the MLP; every projection has a bias.
 *
 * Pins (tests/test_oracle_pins.py): every function here is checked against
 * something other than itself (direct convolution, LN invariants, softmax
 * sums, brute-force attention, single-key MAP, GELU special values, torch
 * float64 library routines, E4M3 against torch's float8 cast).
 */
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <thread>
#include <vector>

namespace {

int g_threads = 0;

int threads() {
  if (g_threads > 0) return g_threads;
  const char* env = std::getenv("ORACLE_THREADS");
  int n = env ? std::atoi(env) : 0;
  if (n <= 0) n = static_cast<int>(std::thread::hardware_concurrency());
  g_threads = n > 0 ? n : 1;
  return g_threads;
}

// Runs f(i) for i in [0, n) spread over the oracle's threads.
template <class F>
void parallel(long n, F f) {
  const int nt = static_cast<int>(std::min<long>(threads(), std::max<long>(n, 1)));
  if (nt <= 1) {
    for (long i = 0; i < n; ++i) f(i);
    return;
  }
  std::vector<std::thread> pool;
  for (int t = 0; t < nt; ++t)
    pool.emplace_back([=] {
      for (long i = t; i < n; i += nt) f(i);
    });
  for (auto& th : pool) th.join();
}

// OCP OFP8 E4M3 ("e4m3fn"): bias 7, no infinities, largest finite 448,
// smallest normal 2^-6, subnormal spacing 2^-9. Round to nearest even,
// saturate finite values to +-448.
float e4m3_value(float x) {
  if (std::isnan(x)) return x;
  const float a = std::fabs(x);
  float r;
  if (a >= 448.0f) {
    r = 448.0f;
  } else if (a < 0.015625f) {  // below 2^-6: fixed quantum 2^-9
    r = std::nearbyint(a * 512.0f) / 512.0f;
  } else {
    int ex;
    std::frexp(a, &ex);                               // a in [2^(ex-1), 2^ex)
    const float quantum = std::ldexp(1.0f, ex - 4);   // 3 fraction bits
    r = std::nearbyint(a / quantum) * quantum;
  }
  return std::signbit(x) ? -r : r;
}

// Operand rounding of the FP8 mode: x_hat = E4M3(16 x) / 16.
std::vector<float> fp8_round(const float* x, size_t n) {
  std::vector<float> y(n);
  for (size_t i = 0; i < n; ++i) y[i] = e4m3_value(16.0f * x[i]) / 16.0f;
  return y;
}

double gelu_tanh(double x) {
  const double c = std::sqrt(2.0 / 3.14159265358979323846);
  return 0.5 * x * (1.0 + std::tanh(c * (x + 0.044715 * x * x * x)));
}

// C[M][N] = A[M][K] W[K][N] (+ bias[N]); A has row stride lda.
void linear(const float* A, long lda, const float* W, const float* bias, float* C, long M, long N, long K,
            bool quant) {
  std::vector<float> Aq, Wq;
  if (quant) {
    Aq.resize(size_t(M) * K);
    for (long i = 0; i < M; ++i) {
      std::vector<float> r = fp8_round(A + i * lda, size_t(K));
      std::copy(r.begin(), r.end(), Aq.begin() + i * K);
    }
    Wq = fp8_round(W, size_t(K) * N);
    A = Aq.data();
    lda = K;
    W = Wq.data();
  }
  auto row = [&](long i, long n0, long n1) {
    std::vector<double> acc(size_t(n1 - n0), 0.0);
    const float* a = A + i * lda;
    for (long k = 0; k < K; ++k) {
      const double ak = a[k];
      const float* w = W + k * N;
      for (long n = n0; n < n1; ++n) acc[size_t(n - n0)] += ak * double(w[n]);
    }
    for (long n = n0; n < n1; ++n)
      C[i * N + n] = static_cast<float>(acc[size_t(n - n0)] + (bias ? double(bias[n]) : 0.0));
  };
  if (M >= threads()) {
    parallel(M, [&](long i) { row(i, 0, N); });
  } else {  // few rows (MAP head): split the columns instead
    const long chunk = 64, nchunks = (N + chunk - 1) / chunk;
    parallel(M * nchunks, [&](long t) {
      const long i = t / nchunks, c = t % nchunks;
      row(i, c * chunk, std::min(N, (c + 1) * chunk));
    });
  }
}

void layernorm(const float* x, const float* g, const float* b, float* y, long rows, long width, float eps) {
  parallel(rows, [&](long r) {
    const float* xr = x + r * width;
    double mean = 0.0;
    for (long i = 0; i < width; ++i) mean += xr[i];
    mean /= double(width);
    double var = 0.0;
    for (long i = 0; i < width; ++i) var += (xr[i] - mean) * (xr[i] - mean);
    var /= double(width);
    const double inv = 1.0 / std::sqrt(var + double(eps));
    for (long i = 0; i < width; ++i) y[r * width + i] = static_cast<float>((xr[i] - mean) * inv * g[i] + b[i]);
  });
}

// Multi-head attention over token-major rows: q rows [Tq][ldq], k/v rows
// [Tk][ldk]/[Tk][ldv]; head h uses channels h*dh .. h*dh+dh-1; o rows [Tq][ldo].
void attention_one(const float* q, long ldq, const float* k, long ldk, const float* v, long ldv, float* o, long ldo,
                   long Tq, long Tk, long h, long dh, double scale) {
  std::vector<double> s(static_cast<size_t>(Tk));
  for (long i = 0; i < Tq; ++i) {
    const float* qi = q + i * ldq + h * dh;
    double m = -INFINITY;
    for (long j = 0; j < Tk; ++j) {
      const float* kj = k + j * ldk + h * dh;
      double dot = 0.0;
      for (long d = 0; d < dh; ++d) dot += double(qi[d]) * double(kj[d]);
      s[size_t(j)] = dot * scale;
      m = std::max(m, s[size_t(j)]);
    }
    double l = 0.0;
    for (long j = 0; j < Tk; ++j) {
      s[size_t(j)] = std::exp(s[size_t(j)] - m);
      l += s[size_t(j)];
    }
    for (long d = 0; d < dh; ++d) {
      double acc = 0.0;
      for (long j = 0; j < Tk; ++j) acc += s[size_t(j)] * double(v[j * ldv + h * dh + d]);
      o[i * ldo + h * dh + d] = static_cast<float>(acc / l);
    }
  }
}

}  // namespace

extern "C" {

typedef struct {
  int tokens, patch_dim, width, heads, head_dim, mlp, layers;
  const float *patch_w, *patch_b, *pos;
  const float* const* ln1_g;
  const float* const* ln1_b;
  const float* const* qkv_w;
  const float* const* qkv_b;
  const float* const* out_w;
  const float* const* out_b;
  const float* const* ln2_g;
  const float* const* ln2_b;
  const float* const* fc1_w;
  const float* const* fc1_b;
  const float* const* fc2_w;
  const float* const* fc2_b;
  const float *enc_ln_g, *enc_ln_b;
  const float *probe, *map_q_w, *map_q_b, *map_kv_w, *map_kv_b, *map_out_w, *map_out_b;
  const float *map_ln_g, *map_ln_b, *map_fc1_w, *map_fc1_b, *map_fc2_w, *map_fc2_b;
} oracle_model;

int oracle_threads(void) { return threads(); }
void oracle_set_threads(int n) { g_threads = n; }

float oracle_e4m3(float x) { return e4m3_value(x); }

void oracle_gelu(const float* x, float* y, long n) {
  for (long i = 0; i < n; ++i) y[i] = static_cast<float>(gelu_tanh(x[i]));
}

void oracle_softmax_rows(const float* x, float* y, long rows, long cols) {
  for (long r = 0; r < rows; ++r) {
    double m = -INFINITY, l = 0.0;
    for (long j = 0; j < cols; ++j) m = std::max(m, double(x[r * cols + j]));
    for (long j = 0; j < cols; ++j) l += std::exp(double(x[r * cols + j]) - m);
    for (long j = 0; j < cols; ++j) y[r * cols + j] = static_cast<float>(std::exp(double(x[r * cols + j]) - m) / l);
  }
}

// C = act(A W + bias) + residual; act 0 = none, 1 = GELU (tanh form). W is [K][N].
void oracle_linear(const float* A, const float* W, const float* bias, const float* residual, float* C, long M,
                   long N, long K, int act, int fp8) {
  linear(A, K, W, bias, C, M, N, K, fp8 != 0);
  if (act == 1)
    parallel(M, [&](long i) {
      for (long n = 0; n < N; ++n) C[i * N + n] = static_cast<float>(gelu_tanh(C[i * N + n]));
    });
  if (residual)
    for (long i = 0; i < M * N; ++i) C[i] += residual[i];
}

void oracle_layernorm(const float* x, const float* g, const float* b, float* y, long rows, long width, float eps) {
  layernorm(x, g, b, y, rows, width, eps);
}

// q, k, v, o: [B][T][H*dh] token-major (channel c = h*dh + d).
void oracle_attention(const float* q, const float* k, const float* v, float* o, long B, long H, long T, long dh,
                      float scale) {
  const long ld = H * dh;
  parallel(B * H, [&](long bh) {
    const long b = bh / H, h = bh % H;
    const long off = b * T * ld;
    attention_one(q + off, ld, k + off, ld, v + off, ld, o + off, ld, T, T, h, dh, scale);
  });
}

// Attention with FP8 score products ("FP8 attention and resident image/embedding
// transfers": the QK product on E4M3 operands at scale 2^-4, written quantised by their
// producer): Q and K are rounded to E4M3 values (q_hat = E4M3(16 q) / 16) before the
// scores; softmax and the P V product are as in oracle_attention.
void oracle_attention_qk8(const float* q, const float* k, const float* v, float* o, long B, long H, long T, long dh,
                          float scale) {
  const size_t n = size_t(B) * size_t(T) * size_t(H * dh);
  std::vector<float> q8(n), k8(n);
  for (size_t i = 0; i < n; ++i) {
    q8[i] = e4m3_value(16.0f * q[i]) / 16.0f;
    k8[i] = e4m3_value(16.0f * k[i]) / 16.0f;
  }
  oracle_attention(q8.data(), k8.data(), v, o, B, H, T, dh, scale);
}

// Host packing of whole images into patch rows ("SigLIP ViT benchmark", image-binding
// paragraph: the image is viewed as [batch, patch_y, patch_x, y, x, channel] and
// flattened to [batch, patches, patch_dim]): token t = py * G + px with G = side / p,
// element k = (y * p + x) * C + c of that token is pixel (py * p + y, px * p + x,
// channel c) of the side x side x C image (channel fastest, row-major).
void oracle_pack_patches(const float* img, float* pix, long B, long side, long C, long p) {
  const long G = side / p, T = G * G, P = p * p * C;
  for (long b = 0; b < B; ++b)
    for (long py = 0; py < G; ++py)
      for (long px = 0; px < G; ++px)
        for (long y = 0; y < p; ++y)
          for (long x = 0; x < p; ++x)
            for (long c = 0; c < C; ++c)
              pix[(b * T + py * G + px) * P + (y * p + x) * C + c] =
                  img[((b * side + py * p + y) * side + px * p + x) * C + c];
}

// X[B][T][D] = pix[B][T][P] Wp[P][D] + bp + pos[T][D]
void oracle_patch_embed(const float* pix, const float* Wp, const float* bp, const float* pos, float* X, long B,
                        long T, long P, long D, int fp8) {
  linear(pix, P, Wp, bp, X, B * T, D, P, fp8 != 0);
  for (long b = 0; b < B; ++b)
    for (long t = 0; t < T; ++t)
      for (long n = 0; n < D; ++n) X[(b * T + t) * D + n] += pos[t * D + n];
}

// MAP pooling of the final-LN output xf[B][T][D] -> out[B][D].
void oracle_map_pool(const oracle_model* m, const float* xf, float* out, long B, int fp8) {
  const long T = m->tokens, D = m->width, F = m->mlp, H = m->heads, dh = m->head_dim;
  const bool q8 = fp8 != 0;
  std::vector<float> q(static_cast<size_t>(D)), kv(size_t(T) * 2 * D), a(size_t(B) * D), A(size_t(B) * D),
      y(size_t(B) * D), hdn(size_t(B) * F), mlp(size_t(B) * D);
  linear(m->probe, D, m->map_q_w, m->map_q_b, q.data(), 1, D, D, q8);
  const double scale = 1.0 / std::sqrt(double(dh));
  for (long b = 0; b < B; ++b) {
    linear(xf + b * T * D, D, m->map_kv_w, m->map_kv_b, kv.data(), T, 2 * D, D, q8);
    parallel(H, [&](long h) {
      attention_one(q.data(), D, kv.data(), 2 * D, kv.data() + D, 2 * D, a.data() + b * D, D, 1, T, h, dh, scale);
    });
  }
  linear(a.data(), D, m->map_out_w, m->map_out_b, A.data(), B, D, D, q8);
  layernorm(A.data(), m->map_ln_g, m->map_ln_b, y.data(), B, D, 1e-6f);
  linear(y.data(), D, m->map_fc1_w, m->map_fc1_b, hdn.data(), B, F, D, q8);
  for (auto& e : hdn) e = static_cast<float>(gelu_tanh(e));
  linear(hdn.data(), F, m->map_fc2_w, m->map_fc2_b, mlp.data(), B, D, F, q8);
  for (long i = 0; i < B * D; ++i) out[i] = A[size_t(i)] + mlp[size_t(i)];
}

// Whole encoder: pix[B][T][P] -> out[B][D] (the [B,1,D] pooled embedding).
// If xf_out is non-null it receives the final-LN output [B][T][D].
// fp8 bit 0: dense-GEMM operands rounded to E4M3 (the FP8 GEMM mode); bit 1: Q and K
// rounded to E4M3 before the attention scores (FP8 attention products).
void oracle_encode(const oracle_model* m, const float* pix, float* out, long B, int layers, int fp8,
                   float* xf_out) {
  const long T = m->tokens, D = m->width, F = m->mlp, H = m->heads, dh = m->head_dim, M = B * T;
  const bool q8 = (fp8 & 1) != 0, qk8 = (fp8 & 2) != 0;
  fp8 &= 1;
  std::vector<float> X(size_t(M) * D), Y(size_t(M) * D), QKV(size_t(M) * 3 * D), O(size_t(M) * D),
      tmp(size_t(M) * D), Hd(size_t(M) * F);
  oracle_patch_embed(pix, m->patch_w, m->patch_b, m->pos, X.data(), B, T, m->patch_dim, D, fp8);
  const double scale = 1.0 / std::sqrt(double(dh));
  for (int l = 0; l < layers; ++l) {
    layernorm(X.data(), m->ln1_g[l], m->ln1_b[l], Y.data(), M, D, 1e-6f);
    linear(Y.data(), D, m->qkv_w[l], m->qkv_b[l], QKV.data(), M, 3 * D, D, q8);
    if (qk8)  // Q and K columns of every row to E4M3 values
      parallel(M, [&](long i) {
        for (long c = 0; c < 2 * D; ++c) {
          float& x = QKV[size_t(i * 3 * D + c)];
          x = e4m3_value(16.0f * x) / 16.0f;
        }
      });
    parallel(B * H, [&](long bh) {
      const long b = bh / H, h = bh % H;
      const float* base = QKV.data() + b * T * 3 * D;
      attention_one(base, 3 * D, base + D, 3 * D, base + 2 * D, 3 * D, O.data() + b * T * D, D, T, T, h, dh, scale);
    });
    linear(O.data(), D, m->out_w[l], m->out_b[l], tmp.data(), M, D, D, q8);
    for (long i = 0; i < M * D; ++i) X[size_t(i)] += tmp[size_t(i)];
    layernorm(X.data(), m->ln2_g[l], m->ln2_b[l], Y.data(), M, D, 1e-6f);
    linear(Y.data(), D, m->fc1_w[l], m->fc1_b[l], Hd.data(), M, F, D, q8);
    parallel(M, [&](long i) {
      for (long n = 0; n < F; ++n) Hd[size_t(i * F + n)] = static_cast<float>(gelu_tanh(Hd[size_t(i * F + n)]));
    });
    linear(Hd.data(), F, m->fc2_w[l], m->fc2_b[l], tmp.data(), M, D, F, q8);
    for (long i = 0; i < M * D; ++i) X[size_t(i)] += tmp[size_t(i)];
  }
  layernorm(X.data(), m->enc_ln_g, m->enc_ln_b, Y.data(), M, D, 1e-6f);
  if (xf_out) std::memcpy(xf_out, Y.data(), sizeof(float) * size_t(M) * D);
  oracle_map_pool(m, Y.data(), out, B, fp8);
}

}  // extern "C"
