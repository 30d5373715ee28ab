// C ABI of the library (include/sv.h): resident weights, cached workspaces,
// the forward-pass orchestration and the per-op entry points. Host code only;
// every step of the forward pass runs in this library's kernels.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <tuple>
#include <memory>
#include <string>
#include <utility>
#include <vector>

#include "../../synth/synth.h"
#include "sv_internal.h"

namespace sv {
namespace {

thread_local std::string g_err;

struct Runtime {
  bool ready = false;
  int device = -1;
  int sms = 0;
  int* dev_err = nullptr;
};
Runtime g_rt;
long long g_launches = 0;

// ------------------------------------------------------------ profiling
struct ProfRec {
  int kind;
  double flops, bytes;
  cudaEvent_t e0, e1;
};
bool g_prof_on = false;
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_ev_pool;

cudaEvent_t get_event() {
  if (!g_ev_pool.empty()) {
    cudaEvent_t e = g_ev_pool.back();
    g_ev_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

using Launch = LaunchScope;

// ------------------------------------------------------------ model state
struct Dims {
  int T = 0, P = 0, D = 0, H = 0, F = 0, L = 0, Kp = 0;
};

struct LayerW {
  __half *ln1_g, *ln1_b, *qkv_w, *qkv_b, *out_w, *out_b, *ln2_g, *ln2_b, *fc1_w, *fc1_b, *fc2_w, *fc2_b;
  uint8_t *qkv_w8, *out_w8, *fc1_w8, *fc2_w8;
  // LayerNorms folded into the F16 QKV and MLP-up GEMMs: qkv_w / fc1_w hold W * gamma
  // (the E4M3 copies keep W); the GEMMs' extra K block rows [N, 16] and combined biases
  __half *qkv_aug, *qkv_bf, *fc1_aug, *fc1_bf;
};

// One parameter tensor as drawn (synth order): its resident F16 copy ([N, kpad]
// K-major for a dense weight, else row-major) and its E4M3 copy, if any.
struct TensorRec {
  int rows = 0, cols = 0;  // logical [rows, cols] (a dense weight: [K, N])
  bool matrix = false;
  int kpad = 0;
  const __half* p16 = nullptr;
  const uint8_t* p8 = nullptr;
};

struct Weights {
  bool ready = false;
  Dims d;
  std::vector<TensorRec> tensors;
  void* arena = nullptr;
  void* fold = nullptr;  // extra K block rows and combined biases of the folded LayerNorms
  __half *patch_w = nullptr, *patch_b = nullptr, *pos = nullptr;
  uint8_t* patch_w8 = nullptr;
  std::vector<LayerW> layers;
  __half *enc_ln_g = nullptr, *enc_ln_b = nullptr, *probe = nullptr, *mq_w = nullptr, *mq_b = nullptr,
         *mkv_w = nullptr, *mkv_b = nullptr, *mo_w = nullptr, *mo_b = nullptr, *mln_g = nullptr, *mln_b = nullptr,
         *mfc1_w = nullptr, *mfc1_b = nullptr, *mfc2_w = nullptr, *mfc2_b = nullptr;
  uint8_t *probe8 = nullptr, *mq_w8 = nullptr, *mkv_w8 = nullptr, *mo_w8 = nullptr, *mfc1_w8 = nullptr,
          *mfc2_w8 = nullptr;
};
Weights g_w;

// One GEMM of the path: operand and epilogue tensor maps, epilogue, logical K.
struct GemmCall {
  GemmOperands g;
  GemmEpi e;
  int k = 0;
};

// Buffers and operand maps of the MAP head for one batch size and dtype.
struct MapPlan {
  GemmCall q, kv, out, fc1, fc2;
  __half* qv = nullptr;  // [D] projected probe
  __half* KV = nullptr;  // [B*T, 2D]
  void* a = nullptr;     // [B, D] pooled attention (f16 / e4m3)
  __half* A = nullptr;   // [B, D]
  void* Ya = nullptr;    // [B, D] LN(A)
  void* Ha = nullptr;    // [B, F]
};

// Workspace and operand maps of the whole forward pass for one batch size and dtype.
struct Plan {
  int B = 0, fp8 = 0;
  int qkv_calls = 1;     // GEMMs per layer for Q, K, V: 1 fused, or 3 (SV_ENCODE_UNFUSED_QKV)
  int qk8 = 0;           // scores on E4M3 Q and K (SV_ENCODE_FP8_ATTENTION)
  bool fold_ln = false;  // LN1 / LN2 folded into the QKV / MLP-up GEMMs (F16 operands)
  void* mem = nullptr;
  size_t bytes = 0;
  void* A0 = nullptr;     // [M, Kp] staged pixels
  __half* X = nullptr;    // [M, D] residual stream
  void* Y = nullptr;       // [M, D] LayerNorm output (GEMM operand)
  float* ln_r = nullptr;    // [M] 1/std of each row (F16 path: LayerNorm folded into the GEMMs)
  __half* ln_aug = nullptr;  // [M, 16] the folded GEMMs' extra K block (-mean)
  float2* ln_part = nullptr;  // [M, kMaxLnTiles] per-tile row statistics from the GEMMs that write X
  __half* QKV = nullptr;  // head-blocked Q/K/V for attention; the MAP KV projection reuses it row-major
  void* O = nullptr;      // [M, D] attention output (GEMM operand)
  void* Hh = nullptr;     // [M, F] GELU output (GEMM operand)
  float* ws = nullptr;    // partial sums of the GEMMs that split K (small batches)
  size_t ws_bytes = 0;
  GemmCall patch;
  std::vector<GemmCall> qkv, out, fc1, fc2;
  MapPlan map;
};
std::map<std::tuple<int, int, int>, std::unique_ptr<Plan>> g_plans;  // sv_encode: (batch, dtype, flags)
std::map<std::pair<int, int>, std::unique_ptr<Plan>> g_map_plans;  // sv_map_pool
void* g_attn_scratch = nullptr;  // head-blocked copy of sv_attention's input
size_t g_attn_scratch_bytes = 0;
void* g_lng_scratch = nullptr;  // sv_ln_gemm: scaled weights, column sums, biases, row statistics
size_t g_lng_scratch_bytes = 0;
void* g_gemm_ws = nullptr;  // sv_gemm_bias_act: partial sums of a GEMM that splits K
size_t g_gemm_ws_bytes = 0;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
// Step graphs of sv_encode: one per (pixels, out, batch, layers, dtype, flags) seen at
// least twice (captured on the second call, replayed from the third on).
struct StepGraph {
  const void* pixels = nullptr;
  const void* out = nullptr;
  int B = 0, layers = 0, fp8 = 0, flags = 0;
  int calls = 0;                    // calls so far with this key
  bool eager_only = false;          // the capture was refused
  cudaGraphExec_t exec = nullptr;   // the captured launch sequence
  long long launches = 0;           // kernels in it
  unsigned long long last_use = 0;  // for eviction
};
constexpr size_t kMaxStepGraphs = 8;
std::vector<StepGraph> g_graphs;
unsigned long long g_graph_clock = 0;
cudaStream_t g_capture_stream = nullptr;

void free_graphs() {
  for (StepGraph& g : g_graphs)
    if (g.exec) cudaGraphExecDestroy(g.exec);
  g_graphs.clear();
}


void free_plans() {
  free_graphs();  // they launch into the plans' workspaces
  for (auto& kv : g_plans) cudaFree(kv.second->mem);
  for (auto& kv : g_map_plans) cudaFree(kv.second->mem);
  g_plans.clear();
  g_map_plans.clear();
  if (g_attn_scratch) cudaFree(g_attn_scratch);
  g_attn_scratch = nullptr;
  g_attn_scratch_bytes = 0;
  if (g_lng_scratch) cudaFree(g_lng_scratch);
  g_lng_scratch = nullptr;
  g_lng_scratch_bytes = 0;
  if (g_gemm_ws) cudaFree(g_gemm_ws);
  g_gemm_ws = nullptr;
  g_gemm_ws_bytes = 0;
}

void free_weights() {
  free_plans();
  if (g_w.arena) cudaFree(g_w.arena);
  if (g_w.fold) cudaFree(g_w.fold);
  g_w = Weights();
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

#define SV_CHECK_CUDA(call, what)                      \
  do {                                                 \
    cudaError_t e_ = (call);                           \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

#define SV_TRY(call)            \
  do {                          \
    sv_status s_ = (call);      \
    if (s_ != SV_OK) return s_; \
  } while (0)

// ------------------------------------------------------------ weights upload
sv_status init_weights(uint64_t seed, const Dims& d) {
  free_weights();
  SV_TRY(ensure_runtime());
  synth_dims sd;
  sd.tokens = d.T;
  sd.patch_dim = d.P;
  sd.width = d.D;
  sd.heads = d.H;
  sd.mlp = d.F;
  sd.layers = d.L;
  const int n = synth_tensor_count(&sd);

  // Every dense weight is stored [N, Kpad] K-major in F16, plus an E4M3 copy.
  struct Slot {
    synth_tensor info;
    bool matrix;
    int kpad;
    size_t off16, off8;
  };
  std::vector<Slot> slots(static_cast<size_t>(n));
  size_t total = 0, max_elems = 0;
  for (int id = 0; id < n; ++id) {
    Slot& s = slots[size_t(id)];
    synth_tensor_info(&sd, id, &s.info);
    const std::string name = s.info.name;
    s.matrix = name.size() > 2 && name.compare(name.size() - 2, 2, "_w") == 0;
    s.kpad = s.matrix ? (name == "patch_w" ? d.Kp : s.info.rows) : s.info.rows;
    const size_t elems = size_t(s.info.cols) * size_t(s.kpad);
    max_elems = elems > max_elems ? elems : max_elems;
    s.off16 = total;
    total = align_up(total + 2 * elems, 256);
    s.off8 = 0;
    if (s.matrix || name == "probe") {
      s.off8 = total;
      total = align_up(total + elems, 256);
    }
  }
  void* arena = nullptr;
  cudaError_t e = cudaMalloc(&arena, total);
  if (e != cudaSuccess) {
    cudaGetLastError();
    set_error("cudaMalloc of %zu bytes for weights failed: %s", total, cudaGetErrorString(e));
    return SV_ERR_OOM;
  }
  g_w.arena = arena;
  g_w.d = d;
  g_w.layers.assign(size_t(d.L), LayerW{});
  std::vector<uint16_t> host(max_elems);
  char* base = static_cast<char*>(arena);
  for (int id = 0; id < n; ++id) {
    Slot& s = slots[size_t(id)];
    const std::string name = s.info.name;
    const size_t elems = size_t(s.info.cols) * size_t(s.kpad);
    const int rc = s.matrix ? synth_fill_tensor_f16_t(seed, &sd, id, host.data(), s.kpad)
                            : synth_fill_tensor_f16(seed, &sd, id, host.data());
    if (rc != 0) {
      set_error("synthetic generator failed for tensor %s", name.c_str());
      return SV_ERR_INVALID_ARG;
    }
    __half* p16 = reinterpret_cast<__half*>(base + s.off16);
    SV_CHECK_CUDA(cudaMemcpy(p16, host.data(), 2 * elems, cudaMemcpyHostToDevice), "weight upload");
    uint8_t* p8 = s.off8 ? reinterpret_cast<uint8_t*>(base + s.off8) : nullptr;
    if (p8) SV_TRY(quantize_launch(p16, p8, elems, nullptr));
    TensorRec rec;
    rec.rows = s.info.rows;
    rec.cols = s.info.cols;
    rec.matrix = s.matrix;
    rec.kpad = s.kpad;
    rec.p16 = p16;
    rec.p8 = p8;
    g_w.tensors.push_back(rec);
    const int l = s.info.layer;
    if (l >= 0) {
      LayerW& w = g_w.layers[size_t(l)];
      if (name == "ln1_g") w.ln1_g = p16;
      else if (name == "ln1_b") w.ln1_b = p16;
      else if (name == "qkv_w") w.qkv_w = p16, w.qkv_w8 = p8;
      else if (name == "qkv_b") w.qkv_b = p16;
      else if (name == "out_w") w.out_w = p16, w.out_w8 = p8;
      else if (name == "out_b") w.out_b = p16;
      else if (name == "ln2_g") w.ln2_g = p16;
      else if (name == "ln2_b") w.ln2_b = p16;
      else if (name == "fc1_w") w.fc1_w = p16, w.fc1_w8 = p8;
      else if (name == "fc1_b") w.fc1_b = p16;
      else if (name == "fc2_w") w.fc2_w = p16, w.fc2_w8 = p8;
      else if (name == "fc2_b") w.fc2_b = p16;
    } else {
      if (name == "patch_w") g_w.patch_w = p16, g_w.patch_w8 = p8;
      else if (name == "patch_b") g_w.patch_b = p16;
      else if (name == "pos") g_w.pos = p16;
      else if (name == "enc_ln_g") g_w.enc_ln_g = p16;
      else if (name == "enc_ln_b") g_w.enc_ln_b = p16;
      else if (name == "probe") g_w.probe = p16, g_w.probe8 = p8;
      else if (name == "map_q_w") g_w.mq_w = p16, g_w.mq_w8 = p8;
      else if (name == "map_q_b") g_w.mq_b = p16;
      else if (name == "map_kv_w") g_w.mkv_w = p16, g_w.mkv_w8 = p8;
      else if (name == "map_kv_b") g_w.mkv_b = p16;
      else if (name == "map_out_w") g_w.mo_w = p16, g_w.mo_w8 = p8;
      else if (name == "map_out_b") g_w.mo_b = p16;
      else if (name == "map_ln_g") g_w.mln_g = p16;
      else if (name == "map_ln_b") g_w.mln_b = p16;
      else if (name == "map_fc1_w") g_w.mfc1_w = p16, g_w.mfc1_w8 = p8;
      else if (name == "map_fc1_b") g_w.mfc1_b = p16;
      else if (name == "map_fc2_w") g_w.mfc2_w = p16, g_w.mfc2_w8 = p8;
      else if (name == "map_fc2_b") g_w.mfc2_b = p16;
    }
  }
  // Fold LN1 into the QKV weights and LN2 into the MLP-up weights (F16 path); the
  // E4M3 copies were quantised from the unscaled weights above.
  {
    const size_t per_layer = size_t(3 * d.D + d.F) * 17;  // halves: [N, 16] rows + [N] biases
    void* fold = nullptr;
    e = cudaMalloc(&fold, per_layer * size_t(d.L) * sizeof(__half));
    if (e != cudaSuccess) {
      cudaGetLastError();
      set_error("cudaMalloc for the folded LayerNorm constants failed: %s", cudaGetErrorString(e));
      return SV_ERR_OOM;
    }
    g_w.fold = fold;
    __half* f = static_cast<__half*>(fold);
    for (int l = 0; l < d.L; ++l) {
      LayerW& w = g_w.layers[size_t(l)];
      w.qkv_aug = f;
      w.fc1_aug = f + size_t(3 * d.D) * 16;
      w.qkv_bf = f + size_t(3 * d.D + d.F) * 16;
      w.fc1_bf = w.qkv_bf + 3 * d.D;
      f += per_layer;
      SV_TRY(fold_ln_launch(w.qkv_w, w.ln1_g, w.ln1_b, w.qkv_b, w.qkv_aug, w.qkv_bf, 3 * d.D, d.D, nullptr));
      SV_TRY(fold_ln_launch(w.fc1_w, w.ln2_g, w.ln2_b, w.fc1_b, w.fc1_aug, w.fc1_bf, d.F, d.D, nullptr));
    }
  }
  SV_CHECK_CUDA(cudaDeviceSynchronize(), "weight initialisation");
  g_w.ready = true;
  return SV_OK;
}

// ------------------------------------------------------------ plans
// Two passes over the same sequence of take() calls: the first (base null)
// sizes the workspace, the second hands out pointers into it.
struct Carver {
  char* base;
  size_t off = 0;
  void* take(size_t bytes) {
    void* p = base ? base + off : nullptr;
    off = align_up(off + bytes, 256);
    return p;
  }
};

// K ranges a small-M, long-K GEMM may be split into (given a partial-sum workspace).
constexpr int kMaxSplits = 8;

// A GEMM call; with a workspace `ws` of `ws_bytes` that holds its partial sums, the GEMM
// may split K.
sv_status make_call(GemmCall* c, const void* A, const void* W, int M, int N, int K, int fp8, const GemmEpi& e,
                    int k_logical, float* ws = nullptr, size_t ws_bytes = 0) {
  c->e = e;
  c->k = k_logical;
  const int splits = (ws && gemm_splitk_ws_bytes_for(M, N, K, fp8, kMaxSplits) <= ws_bytes) ? kMaxSplits : 1;
  SV_TRY(gemm_prepare(&c->g, A, W, M, N, K, fp8, true, splits));
  if (c->g.k_splits > 1) c->e.ws = ws;
  return gemm_bind_epilogue(&c->g, c->e);
}

// Largest split-K workspace over the MAP head's GEMMs for B images.
size_t map_ws_bytes(int B, int fp8) {
  const Dims& d = g_w.d;
  const size_t a = gemm_splitk_ws_bytes_for(1, d.D, d.D, fp8, kMaxSplits);
  const size_t b = gemm_splitk_ws_bytes_for(B * d.T, 2 * d.D, d.D, fp8, kMaxSplits);
  const size_t c = gemm_splitk_ws_bytes_for(B, d.D, d.D, fp8, kMaxSplits);
  const size_t e = gemm_splitk_ws_bytes_for(B, d.F, d.D, fp8, kMaxSplits);
  const size_t f = gemm_splitk_ws_bytes_for(B, d.D, d.F, fp8, kMaxSplits);
  return std::max(std::max(std::max(a, b), std::max(c, e)), f);
}

GemmEpi epi(const __half* bias, void* out, float scale, int act = SV_ACT_NONE, int out_e4m3 = 0,
            const __half* residual = nullptr) {
  GemmEpi e;
  e.bias = bias;
  e.out = out;
  e.scale = scale;
  e.act = act;
  e.out_e4m3 = out_e4m3;
  e.residual = residual;
  return e;
}

// Buffers of the MAP head (carved from `c`); xf is the encoder-output operand.
// The final projection's output is the caller's buffer: it is bound per call.
sv_status build_map(MapPlan& m, Carver& c, const void* xf, int B, int fp8, bool carve_kv, __half* kv_alias,
                    float* ws, size_t ws_bytes) {
  const Dims& d = g_w.d;
  const size_t eb = fp8 ? 1 : 2;
  m.qv = static_cast<__half*>(c.take(size_t(d.D) * 2));
  m.KV = carve_kv ? static_cast<__half*>(c.take(size_t(B) * d.T * 2 * d.D * 2)) : kv_alias;
  m.a = c.take(size_t(B) * d.D * eb);
  m.A = static_cast<__half*>(c.take(size_t(B) * d.D * 2));
  m.Ya = c.take(size_t(B) * d.D * eb);
  m.Ha = c.take(size_t(B) * d.F * eb);
  if (!c.base) return SV_OK;
  const float sc = fp8 ? 1.0f / 256.0f : 1.0f;
  const int D = d.D, F = d.F;
  SV_TRY(make_call(&m.q, fp8 ? (const void*)g_w.probe8 : g_w.probe, fp8 ? (const void*)g_w.mq_w8 : g_w.mq_w, 1, D, D,
                   fp8, epi(g_w.mq_b, m.qv, sc), D, ws, ws_bytes));
  SV_TRY(make_call(&m.kv, xf, fp8 ? (const void*)g_w.mkv_w8 : g_w.mkv_w, B * d.T, 2 * D, D, fp8,
                   epi(g_w.mkv_b, m.KV, sc), D, ws, ws_bytes));
  SV_TRY(make_call(&m.out, m.a, fp8 ? (const void*)g_w.mo_w8 : g_w.mo_w, B, D, D, fp8, epi(g_w.mo_b, m.A, sc), D, ws,
                   ws_bytes));
  SV_TRY(make_call(&m.fc1, m.Ya, fp8 ? (const void*)g_w.mfc1_w8 : g_w.mfc1_w, B, F, D, fp8,
                   epi(g_w.mfc1_b, m.Ha, sc, SV_ACT_GELU_TANH, fp8), D, ws, ws_bytes));
  // the final projection's output is bound per call (run_map)
  m.fc2.e = epi(g_w.mfc2_b, nullptr, sc, SV_ACT_NONE, 0, m.A);
  m.fc2.k = F;
  const int splits = (ws && gemm_splitk_ws_bytes_for(B, D, F, fp8, kMaxSplits) <= ws_bytes) ? kMaxSplits : 1;
  SV_TRY(gemm_prepare(&m.fc2.g, m.Ha, fp8 ? (const void*)g_w.mfc2_w8 : g_w.mfc2_w, B, D, F, fp8, true, splits));
  if (m.fc2.g.k_splits > 1) m.fc2.e.ws = ws;
  return SV_OK;
}

sv_status alloc_carved(Carver& c, void** mem, size_t* bytes) {
  cudaError_t e = cudaMalloc(mem, c.off);
  if (e != cudaSuccess) {
    cudaGetLastError();
    set_error("cudaMalloc of %zu bytes for the workspace failed: %s", c.off, cudaGetErrorString(e));
    return SV_ERR_OOM;
  }
  // Defined contents for every buffer (pads and unused tails read as zero).
  SV_CHECK_CUDA(cudaMemset(*mem, 0, c.off), "workspace clear");
  *bytes = c.off;
  c.base = static_cast<char*>(*mem);
  c.off = 0;
  return SV_OK;
}

sv_status get_plan(int B, int fp8, int flags, Plan** out) {
  const auto key = std::make_tuple(B, fp8, flags);
  auto it = g_plans.find(key);
  if (it != g_plans.end()) {
    *out = it->second.get();
    return SV_OK;
  }
  const Dims& d = g_w.d;
  const size_t M = size_t(B) * d.T, eb = fp8 ? 1 : 2;
  std::unique_ptr<Plan> p(new Plan());
  p->B = B;
  p->fp8 = fp8;
  p->qkv_calls = (flags & SV_ENCODE_UNFUSED_QKV) ? 3 : 1;
  p->qk8 = (flags & SV_ENCODE_FP8_ATTENTION) ? 1 : 0;
  p->fold_ln = !fp8;
  // split-K partial sums: the largest need over the plan's GEMMs (0 at large batches)
  {
    const int Mi = int(M), wq = 3 * d.D / p->qkv_calls;
    size_t need = map_ws_bytes(B, fp8);
    const int shapes[5][3] = {{Mi, d.D, d.Kp}, {Mi, wq, d.D}, {Mi, d.D, d.D}, {Mi, d.F, d.D}, {Mi, d.D, d.F}};
    for (const auto& sh : shapes) need = std::max(need, gemm_splitk_ws_bytes_for(sh[0], sh[1], sh[2], fp8, kMaxSplits));
    p->ws_bytes = need;
  }
  Carver c{nullptr};
  for (int pass = 0; pass < 2; ++pass) {
    p->ws = p->ws_bytes ? static_cast<float*>(c.take(p->ws_bytes)) : nullptr;
    p->A0 = c.take(M * d.Kp * eb);
    p->X = static_cast<__half*>(c.take(M * d.D * 2));
    p->Y = c.take(M * d.D * eb);
    p->ln_r = static_cast<float*>(c.take(M * sizeof(float)));
    p->ln_aug = static_cast<__half*>(c.take(M * 16 * sizeof(__half)));
    p->ln_part = static_cast<float2*>(c.take(M * kMaxLnTiles * sizeof(float2)));
    const size_t qkv_bytes = attention_blocked_bytes(B, d.T, d.H);
    p->QKV = static_cast<__half*>(c.take(qkv_bytes > M * 3 * d.D * 2 ? qkv_bytes : M * 3 * d.D * 2));
    p->O = c.take(M * d.D * eb);
    p->Hh = c.take(M * d.F * eb);
    SV_TRY(build_map(p->map, c, p->Y, B, fp8, false, p->QKV, p->ws, p->ws_bytes));
    if (pass == 0) {
      sv_status st = alloc_carved(c, &p->mem, &p->bytes);
      if (st != SV_OK) return st;
    }
  }
  const int Mi = int(M);
  const float sc = fp8 ? 1.0f / 256.0f : 1.0f;
  sv_status st = SV_OK;
  auto fail = [&](sv_status s) {
    cudaFree(p->mem);
    return s;
  };
  GemmEpi pe = epi(g_w.patch_b, p->X, sc);
  pe.pos = g_w.pos;
  pe.pos_rows = d.T;
  // F16: the GEMMs that write X also write its row statistics for the next LayerNorm
  if (p->fold_ln) pe.ln_part = p->ln_part;
  if ((st = make_call(&p->patch, p->A0, fp8 ? (const void*)g_w.patch_w8 : g_w.patch_w, Mi, d.D, d.Kp, fp8, pe, d.P,
                      p->ws, p->ws_bytes)))
    return fail(st);
  p->qkv.resize(size_t(d.L) * size_t(p->qkv_calls));
  p->out.resize(size_t(d.L));
  p->fc1.resize(size_t(d.L));
  p->fc2.resize(size_t(d.L));
  for (int l = 0; l < d.L; ++l) {
    const LayerW& w = g_w.layers[size_t(l)];
    const size_t i = size_t(l);
    // F16: LN1 / LN2 folded into the QKV / MLP-up GEMMs, which read X itself; E4M3:
    // the LayerNorm kernels write the quantised operand Y
    GemmEpi fe = epi(p->fold_ln ? w.fc1_bf : w.fc1_b, p->Hh, sc, SV_ACT_GELU_TANH, fp8);
    if (p->fold_ln) {
      fe.ln_r = p->ln_r;
      fe.ln_aug_a = p->ln_aug;
      fe.ln_aug_w = w.fc1_aug;
    }
    const void* ln_in = p->fold_ln ? static_cast<const void*>(p->X) : p->Y;
    // Q, K, V: one fused GEMM over the [3D, D] weight, or (SV_ENCODE_UNFUSED_QKV) three
    // over its row slices, each writing its third of the head-blocked layout
    const int nq = p->qkv_calls, wq = 3 * d.D / nq;
    for (int j = 0; j < nq && st == SV_OK; ++j) {
      const size_t r0 = size_t(j) * wq;  // first weight row (output column) of this GEMM
      GemmEpi qe = epi((p->fold_ln ? w.qkv_bf : w.qkv_b) + r0, p->QKV, sc);
      if (p->fold_ln) {
        qe.ln_r = p->ln_r;
        qe.ln_aug_a = p->ln_aug;
        qe.ln_aug_w = w.qkv_aug + r0 * 16;
      }
      qe.blk_out = p->QKV;
      qe.blk_T = d.T;
      qe.blk_H = d.H;
      qe.blk_B = B;
      qe.blk_col0 = int(r0);
      qe.blk_qk8 = p->qk8;
      const void* wptr = fp8 ? static_cast<const void*>(w.qkv_w8 + r0 * d.D) : static_cast<const void*>(w.qkv_w + r0 * d.D);
      st = make_call(&p->qkv[i * size_t(nq) + size_t(j)], ln_in, wptr, Mi, wq, d.D, fp8, qe, d.D, p->ws, p->ws_bytes);
    }
    GemmEpi oe = epi(w.out_b, p->X, sc, SV_ACT_NONE, 0, p->X);
    GemmEpi de = epi(w.fc2_b, p->X, sc, SV_ACT_NONE, 0, p->X);
    if (p->fold_ln) oe.ln_part = de.ln_part = p->ln_part;
    if (st ||
        (st = make_call(&p->out[i], p->O, fp8 ? (const void*)w.out_w8 : w.out_w, Mi, d.D, d.D, fp8, oe, d.D, p->ws,
                        p->ws_bytes)) ||
        (st = make_call(&p->fc1[i], ln_in, fp8 ? (const void*)w.fc1_w8 : w.fc1_w, Mi, d.F, d.D, fp8, fe, d.D, p->ws,
                        p->ws_bytes)) ||
        (st = make_call(&p->fc2[i], p->Hh, fp8 ? (const void*)w.fc2_w8 : w.fc2_w, Mi, d.D, d.F, fp8, de, d.F, p->ws,
                        p->ws_bytes)))
      return fail(st);
    // MLP down with every tile split (small batches): its reduction finishes the next
    // LayerNorm's statistics itself, so the encoder skips that finalize launch
    if (p->fold_ln && p->fc2[i].g.k_splits > 1 && p->fc2[i].g.n_main == 0 && (d.D + 255) / 256 <= 8) {
      p->fc2[i].e.ln_part = nullptr;
      p->fc2[i].e.ln_r_out = p->ln_r;
      p->fc2[i].e.ln_aug_out = p->ln_aug;
    }
  }
  *out = p.get();
  g_plans[key] = std::move(p);
  return SV_OK;
}

// ------------------------------------------------------------ launches with accounting
double gemm_flops(const GemmOperands& g, int k_logical) { return 2.0 * g.M * double(g.N) * double(k_logical); }
double gemm_bytes(const GemmOperands& g, const GemmEpi& e, int k_logical) {
  const double eb = g.fp8 ? 1.0 : 2.0;
  double b = (double(g.M) + double(g.N)) * k_logical * eb + double(g.M) * g.N * (e.out_e4m3 ? 1.0 : 2.0);
  if (e.residual) b += double(g.M) * g.N * 2.0;
  return b;
}

sv_status run_gemm(const GemmCall& c, cudaStream_t s) {
  if (c.g.k_splits > 1) {  // two launches: the K ranges' partial sums, then their reduction and the epilogue
    const double ws = double(gemm_splitk_ws_bytes(c.g));
    const double eb = c.g.fp8 ? 1.0 : 2.0;
    {
      Launch L(kKindGemm, gemm_flops(c.g, c.k), (double(c.g.M) + double(c.g.N)) * c.k * eb + ws, s);
      SV_TRY(gemm_launch(c.g, c.e, s, 0));
    }
    Launch L(kKindGemm, 0.0, ws + gemm_bytes(c.g, c.e, 0), s);
    return gemm_launch(c.g, c.e, s, 1);
  }
  Launch L(kKindGemm, gemm_flops(c.g, c.k), gemm_bytes(c.g, c.e, c.k), s);
  return gemm_launch(c.g, c.e, s);
}

// LayerNorm statistics of X from the row statistics its producing GEMM wrote.
sv_status run_ln_finalize(const Plan& p, const GemmCall& producer, int rows, cudaStream_t s) {
  const int D = g_w.d.D, tiles = (D + producer.g.bn - 1) / producer.g.bn;
  Launch L(kKindLN, 8.0 * rows * tiles, double(rows) * (tiles * 8.0 + 36.0), s);
  return ln_finalize_launch(p.ln_part, tiles, producer.g.bn, p.ln_r, p.ln_aug, rows, D, 1e-6f, s);
}

sv_status run_ln(const __half* x, const __half* gm, const __half* bt, void* y, int rows, int out_e4m3,
                 cudaStream_t s) {
  const int D = g_w.d.D;
  Launch L(kKindLN, 8.0 * rows * D, double(rows) * D * (2.0 + (out_e4m3 ? 1.0 : 2.0)), s);
  return layernorm_launch(x, gm, bt, y, rows, D, 1e-6f, out_e4m3, s);
}

sv_status run_map(MapPlan& m, int B, int fp8, __half* out, cudaStream_t s) {
  const Dims& d = g_w.d;
  SV_TRY(run_gemm(m.q, s));
  SV_TRY(run_gemm(m.kv, s));
  {
    Launch L(kKindMapAttn, 4.0 * B * d.T * double(d.D), double(B) * d.T * 2 * d.D * 2.0, s);
    SV_TRY(map_attn_launch(m.qv, m.KV, m.a, B, d.T, d.H, 1.0f / std::sqrt(72.0f), fp8, s));
  }
  SV_TRY(run_gemm(m.out, s));
  {
    Launch L(kKindLN, 8.0 * B * d.D, double(B) * d.D * 3.0, s);
    SV_TRY(layernorm_launch(m.A, g_w.mln_g, g_w.mln_b, m.Ya, B, d.D, 1e-6f, fp8, s));
  }
  SV_TRY(run_gemm(m.fc1, s));
  if (m.fc2.e.out != out) {  // the caller's output buffer: rebind the final projection's output map
    m.fc2.e.out = out;
    SV_TRY(gemm_bind_epilogue(&m.fc2.g, m.fc2.e));
  }
  return run_gemm(m.fc2, s);
}

// The forward pass. stop >= 0 (a test hook, see sv_debug_encode_stage) returns after
// that sv_stage of the last layer instead of running to the end.
sv_status encode(Plan& p, const __half* pixels, __half* out, int layers, cudaStream_t s, int stop = -1) {
  const Dims& d = g_w.d;
  const int B = p.B, fp8 = p.fp8;
  const int M = B * d.T;
  {
    Launch L(kKindOther, 0.0, double(M) * (d.P * 2.0 + d.Kp * (fp8 ? 1.0 : 2.0)), s);
    SV_TRY(pad_pixels_launch(pixels, p.A0, M, d.P, d.Kp, fp8, s));
  }
  SV_TRY(run_gemm(p.patch, s));
  if (stop == SV_STAGE_PATCH) return SV_OK;
  for (int l = 0; l < layers; ++l) {
    const LayerW& w = g_w.layers[size_t(l)];
    const size_t i = size_t(l);
    const bool last = l == layers - 1;
    // (after a split MLP-down GEMM whose reduction finished the statistics, nothing to do)
    if (!(p.fold_ln && l > 0 && p.fc2[i - 1].e.ln_r_out))
      SV_TRY(p.fold_ln ? run_ln_finalize(p, l == 0 ? p.patch : p.fc2[i - 1], M, s)
                       : run_ln(p.X, w.ln1_g, w.ln1_b, p.Y, M, fp8, s));
    for (int j = 0; j < p.qkv_calls; ++j) SV_TRY(run_gemm(p.qkv[i * size_t(p.qkv_calls) + size_t(j)], s));
    if (last && stop == SV_STAGE_QKV) return SV_OK;
    {
      Launch L(kKindAttn, 4.0 * B * d.H * double(d.T) * double(d.T) * 72.0,
               double(M) * d.D * (2 * (p.qk8 ? 1.0 : 2.0) + 2.0) + double(M) * d.D * (fp8 ? 1.0 : 2.0), s);
      SV_TRY(attention_launch(p.QKV, p.O, B, d.T, d.H, 1.0f / std::sqrt(72.0f), fp8, p.qk8, s));
    }
    if (last && stop == SV_STAGE_ATTENTION) return SV_OK;
    SV_TRY(run_gemm(p.out[i], s));
    if (last && stop == SV_STAGE_OUT_PROJ) return SV_OK;
    SV_TRY(p.fold_ln ? run_ln_finalize(p, p.out[i], M, s) : run_ln(p.X, w.ln2_g, w.ln2_b, p.Y, M, fp8, s));
    SV_TRY(run_gemm(p.fc1[i], s));
    if (last && stop == SV_STAGE_MLP_UP) return SV_OK;
    SV_TRY(run_gemm(p.fc2[i], s));
    if (last && stop == SV_STAGE_MLP_DOWN) return SV_OK;
  }
  SV_TRY(run_ln(p.X, g_w.enc_ln_g, g_w.enc_ln_b, p.Y, M, fp8, s));
  if (stop == SV_STAGE_FINAL_LN) return SV_OK;
  return run_map(p.map, B, fp8, out, s);
}

// sv_encode's launches: one by one on the first call with a key (which also creates the
// workspace, kernel attributes and tensor maps the capture relies on), and whenever
// profiling or SV_ENCODE_EAGER asks for it; captured into a CUDA graph on an internal
// stream on the second call; that graph launched on the caller's stream from then on.
sv_status encode_step(Plan& p, const __half* pixels, __half* out, int layers, int flags, cudaStream_t s) {
  if (g_prof_on || (flags & SV_ENCODE_EAGER)) return encode(p, pixels, out, layers, s);
  // a caller capturing its own stream records the kernels themselves
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
    cudaGetLastError();
    return encode(p, pixels, out, layers, s);
  }
  StepGraph* g = nullptr;
  for (StepGraph& x : g_graphs)
    if (x.pixels == pixels && x.out == out && x.B == p.B && x.layers == layers && x.fp8 == p.fp8 && x.flags == flags)
      g = &x;
  if (!g) {
    if (g_graphs.size() >= kMaxStepGraphs) {  // drop the least recently used
      auto old = std::min_element(g_graphs.begin(), g_graphs.end(), [](const StepGraph& a, const StepGraph& b) {
        return a.last_use < b.last_use;
      });
      if (old->exec) cudaGraphExecDestroy(old->exec);
      g_graphs.erase(old);
    }
    StepGraph n;
    n.pixels = pixels;
    n.out = out;
    n.B = p.B;
    n.layers = layers;
    n.fp8 = p.fp8;
    n.flags = flags;
    g_graphs.push_back(n);
    g = &g_graphs.back();
  }
  g->last_use = ++g_graph_clock;
  if (++g->calls == 1 || g->eager_only) return encode(p, pixels, out, layers, s);
  if (!g->exec) {
    if (!g_capture_stream)
      SV_CHECK_CUDA(cudaStreamCreateWithFlags(&g_capture_stream, cudaStreamNonBlocking), "cudaStreamCreate(capture)");
    SV_CHECK_CUDA(cudaStreamBeginCapture(g_capture_stream, cudaStreamCaptureModeThreadLocal), "cudaStreamBeginCapture");
    const long long before = g_launches;
    const sv_status st = encode(p, pixels, out, layers, g_capture_stream);
    cudaGraph_t graph = nullptr;
    const cudaError_t ce = cudaStreamEndCapture(g_capture_stream, &graph);
    const long long n = g_launches - before;
    g_launches = before;  // counted when the graph is launched
    cudaGraphExec_t exec = nullptr;
    cudaError_t ie = cudaErrorUnknown;
    if (st == SV_OK && ce == cudaSuccess) ie = cudaGraphInstantiate(&exec, graph, 0);
    if (graph) cudaGraphDestroy(graph);
    if (st != SV_OK) return st;
    if (ie != cudaSuccess) {  // capture or instantiation refused: this key runs one by one
      cudaGetLastError();
      g->eager_only = true;
      return encode(p, pixels, out, layers, s);
    }
    g->exec = exec;
    g->launches = n;
  }
  SV_CHECK_CUDA(cudaGraphLaunch(g->exec, s), "cudaGraphLaunch(encode step)");
  g_launches += g->launches;
  return SV_OK;
}

sv_status check_ready() {
  if (!g_w.ready) {
    set_error("weights are not initialised: call sv_init_weights first");
    return SV_ERR_NOT_INITIALIZED;
  }
  return SV_OK;
}

}  // namespace

// ------------------------------------------------------------ shared helpers
void set_error(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
}

sv_status cuda_fail(cudaError_t e, const char* what) {
  set_error("%s: %s", what, cudaGetErrorString(e));
  return e == cudaErrorMemoryAllocation ? SV_ERR_OOM : SV_ERR_CUDA;
}

sv_status ensure_runtime() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (g_rt.ready && g_rt.device == dev) return SV_OK;
  if (g_rt.ready && g_rt.device != dev) {
    set_error("the library was initialised on device %d; device %d is current", g_rt.device, dev);
    return SV_ERR_INVALID_ARG;
  }
  int sms = 0, major = 0, minor = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) {
    set_error("this library is built for sm_103a; device %d is sm_%d%d", dev, major, minor);
    return SV_ERR_UNSUPPORTED;
  }
  int* err = nullptr;
  e = cudaMalloc(&err, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(error word)");
  e = cudaMemset(err, 0, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(error word)");
  g_rt.device = dev;
  g_rt.sms = sms;
  g_rt.dev_err = err;
  g_rt.ready = true;
  return SV_OK;
}

sv_status map_weights_view(MapWeightsView* v) {
  SV_TRY(check_ready());
  const Dims& d = g_w.d;
  v->T = d.T;
  v->D = d.D;
  v->H = d.H;
  v->F = d.F;
  v->probe = g_w.probe;
  v->q_w = g_w.mq_w;
  v->q_b = g_w.mq_b;
  v->kv_w = g_w.mkv_w;
  v->kv_b = g_w.mkv_b;
  v->out_w = g_w.mo_w;
  v->out_b = g_w.mo_b;
  v->ln_g = g_w.mln_g;
  v->ln_b = g_w.mln_b;
  v->fc1_w = g_w.mfc1_w;
  v->fc1_b = g_w.mfc1_b;
  v->fc2_w = g_w.mfc2_w;
  v->fc2_b = g_w.mfc2_b;
  v->probe8 = g_w.probe8;
  v->q_w8 = g_w.mq_w8;
  v->kv_w8 = g_w.mkv_w8;
  v->out_w8 = g_w.mo_w8;
  v->fc1_w8 = g_w.mfc1_w8;
  v->fc2_w8 = g_w.mfc2_w8;
  return SV_OK;
}

int* dev_err() { return g_rt.dev_err; }
int num_sms() { return g_rt.sms; }

LaunchScope::LaunchScope(int kind, double flops, double bytes, cudaStream_t s) : on_(g_prof_on) {
  ++g_launches;
  if (on_) {
    ProfRec r{kind, flops, bytes, get_event(), get_event()};
    cudaEventRecord(r.e0, s);
    g_prof.push_back(r);
    stream_ = s;
  }
}

LaunchScope::~LaunchScope() {
  if (on_) cudaEventRecord(g_prof.back().e1, stream_);
}

}  // namespace sv

using namespace sv;

extern "C" {

sv_status sv_init_weights(uint64_t seed) { return sv_init_weights_dims(seed, 729, 588, 1152, 16, 4304, 27); }

sv_status sv_init_weights_dims(uint64_t seed, int tokens, int patch_dim, int width, int heads, int mlp, int layers) {
  if (tokens < 1 || patch_dim < 1 || patch_dim > 4096 || heads < 1 || layers < 1 || layers > 64 || mlp < 16) {
    set_error("sv_init_weights_dims: sizes out of range");
    return SV_ERR_INVALID_ARG;
  }
  if (width != heads * 72 || width % 16 != 0 || mlp % 16 != 0 || patch_dim % 4 != 0 || width > 4096) {
    set_error("sv_init_weights_dims: needs width == heads*72, width %% 16 == 0, mlp %% 16 == 0, patch_dim %% 4 == 0");
    return SV_ERR_UNSUPPORTED;
  }
  Dims d;
  d.T = tokens;
  d.P = patch_dim;
  d.D = width;
  d.H = heads;
  d.F = mlp;
  d.L = layers;
  d.Kp = int(align_up(size_t(patch_dim), 16));
  return init_weights(seed, d);
}

sv_status sv_model_dims(int* tokens, int* patch_dim, int* width, int* heads, int* mlp, int* layers) {
  SV_TRY(check_ready());
  const Dims& d = g_w.d;
  if (tokens) *tokens = d.T;
  if (patch_dim) *patch_dim = d.P;
  if (width) *width = d.D;
  if (heads) *heads = d.H;
  if (mlp) *mlp = d.F;
  if (layers) *layers = d.L;
  return SV_OK;
}

size_t sv_weights_count(void) {
  if (!g_w.ready) return 0;
  size_t n = 0;
  for (const TensorRec& t : g_w.tensors) n += size_t(t.rows) * size_t(t.cols);
  return n;
}

size_t sv_weights_count_e4m3(void) {
  if (!g_w.ready) return 0;
  size_t n = 0;
  for (const TensorRec& t : g_w.tensors)
    if (t.p8) n += size_t(t.rows) * size_t(t.cols);
  return n;
}

sv_status sv_export_weights(float* host_dst, size_t n_floats) {
  SV_TRY(check_ready());
  const size_t need = sv_weights_count();
  if (!host_dst || n_floats < need) {
    set_error("sv_export_weights: needs a host buffer of %zu floats (got %zu)", need, n_floats);
    return SV_ERR_INVALID_ARG;
  }
  SV_CHECK_CUDA(cudaDeviceSynchronize(), "sv_export_weights");
  std::vector<uint16_t> h;
  float* dst = host_dst;
  for (const TensorRec& t : g_w.tensors) {
    // a dense weight is resident as [N, kpad] (K-major); the logical layout is [K, N]
    const size_t stored = t.matrix ? size_t(t.cols) * size_t(t.kpad) : size_t(t.rows) * size_t(t.cols);
    h.resize(stored);
    SV_CHECK_CUDA(cudaMemcpy(h.data(), t.p16, 2 * stored, cudaMemcpyDeviceToHost), "sv_export_weights copy");
    for (int r = 0; r < t.rows; ++r)
      for (int c = 0; c < t.cols; ++c) {
        const uint16_t bits = t.matrix ? h[size_t(c) * size_t(t.kpad) + size_t(r)] : h[size_t(r) * size_t(t.cols) + size_t(c)];
        __half_raw raw;
        raw.x = bits;
        dst[size_t(r) * size_t(t.cols) + size_t(c)] = __half2float(__half(raw));
      }
    dst += size_t(t.rows) * size_t(t.cols);
  }
  return SV_OK;
}

sv_status sv_export_weights_e4m3(uint8_t* host_dst, size_t n_bytes) {
  SV_TRY(check_ready());
  const size_t need = sv_weights_count_e4m3();
  if (!host_dst || n_bytes < need) {
    set_error("sv_export_weights_e4m3: needs a host buffer of %zu bytes (got %zu)", need, n_bytes);
    return SV_ERR_INVALID_ARG;
  }
  SV_CHECK_CUDA(cudaDeviceSynchronize(), "sv_export_weights_e4m3");
  std::vector<uint8_t> h;
  uint8_t* dst = host_dst;
  for (const TensorRec& t : g_w.tensors) {
    if (!t.p8) continue;
    const size_t stored = t.matrix ? size_t(t.cols) * size_t(t.kpad) : size_t(t.rows) * size_t(t.cols);
    h.resize(stored);
    SV_CHECK_CUDA(cudaMemcpy(h.data(), t.p8, stored, cudaMemcpyDeviceToHost), "sv_export_weights_e4m3 copy");
    for (int r = 0; r < t.rows; ++r)
      for (int c = 0; c < t.cols; ++c)
        dst[size_t(r) * size_t(t.cols) + size_t(c)] =
            t.matrix ? h[size_t(c) * size_t(t.kpad) + size_t(r)] : h[size_t(r) * size_t(t.cols) + size_t(c)];
    dst += size_t(t.rows) * size_t(t.cols);
  }
  return SV_OK;
}

sv_status sv_encode_ex(const void* pixels, void* out, int batch, int layers, int gemm_dtype, int flags,
                       void* stream) {
  SV_TRY(check_ready());
  if (!pixels || !out || batch < 1 || layers < 1 || layers > g_w.d.L ||
      (gemm_dtype != SV_GEMM_F16 && gemm_dtype != SV_GEMM_E4M3) || (flags & ~(SV_ENCODE_UNFUSED_QKV | SV_ENCODE_FP8_ATTENTION | SV_ENCODE_EAGER))) {
    set_error("sv_encode: bad arguments (batch %d, layers %d of %d, gemm_dtype %d, flags %d)", batch, layers,
              g_w.d.L, gemm_dtype, flags);
    return SV_ERR_INVALID_ARG;
  }
  if (!aligned(pixels, 8) || !aligned(out, 16)) {
    set_error("sv_encode: pixels must be 8-byte and out 16-byte aligned");
    return SV_ERR_INVALID_ARG;
  }
  if (long(batch) * g_w.d.T > (1L << 30)) {
    set_error("sv_encode: batch too large");
    return SV_ERR_INVALID_ARG;
  }
  Plan* p = nullptr;
  const int plan_flags = flags & ~SV_ENCODE_EAGER;
  SV_TRY(get_plan(batch, gemm_dtype, plan_flags, &p));
  return encode_step(*p, static_cast<const __half*>(pixels), static_cast<__half*>(out), layers,
                     plan_flags | (flags & SV_ENCODE_EAGER), static_cast<cudaStream_t>(stream));
}

sv_status sv_encode(const void* pixels, void* out, int batch, int layers, int gemm_dtype, void* stream) {
  return sv_encode_ex(pixels, out, batch, layers, gemm_dtype, 0, stream);
}

sv_status sv_gemm_bias_act(const void* A, const void* W, const void* bias, const void* pos, int pos_rows,
                           const void* residual, void* C, int M, int N, int K, int act, int in_dtype, int out_dtype,
                           float scale_a, float scale_w, void* stream) {
  const float scale = scale_a * scale_w;
  if (!A || !W || !C || M < 1 || N < 16 || K < 16 || N % 16 || K % 16 || (act != 0 && act != 1) ||
      (in_dtype != 0 && in_dtype != 1) || (out_dtype != 0 && out_dtype != 1) || (pos && pos_rows < 1) ||
      !std::isfinite(scale)) {
    set_error("sv_gemm_bias_act: bad arguments (M %d N %d K %d; N and K must be multiples of 16)", M, N, K);
    return SV_ERR_INVALID_ARG;
  }
  if (!aligned(A, 16) || !aligned(W, 16) || !aligned(C, 16) || !aligned(bias, 16) || !aligned(pos, 16) ||
      !aligned(residual, 16)) {
    set_error("sv_gemm_bias_act: all pointers must be 16-byte aligned");
    return SV_ERR_INVALID_ARG;
  }
  SV_TRY(ensure_runtime());
  GemmEpi e = epi(static_cast<const __half*>(bias), C, scale, act, out_dtype, static_cast<const __half*>(residual));
  e.pos = static_cast<const __half*>(pos);
  e.pos_rows = pos_rows;
  // a small-M, long-K GEMM splits K: its partial sums go to a library buffer that grows
  // to the largest need seen (freed by sv_shutdown)
  const size_t need = gemm_splitk_ws_bytes_for(M, N, K, in_dtype, kMaxSplits);
  if (need > g_gemm_ws_bytes) {
    if (g_gemm_ws) {
      SV_CHECK_CUDA(cudaDeviceSynchronize(), "sv_gemm_bias_act");
      cudaFree(g_gemm_ws);
      g_gemm_ws = nullptr;
      g_gemm_ws_bytes = 0;
    }
    cudaError_t ce = cudaMalloc(&g_gemm_ws, need);
    if (ce != cudaSuccess) {
      cudaGetLastError();
      set_error("sv_gemm_bias_act: cudaMalloc of %zu bytes for the split-K partial sums failed", need);
      return SV_ERR_OOM;
    }
    g_gemm_ws_bytes = need;
  }
  GemmCall c;
  SV_TRY(make_call(&c, A, W, M, N, K, in_dtype, e, K, static_cast<float*>(g_gemm_ws), g_gemm_ws_bytes));
  return run_gemm(c, static_cast<cudaStream_t>(stream));
}

sv_status sv_ln_gemm(const void* x, const void* gamma, const void* beta, float eps, const void* W, const void* bias,
                     void* C, int M, int N, int K, int act, void* stream) {
  if (!x || !gamma || !beta || !W || !C || M < 1 || N < 16 || N % 16 || K < 16 || K % 16 || K > 4096 ||
      !(eps >= 0.0f) || (act != 0 && act != 1)) {
    set_error("sv_ln_gemm: bad arguments (M %d N %d K %d; N, K multiples of 16, K <= 4096)", M, N, K);
    return SV_ERR_INVALID_ARG;
  }
  if (!aligned(x, 16) || !aligned(gamma, 16) || !aligned(beta, 16) || !aligned(W, 16) || !aligned(bias, 16) ||
      !aligned(C, 16)) {
    set_error("sv_ln_gemm: pointers must be 16-byte aligned");
    return SV_ERR_INVALID_ARG;
  }
  SV_TRY(ensure_runtime());
  // scratch: W * gamma [N, K] | W's extra K block [N, 16] | biases [N] | x's extra K block
  // [M, 16] (all f16) | 1/std [M] f32
  const size_t off_wa = align_up(size_t(N) * K * 2, 256), off_b = align_up(off_wa + size_t(N) * 32, 256),
               off_xa = align_up(off_b + size_t(N) * 2, 256), off_r = align_up(off_xa + size_t(M) * 32, 256),
               need = off_r + size_t(M) * 4;
  if (need > g_lng_scratch_bytes) {  // grows monotonically; freed by sv_shutdown
    if (g_lng_scratch) {
      SV_CHECK_CUDA(cudaDeviceSynchronize(), "sv_ln_gemm");
      cudaFree(g_lng_scratch);
      g_lng_scratch = nullptr;
      g_lng_scratch_bytes = 0;
    }
    cudaError_t e = cudaMalloc(&g_lng_scratch, need);
    if (e != cudaSuccess) {
      cudaGetLastError();
      set_error("sv_ln_gemm: cudaMalloc of %zu bytes failed", need);
      return SV_ERR_OOM;
    }
    g_lng_scratch_bytes = need;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* sc = static_cast<char*>(g_lng_scratch);
  __half* w2 = reinterpret_cast<__half*>(sc);
  __half* wa = reinterpret_cast<__half*>(sc + off_wa);
  __half* bf = reinterpret_cast<__half*>(sc + off_b);
  __half* xa = reinterpret_cast<__half*>(sc + off_xa);
  float* rr = reinterpret_cast<float*>(sc + off_r);
  SV_CHECK_CUDA(cudaMemcpyAsync(w2, W, size_t(N) * K * 2, cudaMemcpyDeviceToDevice, s), "sv_ln_gemm weight copy");
  {
    Launch L(kKindOther, 0.0, double(N) * K * 4.0, s);
    SV_TRY(fold_ln_launch(w2, static_cast<const __half*>(gamma), static_cast<const __half*>(beta),
                          static_cast<const __half*>(bias), wa, bf, N, K, s));
  }
  {
    Launch L(kKindLN, 4.0 * M * K, double(M) * (K * 2.0 + 8.0), s);
    SV_TRY(ln_stats_launch(static_cast<const __half*>(x), rr, xa, M, K, eps, s));
  }
  GemmEpi e = epi(bf, C, 1.0f, act);
  e.ln_r = rr;
  e.ln_aug_a = xa;
  e.ln_aug_w = wa;
  GemmCall c;
  SV_TRY(make_call(&c, x, w2, M, N, K, 0, e, K));
  return run_gemm(c, s);
}

sv_status sv_pack_patches(const void* images, void* pixels, int batch, int image_side, int channels, int patch,
                          void* stream) {
  if (!images || !pixels || batch < 1 || patch < 1 || channels < 1 || image_side < patch || image_side % patch ||
      (patch * channels) % 2 || image_side > 65536) {
    set_error("sv_pack_patches: bad arguments (side %d must be a multiple of patch %d; patch * channels even)",
              image_side, patch);
    return SV_ERR_INVALID_ARG;
  }
  if (!aligned(images, 4) || !aligned(pixels, 4)) {
    set_error("sv_pack_patches: pointers must be 4-byte aligned");
    return SV_ERR_INVALID_ARG;
  }
  SV_TRY(ensure_runtime());
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Launch L(kKindOther, 0.0, double(batch) * image_side * image_side * channels * 4.0, s);
  return pack_patches_launch(static_cast<const __half*>(images), static_cast<__half*>(pixels), batch, image_side,
                             channels, patch, s);
}

sv_status sv_layernorm(void* x, const void* residual, const void* gamma, const void* beta, void* y, int rows,
                       int width, float eps, int out_dtype, void* stream) {
  if (!x || !gamma || !beta || !y || rows < 1 || width < 8 || width > 4096 || width % 8 || !(eps >= 0.0f) ||
      (out_dtype != 0 && out_dtype != 1)) {
    set_error("sv_layernorm: bad arguments (rows %d, width %d)", rows, width);
    return SV_ERR_INVALID_ARG;
  }
  if (!aligned(x, 16) || !aligned(residual, 16) || !aligned(gamma, 16) || !aligned(beta, 16) || !aligned(y, 16)) {
    set_error("sv_layernorm: pointers must be 16-byte aligned");
    return SV_ERR_INVALID_ARG;
  }
  SV_TRY(ensure_runtime());
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const double rb = residual ? 4.0 : 0.0;  // the residual read and the sum written back
  Launch L(kKindLN, 8.0 * rows * width, double(rows) * width * (2.0 + rb + (out_dtype ? 1.0 : 2.0)), s);
  if (residual)
    return layernorm_residual_launch(static_cast<__half*>(x), static_cast<const __half*>(residual),
                                     static_cast<const __half*>(gamma), static_cast<const __half*>(beta), y, rows,
                                     width, eps, out_dtype, s);
  return layernorm_launch(static_cast<const __half*>(x), static_cast<const __half*>(gamma),
                          static_cast<const __half*>(beta), y, rows, width, eps, out_dtype, s);
}

sv_status sv_attention(const void* qkv, void* o, int batch, int heads, int tokens, int head_dim, float scale,
                       int out_dtype, void* stream) {
  return sv_attention_ex(qkv, o, batch, heads, tokens, head_dim, scale, out_dtype, 0, stream);
}

}  // extern "C"

namespace sv {
namespace {
// Shared checks of the attention entry points, and their scratch buffer: the
// head-blocked copy of the operands, grown to the largest call, freed by sv_shutdown.
sv_status attention_args(const char* fn, const void* o, int batch, int heads, int tokens, int head_dim, float* scale,
                         int out_dtype, int flags) {
  if (!o || batch < 1 || heads < 1 || tokens < 1 || batch > 65535 || !std::isfinite(*scale) ||
      (out_dtype != 0 && out_dtype != 1) || (flags & ~SV_ATTENTION_QK_E4M3)) {
    set_error("%s: bad arguments", fn);
    return SV_ERR_INVALID_ARG;
  }
  if (head_dim != 72) {
    set_error("%s: head_dim %d is not supported (72 only)", fn, head_dim);
    return SV_ERR_UNSUPPORTED;
  }
  if (!aligned(o, 16)) {
    set_error("%s: pointers must be 16-byte aligned", fn);
    return SV_ERR_INVALID_ARG;
  }
  if (*scale <= 0.0f) *scale = 1.0f / std::sqrt(float(head_dim));  // scaled dot-product attention
  return SV_OK;
}

sv_status attention_scratch(size_t need, const char* fn) {
  if (need <= g_attn_scratch_bytes) return SV_OK;
  if (g_attn_scratch) {
    SV_CHECK_CUDA(cudaDeviceSynchronize(), fn);
    cudaFree(g_attn_scratch);
    g_attn_scratch = nullptr;
    g_attn_scratch_bytes = 0;
  }
  cudaError_t e = cudaMalloc(&g_attn_scratch, need);
  if (e != cudaSuccess) {
    cudaGetLastError();
    set_error("%s: cudaMalloc of %zu bytes failed", fn, need);
    return SV_ERR_OOM;
  }
  g_attn_scratch_bytes = need;
  return SV_OK;
}

sv_status attention_on_scratch(void* o, int batch, int heads, int tokens, float scale, int out_dtype, int flags,
                               cudaStream_t s) {
  Launch L(kKindAttn, 4.0 * batch * heads * double(tokens) * tokens * 72.0, 0.0, s);
  return attention_launch(g_attn_scratch, o, batch, tokens, heads, scale, out_dtype, flags & SV_ATTENTION_QK_E4M3,
                          s);
}
}  // namespace
}  // namespace sv

extern "C" {

sv_status sv_attention_ex(const void* qkv, void* o, int batch, int heads, int tokens, int head_dim, float scale,
                          int out_dtype, int flags, void* stream) {
  SV_TRY(attention_args("sv_attention", o, batch, heads, tokens, head_dim, &scale, out_dtype, flags));
  if (!qkv || !aligned(qkv, 16)) {
    set_error("sv_attention: qkv must be a 16-byte aligned pointer");
    return SV_ERR_INVALID_ARG;
  }
  SV_TRY(ensure_runtime());
  SV_TRY(attention_scratch(attention_blocked_bytes(batch, tokens, heads), "sv_attention"));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  {
    Launch L(kKindOther, 0.0, double(batch) * tokens * 3 * heads * 72 * 4.0, s);
    SV_TRY(attention_repack_launch(static_cast<const __half*>(qkv), g_attn_scratch, batch, tokens, heads,
                                   flags & SV_ATTENTION_QK_E4M3, s));
  }
  return attention_on_scratch(o, batch, heads, tokens, scale, out_dtype, flags, s);
}

sv_status sv_attention_heads(const void* q, const void* k, const void* v, void* o, int batch, int heads, int tokens,
                             int head_dim, int head_stride, float scale, int out_dtype, int flags, void* stream) {
  SV_TRY(attention_args("sv_attention_heads", o, batch, heads, tokens, head_dim, &scale, out_dtype, flags));
  if (!q || !k || !v || !aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || head_stride < head_dim ||
      head_stride % 8 || head_stride > 4096) {
    set_error("sv_attention_heads: q, k, v must be 16-byte aligned and head_stride (%d) a multiple of 8 in "
              "[head_dim, 4096]", head_stride);
    return SV_ERR_INVALID_ARG;
  }
  SV_TRY(ensure_runtime());
  SV_TRY(attention_scratch(attention_blocked_bytes(batch, tokens, heads), "sv_attention_heads"));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  {
    Launch L(kKindOther, 0.0, double(batch) * tokens * 3 * heads * 72 * 4.0, s);
    SV_TRY(attention_repack_heads_launch(static_cast<const __half*>(q), static_cast<const __half*>(k),
                                         static_cast<const __half*>(v), g_attn_scratch, batch, tokens, heads,
                                         head_stride, flags & SV_ATTENTION_QK_E4M3, s));
  }
  return attention_on_scratch(o, batch, heads, tokens, scale, out_dtype, flags, s);
}

sv_status sv_map_pool(const void* x, void* out, int batch, int gemm_dtype, void* stream) {
  SV_TRY(check_ready());
  if (!x || !out || batch < 1 || (gemm_dtype != 0 && gemm_dtype != 1)) {
    set_error("sv_map_pool: bad arguments");
    return SV_ERR_INVALID_ARG;
  }
  if (!aligned(x, 16) || !aligned(out, 16)) {
    set_error("sv_map_pool: pointers must be 16-byte aligned");
    return SV_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Dims& d = g_w.d;
  const int fp8 = gemm_dtype;
  const auto key = std::make_pair(batch, fp8);
  auto it = g_map_plans.find(key);
  Plan* p = nullptr;
  if (it == g_map_plans.end()) {
    std::unique_ptr<Plan> np(new Plan());
    np->B = batch;
    np->fp8 = fp8;
    Carver c{nullptr};
    np->ws_bytes = map_ws_bytes(batch, fp8);
    for (int pass = 0; pass < 2; ++pass) {
      np->ws = np->ws_bytes ? static_cast<float*>(c.take(np->ws_bytes)) : nullptr;
      np->Y = fp8 ? c.take(size_t(batch) * d.T * d.D) : nullptr;  // quantised copy of x
      if (c.base && !fp8) np->Y = const_cast<void*>(x);
      SV_TRY(build_map(np->map, c, np->Y ? np->Y : x, batch, fp8, true, nullptr, np->ws, np->ws_bytes));
      if (pass == 0) SV_TRY(alloc_carved(c, &np->mem, &np->bytes));
    }
    p = np.get();
    g_map_plans[key] = std::move(np);
  } else {
    p = it->second.get();
    if (!fp8 && p->Y != x) {  // the KV operand map follows the caller's buffer
      SV_TRY(gemm_prepare(&p->map.kv.g, x, g_w.mkv_w, batch * d.T, 2 * d.D, d.D, 0));
      SV_TRY(gemm_bind_epilogue(&p->map.kv.g, p->map.kv.e));
      p->Y = const_cast<void*>(x);
    }
  }
  if (fp8) {
    Launch L(kKindOther, 0.0, double(batch) * d.T * d.D * 3.0, s);
    SV_TRY(quantize_launch(static_cast<const __half*>(x), static_cast<uint8_t*>(p->Y), size_t(batch) * d.T * d.D, s));
  }
  return run_map(p->map, batch, fp8, static_cast<__half*>(out), s);
}

sv_status sv_quantize_e4m3(const void* x, void* y, size_t n, void* stream) {
  if (!x || !y || n % 16 || !aligned(x, 16) || !aligned(y, 16)) {
    set_error("sv_quantize_e4m3: needs n %% 16 == 0 and 16-byte aligned pointers");
    return SV_ERR_INVALID_ARG;
  }
  SV_TRY(ensure_runtime());
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Launch L(kKindOther, 0.0, double(n) * 3.0, s);
  return quantize_launch(static_cast<const __half*>(x), static_cast<uint8_t*>(y), n, s);
}

sv_status sv_make_pixels(uint64_t seed, int batch, void* dev_dst, void* stream) {
  SV_TRY(check_ready());
  if (!dev_dst || batch < 1) {
    set_error("sv_make_pixels: bad arguments");
    return SV_ERR_INVALID_ARG;
  }
  const Dims& d = g_w.d;
  std::vector<uint16_t> host(size_t(batch) * d.T * d.P);
  synth_pixels_f16(seed, batch, d.T, d.P, host.data());
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  SV_CHECK_CUDA(cudaMemcpyAsync(dev_dst, host.data(), host.size() * 2, cudaMemcpyHostToDevice, s), "pixel upload");
  SV_CHECK_CUDA(cudaStreamSynchronize(s), "pixel upload");
  return SV_OK;
}

sv_status sv_sync(void* stream) {
  SV_TRY(ensure_runtime());
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "sv_sync");
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "sv_sync (pending error)");
  int flag = 0;
  e = cudaMemcpy(&flag, g_rt.dev_err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "sv_sync (error word)");
  if (flag) {
    cudaMemset(g_rt.dev_err, 0, sizeof(int));
    set_error("a kernel gave up a bounded wait (device error word 0x%x); its outputs are undefined", flag);
    return SV_ERR_TIMEOUT;
  }
  return SV_OK;
}

const char* sv_last_error(void) { return g_err.c_str(); }

long long sv_launch_count(void) {
  const long long n = g_launches;
  g_launches = 0;
  return n;
}

sv_status sv_profile_enable(int on) {
  g_prof_on = on != 0;
  return SV_OK;
}

sv_status sv_profile_read(int kind, double* ms, double* flops, double* bytes, long long* launches) {
  if (kind < 0 || kind >= kNumKinds) {
    set_error("sv_profile_read: kind %d out of range", kind);
    return SV_ERR_INVALID_ARG;
  }
  SV_CHECK_CUDA(cudaDeviceSynchronize(), "sv_profile_read");
  double t = 0, f = 0, b = 0;
  long long n = 0;
  std::vector<ProfRec> keep;
  for (const ProfRec& r : g_prof) {
    if (r.kind != kind) {
      keep.push_back(r);
      continue;
    }
    float x = 0;
    cudaEventElapsedTime(&x, r.e0, r.e1);
    t += x;
    f += r.flops;
    b += r.bytes;
    ++n;
    g_ev_pool.push_back(r.e0);
    g_ev_pool.push_back(r.e1);
  }
  g_prof.swap(keep);
  if (ms) *ms = t;
  if (flops) *flops = f;
  if (bytes) *bytes = b;
  if (launches) *launches = n;
  return SV_OK;
}

sv_status sv_debug_fill_workspace(int batch, int gemm_dtype, int byte_value) {
  SV_TRY(check_ready());
  if (batch < 1 || (gemm_dtype != 0 && gemm_dtype != 1)) {
    set_error("sv_debug_fill_workspace: bad arguments");
    return SV_ERR_INVALID_ARG;
  }
  Plan* p = nullptr;
  SV_TRY(get_plan(batch, gemm_dtype, 0, &p));
  SV_CHECK_CUDA(cudaMemset(p->mem, byte_value & 0xFF, p->bytes), "sv_debug_fill_workspace");
  SV_CHECK_CUDA(cudaDeviceSynchronize(), "sv_debug_fill_workspace");
  return SV_OK;
}

sv_status sv_debug_wait_timeout(unsigned int limit_us, void* stream) {
  if (limit_us == 0 || limit_us > 2000000u) {
    set_error("sv_debug_wait_timeout: limit must be in 1..2000000 us");
    return SV_ERR_INVALID_ARG;
  }
  SV_TRY(ensure_runtime());
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Launch L(kKindOther, 0.0, 0.0, s);
  return wait_probe_launch(limit_us, s);
}

sv_status sv_debug_encode_stage(const void* pixels, int batch, int layers, int gemm_dtype, int flags, int stage,
                                void* dst, size_t dst_bytes, void* stream) {
  SV_TRY(check_ready());
  const Dims& d = g_w.d;
  if (!pixels || !dst || batch < 1 || layers < 1 || layers > d.L || stage < SV_STAGE_PATCH ||
      stage > SV_STAGE_FINAL_LN || (gemm_dtype != SV_GEMM_F16 && gemm_dtype != SV_GEMM_E4M3) ||
      (flags & ~(SV_ENCODE_UNFUSED_QKV | SV_ENCODE_FP8_ATTENTION | SV_ENCODE_EAGER)) || !aligned(pixels, 8) ||
      !aligned(dst, 16)) {
    set_error("sv_debug_encode_stage: bad arguments");
    return SV_ERR_INVALID_ARG;
  }
  if (stage == SV_STAGE_QKV && (flags & SV_ENCODE_FP8_ATTENTION)) {
    set_error("sv_debug_encode_stage: the QKV stage with E4M3 Q and K is not supported");
    return SV_ERR_UNSUPPORTED;
  }
  const size_t M = size_t(batch) * d.T, eb = gemm_dtype == SV_GEMM_E4M3 ? 1 : 2;
  size_t bytes = 0;
  switch (stage) {
    case SV_STAGE_PATCH:
    case SV_STAGE_OUT_PROJ:
    case SV_STAGE_MLP_DOWN: bytes = M * d.D * 2; break;
    case SV_STAGE_QKV: bytes = M * 3 * d.D * 2; break;
    case SV_STAGE_ATTENTION:
    case SV_STAGE_FINAL_LN: bytes = M * d.D * eb; break;
    default: bytes = M * d.F * eb; break;  // SV_STAGE_MLP_UP
  }
  if (dst_bytes < bytes) {
    set_error("sv_debug_encode_stage: stage %d needs %zu bytes (got %zu)", stage, bytes, dst_bytes);
    return SV_ERR_INVALID_ARG;
  }
  Plan* p = nullptr;
  SV_TRY(get_plan(batch, gemm_dtype, flags & ~SV_ENCODE_EAGER, &p));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  SV_TRY(encode(*p, static_cast<const __half*>(pixels), nullptr, layers, s, stage));
  const void* src = stage == SV_STAGE_ATTENTION ? p->O
                    : stage == SV_STAGE_MLP_UP  ? p->Hh
                    : stage == SV_STAGE_FINAL_LN ? p->Y
                                                 : static_cast<const void*>(p->X);
  if (stage == SV_STAGE_QKV) {
    Launch L(kKindOther, 0.0, double(bytes) * 2.0, s);
    return attention_unpack_launch(p->QKV, static_cast<__half*>(dst), batch, d.T, d.H, s);
  }
  SV_CHECK_CUDA(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s), "sv_debug_encode_stage copy");
  return SV_OK;
}

void sv_shutdown(void) {
  if (g_rt.ready) cudaDeviceSynchronize();
  map_static_forget();
  free_weights();
  for (const ProfRec& r : g_prof) {
    cudaEventDestroy(r.e0);
    cudaEventDestroy(r.e1);
  }
  g_prof.clear();
  for (cudaEvent_t e : g_ev_pool) cudaEventDestroy(e);
  g_ev_pool.clear();
  if (g_capture_stream) cudaStreamDestroy(g_capture_stream);
  g_capture_stream = nullptr;
  if (g_rt.dev_err) cudaFree(g_rt.dev_err);
  g_rt = Runtime();
}

}  // extern "C"
