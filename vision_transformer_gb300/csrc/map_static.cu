// MAP pooling that allocates no device memory of its own.
//
// sv_map_pool keeps a workspace that the library allocates with cudaMalloc on
// first use. Some callers cannot let a library allocate at call time: code
// whose allocator owns all of device memory (a framework's caching
// allocator, a memory pool sized up front), code running under a strict
// memory budget, or code that must not block on the driver's allocator while
// other work is in flight. This variant runs the same head with its scratch in
// one fixed array compiled into the library (kStaticScratchBytes). The array
// takes device memory once this file's code is loaded into a device's context
// (under CUDA's default lazy loading: at the first call of this entry point on
// that device) and keeps it until the context is destroyed.
//
// The array's host-side name is not a device address. The first call on a
// device asks the runtime for the array's device address with
// cudaGetSymbolAddress (with that device current) and keeps it; only that
// address is handed to kernels. The first call on a device should therefore
// come before any stream capture on that device. sv_shutdown forgets the kept
// addresses (map_static_forget), so a context destroyed after sv_shutdown is
// looked up anew.
//
// All calls share the one array and it keeps the previous call's contents;
// every buffer in it is written before it is read within a call, so nothing
// needs clearing. Two calls whose work overlaps on the GPU (different streams,
// or different threads) race on the array.
#include <cmath>

#include "sv_internal.h"

namespace sv {

// 8 MiB: one image's K/V projections (3.4 MB at width 1152), its E4M3 copy
// (0.8 MB) and 15.5 KB per pooled image.
constexpr size_t kStaticScratchBytes = size_t(8) << 20;
constexpr int kStaticMaxBatch = 256;

static __device__ __align__(256) unsigned char g_map_scratch[kStaticScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
void* g_scratch_dev[kMaxDevices] = {};

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Scratch layout for `batch` images: [q D][KV T x 2D][x8 T x D][a B x D][A B x D][Ya B x D][Ha B x F].
struct Layout {
  size_t q, kv, x8, a, A, Ya, Ha, end;
};

Layout layout(const MapWeightsView& w, int batch, int fp8) {
  const size_t eb = fp8 ? 1 : 2;
  Layout l;
  size_t off = 0;
  l.q = off;
  off = up256(off + size_t(w.D) * 2);
  l.kv = off;
  off = up256(off + size_t(w.T) * 2 * w.D * 2);
  l.x8 = off;
  off = up256(off + (fp8 ? size_t(w.T) * w.D : 0));
  l.a = off;
  off = up256(off + size_t(batch) * w.D * eb);
  l.A = off;
  off = up256(off + size_t(batch) * w.D * 2);
  l.Ya = off;
  off = up256(off + size_t(batch) * w.D * eb);
  l.Ha = off;
  off = up256(off + size_t(batch) * w.F * eb);
  l.end = off;
  return l;
}

sv_status scratch_address(char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "sv_map_pool_static: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("sv_map_pool_static: device %d is beyond the %d devices this entry point tracks", dev, kMaxDevices);
    return SV_ERR_UNSUPPORTED;
  }
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_map_scratch);
    if (e != cudaSuccess || !p) return cuda_fail(e, "sv_map_pool_static: cudaGetSymbolAddress");
    g_scratch_dev[dev] = p;
  }
  *out = static_cast<char*>(g_scratch_dev[dev]);
  return SV_OK;
}

// One GEMM launch with its accounting (launch count, profile records).
sv_status run(const GemmOperands& g, const GemmEpi& e, int k_logical, cudaStream_t s) {
  const double eb = g.fp8 ? 1.0 : 2.0;
  double bytes = (double(g.M) + double(g.N)) * k_logical * eb + double(g.M) * g.N * (e.out_e4m3 ? 1.0 : 2.0);
  if (e.residual) bytes += double(g.M) * g.N * 2.0;
  LaunchScope L(kKindGemm, 2.0 * g.M * double(g.N) * double(k_logical), bytes, s);
  return gemm_launch(g, e, s);
}

#define SV_TRY_S(call)          \
  do {                          \
    sv_status s_ = (call);      \
    if (s_ != SV_OK) return s_; \
  } while (0)

}  // namespace

void map_static_forget() {
  for (void*& p : g_scratch_dev) p = nullptr;
}

}  // namespace sv

using namespace sv;

extern "C" sv_status sv_map_pool_static(const void* x, void* out, int batch, int gemm_dtype, void* stream) {
  MapWeightsView w;
  SV_TRY_S(map_weights_view(&w));
  if (!x || !out || batch < 1 || (gemm_dtype != 0 && gemm_dtype != 1)) {
    set_error("sv_map_pool_static: bad arguments");
    return SV_ERR_INVALID_ARG;
  }
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) % 16) {
    set_error("sv_map_pool_static: pointers must be 16-byte aligned");
    return SV_ERR_INVALID_ARG;
  }
  const int fp8 = gemm_dtype;
  const Layout l = layout(w, batch, fp8);
  if (batch > kStaticMaxBatch || l.end > kStaticScratchBytes) {
    set_error("sv_map_pool_static: batch %d needs %zu bytes of scratch; the static buffer holds %zu bytes and "
              "at most %d images per call",
              batch, l.end, kStaticScratchBytes, kStaticMaxBatch);
    return SV_ERR_INVALID_ARG;
  }
  char* s = nullptr;
  SV_TRY_S(scratch_address(&s));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t eb = fp8 ? 1 : 2;
  __half* q = reinterpret_cast<__half*>(s + l.q);
  __half* kv = reinterpret_cast<__half*>(s + l.kv);
  uint8_t* x8 = reinterpret_cast<uint8_t*>(s + l.x8);
  void* a = s + l.a;
  __half* A = reinterpret_cast<__half*>(s + l.A);
  void* Ya = s + l.Ya;
  void* Ha = s + l.Ha;
  const float sc = fp8 ? 1.0f / 256.0f : 1.0f;
  const float attn_scale = 1.0f / std::sqrt(72.0f);

  GemmOperands g;
  GemmEpi e;
  e.scale = sc;
  // q = probe . Wq + bq (shared by every image)
  SV_TRY_S(gemm_prepare(&g, fp8 ? (const void*)w.probe8 : w.probe, fp8 ? (const void*)w.q_w8 : w.q_w, 1, w.D, w.D,
                        fp8));
  e.bias = w.q_b;
  e.out = q;
  SV_TRY_S(gemm_bind_epilogue(&g, e));
  SV_TRY_S(run(g, e, w.D, st));
  // one image at a time: [K V] = x_b . Wkv + bkv, then the single-query attention into a[b]
  const size_t img = size_t(w.T) * w.D;
  for (int b = 0; b < batch; ++b) {
    const __half* xb = static_cast<const __half*>(x) + size_t(b) * img;
    const void* A_op = xb;
    if (fp8) {
      LaunchScope L(kKindOther, 0.0, double(img) * 3.0, st);
      SV_TRY_S(quantize_launch(xb, x8, img, st));
      A_op = x8;
    }
    SV_TRY_S(gemm_prepare(&g, A_op, fp8 ? (const void*)w.kv_w8 : w.kv_w, w.T, 2 * w.D, w.D, fp8));
    e.bias = w.kv_b;
    e.out = kv;
    SV_TRY_S(gemm_bind_epilogue(&g, e));
    SV_TRY_S(run(g, e, w.D, st));
    LaunchScope L(kKindMapAttn, 4.0 * w.T * double(w.D), double(w.T) * 2 * w.D * 2.0, st);
    SV_TRY_S(map_attn_launch(q, kv, static_cast<char*>(a) + size_t(b) * w.D * eb, 1, w.T, w.H, attn_scale, fp8,
                             st));
  }
  // A = a . Wo + bo;  out = A + W2 gelu(W1 LN(A) + b1) + b2
  SV_TRY_S(gemm_prepare(&g, a, fp8 ? (const void*)w.out_w8 : w.out_w, batch, w.D, w.D, fp8));
  e.bias = w.out_b;
  e.out = A;
  SV_TRY_S(gemm_bind_epilogue(&g, e));
  SV_TRY_S(run(g, e, w.D, st));
  {
    LaunchScope L(kKindLN, 8.0 * batch * w.D, double(batch) * w.D * 3.0, st);
    SV_TRY_S(layernorm_launch(A, w.ln_g, w.ln_b, Ya, batch, w.D, 1e-6f, fp8, st));
  }
  SV_TRY_S(gemm_prepare(&g, Ya, fp8 ? (const void*)w.fc1_w8 : w.fc1_w, batch, w.F, w.D, fp8));
  e.bias = w.fc1_b;
  e.act = SV_ACT_GELU_TANH;
  e.out_e4m3 = fp8;
  e.out = Ha;
  SV_TRY_S(gemm_bind_epilogue(&g, e));
  SV_TRY_S(run(g, e, w.D, st));
  SV_TRY_S(gemm_prepare(&g, Ha, fp8 ? (const void*)w.fc2_w8 : w.fc2_w, batch, w.D, w.F, fp8));
  e.bias = w.fc2_b;
  e.act = SV_ACT_NONE;
  e.out_e4m3 = 0;
  e.residual = A;
  e.out = out;
  SV_TRY_S(gemm_bind_epilogue(&g, e));
  return run(g, e, w.F, st);
}
