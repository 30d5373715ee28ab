// Declarations shared by the library's translation units (not part of the ABI).
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/sv.h"

namespace sv {

// ---- runtime state helpers (api.cu)
void set_error(const char* fmt, ...);
sv_status cuda_fail(cudaError_t e, const char* what);
sv_status ensure_runtime();  // device error word, SM count
int* dev_err();
int num_sms();

enum KernelKind { kKindGemm = 0, kKindAttn = 1, kKindLN = 2, kKindMapAttn = 3, kKindOther = 4, kNumKinds = 5 };

// Accounting of one library launch (api.cu): counts it for sv_launch_count and,
// while profiling is on, brackets it with CUDA events on its stream for
// sv_profile_read. Construct it right before the launch; it closes at scope end.
class LaunchScope {
 public:
  LaunchScope(int kind, double flops, double bytes, cudaStream_t s);
  ~LaunchScope();
  LaunchScope(const LaunchScope&) = delete;
  LaunchScope& operator=(const LaunchScope&) = delete;

 private:
  bool on_;
  cudaStream_t stream_ = nullptr;
};

// Kernel attributes (dynamic shared memory limits) are set once per device; device
// ordinals at or above this bound set them on every launch.
constexpr int kMaxAttrDevices = 64;

// Forgets the device addresses sv_map_pool_static has looked up (map_static.cu);
// called by sv_shutdown.
void map_static_forget();

// Read-only view of the resident MAP-head weights and model sizes (api.cu).
struct MapWeightsView {
  int T, D, H, F;
  const __half *probe, *q_w, *q_b, *kv_w, *kv_b, *out_w, *out_b, *ln_g, *ln_b, *fc1_w, *fc1_b, *fc2_w, *fc2_b;
  const uint8_t *probe8, *q_w8, *kv_w8, *out_w8, *fc1_w8, *fc2_w8;
};
sv_status map_weights_view(MapWeightsView* v);

// ---- tensor maps (gemm_tc.cu)
sv_status make_tmap(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* ptr, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle sw);

// ---- GEMM: C = epilogue(A[M,K] . W[N,K]^T)
struct GemmEpi {
  const __half* bias = nullptr;      // [N]
  const __half* pos = nullptr;       // [pos_rows, N], added by row m % pos_rows
  int pos_rows = 1;
  const __half* residual = nullptr;  // [M, N]
  void* out = nullptr;               // [M, N] f16 or e4m3
  int act = SV_ACT_NONE;
  int out_e4m3 = 0;
  float scale = 1.0f;
  // Head-blocked output for attention (replaces the row-major store when set):
  // see attention_blocked_bytes. `out` must still name a buffer of >= M*N f16.
  void* blk_out = nullptr;
  int blk_T = 0, blk_H = 0, blk_B = 0;
  int blk_col0 = 0;  // this GEMM's column 0 is column blk_col0 of the fused [Q | K | V] output
  int blk_qk8 = 0;   // Q and K written as E4M3 (value x 16) in their blocks, for FP8 score products
  // LayerNorm of A folded in (A is the LayerNorm input, W already scaled by gamma):
  // the GEMM runs one more K block of 16, ln_aug_a [M, 16] . ln_aug_w [N, 16]^T =
  // -mean_m s_n, and the epilogue scales row m by ln_r[m] before adding `bias` (b').
  // F16 operands only.
  const float* ln_r = nullptr;         // [M]
  const __half* ln_aug_a = nullptr;    // [M, 16]
  const __half* ln_aug_w = nullptr;    // [N, 16]
  // Row statistics of the output for the next LayerNorm: for each row m, column tile
  // t (bn columns, the last one N - t bn) and half h (the tile's 32-column chunks
  // c = h, h + 2, ...; absent when the tile has no such chunk),
  // ln_part[(m * n_tiles + t) * 2 + h] = (mean, sum of squared deviations from that
  // mean) of those F32 results (after bias, positions and residual).
  // ln_finalize_launch merges them.
  float2* ln_part = nullptr;
  // Partial sums of a GEMM that splits K (GemmOperands::k_splits > 1): at least
  // gemm_splitk_ws_bytes(g) bytes, used by gemm_launch and free again when its work ends.
  float* ws = nullptr;
  // With every tile split (k_splits > 1, n_main 0; at most 8 column tiles) the reduction
  // can finish the row statistics itself, in place of ln_part and ln_finalize_launch:
  // ln_r_out[m] = 1/sqrt(var + ln_eps) and ln_aug_out[m, 0..15] = (-mean_hi, -mean_hi,
  // -mean_lo, 0, ...) over the row's N results.
  float* ln_r_out = nullptr;
  __half* ln_aug_out = nullptr;
  float ln_eps = 1e-6f;
};
// Statistics entries per row that GemmEpi::ln_part can hold (two per column tile:
// 1152 columns in tiles of >= 64).
constexpr int kMaxLnTiles = 64;

// The operand side of a GEMM: tensor maps for A and W plus the sizes.
struct GemmOperands {
  CUtensorMap ta, tw, tc, tr;  // A, W, output, residual
  CUtensorMap tw_tail;         // W rows of the narrow last column tile (CTA pairs)
  CUtensorMap ta_aug, tw_aug;  // the extra K block of a folded LayerNorm
  CUtensorMap tw_aug_tail;     // its W rows for the narrow last column tile (CTA pairs)
  CUtensorMap tws;             // split-K partial-sum workspace (row-major F32)
  int has_aug = 0;
  int tail_n = 0;              // MMA N of the narrow last column tile, 0 if all tiles are full
  int tail_last = 0;           // narrow tiles after all full ones in the work order
  int M = 0, N = 0, K = 0;
  int fp8 = 0;
  int bn = 0;
  int mc = 0;  // CTA pairs (clusters of 2) sharing one 256-row MMA
  int atoms = 1;  // 128-byte swizzle rows of K per pipeline stage (1 or 2)
  int k_splits = 1;  // K ranges run by separate CTAs (pairs), summed by a reduction kernel
  int kb_split = 0;  // pipeline stages of K per range
  int n_main = 0;    // with k_splits > 1: tile items below n_main run whole (the rest split)
  int has_res = 0;
  const void* out = nullptr;  // epilogue buffers the output / residual maps describe
  const void* res = nullptr;
  const float* ws = nullptr;  // the split-K workspace the map tws describes
  int out_e4m3 = 0;
};

// Tensor map of a K-major operand [rows, K] (row stride = K elements) with the
// 128-byte swizzle the GEMM expects, box [box_rows, 128 bytes].
sv_status gemm_operand_map(CUtensorMap* m, const void* ptr, int rows, int K, int fp8, int box_rows);
int gemm_pick_bn(int M, int N, int K, bool mc, double* t_best, int sms);
// allow_pair = false keeps single-CTA tiles; max_splits > 1 lets a small-M, long-K GEMM
// split K into up to that many ranges (the caller then provides GemmEpi::ws).
sv_status gemm_prepare(GemmOperands* g, const void* A, const void* W, int M, int N, int K, int fp8,
                       bool allow_pair = true, int max_splits = 1);
// Workspace bytes of a prepared GEMM's split-K partial sums (0 without a split), and the
// same for the shape that gemm_prepare(..., true, max_splits) would choose.
size_t gemm_splitk_ws_bytes(const GemmOperands& g);
size_t gemm_splitk_ws_bytes_for(int M, int N, int K, int fp8, int max_splits);
// Builds the output / residual tensor maps for the epilogue's buffers (must precede gemm_launch).
sv_status gemm_bind_epilogue(GemmOperands* g, const GemmEpi& e);
// part: -1 every launch; with split K, 0 only the GEMM and 1 only the reduction (each
// with its own launch accounting).
sv_status gemm_launch(const GemmOperands& g, const GemmEpi& e, cudaStream_t s, int part = -1);

// Launches kern with programmatic stream serialization (the kernel must call
// pdl_wait() before touching global memory; see ptx.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ---- attention (attention.cu)
// Head-blocked Q/K/V: block (which, b, h, tile) at index ((which*B + b)*H + h)*tiles + tile
// (which 0 = Q, 1 = K, 2 = V; tiles of 128 tokens), each block 9 column groups x 128 rows x
// 8 f16 (2048 bytes per group: row r of group cg at cg*2048 + r*16). Rows past the last
// token of an image are never written or read as data.
// E4M3 Q / K (qk8, FP8 score products): the same block positions, each using its first
// 5 groups of 128 rows x 16 values E4M3(16 x) (row r of group g at g*2048 + r*16; group 4
// holds columns 64..71 and eight zero bytes).
size_t attention_blocked_bytes(int B, int T, int H);
// Row-major [B, T, 3*H*72] f16 -> head-blocked (qk8: Q and K quantised to E4M3).
sv_status attention_repack_launch(const __half* qkv, void* blocked, int B, int T, int H, int qk8, cudaStream_t s);
// Per-head q, k, v [B, H, T, stride] f16 (first 72 values of each row used) -> head-blocked.
sv_status attention_repack_heads_launch(const __half* q, const __half* k, const __half* v, void* blocked, int B,
                                        int T, int H, int stride, int qk8, cudaStream_t s);
// Head-blocked F16 Q, K, V -> row-major [B, T, 3*H*72] f16 (the inverse of the repack).
sv_status attention_unpack_launch(const void* blocked, __half* qkv, int B, int T, int H, cudaStream_t s);
// o: [B, T, H*72] f16 / e4m3. qk8: Q and K blocks are E4M3, S = Q K^T on E4M3 operands.
sv_status attention_launch(const void* blocked, void* o, int B, int T, int H, float scale, int out_e4m3, int qk8,
                           cudaStream_t s);

// ---- elementwise (elementwise.cu)
sv_status layernorm_launch(const __half* x, const __half* g, const __half* b, void* y, int rows, int width,
                           float eps, int out_e4m3, cudaStream_t s);
// The same on x + res (F16 sum, written back to x).
sv_status layernorm_residual_launch(__half* x, const __half* res, const __half* g, const __half* b, void* y, int rows,
                                    int width, float eps, int out_e4m3, cudaStream_t s);
// Row statistics only, for a LayerNorm folded into a GEMM: r[m] = 1/sqrt(var + eps)
// and aug[m, 0..15] = (-mean_hi, -mean_hi, -mean_lo, 0, ...) in F16.
sv_status ln_stats_launch(const __half* x, float* r, __half* aug, int rows, int width, float eps, cudaStream_t s);
// The same r and aug from a GEMM epilogue's per-tile row statistics (GemmEpi::ln_part):
// part[rows, tiles, 2] of (mean, M2) over the two chunk sets of tiles of tile_w columns
// (the last width - (tiles-1) tile_w).
sv_status ln_finalize_launch(const float2* part, int tiles, int tile_w, float* r, __half* aug, int rows, int width,
                             float eps, cudaStream_t s);
// W <- W * gamma (per column k, in place, F16); w_aug[n, 0..15] = (s_hi, s_lo, s_hi, 0, ...)
// with s = sum_k W'[n, k]; b_out[n] = b[n] (0 if null) + sum_k beta[k] W[n, k] (original W), F16.
sv_status fold_ln_launch(__half* W, const __half* gamma, const __half* beta, const __half* b, __half* w_aug,
                         __half* b_out, int N, int K, cudaStream_t s);
sv_status pack_patches_launch(const __half* img, __half* pix, int B, int side, int C, int p, cudaStream_t s);
sv_status pad_pixels_launch(const __half* pix, void* out, long rows, int P, int Kp, int out_e4m3, cudaStream_t s);
sv_status quantize_launch(const __half* x, uint8_t* y, size_t n, cudaStream_t s);
sv_status wait_probe_launch(unsigned int limit_us, cudaStream_t s);
sv_status map_attn_launch(const __half* q, const __half* kv, void* out, int B, int T, int H, float scale,
                          int out_e4m3, cudaStream_t s);

}  // namespace sv
