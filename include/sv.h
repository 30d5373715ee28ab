/*
 * sv.h — C ABI of the GB300 (sm_103a) SigLIP So400m/14 image-encoder library.
 *
 * The library runs the forward pass of the So400m/14 vision tower at 378 px
 * with MAP pooling, on one GPU, in hand-written CUDA kernels: tcgen05/TMEM
 * tensor-core GEMMs fed by TMA with fused epilogues, a fused flash-style
 * attention, a warp-per-row LayerNorm and a single-query MAP attention.
 *
 * What the network computes follows the "SigLIP ViT benchmark" page
 * (network paragraph, flowchart, precision paragraph, "fused QKV" section);
 * the pixel/embedding interface follows the "FP8 attention and resident
 * image/embedding transfers" page ("Host transfer mechanism": host-packed F16
 * patches in, an F16 embedding out).
 *
 * Conventions for every entry point:
 *  - Tensor pointers are DEVICE pointers owned by the caller (e.g. torch
 *    tensors), contiguous, row-major, and 16-byte aligned unless stated.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls are
 *    asynchronous: SV_OK means the work was enqueued. Asynchronous faults and
 *    device-side wait time-outs are reported by sv_sync().
 *  - Argument, shape and alignment violations return SV_ERR_INVALID_ARG or
 *    SV_ERR_UNSUPPORTED before anything is launched; nothing is reinterpreted
 *    silently (LayerNorm/Add paragraph: unsupported storage is rejected).
 *  - No C++ exception crosses this boundary. sv_last_error() describes the
 *    last failure on the calling thread.
 *  - Element types: "f16" is IEEE binary16. "e4m3" is the OCP FP8 E4M3 code
 *    (e4m3fn) of 16*x, i.e. the pages' FP8 operand at scale 2^-4: the stored
 *    byte q represents q * 2^-4 ("SigLIP ViT benchmark", FP8 example
 *    --fp8-scale=-4; saturating, round-to-nearest-even conversion).
 *  - The library works on the CUDA device that is current when it is first
 *    used; later calls must be made with that device current.
 */
#ifndef SV_H
#define SV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SV_OK = 0,
  SV_ERR_INVALID_ARG = 1,     /* bad pointer, size, alignment or enum value */
  SV_ERR_UNSUPPORTED = 2,     /* a shape/layout this library does not implement */
  SV_ERR_NOT_INITIALIZED = 3, /* weights not initialised (sv_init_*) */
  SV_ERR_CUDA = 4,            /* a CUDA runtime/driver call failed */
  SV_ERR_OOM = 5,             /* device or host allocation failed */
  SV_ERR_TIMEOUT = 6          /* a kernel gave up a bounded wait (see sv_sync) */
} sv_status;

typedef enum { SV_GEMM_F16 = 0, SV_GEMM_E4M3 = 1 } sv_gemm_dtype;
typedef enum { SV_DT_F16 = 0, SV_DT_E4M3 = 1 } sv_dtype;
typedef enum { SV_ACT_NONE = 0, SV_ACT_GELU_TANH = 1 } sv_act;

/* ---------------------------------------------------------------- weights */

/*
 * Draws the full So400m/14 parameter set (27 layers + MAP head; 428 M
 * parameters) from `seed` with the generator in synth/synth.h (Gaussian
 * Xavier weights, N(0, 0.01^2) biases, N(0, 1/1152) positional embedding and
 * probe, LayerNorm scale 1 and bias 0: "SigLIP ViT benchmark", initialisation
 * paragraph), rounds them to F16 and uploads them to the current device,
 * together with an E4M3 copy of every dense-GEMM weight (codes of 16 w).
 * The weights are library-owned and resident until sv_shutdown() or the next
 * sv_init_*; re-initialisation frees the previous set. Synchronous.
 * Errors: SV_ERR_OOM, SV_ERR_CUDA.
 */
sv_status sv_init_weights(uint64_t seed);

/*
 * Same as sv_init_weights for other widths of the same graph, e.g. the pages'
 * reduced "vit-small" graph (tokens 4, width 144, 2 heads, MLP 288) or the
 * four-token full-width diagnostic (tokens 4, width 1152, 16 heads, MLP 4304)
 * ("SigLIP ViT benchmark", --vit-small paragraph and "four-token diagnostic").
 * Requirements: width == heads * 72 (head width 72, the only head width the
 * attention kernel implements), width % 16 == 0, width <= 4096, mlp % 16 == 0,
 * patch_dim % 4 == 0, 1 <= patch_dim <= 4096, 1 <= tokens, 1 <= layers <= 64.
 * Errors: SV_ERR_UNSUPPORTED for other shapes; SV_ERR_OOM, SV_ERR_CUDA.
 */
sv_status sv_init_weights_dims(uint64_t seed, int tokens, int patch_dim, int width, int heads, int mlp,
                               int layers);

/* Model dimensions of the resident weights (any pointer may be NULL). */
sv_status sv_model_dims(int* tokens, int* patch_dim, int* width, int* heads, int* mlp, int* layers);

/*
 * Number of parameter values of the resident model (0 before sv_init_*): the
 * sum over its tensors of rows x cols, in the tensor order of synth/synth.h.
 */
size_t sv_weights_count(void);

/*
 * Copies the resident parameters back to the host: every tensor in the order
 * of synth/synth.h, each in its logical row-major layout ([fan_in, fan_out] for
 * a dense weight, i.e. the transpose of the [N, K] copy the GEMMs read; the K
 * padding of the patch weight is left out), each F16 value widened to F32
 * exactly. This is what the pages' resident loop saves as its reference
 * weights ("FP8 attention and resident image/embedding transfers", Resident
 * inference loop). The QKV and MLP-up weights are resident with their
 * LayerNorm scale folded in (gamma_k W[k][n], rounded to F16 once), which is W
 * itself for the scale-1 initialisation.
 * host_dst: caller-owned host memory of at least n_floats = sv_weights_count()
 * values. Synchronous. Errors: SV_ERR_NOT_INITIALIZED; SV_ERR_INVALID_ARG if
 * host_dst is NULL or n_floats is too small; SV_ERR_CUDA.
 */
sv_status sv_export_weights(float* host_dst, size_t n_floats);

/* Number of bytes sv_export_weights_e4m3 writes (0 before sv_init_*). */
size_t sv_weights_count_e4m3(void);

/*
 * Copies the E4M3 copies of the resident weights back to the host: the dense
 * weights and the MAP probe (the tensors an E4M3 GEMM reads), in the order of
 * synth/synth.h, each in its logical row-major layout as in sv_export_weights,
 * one E4M3 code of 16 w per byte. host_dst: at least sv_weights_count_e4m3()
 * bytes. Synchronous. Errors: as sv_export_weights.
 */
sv_status sv_export_weights_e4m3(uint8_t* host_dst, size_t n_bytes);

/* ---------------------------------------------------------------- forward */

/*
 * The whole forward pass: pixels [batch, tokens, patch_dim] f16 (patches in
 * [patch_y, patch_x, y, x, channel] order: "SigLIP ViT benchmark", image
 * binding paragraph) -> out [batch, 1, width] f16 (the pooled embedding with
 * its singleton probe axis). Runs the patch-embedding GEMM with bias and
 * positional embedding, the first `layers` encoder layers (1..L of the
 * resident weights), the final LayerNorm and MAP pooling.
 * gemm_dtype SV_GEMM_F16: F16 operands, F32 accumulation. SV_GEMM_E4M3: every
 * dense-GEMM operand in E4M3 at scale 2^-4 (activations quantised by the
 * kernel that produces them), F32 accumulation; LayerNorm statistics,
 * softmax and attention accumulation stay F32 and the residual stream F16 in
 * both modes ("SigLIP ViT benchmark", precision paragraph). With F16 the
 * encoder's LayerNorms are folded into the QKV and MLP-up projections (gamma in
 * the weights, beta in the bias, the mean subtracted by the tensor core, 1/std
 * in the epilogue), their row statistics taken from the epilogues of the GEMMs
 * that write the residual stream.
 * `pixels` needs only 8-byte alignment. The first call at a given batch size
 * and gemm_dtype allocates and caches a device workspace (freed by
 * sv_shutdown); later calls allocate nothing.
 * Launches: the first call with given (pixels, out, batch, layers, gemm_dtype,
 * flags) launches its kernels one by one; the second captures the same launch
 * sequence into a CUDA graph (on an internal stream) and later calls with the
 * same arguments launch that graph on `stream`: one host call per step, with
 * identical results. The graphs name the caller's buffers by address, so a
 * buffer freed and reallocated at the same address must keep its role; the
 * graphs are dropped by sv_init_weights and sv_shutdown. Calls made while
 * profiling is on (sv_profile_enable), or on a stream the caller is capturing
 * into a graph of its own, launch one by one.
 * Errors: SV_ERR_NOT_INITIALIZED, SV_ERR_INVALID_ARG, SV_ERR_OOM, SV_ERR_CUDA.
 */
sv_status sv_encode(const void* pixels, void* out, int batch, int layers, int gemm_dtype, void* stream);

/* Options of sv_encode_ex. */
typedef enum {
  /* Q, K and V as three 1152 -> 1152 GEMMs over the row slices of the fused
   * weight instead of one 1152 -> 3456 GEMM (the pages' fused-QKV comparison:
   * "Fused QKV projection" section, which measured fusion as about 7.6% faster).
   * The results are the same; only the launch structure differs. */
  SV_ENCODE_UNFUSED_QKV = 1,
  /* FP8 attention products ("FP8 attention and resident image/embedding
   * transfers", Projected attention and Full 27-layer ViT): every encoder
   * layer's scores S = Q K^T are computed on E4M3 operands at scale 2^-4
   * (Q and K written as E4M3(16 x) by the QKV projection's epilogue, the
   * producer-side quantisation those pages name as the profitable form).
   * Softmax, the P V product (F16) and the output precision are unchanged; the
   * MAP head's single-query attention is not affected. Combines with either
   * gemm_dtype. */
  SV_ENCODE_FP8_ATTENTION = 2,
  /* Launch the kernels one by one on every call (no step graph; see sv_encode).
   * The results are the same. */
  SV_ENCODE_EAGER = 4
} sv_encode_flags;

/*
 * sv_encode with options: flags is 0 (exactly sv_encode) or any OR of
 * SV_ENCODE_UNFUSED_QKV, SV_ENCODE_FP8_ATTENTION and SV_ENCODE_EAGER.
 * Each (batch, gemm_dtype, flags without SV_ENCODE_EAGER) combination has its
 * own cached workspace.
 * Errors: as sv_encode; unknown flag bits -> SV_ERR_INVALID_ARG.
 */
sv_status sv_encode_ex(const void* pixels, void* out, int batch, int layers, int gemm_dtype, int flags,
                       void* stream);

/*
 * Packs whole images into the patch rows sv_encode takes ("SigLIP ViT
 * benchmark", image-binding paragraph: the host-side step that views an image
 * as [batch, patch_y, patch_x, y, x, channel] and flattens it to [batch, 729,
 * 588]), on the GPU. images: f16 [batch, image_side, image_side, channels]
 * (row-major, channel fastest; normalisation stays with the caller, as on the
 * pages); pixels: f16 [batch, (image_side/patch)^2, patch*patch*channels] with
 * element (y*patch + x)*channels + c of token py*(image_side/patch) + px equal
 * to pixel (py*patch + y, px*patch + x, c). For So400m/14 at 378 px:
 * image_side 378, channels 3, patch 14 -> [batch, 729, 588]. A pure layout change.
 * Requirements: image_side % patch == 0; patch*channels even; pointers 4-byte
 * aligned. Errors: SV_ERR_INVALID_ARG, SV_ERR_CUDA.
 */
sv_status sv_pack_patches(const void* images, void* pixels, int batch, int image_side, int channels, int patch,
                          void* stream);

/* ---------------------------------------------------------------- per-op */

/*
 * C[M,N] = out_cast( act(scale * (A[M,K] . W[N,K]^T) + bias[N] + pos[m % pos_rows, N]) + residual[M,N] )
 * A dense projection with its fused epilogue ("SigLIP ViT benchmark":
 * projections with bias, GELU, residual adds). W is stored [N, K] (K-major,
 * i.e. the transpose of the logical [fan_in, fan_out] weight).
 *   scale = scale_a * scale_w, the dequantisation scales of the two operands.
 *   in_dtype SV_GEMM_F16: A, W f16 (scales 1); SV_GEMM_E4M3: A, W e4m3 codes of
 *     16 a and 16 w, so the caller passes scale_a = scale_w = 2^-4.
 *   bias: f16 [N] or NULL. pos: f16 [pos_rows, N] or NULL (added by row
 *     m % pos_rows: the positional embedding of the patch-embedding GEMM).
 *   residual: f16 [M, N] or NULL; it may alias C (each element is read
 *     before it is written, by the same thread).
 *   act: sv_act (applied before the residual add).
 *   out_dtype: SV_DT_F16, or SV_DT_E4M3 (codes of 16*y).
 * With K >= 2048 the GEMM may split K into ranges: at small M every output tile
 * (e.g. the 729 x 1152 x 4304 MLP-down projection of one image), otherwise, with F16
 * operands, the tiles of a short last round of its tile schedule (e.g. 23,328 rows).
 * Two launches; the ranges' F32 partial sums go to a library-owned device buffer that
 * grows to the largest need seen (a cudaMalloc on such a call; freed by sv_shutdown)
 * and are added in a fixed order, so repeated calls give identical bits. Calls on
 * different streams that split K share that buffer and must not overlap.
 * Requirements: M >= 1; N >= 16 and N % 16 == 0; K >= 16 and K % 16 == 0;
 * every pointer 16-byte aligned.
 * Errors: SV_ERR_INVALID_ARG, SV_ERR_OOM, SV_ERR_CUDA.
 */
sv_status sv_gemm_bias_act(const void* A, const void* W, const void* bias, const void* pos, int pos_rows,
                           const void* residual, void* C, int M, int N, int K, int act, int in_dtype, int out_dtype,
                           float scale_a, float scale_w, void* stream);

/*
 * y = (x - mean) / sqrt(var + eps) * gamma + beta per row, mean and biased
 * centred variance in F32 ("SigLIP ViT benchmark", LayerNorm paragraph), with an
 * optional residual add in front ("SigLIP ViT benchmark", LayerNorm/Add
 * paragraph: the residual adds of the encoder; "Performance follow-up": LN and
 * Add as the follow-up targets).
 * x: f16 [rows, width]. residual: f16 [rows, width] or NULL; when given, each
 *   row is first replaced by x + residual (added in F32, rounded to F16 once),
 *   which is written back to x, and y is the LayerNorm of that F16 sum.
 * gamma, beta: f16 [width]; y: [rows, width] f16 or e4m3 (out_dtype); y must
 * not overlap x or residual. Requirements: width % 8 == 0, 8 <= width <= 4096;
 * pointers 16-byte aligned.
 */
sv_status sv_layernorm(void* x, const void* residual, const void* gamma, const void* beta, void* y, int rows,
                       int width, float eps, int out_dtype, void* stream);

/*
 * C[M,N] = act(LayerNorm(x)[M,K] . W[N,K]^T + bias[N]), F16 in and out: a
 * pre-normalised projection ("SigLIP ViT benchmark": the LN1 -> QKV and
 * LN2 -> MLP-up pairs of each layer) with the LayerNorm folded into the GEMM
 * instead of written out: the row mean and 1/sqrt(var + eps) (F32, centred
 * variance) come from a statistics pass over x, W is scaled by gamma, and the
 * epilogue applies r (x . W' - mean * colsum(W')) + bias + W . beta in F32 before
 * the activation. This is what sv_encode runs in F16 mode.
 * x: f16 [M, K]; gamma, beta: f16 [K]; W: f16 [N, K] (K-major); bias: f16 [N]
 * or NULL; C: f16 [M, N]; act: sv_act.
 * Requirements: M >= 1; N, K multiples of 16; K <= 4096; pointers 16-byte
 * aligned. The call keeps a scratch buffer (scaled weights and statistics) that
 * grows to the largest call and is freed by sv_shutdown.
 * Errors: SV_ERR_INVALID_ARG, SV_ERR_OOM, SV_ERR_CUDA.
 */
sv_status sv_ln_gemm(const void* x, const void* gamma, const void* beta, float eps, const void* W, const void* bias,
                     void* C, int M, int N, int K, int act, void* stream);

/*
 * Multi-head self-attention with F32 softmax and accumulation ("SigLIP ViT
 * benchmark", precision paragraph; padding is never read as data: "SigLIP
 * optimized execution and PV padding", cause and fix).
 * qkv: f16 [batch, tokens, 3 * heads * head_dim], the fused projection output:
 *   columns [Q | K | V], head h at columns h*head_dim .. h*head_dim+head_dim-1
 *   inside each third ("fused QKV" section: slices with head views).
 * o: [batch, tokens, heads * head_dim] f16 or e4m3 (out_dtype), head h at
 *   columns h*head_dim.. (heads concatenated).
 * o_h = softmax(scale * Q_h K_h^T) V_h; scale <= 0 selects 1 / sqrt(head_dim)
 * (scaled dot-product attention). Requirements: head_dim == 72, tokens >= 1,
 * heads >= 1. The call keeps a scratch buffer (the head-blocked copy of qkv) that
 * grows to the largest call and is freed by sv_shutdown. One of two kernels with the
 * same arithmetic runs, chosen by the launch's size (sv_debug_attention_plan).
 */
sv_status sv_attention(const void* qkv, void* o, int batch, int heads, int tokens, int head_dim, float scale,
                       int out_dtype, void* stream);

/* Options of sv_attention_ex. */
typedef enum {
  /* Scores on E4M3 operands: Q and K rounded to E4M3 at scale 2^-4 (stored as
   * E4M3(16 x)) before S = Q K^T ("FP8 attention and resident image/embedding
   * transfers", Projected attention); everything else as sv_attention. */
  SV_ATTENTION_QK_E4M3 = 1
} sv_attention_flags;

/*
 * sv_attention with options: flags is 0 (exactly sv_attention) or
 * SV_ATTENTION_QK_E4M3. Errors: as sv_attention; unknown flag bits ->
 * SV_ERR_INVALID_ARG.
 */
sv_status sv_attention_ex(const void* qkv, void* o, int batch, int heads, int tokens, int head_dim, float scale,
                          int out_dtype, int flags, void* stream);

/*
 * The same attention with Q, K and V given per head: q, k, v: f16 [batch, heads,
 * tokens, head_stride], head_stride >= head_dim values per row of which the
 * first head_dim are used (e.g. 80: the head width 72 padded to the tensor
 * core's step; the pad values are never read). o, scale, out_dtype and flags as
 * in sv_attention_ex. Requirements: head_dim == 72, head_stride % 8 == 0,
 * head_stride <= 4096; pointers 16-byte aligned.
 */
sv_status sv_attention_heads(const void* q, const void* k, const void* v, void* o, int batch, int heads, int tokens,
                             int head_dim, int head_stride, float scale, int out_dtype, int flags, void* stream);

/*
 * MAP pooling head with the resident weights ("SigLIP ViT benchmark":
 * shared learned probe, its own Q projection, the fused KV projection,
 * multi-head cross-attention, output projection, LayerNorm/MLP residual).
 * x: f16 [batch, tokens, width], the final-LayerNorm output. out: f16
 * [batch, 1, width]. gemm_dtype as in sv_encode (with E4M3 the input is
 * quantised first).
 */
sv_status sv_map_pool(const void* x, void* out, int batch, int gemm_dtype, void* stream);

/*
 * sv_map_pool without any device allocation by the library. The pages have no
 * counterpart: this entry point exists for callers that cannot let a library
 * call cudaMalloc at run time, e.g. a framework whose caching allocator or
 * pre-sized pool owns the device memory, or a service with a fixed memory
 * budget. Same arguments, computation and results as sv_map_pool (it uses the
 * resident weights of sv_init_weights, which the caller sets up beforehand);
 * images are pooled one at a time, so it is slower for large batches.
 * Its scratch is one static device array of 8 MiB compiled into the library.
 * The array is placed in a device's memory when the library's code is loaded
 * into that device's context (with CUDA's default lazy loading, at the first
 * sv_map_pool_static call on the device) and stays there until the context is
 * destroyed. With the So400m/14 sizes that admits 1..256 images per call;
 * larger batches (or models whose scratch would not fit) are rejected with
 * SV_ERR_INVALID_ARG. The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current and keeps it; make
 * that first call before any stream capture. sv_shutdown forgets the kept
 * addresses: a caller that resets or destroys a device's context must call
 * sv_shutdown before doing so. All calls share the array, and it keeps the
 * previous call's contents: calls whose GPU work overlaps (other streams or
 * threads) race on it and must be serialised by the caller.
 */
sv_status sv_map_pool_static(const void* x, void* out, int batch, int gemm_dtype, void* stream);

/* y[i] = e4m3 code of 16 * x[i] (saturating, round to nearest even); x f16, n % 16 == 0. */
sv_status sv_quantize_e4m3(const void* x, void* y, size_t n, void* stream);

/* ---------------------------------------------------------------- utilities */

/* Pixels [batch, tokens, patch_dim] f16 uniform in [-1, 1] from `seed` (synth/synth.h), written to dev_dst. */
sv_status sv_make_pixels(uint64_t seed, int batch, void* dev_dst, void* stream);

/*
 * Waits for `stream`, then reports any asynchronous CUDA error and the
 * library's device error word: SV_ERR_TIMEOUT if a kernel gave up a bounded
 * wait (the kernel then returned without finishing; its outputs are
 * undefined). Clears the error word.
 */
sv_status sv_sync(void* stream);

/* Thread-local description of the last error; valid until the next call on this thread. */
const char* sv_last_error(void);

/* Number of kernels the library has launched since the last call (and resets the count). */
long long sv_launch_count(void);

/*
 * Kernel timing for roofline reports. While enabled, each library launch is
 * bracketed by CUDA events on its stream. sv_profile_read returns, for one
 * kernel class (0 GEMM, 1 attention, 2 LayerNorm, 3 MAP attention, 4 other),
 * the summed device milliseconds, the algorithmic FLOPs and bytes of those
 * launches and their count, then resets that class. It synchronises the device.
 */
sv_status sv_profile_enable(int on);
sv_status sv_profile_read(int kind, double* ms, double* flops, double* bytes, long long* launches);

/* ---------------------------------------------------------------- test hooks */

/*
 * Fills the cached sv_encode workspace for (batch, gemm_dtype) with
 * `byte_value` (creating it if needed), so a test can show that no kernel
 * reads a buffer it has not written in the same call (0xFF makes every F16
 * and E4M3 value a NaN). This is the device analogue of the pages' NaN-poison
 * experiments ("Profile layout diagnosis": NaN in padding tails turned every
 * output NaN). Synchronous.
 */
sv_status sv_debug_fill_workspace(int batch, int gemm_dtype, int byte_value);

/*
 * Launches a one-thread kernel that waits on an mbarrier nothing completes,
 * with the given limit (1 us .. 2 s). The wait gives up, sets the device error
 * word and the kernel returns, so the next sv_sync reports SV_ERR_TIMEOUT and
 * the context stays usable. Exercises the bounded-wait path every kernel uses.
 */
sv_status sv_debug_wait_timeout(unsigned int limit_us, void* stream);

/*
 * The launch plan sv_gemm_bias_act / sv_encode give an M x N x K GEMM on a GPU with
 * `sms` SMs, computed on the host alone (no device needed): out[0..7] = tile width,
 * CTA pairs (0/1), 128-byte rows of K per pipeline stage, width of a narrower last
 * column tile (0: none), narrow tiles scheduled last (0/1), K ranges (1: K not split),
 * pipeline stages per K range, and the tiles that run whole before the split ones (0
 * with a split: every tile split). *ws_bytes (if not NULL): the split-K partial-sum
 * workspace. max_splits: 1 as for a caller without a workspace, 8 as sv_encode and
 * sv_gemm_bias_act use. gemm_dtype: sv_gemm_dtype. Errors: SV_ERR_INVALID_ARG.
 */
sv_status sv_debug_gemm_plan(int M, int N, int K, int gemm_dtype, int sms, int max_splits, int* out,
                             size_t* ws_bytes);

/*
 * Attention kernels ("SigLIP ViT benchmark", attention paragraph: softmax(Q K^T / sqrt(72)) V
 * per head). Every attention launch (sv_attention*, sv_encode) runs one of two kernels with
 * the same arithmetic: 1 = items of two 128-query tiles per CTA, 2 = items of one 128-query
 * tile with three score tiles in tensor memory. By size (choice 0, the default) the second
 * runs when all of a launch's one-tile items, ceil(tokens / 128) x heads x batch, fit in one
 * round of the SMs (one image of 729 tokens and 16 heads: 96 items), the first otherwise.
 * sv_debug_attention_kernel(1 or 2) forces one kernel for later launches of this process,
 * for tests that cover both on the same sizes; step graphs that sv_encode captured before
 * keep the kernel they were captured with. Errors: SV_ERR_INVALID_ARG (choice not 0, 1, 2).
 */
sv_status sv_debug_attention_kernel(int choice);

/*
 * The kernel (*kernel: 1 or 2, as above) and the number of persistent CTAs (*grid) that an
 * attention launch over `batch` images of `tokens` tokens and `heads` heads takes on a GPU
 * with `sms` SMs under the current choice; computed on the host alone (no device needed).
 * Errors: SV_ERR_INVALID_ARG (a size < 1, or a NULL output).
 */
sv_status sv_debug_attention_plan(int batch, int tokens, int heads, int sms, int* kernel, int* grid);

/* Stages of the forward pass that sv_debug_encode_stage can stop after. */
typedef enum {
  SV_STAGE_PATCH = 0,     /* X after the patch embedding: f16 [batch*tokens, width] */
  SV_STAGE_QKV = 1,       /* [Q | K | V] of the last layer, row-major f16 [batch*tokens, 3*width] */
  SV_STAGE_ATTENTION = 2, /* attention output O of the last layer: [batch*tokens, width] */
  SV_STAGE_OUT_PROJ = 3,  /* X after the output projection + residual of the last layer (f16) */
  SV_STAGE_MLP_UP = 4,    /* GELU output of the last layer's MLP: [batch*tokens, mlp] */
  SV_STAGE_MLP_DOWN = 5,  /* X after the last layer (f16) */
  SV_STAGE_FINAL_LN = 6   /* output of the final LayerNorm: [batch*tokens, width] */
} sv_stage;

/*
 * Test hook for per-stage parity: runs sv_encode_ex's launches one by one for
 * `batch` images through `layers` layers, stops after `stage` (of the last
 * layer), and copies that stage's output tensor into dst (caller-owned device
 * memory of at least dst_bytes; the sizes and types are in sv_stage: f16, or for
 * O, the MLP hidden and the final LayerNorm with gemm_dtype SV_GEMM_E4M3 the
 * e4m3 codes the next GEMM reads). SV_STAGE_QKV with SV_ENCODE_FP8_ATTENTION
 * (E4M3 Q and K) is not supported. Uses the cached workspace of
 * (batch, gemm_dtype, flags) and the caller's stream; the output buffer of
 * sv_encode is not written.
 * Errors: as sv_encode_ex; SV_ERR_INVALID_ARG if dst_bytes is too small.
 */
sv_status sv_debug_encode_stage(const void* pixels, int batch, int layers, int gemm_dtype, int flags, int stage,
                                void* dst, size_t dst_bytes, void* stream);

/* Frees the weights, workspaces and events; the library can be re-initialised. */
void sv_shutdown(void);

#ifdef __cplusplus
}
#endif
#endif /* SV_H */
