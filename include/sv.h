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
 *   in_dtype SV_GEMM_F16: A, W f16; SV_GEMM_E4M3: A, W e4m3 codes and the
 *     caller passes scale = 2^-8 to undo the two 2^4 operand scales.
 *   bias: f16 [N] or NULL. pos: f16 [pos_rows, N] or NULL (added by row
 *     m % pos_rows: the positional embedding of the patch-embedding GEMM).
 *   residual: f16 [M, N] or NULL; it may alias C (each element is read
 *     before it is written, by the same thread).
 *   act: sv_act (applied before the residual add).
 *   out_dtype: SV_DT_F16, or SV_DT_E4M3 (codes of 16*y).
 * Requirements: M >= 1; N >= 16 and N % 16 == 0; K >= 16 and K % 16 == 0;
 * every pointer 16-byte aligned.
 * Errors: SV_ERR_INVALID_ARG, SV_ERR_CUDA.
 */
sv_status sv_gemm_bias_act(const void* A, const void* W, const void* bias, const void* pos, int pos_rows,
                           const void* residual, void* C, int M, int N, int K, int act, int in_dtype, int out_dtype,
                           float scale, void* stream);

/*
 * y = (x - mean) / sqrt(var + eps) * gamma + beta per row, mean and biased
 * centred variance in F32 ("SigLIP ViT benchmark", LayerNorm paragraph).
 * x: f16 [rows, width]; gamma, beta: f16 [width]; y: [rows, width] f16 or
 * e4m3 (out_dtype). Requirements: width % 8 == 0, 8 <= width <= 4096.
 */
sv_status sv_layernorm(const void* x, const void* gamma, const void* beta, void* y, int rows, int width, float eps,
                       int out_dtype, void* stream);

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
 * o_h = softmax(scale * Q_h K_h^T) V_h. Requirements: head_dim == 72,
 * tokens >= 1, heads >= 1.
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
 * Its scratch is one static device array of 8 MiB compiled into the library,
 * held by every GPU that loads the library until the process exits. With the
 * So400m/14 sizes that admits 1..256 images per call; larger batches (or
 * models whose scratch would not fit) are rejected with SV_ERR_INVALID_ARG.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before
 * any stream capture. All calls share the array: calls whose GPU work overlaps
 * (other streams or threads) race and must be serialised by the caller.
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

/* Frees the weights, workspaces and events; the library can be re-initialised. */
void sv_shutdown(void);

#ifdef __cplusplus
}
#endif
#endif /* SV_H */
