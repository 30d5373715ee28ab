/*
 * synth — seeded synthetic inputs for the So400m/14 SigLIP image encoder.
 *
 * This module is the ONE piece of code shared by the CUDA library and by the
 * CPU oracle that checks it. It holds no step of the network's arithmetic:
 * it only draws the random parameters and pixels that both sides consume,
 * already rounded to IEEE binary16 (the network stores every parameter in
 * F16, "SigLIP ViT benchmark" page, precision paragraph).
 *
 * Initialisation recipe ("SigLIP ViT benchmark" page, initialisation
 * paragraph, with the plainest reading of what it leaves open):
 *   - dense weights: Gaussian Xavier, std = sqrt(2 / (fan_in + fan_out)),
 *     fan_in = K (input width), fan_out = N (output width) of that matrix;
 *     a fused projection ([Wq|Wk|Wv], MAP [Wk|Wv]) keeps the per-slice
 *     variance, i.e. std = sqrt(2 / (D + D)) ("fused QKV" section);
 *   - biases: N(0, 0.01^2) ("tiny Gaussian values");
 *   - positional embedding and MAP probe: N(0, 1/D) (std 1/sqrt(width));
 *   - LayerNorm scale 1, bias 0;
 *   - pixels: uniform in [-1, 1], laid out [batch, 729, 588] with the 588
 *     values of a patch in (y, x, channel) order.
 *
 * Random numbers: SplitMix64 (Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014) used as a counter-based
 * generator. Stream key for a tag:  s = mix(seed ^ (0xD1B54A32D192ED03 * (tag + 1))).
 * Draw i of that stream:            x_i = mix(s + (i + 1) * 0x9E3779B97F4A7C15).
 * mix() is SplitMix64's output finaliser. Uniform: u_i = ((x_i >> 11) + 0.5) * 2^-53.
 * Normal i (Box-Muller, cosine branch): z_i = sqrt(-2 ln u_{2i}) * cos(2 pi u_{2i+1}).
 * Every value is computed in double and rounded once to F16 (round to nearest
 * even, overflow to infinity).
 *
 * Tensor order (tag = index below; D width, P patch values, T tokens, F MLP
 * width, L layers). Logical shapes are [fan_in, fan_out] = [K, N], row-major.
 *    0 patch_w [P,D]   1 patch_b [D]   2 pos [T,D]
 *    per layer l, tag 3 + 12 l + j:
 *      j=0 ln1_g [D]  1 ln1_b [D]  2 qkv_w [D,3D]  3 qkv_b [3D]  4 out_w [D,D]
 *      5 out_b [D]    6 ln2_g [D]  7 ln2_b [D]     8 fc1_w [D,F] 9 fc1_b [F]
 *      10 fc2_w [F,D] 11 fc2_b [D]
 *    then tag 3 + 12 L + j:
 *      j=0 enc_ln_g [D]  1 enc_ln_b [D]  2 probe [1,D]  3 map_q_w [D,D]  4 map_q_b [D]
 *      5 map_kv_w [D,2D] 6 map_kv_b [2D] 7 map_out_w [D,D] 8 map_out_b [D]
 *      9 map_ln_g [D]    10 map_ln_b [D] 11 map_fc1_w [D,F] 12 map_fc1_b [F]
 *      13 map_fc2_w [F,D] 14 map_fc2_b [D]
 * Pixels use tag 0x50495845 ("PIXE"); value k of token t of image b is draw
 * (b*T + t)*P + k, so a larger batch extends a smaller one.
 */
#ifndef SYNTH_H
#define SYNTH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int tokens;     /* T: patches per image (729 for 378x378 / 14) */
  int patch_dim;  /* P: values per patch (588 = 14*14*3) */
  int width;      /* D: 1152 */
  int heads;      /* H: 16 */
  int mlp;        /* F: 4304 */
  int layers;     /* L: 27 */
} synth_dims;

/* Distribution kinds */
enum { SYNTH_NORMAL = 0, SYNTH_CONST = 1 };

typedef struct {
  char name[32];
  int layer;      /* encoder layer index, or -1 */
  int rows;       /* K (fan_in); 1 for vectors */
  int cols;       /* N (fan_out) */
  int kind;       /* SYNTH_NORMAL or SYNTH_CONST */
  double mean;    /* constant value for SYNTH_CONST */
  double std;
} synth_tensor;

#define SYNTH_PIXEL_TAG 0x50495845ull

/* The So400m/14 @ 378 px dimensions. */
synth_dims synth_so400m(int layers);

int synth_tensor_count(const synth_dims* d);
/* Returns 0 on success, -1 for an id out of range. */
int synth_tensor_info(const synth_dims* d, int id, synth_tensor* out);

/* Fill a whole tensor (rows*cols values, logical row-major [K][N]) as F16 bits. */
int synth_fill_tensor_f16(uint64_t seed, const synth_dims* d, int id, uint16_t* out);
/* Same values, written transposed: out[n*K + k] = W[k][n] ([N][K], K-major), with each
   row padded to k_stride (>= K) elements; the padding is set to +0. */
int synth_fill_tensor_f16_t(uint64_t seed, const synth_dims* d, int id, uint16_t* out, int k_stride);

/* Pixels [batch][tokens][patch_dim] as F16 bits, uniform in [-1, 1]. */
void synth_pixels_f16(uint64_t seed, int batch, int tokens, int patch_dim, uint16_t* out);

/* Generic streams (also used by tests for per-op inputs). */
void synth_normal_f16(uint64_t seed, uint64_t tag, double mean, double std, uint16_t* out, size_t n);
void synth_uniform_f16(uint64_t seed, uint64_t tag, double lo, double hi, uint16_t* out, size_t n);
/* Draw i as a raw 64-bit value and as a double, for tests of the generator itself. */
uint64_t synth_draw_u64(uint64_t seed, uint64_t tag, uint64_t i);
double synth_draw_normal(uint64_t seed, uint64_t tag, uint64_t i);

/* IEEE binary16 round-to-nearest-even of a double (overflow -> inf). */
uint16_t synth_f16_from_double(double x);

#ifdef __cplusplus
}
#endif
#endif
