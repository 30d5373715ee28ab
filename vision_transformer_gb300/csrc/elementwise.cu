// Memory-bound kernels: LayerNorm, pixel staging, E4M3 quantisation and the
// single-query MAP attention, plus the bounded-wait self-test kernel.
#include <cuda_fp8.h>

#include "ptx.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(16.0f * a, 16.0f * b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(16.0f * c, 16.0f * d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

// LayerNorm, one half-warp per row ("SigLIP ViT benchmark", LayerNorm paragraph):
// mean, then the centred (biased) variance, both in F32 from the row held in
// registers, then the affine map. Each of the 16 lanes owns CPL chunks of 8 values
// (16-byte loads, all issued before any arithmetic); a 1152-wide row is 9 chunks
// per lane. With `res` set the row is first x + res (LayerNorm/Add paragraph: the
// residual add before the normalisation), added in F32 and rounded to F16 once; that
// sum is stored to x_out and normalised. With `stats_r` set only the row statistics are written:
// 1/sqrt(var + eps) to stats_r and, for the consuming GEMM's extra K block, the F16
// row (-mean_hi, -mean_hi, -mean_lo, 0...) to stats_aug (mean_hi + mean_lo = mean to
// about 2^-22 relative).
__device__ __forceinline__ float half_sum(float v) {  // over the 16 lanes of a half-warp
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int CPL>
__global__ void __launch_bounds__(256, CPL <= 9 ? 4 : 1) layernorm_kernel(const __half* x, const __half* __restrict__ res,
                                                        __half* x_out, const __half* __restrict__ g,
                                                        const __half* __restrict__ bta, void* __restrict__ y,
                                                        int rows, int width, float eps, int out_e4m3,
                                                        float* __restrict__ stats_r, __half* __restrict__ stats_aug) {
  pdl_launch_dependents();
  pdl_wait();
  const int hw = threadIdx.x >> 4, hl = threadIdx.x & 15;  // half-warp (row of the block), its lane
  const long row0 = long(blockIdx.x) * 16 + hw;
  const bool live = row0 < rows;
  const long row = live ? row0 : rows - 1;  // dead half-warps shadow a real row (no stores)
  const int chunks = width >> 3;
  const __half* xr = x + row * long(width);
  uint4 u[CPL];
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const int c = hl + 16 * i;
    u[i] = c < chunks ? *(reinterpret_cast<const uint4*>(xr) + c) : make_uint4(0u, 0u, 0u, 0u);
  }
  if (res) {  // x + res, rounded to F16, written back (each lane its own chunks)
    const __half* rr = res + row * long(width);
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int c = hl + 16 * i;
      if (c < chunks) {
        const uint4 ru = __ldg(reinterpret_cast<const uint4*>(rr) + c);
        __half2* xh = reinterpret_cast<__half2*>(&u[i]);
        const __half2* rh = reinterpret_cast<const __half2*>(&ru);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 a = __half22float2(xh[k]), b = __half22float2(rh[k]);
          xh[k] = __floats2half2_rn(a.x + b.x, a.y + b.y);
        }
        if (live) *(reinterpret_cast<uint4*>(x_out + row * long(width)) + c) = u[i];
      }
    }
  }
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const __half2* h = reinterpret_cast<const __half2*>(&u[i]);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __half22float2(h[k]);
      s += f.x + f.y;
    }
  }
  const float mean = half_sum(s) / float(width);
  // keep the row as packed halves between passes (re-converting is cheaper than
  // holding 8 CPL floats live)
#pragma unroll
  for (int i = 0; i < CPL; ++i) asm volatile("" : "+r"(u[i].x), "+r"(u[i].y), "+r"(u[i].z), "+r"(u[i].w));
  float q = 0.0f;
#pragma unroll
  for (int i = 0; i < CPL; ++i)
    if (hl + 16 * i < chunks) {
      const __half2* h = reinterpret_cast<const __half2*>(&u[i]);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __half22float2(h[k]);
        const float d0 = f.x - mean, d1 = f.y - mean;
        q = fmaf(d0, d0, q);
        q = fmaf(d1, d1, q);
      }
    }
  const float var = half_sum(q) / float(width);
  const float rstd = rsqrtf(var + eps);
  if (!live) return;
#pragma unroll
  for (int i = 0; i < CPL; ++i) asm volatile("" : "+r"(u[i].x), "+r"(u[i].y), "+r"(u[i].z), "+r"(u[i].w));
  if (stats_r) {  // statistics only: the normalisation is folded into the consuming GEMM
    if (hl < 2) {  // row of the GEMM's extra K block: (-mean_hi, -mean_hi, -mean_lo, 0, ...)
      const __half hi = __float2half_rn(-mean);
      const __half lo = __float2half_rn(-mean - __half2float(hi));
      const __half2 z = __float2half2_rn(0.0f);
      uint4 w;  // lane 0: columns 0..7, lane 1: columns 8..15
      __half2* h = reinterpret_cast<__half2*>(&w);
      h[0] = hl == 0 ? __halves2half2(hi, hi) : z;
      h[1] = hl == 0 ? __halves2half2(lo, __float2half_rn(0.0f)) : z;
      h[2] = h[3] = z;
      *reinterpret_cast<uint4*>(stats_aug + row * 16 + 8 * hl) = w;
    }
    if (hl == 0) stats_r[row] = rstd;
    return;
  }
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    const int c = hl + 16 * i;
    if (c < chunks) {
      const uint4 gu = __ldg(reinterpret_cast<const uint4*>(g) + c);
      const uint4 bu = __ldg(reinterpret_cast<const uint4*>(bta) + c);
      const __half2* xh = reinterpret_cast<const __half2*>(&u[i]);
      const __half2* gh = reinterpret_cast<const __half2*>(&gu);
      const __half2* bh = reinterpret_cast<const __half2*>(&bu);
      float o[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 xv = __half22float2(xh[k]), gv = __half22float2(gh[k]), bv = __half22float2(bh[k]);
        o[2 * k] = fmaf((xv.x - mean) * rstd, gv.x, bv.x);
        o[2 * k + 1] = fmaf((xv.y - mean) * rstd, gv.y, bv.y);
      }
      if (!out_e4m3) {
        uint4 w;
        __half2* wh = reinterpret_cast<__half2*>(&w);
#pragma unroll
        for (int k = 0; k < 4; ++k) wh[k] = __floats2half2_rn(o[2 * k], o[2 * k + 1]);
        *reinterpret_cast<uint4*>(static_cast<__half*>(y) + row * long(width) + 8 * c) = w;
      } else {
        uint2 w;
        w.x = e4m3x4(o[0], o[1], o[2], o[3]);
        w.y = e4m3x4(o[4], o[5], o[6], o[7]);
        *reinterpret_cast<uint2*>(static_cast<uint8_t*>(y) + row * long(width) + 8 * c) = w;
      }
    }
  }
}

// Whole images [B, side, side, C] f16 (channel fastest) -> patch rows
// [B, G*G, p*p*C] f16 with G = side / p ("SigLIP ViT benchmark", image-binding
// paragraph: [batch, patch_y, patch_x, y, x, channel] flattened): element
// k = (y p + x) C + c of token py G + px is pixel (py p + y, px p + x, c). A token's
// p*C-value run for one patch row y is contiguous in both layouts, so one thread
// moves two values (p*C is even for the 3-channel images of the path).
__global__ void pack_patches_kernel(const __half2* __restrict__ img, __half2* __restrict__ pix, long pairs, int side,
                                    int C, int p) {
  pdl_launch_dependents();
  pdl_wait();
  const long i = long(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= pairs) return;
  const int G = side / p, P = p * p * C, run = p * C;
  const long e = 2 * i;  // first output element of the pair
  const long row = e / P;
  const int k = int(e - row * P);
  const long b = row / (long(G) * G);
  const int t = int(row - b * G * G), py = t / G, px = t - (t / G) * G;
  const int y = k / run, r = k - y * run;  // r: offset inside the run of patch row y
  const long src = ((b * side + py * p + y) * long(side) + px * p) * C + r;
  pix[i] = img[src >> 1];
}

// Pixels [rows, P] f16 -> GEMM operand [rows, Kp] (f16 or e4m3 codes), zero
// columns P..Kp-1 (the K tail both GEMM operands share). One thread per 4 values.
__global__ void pad_pixels_kernel(const __half* __restrict__ pix, void* __restrict__ out, long rows, int P, int Kp,
                                  int out_e4m3) {
  pdl_launch_dependents();
  pdl_wait();
  const long i = long(blockIdx.x) * blockDim.x + threadIdx.x;
  const int cpr = Kp >> 2;
  if (i >= rows * cpr) return;
  const long row = i / cpr;
  const int c = int(i % cpr) * 4;
  uint2 u = make_uint2(0, 0);
  if (c < P) u = *reinterpret_cast<const uint2*>(pix + row * long(P) + c);
  if (!out_e4m3) {
    *reinterpret_cast<uint2*>(static_cast<__half*>(out) + row * long(Kp) + c) = u;
  } else {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(out) + row * long(Kp) + c) = e4m3x4(a.x, a.y, b.x, b.y);
  }
}

// y = e4m3 code of 16 x, 16 values per thread.
__global__ void quantize_kernel(const __half* __restrict__ x, uint8_t* __restrict__ y, size_t n16) {
  const size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n16) return;
  const uint4* src = reinterpret_cast<const uint4*>(x) + 2 * i;
  uint4 w;
  uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4 u = src[h];
    const __half2* hp = reinterpret_cast<const __half2*>(&u);
    const float2 a = __half22float2(hp[0]), b = __half22float2(hp[1]);
    const float2 c = __half22float2(hp[2]), d = __half22float2(hp[3]);
    wp[2 * h] = e4m3x4(a.x, a.y, b.x, b.y);
    wp[2 * h + 1] = e4m3x4(c.x, c.y, d.x, d.y);
  }
  reinterpret_cast<uint4*>(y)[i] = w;
}

// MAP attention: one learned query per head over the T tokens of one image
// ("SigLIP ViT benchmark": the probe's cross-attention). q: [D] f16 (the
// projected probe, shared by every image); kv: [B*T, 2D] f16 (K | V).
// One CTA of 128 threads per (head, image); scores and the F32 softmax in
// shared memory; the weighted V sum split over 14 key groups x 9 column groups.
constexpr int kMapThreads = 128;
constexpr int kMapKeyGroups = 14;

__global__ void __launch_bounds__(kMapThreads) map_attn_kernel(const __half* __restrict__ q,
                                                               const __half* __restrict__ kv, void* __restrict__ out,
                                                               int T, int D, float scale_log2, int out_e4m3) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ float sm[];
  float* s = sm;        // [T]
  float* red = sm + T;  // [kMapKeyGroups][72]
  __shared__ float qf[72];
  __shared__ float wred[4];
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < 72) qf[tid] = __half2float(q[h * 72 + tid]);
  __syncthreads();
  const size_t ld = size_t(2) * size_t(D);
  const __half* base = kv + size_t(b) * size_t(T) * ld;
  float mx = -INFINITY;
  for (int t = tid; t < T; t += kMapThreads) {
    const uint4* kr = reinterpret_cast<const uint4*>(base + size_t(t) * ld + size_t(h) * 72);
    float dot = 0.0f;
#pragma unroll
    for (int g = 0; g < 9; ++g) {
      const uint4 u = __ldg(kr + g);
      const __half2* hp = reinterpret_cast<const __half2*>(&u);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(hp[i]);
        dot = fmaf(f.x, qf[8 * g + 2 * i], dot);
        dot = fmaf(f.y, qf[8 * g + 2 * i + 1], dot);
      }
    }
    s[t] = dot * scale_log2;
    mx = fmaxf(mx, s[t]);
  }
  mx = warp_max(mx);
  if (lane == 0) wred[warp] = mx;
  __syncthreads();
  mx = fmaxf(fmaxf(wred[0], wred[1]), fmaxf(wred[2], wred[3]));
  __syncthreads();
  float sum = 0.0f;
  for (int t = tid; t < T; t += kMapThreads) {
    const float pv = ex2(s[t] - mx);
    s[t] = pv;
    sum += pv;
  }
  sum = warp_sum(sum);
  if (lane == 0) wred[warp] = sum;
  __syncthreads();
  const float l = (wred[0] + wred[1]) + (wred[2] + wred[3]);
  const int grp = tid / 9, cg = tid % 9;
  if (grp < kMapKeyGroups) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int t = grp; t < T; t += kMapKeyGroups) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(base + size_t(t) * ld + size_t(D) + size_t(h) * 72) + cg);
      const __half2* hp = reinterpret_cast<const __half2*>(&u);
      const float pt = s[t];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(hp[i]);
        acc[2 * i] = fmaf(pt, f.x, acc[2 * i]);
        acc[2 * i + 1] = fmaf(pt, f.y, acc[2 * i + 1]);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) red[grp * 72 + cg * 8 + i] = acc[i];
  }
  __syncthreads();
  if (tid < 72) {
    float a = 0.0f;
    for (int g2 = 0; g2 < kMapKeyGroups; ++g2) a += red[g2 * 72 + tid];
    a /= l;
    const size_t o = size_t(b) * size_t(D) + size_t(h) * 72 + tid;
    if (!out_e4m3)
      static_cast<__half*>(out)[o] = __float2half_rn(a);
    else
      static_cast<uint8_t*>(out)[o] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(16.0f * a, __NV_SATFINITE, __NV_E4M3));
  }
}

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// completes; the wait gives up after limit_ns, sets the device error word and
// the kernel returns normally.
__global__ void wait_probe_kernel(unsigned long long limit_ns, int* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
    mbar_wait(smem_u32(&bar), 0, &abort_flag, err, limit_ns);
    mbar_arrive(smem_u32(&bar));  // completes the phase so the barrier is left consistent
  }
}

// LayerNorm statistics from a GEMM epilogue's per-tile partials: each tile has two
// partials, over its 32-column chunks c = 0, 2, ... and c = 1, 3, ... (a partial
// covering no column is absent). kLanes consecutive lanes share a row: 8 for few rows
// (lane j loads the row's partials j, j + 8, ..., all before any arithmetic, so a row's
// loads are in flight together), 1 for many (a thread walks its row's partials in order;
// the other rows' threads hide the latency, and more lanes would only add arithmetic).
// A lane merges its partials, and the lanes' results are merged by shuffles,
// each merge being the pairwise update of Chan, Golub and LeVeque (1979): n = na + nb,
// d = mean_b - mean_a, mean = mean_a + d nb / n, M2 = M2a + M2b + d^2 na nb / n. Then
// var = M2 / width (biased, as the LayerNorm kernel) and the same r / aug outputs as its
// statistics mode.

template <int kLanes>
__global__ void __launch_bounds__(128) ln_finalize_kernel(const float2* __restrict__ part, int tiles, int tile_w,
                                                         float* __restrict__ r, __half* __restrict__ aug,
                                                         int rows, int width, float eps) {
  constexpr int kPerLane = (kMaxLnTiles + kLanes - 1) / kLanes;  // partials one lane may hold
  pdl_launch_dependents();
  pdl_wait();
  const int gt = int(blockIdx.x) * 128 + int(threadIdx.x);
  const int row = gt / kLanes, j = gt % kLanes;
  const bool live = row < rows;
  const int entries = 2 * tiles;
  const float2* pr = part + size_t(live ? row : 0) * size_t(entries);
  float n = 0.0f, mean = 0.0f, m2 = 0.0f;
  // columns of chunks h, h + 2, ... of tile t (the last chunk may be partial)
  auto cols_of = [&](int t, int h) {
    const int w = min(tile_w, width - t * tile_w), chunks = (w + 31) / 32, last = w - 32 * (chunks - 1);
    return 32 * ((chunks - h + 1) / 2) - (((chunks - 1) & 1) == h ? 32 - last : 0);
  };
  if constexpr (kLanes == 1) {
    if (live)
      for (int e = 0; e < entries; ++e) {
        const int cols = cols_of(e >> 1, e & 1);
        if (cols > 0) {
          const float2 q = __ldg(pr + e);
          chan_merge(n, mean, m2, float(cols), q.x, q.y);
        }
      }
  } else {
    float2 q[kPerLane];
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
      const int e = j + i * kLanes;
      q[i] = (live && e < entries) ? __ldg(pr + e) : make_float2(0.0f, 0.0f);
    }
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
      const int e = j + i * kLanes;
      if (!live || e >= entries) break;
      const int cols = cols_of(e >> 1, e & 1);
      if (cols > 0) chan_merge(n, mean, m2, float(cols), q[i].x, q[i].y);
    }
#pragma unroll
    for (int o = 1; o < kLanes; o <<= 1) {
      const float nb = __shfl_xor_sync(0xffffffffu, n, o), mb = __shfl_xor_sync(0xffffffffu, mean, o),
                  m2b = __shfl_xor_sync(0xffffffffu, m2, o);
      chan_merge(n, mean, m2, nb, mb, m2b);
    }
  }
  if (!live || j != 0) return;
  const float rstd = rsqrtf(m2 / float(width) + eps);
  const __half hi = __float2half_rn(-mean);
  const __half lo = __float2half_rn(-mean - __half2float(hi));
  const __half2 z = __float2half2_rn(0.0f);
  uint4 w;
  __half2* h = reinterpret_cast<__half2*>(&w);
  h[0] = __halves2half2(hi, hi);
  h[1] = __halves2half2(lo, __float2half_rn(0.0f));
  h[2] = h[3] = z;
  uint4* dst = reinterpret_cast<uint4*>(aug + size_t(row) * 16);
  dst[0] = w;
  dst[1] = make_uint4(0u, 0u, 0u, 0u);
  r[row] = rstd;
}

// LayerNorm folded into the linear map that consumes it: with y = (x - mu) r . g + be
// (r = 1/sqrt(var + eps)), y . W_n + b_n = r (x . W'_n - mu s_n) + b'_n where
// W'_nk = g_k W_nk (rounded to F16, in place), s_n = sum_k W'_nk and
// b'_n = b_n + sum_k be_k W_nk (stored in F16). The GEMM subtracts mu s_n as one
// extra K block: this row of it is (s_hi, s_lo, s_hi, 0, ...) against the LayerNorm
// input's (-mu_hi, -mu_hi, -mu_lo, 0, ...), so the tensor core adds -mu s exactly up
// to the dropped mu_lo s_lo term. One warp per output row n; sums in F32.
__global__ void __launch_bounds__(256) fold_ln_kernel(__half* __restrict__ W, const __half* __restrict__ g,
                                                      const __half* __restrict__ be, const __half* __restrict__ b,
                                                      __half* __restrict__ w_aug, __half* __restrict__ b_out, int N,
                                                      int K) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long n = long(blockIdx.x) * 8 + warp;
  if (n >= N) return;
  __half* wr = W + n * long(K);
  float s = 0.0f, t = 0.0f;
  for (int k = lane; k < K; k += 32) {
    const float w = __half2float(wr[k]);
    t = fmaf(__half2float(be[k]), w, t);
    const __half wg = __float2half_rn(w * __half2float(g[k]));
    wr[k] = wg;
    s += __half2float(wg);
  }
  s = warp_sum(s);
  t = warp_sum(t);
  if (lane < 2) {  // row of the extra K block: (s_hi, s_lo, s_hi, 0, ...)
    const __half hi = __float2half_rn(s);
    const __half lo = __float2half_rn(s - __half2float(hi));
    const __half2 z = __float2half2_rn(0.0f);
    uint4 u;
    __half2* h = reinterpret_cast<__half2*>(&u);
    h[0] = lane == 0 ? __halves2half2(hi, lo) : z;
    h[1] = lane == 0 ? __halves2half2(hi, __float2half_rn(0.0f)) : z;
    h[2] = h[3] = z;
    *reinterpret_cast<uint4*>(w_aug + n * 16 + 8 * lane) = u;
  }
  if (lane == 0) b_out[n] = __float2half_rn((b ? __half2float(b[n]) : 0.0f) + t);
}

template <int CPL>
void ln_launch(const __half* x, const __half* res, __half* x_out, const __half* g, const __half* b, void* y, int rows,
               int width, float eps, int out_e4m3, float* stats_r, __half* stats_aug, cudaStream_t s) {
  // a launch error stays pending for the caller's cudaGetLastError
  launch_pdl(layernorm_kernel<CPL>, dim3(unsigned((rows + 15) / 16)), dim3(256), 0, s, x, res, x_out, g, b, y, rows,
             width, eps, out_e4m3, stats_r, stats_aug);
}

}  // namespace

namespace {
sv_status ln_any(const __half* x, const __half* res, __half* x_out, const __half* g, const __half* b, void* y, int rows,
                 int width, float eps, int out_e4m3, float* stats_r, __half* stats_aug, cudaStream_t s) {
  const int cpl = (width / 8 + 15) / 16;  // 16-byte chunks per lane of a half-warp
  if (cpl <= 1) ln_launch<1>(x, res, x_out, g, b, y, rows, width, eps, out_e4m3, stats_r, stats_aug, s);
  else if (cpl <= 2) ln_launch<2>(x, res, x_out, g, b, y, rows, width, eps, out_e4m3, stats_r, stats_aug, s);
  else if (cpl <= 4) ln_launch<4>(x, res, x_out, g, b, y, rows, width, eps, out_e4m3, stats_r, stats_aug, s);
  else if (cpl <= 9) ln_launch<9>(x, res, x_out, g, b, y, rows, width, eps, out_e4m3, stats_r, stats_aug, s);
  else if (cpl <= 16) ln_launch<16>(x, res, x_out, g, b, y, rows, width, eps, out_e4m3, stats_r, stats_aug, s);
  else if (cpl <= 32) ln_launch<32>(x, res, x_out, g, b, y, rows, width, eps, out_e4m3, stats_r, stats_aug, s);
  else {
    set_error("layernorm: width %d too large", width);
    return SV_ERR_UNSUPPORTED;
  }
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SV_OK : cuda_fail(e, "layernorm launch");
}
}  // namespace

sv_status layernorm_launch(const __half* x, const __half* g, const __half* b, void* y, int rows, int width,
                           float eps, int out_e4m3, cudaStream_t s) {
  return ln_any(x, nullptr, nullptr, g, b, y, rows, width, eps, out_e4m3, nullptr, nullptr, s);
}

sv_status layernorm_residual_launch(__half* x, const __half* res, const __half* g, const __half* b, void* y, int rows,
                                    int width, float eps, int out_e4m3, cudaStream_t s) {
  return ln_any(x, res, x, g, b, y, rows, width, eps, out_e4m3, nullptr, nullptr, s);
}

sv_status ln_stats_launch(const __half* x, float* stats_r, __half* stats_aug, int rows, int width, float eps,
                          cudaStream_t s) {
  return ln_any(x, nullptr, nullptr, nullptr, nullptr, nullptr, rows, width, eps, 0, stats_r, stats_aug, s);
}

sv_status ln_finalize_launch(const float2* part, int tiles, int tile_w, float* r, __half* aug, int rows, int width,
                             float eps, cudaStream_t s) {
  if (tiles < 1 || 2 * tiles > kMaxLnTiles) {
    set_error("ln_finalize: %d column tiles (at most %d)", tiles, kMaxLnTiles / 2);
    return SV_ERR_UNSUPPORTED;
  }
  const bool few = rows < 16384;
  const long threads = long(rows) * (few ? 8 : 1);
  const dim3 grid(unsigned((threads + 127) / 128));
  cudaError_t e = few ? launch_pdl(ln_finalize_kernel<8>, grid, dim3(128), 0, s, part, tiles, tile_w, r, aug, rows,
                                   width, eps)
                      : launch_pdl(ln_finalize_kernel<1>, grid, dim3(128), 0, s, part, tiles, tile_w, r, aug, rows,
                                   width, eps);
  return e == cudaSuccess ? SV_OK : cuda_fail(e, "ln_finalize launch");
}

sv_status fold_ln_launch(__half* W, const __half* g, const __half* be, const __half* b, __half* w_aug, __half* b_out,
                         int N, int K, cudaStream_t s) {
  fold_ln_kernel<<<unsigned((N + 7) / 8), 256, 0, s>>>(W, g, be, b, w_aug, b_out, N, K);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SV_OK : cuda_fail(e, "fold_ln launch");
}

sv_status pack_patches_launch(const __half* img, __half* pix, int B, int side, int C, int p, cudaStream_t s) {
  const long pairs = long(B) * side * side * C / 2;
  cudaError_t e = launch_pdl(pack_patches_kernel, dim3(unsigned((pairs + 255) / 256)), dim3(256), 0, s,
                             reinterpret_cast<const __half2*>(img), reinterpret_cast<__half2*>(pix), pairs, side, C, p);
  return e == cudaSuccess ? SV_OK : cuda_fail(e, "pack_patches launch");
}

sv_status pad_pixels_launch(const __half* pix, void* out, long rows, int P, int Kp, int out_e4m3, cudaStream_t s) {
  const long n = rows * (Kp / 4);
  cudaError_t e = launch_pdl(pad_pixels_kernel, dim3(unsigned((n + 255) / 256)), dim3(256), 0, s, pix, out, rows, P, Kp,
                             out_e4m3);
  return e == cudaSuccess ? SV_OK : cuda_fail(e, "pad_pixels launch");
}

sv_status quantize_launch(const __half* x, uint8_t* y, size_t n, cudaStream_t s) {
  const size_t n16 = n / 16;
  if (n16 == 0) return SV_OK;
  quantize_kernel<<<unsigned((n16 + 255) / 256), 256, 0, s>>>(x, y, n16);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SV_OK : cuda_fail(e, "quantize launch");
}

sv_status wait_probe_launch(unsigned int limit_us, cudaStream_t s) {
  wait_probe_kernel<<<1, 32, 0, s>>>(1000ull * limit_us, dev_err());
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SV_OK : cuda_fail(e, "wait probe launch");
}

sv_status map_attn_launch(const __half* q, const __half* kv, void* out, int B, int T, int H, float scale,
                          int out_e4m3, cudaStream_t s) {
  const size_t smem = sizeof(float) * (size_t(T) + size_t(kMapKeyGroups) * 72);
  // the attribute is per device: the largest value set so far on each device
  static size_t attr[kMaxAttrDevices] = {};
  int dev = 0;
  cudaError_t de = cudaGetDevice(&dev);
  if (de != cudaSuccess) return cuda_fail(de, "cudaGetDevice(map_attn)");
  if (smem > 48 * 1024 && (dev < 0 || dev >= kMaxAttrDevices || smem > attr[dev])) {
    cudaError_t e = cudaFuncSetAttribute(map_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(map_attn)");
    if (dev >= 0 && dev < kMaxAttrDevices) attr[dev] = smem;
  }
  cudaError_t e = launch_pdl(map_attn_kernel, dim3(unsigned(H), unsigned(B)), dim3(kMapThreads), smem, s, q, kv, out, T,
                             H * 72, scale * 1.4426950408889634f, out_e4m3);
  return e == cudaSuccess ? SV_OK : cuda_fail(e, "map_attn launch");
}

}  // namespace sv
