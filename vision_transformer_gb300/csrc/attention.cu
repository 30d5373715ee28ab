// Fused multi-head self-attention for head width 72 on the tcgen05 tensor cores.
//
// o_h = softmax(scale * Q_h K_h^T) V_h per image and head, F16 operands, F32
// scores, softmax and accumulation, F16 (or E4M3) result ("SigLIP ViT
// benchmark", precision paragraph: F32 softmax/accumulation state, result
// converted back to F16). The 729 x 729 score matrix never leaves the SM
// (flash-style online softmax), which replaces the pages' materialised and
// blocked-merge forms.
//
// Padding contract ("SigLIP optimized execution and PV padding", cause and
// fix: padding columns were once read as data and turned outputs into NaN):
//   - head width 72 is padded to 80 for the MMA K / N steps; the pad columns
//     of every operand tile in shared memory are written as zeros once at
//     kernel start and never loaded from memory;
//   - rows past the image's last token come from the TMA out-of-bounds fill
//     (zeros; the tensor map is bounded per image), and keys past the last
//     token are masked to -inf before the row maximum, so their probability
//     is exactly 0;
//   - query rows past the last token are computed but never stored.
//
// CTA = (128-query tile, head, image), 192 threads:
//   warp 0      TMA: Q once, then K and V tiles of 128 keys into 2 stages;
//   warp 1      TMEM owner + MMA issuer: S_j = Q K_j^T (M 128, N 128, K 80)
//               into TMEM, and O_j = P_j V_j (M 128, N 80, K 128) into TMEM;
//   warps 2..5  softmax: one thread per query row reads its S row from TMEM,
//               writes P_j (F16) to shared memory, and folds O_j into an F32
//               register accumulator with the online-softmax rescale.
// Operand tiles use the no-swizzle core-matrix layout: [column group of 8]
// [row][8 values], i.e. 8x16-byte core matrices, 128 B apart along rows and
// 2048 B apart along the 8-column groups.
#include <cuda_fp8.h>

#include "ptx.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kDh = 72;                      // head width
constexpr int kGroups = 9;                   // 72 / 8 column groups loaded from memory
constexpr int kTileRows = 128;               // queries per CTA, keys per step
constexpr int kGroupBytes = kTileRows * 16;  // 2048: one column group of a tile
constexpr int kOpBytes = 10 * kGroupBytes;   // 80 columns (72 + zero pad)
constexpr int kPBytes = 16 * kGroupBytes;    // 128 keys of probabilities
constexpr int kThreads = 192;

// Shared memory map (offsets from the 1024-aligned base).
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kOpBytes;      // 2 stages
constexpr int kOffV = kOffK + 2 * kOpBytes;  // 2 stages
constexpr int kOffP = kOffV + 2 * kOpBytes;  // 2 buffers
constexpr int kOffBar = kOffP + 2 * kPBytes;
constexpr int kSmem = 1024 + kOffBar + 256;

// TMEM columns: S0 0, S1 128, O0 256, O1 384.
constexpr uint32_t kTmemCols = 512;

struct Params {
  int T, H, D;
  float scale_log2;  // scale * log2(e)
  void* out;
  int out_e4m3;
  int* err;
};

// Barrier indices (8 bytes each).
enum {
  kBarQ = 0,
  kBarKFull = 1,    // +stage
  kBarVFull = 3,    // +stage
  kBarKVEmpty = 5,  // +stage
  kBarSFull = 7,    // +buffer
  kBarSEmpty = 9,   // +buffer
  kBarPFull = 11,   // +buffer
  kBarOFull = 13,   // +buffer
  kBarOEmpty = 15,  // +buffer
  kBarDrain = 17,
  kNumBars = 18
};

__global__ void __launch_bounds__(kThreads, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tm, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kOffBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto bar = [&](int i) { return bar0 + 8u * uint32_t(i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int T = p.T, D = p.D;
  const int nkv = (T + kTileRows - 1) / kTileRows;

  // Zero the pad column group (columns 72..79) of Q and of both K and V stages.
  for (int i = threadIdx.x; i < 5 * (kGroupBytes / 16); i += kThreads) {
    const int t = i / (kGroupBytes / 16), w = i % (kGroupBytes / 16);
    const int off = (t == 0 ? kOffQ : (t <= 2 ? kOffK + (t - 1) * kOpBytes : kOffV + (t - 3) * kOpBytes));
    reinterpret_cast<uint4*>(smem + off + kGroups * kGroupBytes)[w] = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQ), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarKVEmpty + s), 1);
      mbar_init(bar(kBarSFull + s), 1);
      mbar_init(bar(kBarSEmpty + s), 128);  // every softmax thread arrives
      mbar_init(bar(kBarPFull + s), 128);
      mbar_init(bar(kBarOFull + s), 1);
      mbar_init(bar(kBarOEmpty + s), 128);
    }
    mbar_init(bar(kBarDrain), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) prefetch_tmap(&tm);
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // Q tile: columns h*72 .. h*72+71 of the Q third, tokens qt*128 ..
      mbar_arrive_expect_tx(bar(kBarQ), kGroups * kGroupBytes);
      for (int g = 0; g < kGroups; ++g)
        tma_load_3d(sbase + kOffQ + g * kGroupBytes, &tm, bar(kBarQ), h * kDh + 8 * g, qt * kTileRows, b);
      uint32_t issued = 0, issued_phase = 0;
      for (int j = 0; j < nkv; ++j) {
        const int s = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!mbar_wait(bar(kBarKVEmpty + s), ph ^ 1, abort_flag, p.err)) break;
        mbar_arrive_expect_tx(bar(kBarKFull + s), kGroups * kGroupBytes);
        for (int g = 0; g < kGroups; ++g)
          tma_load_3d(sbase + kOffK + s * kOpBytes + g * kGroupBytes, &tm, bar(kBarKFull + s), D + h * kDh + 8 * g,
                      j * kTileRows, b);
        mbar_arrive_expect_tx(bar(kBarVFull + s), kGroups * kGroupBytes);
        for (int g = 0; g < kGroups; ++g)
          tma_load_3d(sbase + kOffV + s * kOpBytes + g * kGroupBytes, &tm, bar(kBarVFull + s),
                      2 * D + h * kDh + 8 * g, j * kTileRows, b);
        issued |= 1u << s;
        issued_phase = (issued_phase & ~(1u << s)) | (ph << s);
      }
      mbar_wait_bounded(bar(kBarQ), 0, p.err);
      for (int s = 0; s < 2; ++s)
        if (issued & (1u << s)) {
          mbar_wait_bounded(bar(kBarKFull + s), (issued_phase >> s) & 1, p.err);
          mbar_wait_bounded(bar(kBarVFull + s), (issued_phase >> s) & 1, p.err);
        }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = make_idesc(128, 128, 0, false);  // S = Q K^T, both K-major
      constexpr uint32_t idesc_o = make_idesc(128, 80, 0, true);    // O = P V, V MN-major
      bool ok = mbar_wait(bar(kBarQ), 0, abort_flag, p.err);
      for (int j = 0; ok && j <= nkv; ++j) {
        if (j < nkv) {
          const int s = j & 1;
          const uint32_t ph = (j >> 1) & 1;
          if (!mbar_wait(bar(kBarKFull + s), ph, abort_flag, p.err) ||
              !mbar_wait(bar(kBarSEmpty + s), ph ^ 1, abort_flag, p.err))
            break;
          tc_fence_after();
          const uint32_t qa = sbase + kOffQ, ka = sbase + kOffK + s * kOpBytes;
#pragma unroll
          for (int kk = 0; kk < 5; ++kk)  // K = 80 in steps of 16 (two column groups)
            mma_f16(tmem + uint32_t(s * 128), make_sdesc(qa + kk * 2 * kGroupBytes, kGroupBytes, 128, 0),
                    make_sdesc(ka + kk * 2 * kGroupBytes, kGroupBytes, 128, 0), idesc_s, kk > 0);
          tc_commit(bar(kBarSFull + s));
        }
        if (j >= 1) {
          const int i = j - 1, s = i & 1;
          const uint32_t ph = (i >> 1) & 1;
          if (!mbar_wait(bar(kBarPFull + s), ph, abort_flag, p.err) ||
              !mbar_wait(bar(kBarVFull + s), ph, abort_flag, p.err) ||
              !mbar_wait(bar(kBarOEmpty + s), ph ^ 1, abort_flag, p.err))
            break;
          tc_fence_after();
          const uint32_t pa = sbase + kOffP + s * kPBytes, va = sbase + kOffV + s * kOpBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // K = 128 keys in steps of 16
            mma_f16(tmem + uint32_t(256 + s * 128), make_sdesc(pa + kk * 2 * kGroupBytes, kGroupBytes, 128, 0),
                    make_sdesc(va + kk * 256, 128, kGroupBytes, 0), idesc_o, kk > 0);
          tc_commit(bar(kBarOFull + s));
          tc_commit(bar(kBarKVEmpty + s));
        }
      }
      tc_commit(bar(kBarDrain));
      mbar_wait_bounded(bar(kBarDrain), 0, p.err);
    }
  } else {
    const int sub = warp & 3;
    const int r = sub * 32 + lane;  // query row within the tile == TMEM lane
    const uint32_t lane_off = uint32_t(sub * 32) << 16;
    float o[kDh];
#pragma unroll
    for (int d = 0; d < kDh; ++d) o[d] = 0.0f;
    float m = -INFINITY;          // running max (log2 units) of the P tiles written so far
    float m_folded = -INFINITY;   // reference max of the accumulator o
    float m_pending = -INFINITY;  // max used for the P tile whose O is not folded yet
    float l = 0.0f;
    bool ok = true;

    auto fold = [&](int i) -> bool {  // o = o * 2^(m_folded - m_i) + O_i
      const int s = i & 1;
      if (!mbar_wait(bar(kBarOFull + s), (i >> 1) & 1, abort_flag, p.err)) return false;
      tc_fence_after();
      const uint32_t ta = tmem + uint32_t(256 + s * 128) + lane_off;
      uint32_t a[32], c[32], e[8];
      tmem_ld32(ta, a);
      tmem_ld32(ta + 32, c);
      tmem_ld8(ta + 64, e);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(bar(kBarOEmpty + s));
      const float f = ex2(m_folded - m_pending);
#pragma unroll
      for (int d = 0; d < 32; ++d) o[d] = fmaf(o[d], f, __uint_as_float(a[d]));
#pragma unroll
      for (int d = 0; d < 32; ++d) o[32 + d] = fmaf(o[32 + d], f, __uint_as_float(c[d]));
#pragma unroll
      for (int d = 0; d < 8; ++d) o[64 + d] = fmaf(o[64 + d], f, __uint_as_float(e[d]));
      m_folded = m_pending;
      return true;
    };

    for (int j = 0; j < nkv && ok; ++j) {
      const int s = j & 1;
      if (!mbar_wait(bar(kBarSFull + s), (j >> 1) & 1, abort_flag, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t ta = tmem + uint32_t(s * 128) + lane_off;
      const int valid = T - j * kTileRows;  // keys of this tile that exist (>= 1)
      // pass 1: row maximum over valid keys
      float mx = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(ta + 32 * c, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (32 * c + i < valid) mx = fmaxf(mx, __uint_as_float(v[i]));
      }
      const float m_new = fmaxf(m, mx * p.scale_log2);
      // pass 2: probabilities, row sum, F16 P tile in shared memory
      uint8_t* pbuf = smem + kOffP + s * kPBytes;
      float sum = 0.0f;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(ta + 32 * c, v);
        tmem_ld_wait();
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint4 w;
          __half2* hw = reinterpret_cast<__half2*>(&w);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int k0 = 32 * c + 8 * g + 2 * i;
            const float p0 = k0 < valid ? ex2(fmaf(__uint_as_float(v[8 * g + 2 * i]), p.scale_log2, -m_new)) : 0.0f;
            const float p1 =
                k0 + 1 < valid ? ex2(fmaf(__uint_as_float(v[8 * g + 2 * i + 1]), p.scale_log2, -m_new)) : 0.0f;
            sum += p0 + p1;
            hw[i] = __floats2half2_rn(p0, p1);
          }
          *reinterpret_cast<uint4*>(pbuf + (4 * c + g) * kGroupBytes + r * 16) = w;
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();  // P (generic-proxy stores) visible to the tensor core
      mbar_arrive(bar(kBarSEmpty + s));
      mbar_arrive(bar(kBarPFull + s));
      l = fmaf(l, ex2(m - m_new), sum);
      m = m_new;
      if (j >= 1 && !fold(j - 1)) {
        ok = false;
        break;
      }
      m_pending = m_new;
    }
    if (ok) ok = fold(nkv - 1);

    const int t = qt * kTileRows + r;
    if (ok && t < T) {
      const float inv = 1.0f / l;
      const size_t row = size_t(b) * size_t(T) + size_t(t);
      if (!p.out_e4m3) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__half*>(p.out) + row * size_t(D) + size_t(h) * kDh);
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
          uint4 w;
          __half2* hw = reinterpret_cast<__half2*>(&w);
#pragma unroll
          for (int i = 0; i < 4; ++i) hw[i] = __floats2half2_rn(o[8 * g + 2 * i] * inv, o[8 * g + 2 * i + 1] * inv);
          dst[g] = w;
        }
      } else {
        uint2* dst = reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.out) + row * size_t(D) + size_t(h) * kDh);
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
          uint2 w;
          __nv_fp8x2_storage_t* q = reinterpret_cast<__nv_fp8x2_storage_t*>(&w);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            q[i] = __nv_cvt_float2_to_fp8x2(
                make_float2(16.0f * o[8 * g + 2 * i] * inv, 16.0f * o[8 * g + 2 * i + 1] * inv), __NV_SATFINITE,
                __NV_E4M3);
          dst[g] = w;
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

sv_status attention_map(CUtensorMap* m, const void* qkv, int B, int T, int H) {
  const uint64_t D3 = uint64_t(3) * uint64_t(H) * kDh;
  const uint64_t dims[3] = {D3, uint64_t(T), uint64_t(B)};
  const uint64_t strides[2] = {D3 * 2, D3 * 2 * uint64_t(T)};
  const uint32_t box[3] = {8, uint32_t(kTileRows), 1};
  return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, qkv, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

sv_status attention_launch(const CUtensorMap& m, void* o, int B, int T, int H, float scale, int out_e4m3,
                           cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attention)");
    attr_set = true;
  }
  Params p;
  p.T = T;
  p.H = H;
  p.D = H * kDh;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.out = o;
  p.out_e4m3 = out_e4m3;
  p.err = dev_err();
  dim3 grid((T + kTileRows - 1) / kTileRows, H, B);
  attention_kernel<<<grid, kThreads, kSmem, s>>>(m, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return SV_OK;
}

}  // namespace sv
