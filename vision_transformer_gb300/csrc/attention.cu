// Fused multi-head self-attention for head width 72 on the tcgen05 tensor cores.
//
// o_h = softmax(scale * Q_h K_h^T) V_h per image and head, F16 operands, F32
// scores, softmax and accumulation, F16 (or E4M3) result ("SigLIP ViT
// benchmark", precision paragraph: F32 softmax/accumulation state, result
// converted back to F16). The 729 x 729 score matrix never leaves the SM
// (flash-style online softmax), which replaces the pages' materialised and
// blocked-merge forms.
//
// Input: Q, K, V in the head-blocked layout written by the QKV projection's
// epilogue (sv_internal.h): each (image, head, 128-token tile) operand is one
// contiguous 18 KB block already in the tensor core's core-matrix order
// (column group of 8, then row, then 8 values), so a tile arrives with one
// bulk copy.
//
// Padding contract ("SigLIP optimized execution and PV padding", cause and
// fix: padding columns were once read as data and turned outputs into NaN):
//   - head width 72 is padded to 80 for the MMA K / N steps: the pad column
//     group of every operand tile in shared memory is never loaded; it is zero
//     for Q and K and (1, 0, ..., 0) for V, so output column 72 is the row sum;
//   - only the rows of existing tokens are copied; every operand buffer is
//     zeroed at kernel start, so rows past the last token hold zeros or values
//     of an earlier tile, never unwritten memory; keys past the last token are
//     masked to -inf before the row maximum, so their probability is exactly 0;
//   - query rows past the last token are computed but never stored.
//
// CTA = (256 queries as two 128-row tiles, head, image), 320 threads:
//   warp 0      bulk copies: Q (both tiles) once, then K and V tiles of 128
//               keys, each into 2 stages with its own release;
//   warp 1      TMEM owner + MMA issuer: per softmax group w, S_w(j) = Q_w K_j^T
//               (M 128, N 128, K 80) and O_w(j) = P_w(j) V_j (M 128, N 80, K 128);
//   warps 2..5  softmax group 0, warps 6..9 softmax group 1: one thread per
//               query row reads its S row from TMEM, writes P (F16) to shared
//               memory and folds O into an F32 register accumulator with the
//               online-softmax rescale; the softmax denominator comes out of
//               the P V product (a column of ones in V's pad group). The two
//               groups ping-pong: while one computes exponentials the tensor
//               core serves the other.
#include <cuda_fp8.h>

#include "ptx.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kDh = 72;                      // head width
constexpr int kGroups = 9;                   // 72 / 8 column groups held in memory
constexpr int kTile = 128;                   // queries per group, keys per step
constexpr int kGroupBytes = kTile * 16;      // 2048: one column group of a tile
constexpr int kBlockBytes = kGroups * kGroupBytes;  // 18432: one operand tile in memory
constexpr int kOpBytes = 10 * kGroupBytes;   // 80 columns in shared memory (72 + zero pad)
constexpr int kPBytes = 16 * kGroupBytes;    // 128 keys of probabilities
constexpr int kThreads = 320;

// Shared memory map (offsets from the 1024-aligned base).
constexpr int kOffQ = 0;                     // 2 query tiles
constexpr int kOffK = kOffQ + 2 * kOpBytes;  // 2 stages
constexpr int kOffV = kOffK + 2 * kOpBytes;  // 2 stages
constexpr int kOffP = kOffV + 2 * kOpBytes;  // one buffer per softmax group
constexpr int kOffBar = kOffP + 2 * kPBytes;
constexpr int kSmem = 1024 + kOffBar + 256;

// TMEM columns: S_w at 128 w, O_w at 256 + 128 w.
constexpr uint32_t kTmemCols = 512;

struct Params {
  const uint8_t* blocked;
  int B, T, H, tiles;
  float scale_log2;  // scale * log2(e)
  void* out;
  int out_e4m3;
  int* err;
};

// Barrier indices (8 bytes each).
enum {
  kBarQ = 0,
  kBarKFull = 1,    // +stage
  kBarKEmpty = 3,   // +stage
  kBarVFull = 5,    // +stage
  kBarVEmpty = 7,   // +stage
  kBarSFull = 9,    // +group
  kBarSEmpty = 11,  // +group: the group has read S into registers
  kBarPFull = 13,   // +group
  kBarOFull = 15,   // +group: O += P V of the group's latest tile has finished
  kBarDrain = 17,
  kNumBars = 18
};

// The reference maximum of a row (log2 units) is raised only when a tile's
// maximum exceeds it by more than this, so P <= 2^8 and O is rescaled rarely.
constexpr float kSlack = 8.0f;

__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// Rows of tile `tile` that hold tokens (0 if the tile starts past the last token).
__device__ __forceinline__ int tile_rows(int T, int tile) {
  const int v = T - tile * kTile;
  return v <= 0 ? 0 : (v < kTile ? v : kTile);
}

// Copies the existing rows of one operand tile; returns the bytes it will deliver.
__device__ __forceinline__ uint32_t copy_tile(uint32_t dst, const uint8_t* src, int rows, uint32_t bar) {
  if (rows == kTile) {
    bulk_copy(dst, src, kBlockBytes, bar);
    return kBlockBytes;
  }
  for (int g = 0; g < kGroups; ++g) bulk_copy(dst + g * kGroupBytes, src + g * kGroupBytes, rows * 16, bar);
  return uint32_t(kGroups * rows * 16);
}

__device__ __forceinline__ uint32_t tile_bytes(int rows) {
  return rows == kTile ? uint32_t(kBlockBytes) : uint32_t(kGroups * rows * 16);
}

__global__ void __launch_bounds__(kThreads, 1) attention_kernel(const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kOffBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto bar = [&](int i) { return bar0 + 8u * uint32_t(i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qpair = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int T = p.T;
  const int nkv = (T + kTile - 1) / kTile;
  // operand block of (which, tile) for this image and head
  auto block = [&](int which, int tile) {
    return p.blocked + (((size_t(which) * p.B + b) * p.H + h) * p.tiles + tile) * size_t(kBlockBytes);
  };

  // Zero every operand buffer (Q, K and V tiles including their pad column group),
  // except V's pad group, whose first column is 1: P V then carries the row sum
  // of P (the softmax denominator, from the same F16 P) in output column 72.
  for (int i = threadIdx.x; i < (6 * kOpBytes) / 16; i += kThreads) {
    const int off = i * 16;
    const bool v_pad = off >= kOffV && ((off - kOffV) % kOpBytes) >= kGroups * kGroupBytes;
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(v_pad ? 0x3C00u : 0u, 0, 0, 0);
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQ), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarKEmpty + s), 1);
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarVEmpty + s), 1);
      mbar_init(bar(kBarSFull + s), 1);
      mbar_init(bar(kBarSEmpty + s), 128);  // every softmax thread of the group arrives
      mbar_init(bar(kBarPFull + s), 128);
      mbar_init(bar(kBarOFull + s), 1);
    }
    mbar_init(bar(kBarDrain), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
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
      // both query tiles on one barrier
      const int qr0 = tile_rows(T, 2 * qpair), qr1 = tile_rows(T, 2 * qpair + 1);
      mbar_arrive_expect_tx(bar(kBarQ), tile_bytes(qr0) + (qr1 ? tile_bytes(qr1) : 0));
      copy_tile(sbase + kOffQ, block(0, 2 * qpair), qr0, bar(kBarQ));
      if (qr1) copy_tile(sbase + kOffQ + kOpBytes, block(0, 2 * qpair + 1), qr1, bar(kBarQ));
      uint32_t issued = 0, issued_phase = 0;  // bit s: K stage s; bit 2+s: V stage s
      for (int j = 0; j < nkv; ++j) {
        const int s = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        const int rows = tile_rows(T, j);
        if (!mbar_wait(bar(kBarKEmpty + s), ph ^ 1, abort_flag, p.err)) break;
        mbar_arrive_expect_tx(bar(kBarKFull + s), tile_bytes(rows));
        copy_tile(sbase + kOffK + s * kOpBytes, block(1, j), rows, bar(kBarKFull + s));
        issued |= 1u << s;
        issued_phase = (issued_phase & ~(1u << s)) | (ph << s);
        if (!mbar_wait(bar(kBarVEmpty + s), ph ^ 1, abort_flag, p.err)) break;
        mbar_arrive_expect_tx(bar(kBarVFull + s), tile_bytes(rows));
        copy_tile(sbase + kOffV + s * kOpBytes, block(2, j), rows, bar(kBarVFull + s));
        issued |= 1u << (2 + s);
        issued_phase = (issued_phase & ~(1u << (2 + s))) | (ph << (2 + s));
      }
      // every copy this thread issued lands before the CTA can exit
      mbar_wait_bounded(bar(kBarQ), 0, p.err);
      for (int s = 0; s < 2; ++s) {
        if (issued & (1u << s)) mbar_wait_bounded(bar(kBarKFull + s), (issued_phase >> s) & 1, p.err);
        if (issued & (4u << s)) mbar_wait_bounded(bar(kBarVFull + s), (issued_phase >> (2 + s)) & 1, p.err);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = make_idesc(128, 128, 0, false);  // S = Q K^T, both K-major
      constexpr uint32_t idesc_o = make_idesc(128, 80, 0, true);    // O = P V, V MN-major
      auto issue_s = [&](int w, int j) -> bool {  // S_w(j) = Q_w K_j^T
        const int s = j & 1;
        if (!mbar_wait(bar(kBarKFull + s), (j >> 1) & 1, abort_flag, p.err)) return false;
        if (!mbar_wait(bar(kBarSEmpty + w), (j & 1) ^ 1, abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t qa = sbase + kOffQ + w * kOpBytes, ka = sbase + kOffK + s * kOpBytes;
#pragma unroll
        for (int kk = 0; kk < 5; ++kk)  // K = 80 in steps of 16 (two column groups)
          mma_f16(tmem + uint32_t(w * 128), make_sdesc(qa + kk * 2 * kGroupBytes, kGroupBytes, 128, 0),
                  make_sdesc(ka + kk * 2 * kGroupBytes, kGroupBytes, 128, 0), idesc_s, kk > 0);
        tc_commit(bar(kBarSFull + w));
        if (w == 1) tc_commit(bar(kBarKEmpty + s));  // both groups have read K_j
        return true;
      };
      auto issue_pv = [&](int w, int j) -> bool {  // O_w += P_w(j) V_j
        const int s = j & 1;
        if (!mbar_wait(bar(kBarPFull + w), j & 1, abort_flag, p.err)) return false;
        if (!mbar_wait(bar(kBarVFull + s), (j >> 1) & 1, abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t pa = sbase + kOffP + w * kPBytes, va = sbase + kOffV + s * kOpBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // K = 128 keys in steps of 16
          mma_f16(tmem + uint32_t(256 + w * 128), make_sdesc(pa + kk * 2 * kGroupBytes, kGroupBytes, 128, 0),
                  make_sdesc(va + kk * 256, 128, kGroupBytes, 0), idesc_o, (j | kk) > 0);
        tc_commit(bar(kBarOFull + w));
        if (w == 1) tc_commit(bar(kBarVEmpty + s));  // both groups have read V_j
        return true;
      };
      // S of the next tile is issued as soon as a group has read its S, so it is
      // computed while that group's softmax of the current tile runs.
      bool ok = mbar_wait(bar(kBarQ), 0, abort_flag, p.err) && issue_s(0, 0) && issue_s(1, 0);
      for (int j = 0; ok && j < nkv; ++j) {
        ok = (j + 1 >= nkv || issue_s(0, j + 1)) && (j + 1 >= nkv || issue_s(1, j + 1)) && issue_pv(0, j) &&
             issue_pv(1, j);
      }
      tc_commit(bar(kBarDrain));
      mbar_wait_bounded(bar(kBarDrain), 0, p.err);
    }
  } else {
    const int w = (warp - 2) >> 2;  // softmax group
    const int sub = warp & 3;       // TMEM lane quarter
    const int r = sub * 32 + lane;  // query row within the group's tile == TMEM lane
    const uint32_t lane_off = uint32_t(sub * 32) << 16;
    const uint32_t s_tm = tmem + uint32_t(w * 128) + lane_off;
    const uint32_t o_tm = tmem + uint32_t(256 + w * 128) + lane_off;
    uint8_t* pbuf = smem + kOffP + w * kPBytes;
    const float sl2 = p.scale_log2;
    // Reference maximum (log2 units) of this row's P tiles and of the O accumulator
    // in TMEM; the softmax denominator accumulates in O's column 72.
    float m = -INFINITY;
    bool ok = true;

    for (int j = 0; j < nkv && ok; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarSFull + w), j & 1, abort_flag, p.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the whole S row in registers (four loads in flight), then S is released
      uint32_t sv[4][32];
      tmem_ld32(s_tm, sv[0]);
      tmem_ld32(s_tm + 32, sv[1]);
      tmem_ld32(s_tm + 64, sv[2]);
      tmem_ld32(s_tm + 96, sv[3]);
      tmem_ld_wait(sv[0]);
      reg_fence(sv[1]);
      reg_fence(sv[2]);
      reg_fence(sv[3]);
      tc_fence_before();
      mbar_arrive(bar(kBarSEmpty + w));
      const int valid = T - j * kTile;  // keys of this tile that exist (>= 1)
      if (valid < kTile) {              // keys past the last token: -inf, so P = 0 exactly
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * c + i >= valid) sv[c][i] = 0xff800000u;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; i += 2) mx = fmax3(mx, __uint_as_float(sv[c][i]), __uint_as_float(sv[c][i + 1]));
      const float m_tile = mx * sl2;
      const bool raise = m_tile > m + kSlack;  // always at j == 0
      const float m_new = raise ? m_tile : m;
      if (j > 0) {
        // O += P(j-1) V has finished: the P buffer is free and O is stable
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarOFull + w), (j - 1) & 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, raise)) {  // O (and its row sum) *= 2^(m - m_new), 1 for kept rows
          const float f = ex2(m - m_new);
#pragma unroll 1
          for (int c = 0; c < 10; ++c) {  // 80 columns, 8 at a time (few live registers)
            uint32_t e[8];
            tmem_ld8(o_tm + 8 * c, e);
            tmem_ld_wait();
            asm volatile("" : "+r"(e[0]), "+r"(e[1]), "+r"(e[2]), "+r"(e[3]), "+r"(e[4]), "+r"(e[5]), "+r"(e[6]),
                         "+r"(e[7]));
#pragma unroll
            for (int i = 0; i < 8; ++i) e[i] = __float_as_uint(__uint_as_float(e[i]) * f);
            tmem_st8(o_tm + 8 * c, e);
          }
          tmem_st_wait();
        }
      }
      m = m_new;
      // P = 2^(scale log2(e) s - m) as the F16 P tile in shared memory
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint4 wv;
          __half2* hw = reinterpret_cast<__half2*>(&wv);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float p0 = ex2(fmaf(__uint_as_float(sv[c][8 * g + 2 * i]), sl2, -m));
            const float p1 = ex2(fmaf(__uint_as_float(sv[c][8 * g + 2 * i + 1]), sl2, -m));
            hw[i] = __floats2half2_rn(p0, p1);
          }
          *reinterpret_cast<uint4*>(pbuf + (4 * c + g) * kGroupBytes + r * 16) = wv;
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();  // P (generic-proxy stores) visible to the tensor core
      mbar_arrive(bar(kBarPFull + w));
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarOFull + w), (nkv - 1) & 1, abort_flag, p.err));

    const int t = (2 * qpair + w) * kTile + r;
    if (ok) {
      tc_fence_after();
      uint32_t a[32], c[32], e[16];
      tmem_ld32(o_tm, a);
      tmem_ld32(o_tm + 32, c);
      tmem_ld16(o_tm + 64, e);
      tmem_ld_wait(a);
      reg_fence(c);
      tmem_ld_wait();
      float o[kDh];
#pragma unroll
      for (int d = 0; d < 32; ++d) o[d] = __uint_as_float(a[d]);
#pragma unroll
      for (int d = 0; d < 32; ++d) o[32 + d] = __uint_as_float(c[d]);
#pragma unroll
      for (int d = 0; d < 8; ++d) o[64 + d] = __uint_as_float(e[d]);
      const float l = __uint_as_float(e[8]);
      if (t < T) {
        const float inv = 1.0f / l;
        const int D = p.H * kDh;
        const size_t row = size_t(b) * size_t(T) + size_t(t);
        if (!p.out_e4m3) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__half*>(p.out) + row * size_t(D) + size_t(h) * kDh);
#pragma unroll
          for (int g = 0; g < kGroups; ++g) {
            uint4 wv;
            __half2* hw = reinterpret_cast<__half2*>(&wv);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              hw[i] = __floats2half2_rn(o[8 * g + 2 * i] * inv, o[8 * g + 2 * i + 1] * inv);
            dst[g] = wv;
          }
        } else {
          uint2* dst = reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.out) + row * size_t(D) + size_t(h) * kDh);
#pragma unroll
          for (int g = 0; g < kGroups; ++g) {
            uint2 wv;
            __nv_fp8x2_storage_t* q = reinterpret_cast<__nv_fp8x2_storage_t*>(&wv);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              q[i] = __nv_cvt_float2_to_fp8x2(
                  make_float2(16.0f * o[8 * g + 2 * i] * inv, 16.0f * o[8 * g + 2 * i + 1] * inv), __NV_SATFINITE,
                  __NV_E4M3);
            dst[g] = wv;
          }
        }
      }
    }
    tmem_ld_wait();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Row-major [B, T, 3 D] -> head-blocked; one thread per 16-byte group of 8 values.
__global__ void repack_kernel(const __half* __restrict__ qkv, uint8_t* __restrict__ blk, int B, int T, int H,
                              int tiles) {
  const int D = H * kDh;
  const long i = long(blockIdx.x) * blockDim.x + threadIdx.x;
  const long per_row = 3L * D / 8;
  if (i >= long(B) * T * per_row) return;
  const long m = i / per_row;
  const int col = int(i - m * per_row) * 8;
  const int bimg = int(m / T), t = int(m - long(bimg) * T);
  const int which = col / D, rem = col - which * D, h = rem / kDh, cg = (rem - h * kDh) >> 3;
  const size_t idx = ((size_t(which) * B + bimg) * H + h) * tiles + (t >> 7);
  *reinterpret_cast<uint4*>(blk + (idx * kGroups + cg) * kGroupBytes + (t & 127) * 16) =
      *reinterpret_cast<const uint4*>(qkv + m * 3 * D + col);
}

}  // namespace

size_t attention_blocked_bytes(int B, int T, int H) {
  return size_t(3) * B * H * ((T + kTile - 1) / kTile) * size_t(kBlockBytes);
}

sv_status attention_repack_launch(const __half* qkv, void* blocked, int B, int T, int H, cudaStream_t s) {
  const long n = long(B) * T * (3L * H * kDh / 8);
  repack_kernel<<<unsigned((n + 255) / 256), 256, 0, s>>>(qkv, static_cast<uint8_t*>(blocked), B, T, H,
                                                           (T + kTile - 1) / kTile);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SV_OK : cuda_fail(e, "attention repack launch");
}

sv_status attention_launch(const void* blocked, void* o, int B, int T, int H, float scale, int out_e4m3,
                           cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attention)");
    attr_set = true;
  }
  Params p;
  p.blocked = static_cast<const uint8_t*>(blocked);
  p.B = B;
  p.T = T;
  p.H = H;
  p.tiles = (T + kTile - 1) / kTile;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.out = o;
  p.out_e4m3 = out_e4m3;
  p.err = dev_err();
  dim3 grid((T + 2 * kTile - 1) / (2 * kTile), H, B);
  attention_kernel<<<grid, kThreads, kSmem, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return SV_OK;
}

}  // namespace sv
