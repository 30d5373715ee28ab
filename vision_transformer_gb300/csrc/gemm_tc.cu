// Dense projection GEMM on the 5th-generation tensor cores (tcgen05 + TMEM),
// with the epilogues of the encoder fused in: bias, positional embedding,
// tanh-GELU, residual add, F16 or E4M3 output.
//
// C[M,N] = epi(A[M,K] . W[N,K]^T): every dense GEMM of the encoder ("SigLIP
// ViT benchmark": the 588->1152 patch embedding, the fused 1152->3456 QKV
// projection, the output projection, the 1152->4304->1152 MLP, and the MAP
// head's Q, KV, output and MLP projections).
//
// Design (one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer: A and W tiles (128-byte swizzled, 128 bytes of
//               K per stage) into a ring of shared-memory stages;
//   warp 1      allocates TMEM and issues tcgen05.mma (M = 128, N = BN) from
//               one thread; the accumulator (F32) lives in TMEM, double
//               buffered so the epilogue of one tile overlaps the next tile's
//               main loop. With two or more row tiles the CTAs run in pairs
//               (clusters of 2) that share one M = 256 MMA (cta_group::2):
//               each CTA stages its 128 rows of A and half of the W tile, the
//               leader issues the MMAs, each CTA's TMEM holds its 128 rows;
//   warps 2..   epilogue, two warps per TMEM lane quarter taking every other
//               32-column chunk (the warp's next chunk's tcgen05.ld in flight
//               during this chunk's math), or three taking every third (each
//               chunk loaded when it starts: E4M3 pairs, 192-wide F16 pairs
//               without statistics); fused math, the 32 x 32 result block
//               staged in swizzled shared memory and written by a TMA store;
//               residual blocks arrive by TMA one chunk ahead; the GEMMs that
//               write the residual stream also leave per-tile row statistics for
//               the next LayerNorm (eight-warp epilogues).
// Split K (long K): at small M, where the tiles would fill few SMs, every tile, and
// otherwise the tiles of a short last wave, become (tile, K range) items; each writes
// its raw F32 sums to a workspace and gemm_splitk_reduce_kernel adds them up in a
// fixed order and applies the epilogue.
// Launched with programmatic stream serialization: the prologue overlaps the
// previous kernel, global memory is touched only after griddepcontrol.wait.
// F16 operands use kind::f16 (K = 16 per instruction); E4M3 operands use
// kind::f8f6f4 (K = 32 per instruction) with the dequantisation scale
// applied to the accumulator. All waits are bounded (ptx.cuh).
#include <cuda_fp8.h>

#include <cstdio>

#include "ptx.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kBM = 128;
constexpr int kSwzBytes = 128;  // one 128-byte swizzle row of K
// Warp 0 loads, warp 1 issues the MMAs, the EPI warps after them run the epilogue:
// 8, two per TMEM lane quarter, each taking every other 32-column chunk of a tile (with
// four warps the epilogue of a K = 1152 tile took about as long as its main loop), or
// 12, three per quarter: for CTA pairs on E4M3 operands (their main loop over a
// K = 1152 tile takes half the time of the F16 one, the epilogue's work per tile is the
// same, and with two per quarter the MMA of the 1152 -> 4304 MLP projection waited about
// 30% of every tile for a free accumulator), and for 192-wide F16 pairs (one tile per
// CTA pair at one image, its epilogue not overlapped: 729 x 3456 x 1152 13.0 -> 12.15
// us). Twelve warps keep no LayerNorm statistics (those GEMMs get eight).
template <int EPI>
constexpr int gemm_threads() {
  return 64 + 32 * EPI;
}
// Widest output tile used with CTA pairs (its TMEM: 2 x BN columns per CTA).
constexpr int kPairMaxBn = 256;
// Suspend limits (ns) of the mbarrier waits of each role. A waiter that polls
// instead keeps taking issue slots and shared-memory cycles from the warps that
// do the work: the epilogue warps wait a whole main loop for each accumulator.
// Measured on the encoder's GEMMs (M = 23,328, F16): suspending waiters made all
// four 6-7% faster.
constexpr uint32_t kSleepProducer = 1000000;
constexpr uint32_t kSleepMma = 1000000;
constexpr uint32_t kSleepEpi = 1000000;

// PAIR: the two CTAs of a cluster share one 256-row MMA (cta_group::2): each
// holds its 128 rows of A and half of the W tile per stage, and the tensor core
// reads the other half from the peer.
// ATOMS: 128-byte swizzle rows of K per stage. Two (fewer, larger stages, half the
// barrier round trips per K) pay for CTA pairs over K = 1152 with L2-resident operands
// (QKV, MLP up: 4-7% faster); one is better where A streams from DRAM (MLP down) or a
// single CTA would be left with two stages (output projection).
template <int BN, bool PAIR, int ATOMS, int EPI>
struct Cfg {
  static constexpr int kAtomA = kBM * kSwzBytes;                   // one swizzle row of the A tile
  static constexpr int kAtomB = (PAIR ? BN / 2 : BN) * kSwzBytes;  // of the W tile (this CTA's rows)
  static constexpr int kStageA = kAtomA * ATOMS;
  static constexpr int kStageB = kAtomB * ATOMS;
  static constexpr int kBKBytes = kSwzBytes * ATOMS;  // K bytes per stage
  static constexpr int kStage = kStageA + kStageB;
  // epilogue staging: per epilogue warp a ring of two 32 x 32 blocks (residual in,
  // result out)
  static constexpr int kEpiBlock = 2048;
  static constexpr int kEpiRing = 2;
  static constexpr int kEpiBytes = EPI * kEpiRing * kEpiBlock;
  // barriers (full / empty per stage, at most 8 stages; 2 + 2 accumulator; drain; per
  // epilogue warp and ring block) and the TMEM address slot
  static constexpr int kBarBytes = (8 * (2 * 8 + 5 + EPI * kEpiRing) + 8 + 63) / 64 * 64;
  static constexpr int kBudget = 232448 - 1024 - kEpiBytes - kBarBytes;
  static constexpr int kStages = kBudget / kStage < 8 ? kBudget / kStage : 8;
  static constexpr int kTmemCols = 2 * BN <= 128 ? 128 : (2 * BN <= 256 ? 256 : 512);
  static constexpr int kSmem = 1024 + kStages * kStage + kEpiBytes + kBarBytes;
  static_assert(kStage % 1024 == 0, "stage must keep 1024-byte alignment");
  static_assert(8 * (2 * kStages + 5 + EPI * kEpiRing) + 8 <= kBarBytes, "barrier area");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

struct Params {
  int M, N, K;
  int m_tiles, n_tiles, k_blocks;
  // n_full column tiles are BN wide; a last, narrower one (N % BN columns) runs its
  // MMAs with N = tail_n; with tail_last the narrow tiles come after all full ones
  int n_full, tail_n, tail_last;
  const __half* bias;
  const __half* pos;
  int pos_rows;
  int has_res;
  int act, out_e4m3;
  float scale;
  // LayerNorm folded in (see GemmEpi): 1/std per row, and one extra K block of 16
  const float* ln_r;
  int ln_aug;
  int* err;
  void* out;  // the output matrix [M, N] (also described by the output tensor map)
  // head-blocked output (fused QKV projection feeding attention), or null
  uint8_t* blk;
  int blk_T, blk_H, blk_B, blk_tiles;
  int blk_col0;  // first column of the fused [Q | K | V] space this GEMM's columns start at
  int blk_qk8;   // Q and K as E4M3 (16 x value): 16-byte groups of 16 columns per row
  float2* ln_part;  // per (row, column tile): (mean, M2) of the results, or null
  // split K: items below n_main are whole tiles; item n_main + q * k_splits + s is K
  // range s (K blocks [s kb_split, min(k_blocks, (s + 1) kb_split))) of tile item
  // n_main + q, whose raw sums go to rows ((q * k_splits + s) * (PAIR ? 2 : 1) + rank) * 128
  // .. + 127 of the [rows, BN] F32 workspace (through tmAa)
  int n_main, k_splits, kb_split;
};

// GELU, tanh form: 0.5 x (1 + tanh(u)), u = sqrt(2/pi) (x + 0.044715 x^3), with
// the hardware tanh (one MUFU operation; relative error about 2^-11, the F16
// output's own rounding). Two values at a time, with the two-lane F32 instructions.
__device__ __forceinline__ void gelu_tanh_x2(float& x0, float& x1) {
  float q0, q1, u0, u1, t0, t1, h0, h1;
  mul_x2(q0, q1, x0, x1, x0, x1);                                  // x^2
  mul_x2(q0, q1, q0, q1, 0.044715f, 0.044715f);                    // 0.044715 x^2
  fma_x2(u0, u1, q0, q1, x0, x1, x0, x1);                          // x + 0.044715 x^3
  mul_x2(u0, u1, u0, u1, 0.7978845608028654f, 0.7978845608028654f);
  asm("tanh.approx.f32 %0, %1;" : "=f"(t0) : "f"(u0));
  asm("tanh.approx.f32 %0, %1;" : "=f"(t1) : "f"(u1));
  mul_x2(h0, h1, x0, x1, 0.5f, 0.5f);
  fma_x2(x0, x1, h0, h1, t0, t1, h0, h1);
}

__device__ __forceinline__ void load8h(const __half* p, float* f) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __half22float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ void add8h(const uint4& v, float* f) {
  const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __half22float2(h[i]);
    add_x2(f[2 * i], f[2 * i + 1], f[2 * i], f[2 * i + 1], t.x, t.y);
  }
}

// Bias of output columns n .. n+31 as four 8-column groups (zero past N or
// without a bias; N is a multiple of 16).
__device__ __forceinline__ void load_bias(const Params& p, int n, uint4 (&bq)[4]) {
#pragma unroll
  for (int g = 0; g < 4; ++g)
    bq[g] = (p.bias && n + 8 * g < p.N) ? __ldg(reinterpret_cast<const uint4*>(p.bias + n + 8 * g))
                                        : make_uint4(0u, 0u, 0u, 0u);
}

// Number of 32-column chunks of tile column block nt that hold columns < N.
__device__ __forceinline__ int tile_chunks(const Params& p, int nt, int bn) {
  const int rem = p.N - nt * bn;
  const int c = (rem + 31) / 32;
  return c < bn / 32 ? c : bn / 32;
}

// Work item `it` -> output tile (mt, nt): row by row, or (tail_last) the full-width
// tiles row by row and then the narrow last column (cheaper MMAs) of every row, which
// then fills the last wave. With PAIR an item is a 256-row
// tile of two vertically adjacent 128-row tiles; the CTA of cluster rank r takes
// m-tile 2 * pair + r.
// mu: the 128-row tile (PAIR: the 256-row pair of tiles) of tile item `it`.
__host__ __device__ __forceinline__ void tile_pos(int it, int row_units, int n_tiles, int n_full, int tail_last,
                                                  int& mu, int& nt) {
  const int full_items = row_units * n_full;
  if (!tail_last) {  // row by row: the tiles of one row share their A rows in L2
    mu = it / n_tiles;
    nt = it - mu * n_tiles;
  } else if (it < full_items) {
    mu = it / n_full;
    nt = it - mu * n_full;
  } else {  // the narrow last column, after every full tile: it fills the last wave
    mu = it - full_items;
    nt = n_full;
  }
}

// The inverse of tile_pos: tile item of row unit mu and column tile nt.
__host__ __device__ __forceinline__ int tile_index(int mu, int nt, int row_units, int n_tiles, int n_full,
                                                   int tail_last) {
  if (!tail_last) return mu * n_tiles + nt;
  return nt < n_full ? mu * n_full + nt : row_units * n_full + mu;
}

template <bool PAIR>
__device__ __forceinline__ void tile_of(const Params& p, int it, int rank, int& mt, int& nt) {
  int mu;
  tile_pos(it, PAIR ? (p.m_tiles + 1) / 2 : p.m_tiles, p.n_tiles, p.n_full, p.tail_last, mu, nt);
  mt = PAIR ? 2 * mu + rank : mu;
}

// SPLIT: 0 whole tiles only; otherwise the items from n_main on are (tile, K range) pairs
// whose raw sums go to the split-K workspace (tmAa describes it; no LayerNorm is folded
// into a split GEMM): 1 every item (n_main = 0), 2 whole tiles first, then split ones.
// EPI: epilogue warps (8 or 12, see gemm_threads).
template <int BN, bool FP8, bool PAIR, int ATOMS, int SPLIT, int EPI>
__global__ void __launch_bounds__(gemm_threads<EPI>(), 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                   const __grid_constant__ CUtensorMap tmWt, const __grid_constant__ CUtensorMap tmC,
                   const __grid_constant__ CUtensorMap tmR, const __grid_constant__ CUtensorMap tmAa,
                   const __grid_constant__ CUtensorMap tmWa, const __grid_constant__ CUtensorMap tmWat,
                   const Params p) {
  constexpr int kEpiWarps = EPI;
  constexpr int kParts = kEpiWarps / 4;  // epilogue warps per TMEM lane quarter
  // With two warps per quarter the TMEM load of a warp's next chunk is issued during
  // this chunk's math. With three (128 registers a thread) each chunk loads its own:
  // measured on the E4M3 encoder, 3.5% faster per step at batch 32 than loading ahead.
  constexpr bool kLdAhead = kParts < 3;
  using C = Cfg<BN, PAIR, ATOMS, kEpiWarps>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* epi = smem + C::kStages * C::kStage;  // [epilogue warp][ring] 32 x 32 blocks
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi + C::kEpiBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::kStages + 5 + kEpiWarps * C::kEpiRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar_full = smem_u32(bars);
  const uint32_t bar_empty = bar_full + 8 * C::kStages;
  const uint32_t bar_tfull = bar_empty + 8 * C::kStages;
  const uint32_t bar_tempty = bar_tfull + 16;
  const uint32_t bar_drain = bar_tempty + 16;
  const uint32_t bar_res = bar_drain + 8;  // [epilogue warp][ring]

  // Work items: tiles, or (PAIR) 256-row tiles shared by the two CTAs of a cluster.
  const int aug_blocks = (!FP8 && p.ln_aug) ? 1 : 0;  // folded LayerNorm's extra K block
  const int rank = PAIR ? int(cluster_ctarank()) : 0;
  const bool leader = rank == 0;
  const int it0 = PAIR ? int(blockIdx.x >> 1) : int(blockIdx.x);
  const int it_step = PAIR ? int(gridDim.x >> 1) : int(gridDim.x);
  const int tile_items = PAIR ? ((p.m_tiles + 1) / 2) * p.n_tiles : p.m_tiles * p.n_tiles;
  const int main_items = SPLIT == 1 ? 0 : (SPLIT == 2 ? p.n_main : tile_items);  // items that are whole tiles
  const int num_items = SPLIT ? main_items + (tile_items - main_items) * p.k_splits : tile_items;
  // item -> tile item; ks = its K range (-1: the whole of K)
  auto item_tile = [&](int it, int& ks) {
    if (!SPLIT || it < main_items) {
      ks = -1;
      return it;
    }
    const int j = it - main_items;
    ks = j % p.k_splits;
    return main_items + j / p.k_splits;
  };
  // K blocks of K range ks: [kb_lo, kb_hi)
  auto k_range = [&](int ks, int& kb_lo, int& kb_hi) {
    if (SPLIT && ks >= 0) {
      kb_lo = ks * p.kb_split;
      kb_hi = min(p.k_blocks, kb_lo + p.kb_split);
    } else {
      kb_lo = 0;
      kb_hi = p.k_blocks;
    }
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);   // PAIR: the leader's producer arms it for both CTAs' bytes
      mbar_init(bar_empty + 8 * s, 1);  // PAIR: released by the leader's MMA commit in both CTAs
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull + 8 * a, 1);
      mbar_init(bar_tempty + 8 * a, (PAIR ? 64 : 32) * kEpiWarps);  // every epilogue thread (of both CTAs) arrives
    }
    mbar_init(bar_drain, 1);
    for (int i = 0; i < kEpiWarps * C::kEpiRing; ++i) mbar_init(bar_res + 8 * i, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmC);
    if (p.has_res) prefetch_tmap(&tmR);
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // both CTAs' barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();  // operands, residual and statistics come from earlier kernels

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_phase = 0;  // stages with loads in flight, and their phase bit
      bool ok = true;
      for (int it = it0; it < num_items && ok; it += it_step) {
        int mt, nt, kb_lo, kb_hi, ks;
        tile_of<PAIR>(p, item_tile(it, ks), rank, mt, nt);
        k_range(ks, kb_lo, kb_hi);
        for (int kb = kb_lo; kb < kb_hi + aug_blocks; ++kb) {
          if (!mbar_wait<kSleepProducer>(bar_empty + 8 * stage, phase ^ 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar_full + 8 * stage;
          const uint32_t sa = smem_u32(smem + stage * C::kStage);
          const int kc = kb * (FP8 ? C::kBKBytes : C::kBKBytes / 2);
          constexpr int kAtomK = FP8 ? kSwzBytes : kSwzBytes / 2;  // K elements of one swizzle row
          if (kb == p.k_blocks) {  // folded LayerNorm: the 16-wide K block (-mean | column sums)
            if (PAIR) {  // each CTA: its 128 rows of the A block, its half of the W block's rows
              const bool narrow = nt == p.n_full && p.tail_n;
              const int wrows = narrow ? p.tail_n / 2 : BN / 2;
              const uint32_t fb_lead = mapa_shared(fb, 0);
              if (leader) mbar_arrive_expect_tx(fb, 2 * (kBM + wrows) * 32);
              tma_load_2d_pair(sa, &tmAa, fb_lead, 0, mt * kBM);
              tma_load_2d_pair(sa + C::kStageA, narrow ? &tmWat : &tmWa, fb_lead, 0, nt * BN + rank * wrows);
            } else {
              mbar_arrive_expect_tx(fb, (kBM + BN) * 32);
              tma_load_2d(sa, &tmAa, fb, 0, mt * kBM);
              tma_load_2d(sa + C::kStageA, &tmWa, fb, 0, nt * BN);
            }
          } else if (PAIR) {  // both CTAs' copies complete on the leader's barrier
            const uint32_t fb_lead = mapa_shared(fb, 0);
            if (nt == p.n_full && p.tail_n) {  // narrow tile: each CTA holds tail_n / 2 W rows
              if (leader) mbar_arrive_expect_tx(fb, 2 * (C::kStageA + (p.tail_n / 2) * C::kBKBytes));
#pragma unroll
              for (int a = 0; a < ATOMS; ++a) {
                tma_load_2d_pair(sa + a * C::kAtomA, &tmA, fb_lead, kc + a * kAtomK, mt * kBM);
                tma_load_2d_pair(sa + C::kStageA + a * C::kAtomB, &tmWt, fb_lead, kc + a * kAtomK,
                                 nt * BN + rank * (p.tail_n / 2));
              }
            } else {
              if (leader) mbar_arrive_expect_tx(fb, 2 * C::kStage);
#pragma unroll
              for (int a = 0; a < ATOMS; ++a) {
                tma_load_2d_pair(sa + a * C::kAtomA, &tmA, fb_lead, kc + a * kAtomK, mt * kBM);
                tma_load_2d_pair(sa + C::kStageA + a * C::kAtomB, &tmW, fb_lead, kc + a * kAtomK,
                                 nt * BN + rank * (BN / 2));
              }
            }
          } else {
            mbar_arrive_expect_tx(fb, C::kStage);
#pragma unroll
            for (int a = 0; a < ATOMS; ++a) {
              tma_load_2d(sa + a * C::kAtomA, &tmA, fb, kc + a * kAtomK, mt * kBM);
              tma_load_2d(sa + C::kStageA + a * C::kAtomB, &tmW, fb, kc + a * kAtomK, nt * BN);
            }
          }
          issued |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Every copy this thread issued lands (and, under PAIR, every stage release of the
      // leader's MMA lands in this CTA) before the CTA can exit; immediate on the normal path.
      for (int st = 0; st < C::kStages; ++st)
        if (issued & (1u << st)) {
          if (PAIR)
            mbar_wait_bounded(bar_empty + 8 * st, (issued_phase >> st) & 1, p.err);
          else
            mbar_wait_bounded(bar_full + 8 * st, (issued_phase >> st) & 1, p.err);
        }
      // After an abort under PAIR, copies issued toward stages nobody consumes may
      // still be in flight: give them time to land (about 100 us) before leaving.
      if (PAIR && *abort_flag) {
        const unsigned long long t0 = globaltimer();
        while (globaltimer() - t0 < 100000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      constexpr uint32_t idesc_full = make_idesc(PAIR ? 2 * kBM : kBM, BN, 0, false);
      const uint32_t idesc_tail = make_idesc(PAIR ? 2 * kBM : kBM, p.tail_n ? p.tail_n : BN, 0, false);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int it = it0; it < num_items && ok; it += it_step, ++local) {
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        int mt_i, nt_i, kb_lo, kb_hi, ks;
        tile_of<PAIR>(p, item_tile(it, ks), rank, mt_i, nt_i);
        k_range(ks, kb_lo, kb_hi);
        const uint32_t idesc = (nt_i == p.n_full && p.tail_n) ? idesc_tail : idesc_full;
        if (!mbar_wait<kSleepMma>(bar_tempty + 8 * acc, acc_phase ^ 1, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + uint32_t(acc * BN);
        for (int kb = kb_lo; kb < kb_hi + aug_blocks; ++kb) {
          if (!mbar_wait<kSleepMma>(bar_full + 8 * stage, phase, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * C::kStage);
          const uint32_t sb = sa + C::kStageA;
          if (!FP8 && kb == p.k_blocks) {
            // 32-byte rows with the 32-byte swizzle: 8-row groups 256 bytes apart
            if (PAIR)
              mma_f16_pair(d, make_sdesc(sa, 16, 256, 6), make_sdesc(sb, 16, 256, 6), idesc, 1u);
            else
              mma_f16(d, make_sdesc(sa, 16, 256, 6), make_sdesc(sb, 16, 256, 6), idesc, 1u);
          } else
#pragma unroll
          for (int j = 0; j < 4 * ATOMS; ++j) {  // 4 instructions x 32 bytes of K per swizzle row
            const uint64_t ad = make_sdesc(sa + (j >> 2) * C::kAtomA + 32 * (j & 3), 16, 1024, 2);
            const uint64_t bd = make_sdesc(sb + (j >> 2) * C::kAtomB + 32 * (j & 3), 16, 1024, 2);
            const uint32_t accum = ((kb - kb_lo) | j) != 0;
            if (PAIR) {
              if (FP8)
                mma_f8_pair(d, ad, bd, idesc, accum);
              else
                mma_f16_pair(d, ad, bd, idesc, accum);
            } else {
              if (FP8)
                mma_f8(d, ad, bd, idesc, accum);
              else
                mma_f16(d, ad, bd, idesc, accum);
            }
          }
          // frees the stage (in both CTAs under PAIR) when these MMAs finish
          if (PAIR)
            tc_commit_pair_mc(bar_empty + 8 * stage, uint16_t(3));
          else
            tc_commit(bar_empty + 8 * stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok) {
          if (PAIR)
            tc_commit_pair_mc(bar_tfull + 8 * acc, uint16_t(3));
          else
            tc_commit(bar_tfull + 8 * acc);
        }
      }
      // All MMAs this thread issued complete before TMEM is released.
      if (PAIR)
        tc_commit_pair_mc(bar_drain, uint16_t(1));
      else
        tc_commit(bar_drain);
      mbar_wait_bounded(bar_drain, 0, p.err);
      // Under PAIR the epilogues of both CTAs release accumulators on this CTA's
      // barriers: wait for the last releases so none lands after this CTA exits.
      if (PAIR)
        for (int a = 0; a < 2 && a < local; ++a) {
          const int last = (local - 1 - a) >= 0 ? ((local - 1 - a) >> 1) : 0;  // use index of the last use of acc
          const int acc = (local - 1 - a) & 1;
          mbar_wait_bounded(bar_tempty + 8 * acc, uint32_t(last) & 1, p.err);
        }
    }
  } else {
    // Epilogue: warp ew owns TMEM lanes 32*sub .. +31, i.e. rows row0 .. row0+31 of
    // each tile, and of them the 32-column chunks c = part, part + kParts, ...; each chunk is
    // staged as a 32 x 32 block in shared memory (64-byte rows with the 64-byte swizzle
    // for F16, 32-byte rows with the 32-byte swizzle for E4M3) and written by one TMA
    // store, which also clips the M / N tails.
    const int sub = warp & 3, ew = warp - 2, part = ew >> 2;
    // Ring of kEpiRing blocks per warp; chunk q (counted over all of this warp's chunks)
    // uses block q % kEpiRing. With a residual, the residual block of chunk q is
    // loaded there kResAhead chunks ahead, the result overwrites it in place and the
    // TMA store of the result reads it; the load of chunk q + kResAhead reuses the
    // block of chunk q + kResAhead - kEpiRing once that chunk's store has read it.
    constexpr int kResAhead = C::kEpiRing - 1;
    uint8_t* ring = epi + ew * C::kEpiRing * C::kEpiBlock;
    const uint32_t rbar = bar_res + 8 * C::kEpiRing * ew;
    // residual loads in flight per block, with the phase parity that completes them
    uint32_t res_issued = 0, res_par = 0;
    // prefetch cursor: next chunk whose residual is to be loaded (work item, chunk, counter)
    int pit = it0, pc = part, pq = 0;
    auto prefetch_upto = [&](int qmax) {  // issue residual loads for chunks pq .. qmax
      while (p.has_res && pq <= qmax && pit < main_items) {  // split items read no residual
        int mt2, nt2;
        tile_of<PAIR>(p, pit, rank, mt2, nt2);
        if (pc >= tile_chunks(p, nt2, BN)) {  // no (more) chunks of this warp in the tile
          pc = part;
          pit += it_step;
          continue;
        }
        const int kb = pq % C::kEpiRing;
        res_issued |= 1u << kb;
        res_par = (res_par & ~(1u << kb)) | ((uint32_t(pq / C::kEpiRing) & 1u) << kb);
        if (lane == 0) {
          bulk_wait_read<C::kEpiRing - 1 - kResAhead>();  // the store that last read this block is done
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(rbar + 8 * kb, C::kEpiBlock);
          tma_load_2d(smem_u32(ring + kb * C::kEpiBlock), &tmR, rbar + 8 * kb, nt2 * BN + 32 * pc,
                      mt2 * kBM + sub * 32);
        }
        ++pq;
        pc += kParts;
      }
    };
    prefetch_upto(kResAhead - 1);
    int q = 0;  // chunk counter of this warp: selects blocks and parities
    int local = 0;
    bool ok = true;
    const uint32_t tempty_lead0 = PAIR ? mapa_shared(bar_tempty, 0) : bar_tempty;
    for (int it = it0; it < num_items && ok; it += it_step, ++local) {
      int mt, nt, ks;
      const int ti = item_tile(it, ks);
      tile_of<PAIR>(p, ti, rank, mt, nt);
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      const int row0 = mt * kBM + sub * 32;
      const int row = row0 + lane;
      const int n0 = nt * BN;
      const int nch = tile_chunks(p, nt, BN);
      // folded LayerNorm: 1/std of this row (requested before the accumulator wait, so
      // its latency hides behind it) joins the dequantisation scale
      const float row_scale = p.ln_r ? p.scale * __ldg(p.ln_r + (row < p.M ? row : p.M - 1)) : p.scale;
      // every lane waits; the outcome is made warp-uniform so warp-collective steps stay converged
      if (!__all_sync(0xffffffffu, mbar_wait<kSleepEpi>(bar_tfull + 8 * acc, acc_phase, abort_flag, p.err))) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + uint32_t(acc * BN) + (uint32_t(sub * 32) << 16);
      if (SPLIT && ks >= 0) {  // this K range's raw sums: each 32 x 32 F32 chunk staged in the
                               // warp's 4 KB (128-byte swizzle), one TMA store to the workspace
        const int wrow = (((ti - main_items) * p.k_splits + ks) * (PAIR ? 2 : 1) + rank) * kBM + sub * 32;
        for (int c = part; c < nch; c += kParts) {
          if (lane == 0) bulk_wait_read<0>();  // the previous chunk's store has read the block
          __syncwarp();
          uint32_t pr[32];
          tmem_ld32(tbase + 32 * c, pr);
          tmem_ld_wait(pr);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(ring + lane * 128 + 16 * (u ^ (lane & 7))) =
                make_uint4(pr[4 * u], pr[4 * u + 1], pr[4 * u + 2], pr[4 * u + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmAa, smem_u32(ring), 32 * c, wrow);
            bulk_commit();
          }
        }
        tc_fence_before();
        if (PAIR)
          mbar_arrive_cluster(tempty_lead0 + 8 * acc);
        else
          mbar_arrive(bar_tempty + 8 * acc);
        continue;
      }
      // The TMEM load and the bias of chunk c + 1 are issued as soon as chunk c's
      // accumulators are in registers, so their latency hides behind chunk c's math.
      uint32_t r[32];
      uint4 bq[4];
      if (part < nch) {
        if (kLdAhead) tmem_ld32(tbase + 32 * part, r);
        load_bias(p, n0 + 32 * part, bq);
      }
      // row statistics of this tile for the next LayerNorm: sums of x - x0 and of its
      // square, x0 = the row's first value in the tile (a shift that keeps the sums small)
      float st_x0 = 0.0f, st_s1 = 0.0f, st_s2 = 0.0f, st_s1b = 0.0f, st_s2b = 0.0f;
#pragma unroll 1
      for (int c = part; c < nch; c += kParts, ++q) {
        const int kb = q % C::kEpiRing;
        uint8_t* blk = ring + kb * C::kEpiBlock;
        prefetch_upto(q + kResAhead);
        const int n = n0 + 32 * c;
        const int ngroups = min(4, (p.N - n) / 8);  // groups of 8 columns below N
        if (!kLdAhead) tmem_ld32(tbase + 32 * c, r);
        tmem_ld_wait(r);
        float v[32];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const __half2* h = reinterpret_cast<const __half2*>(&bq[g]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 t = __half22float2(h[i]);
            fma_x2(v[8 * g + 2 * i], v[8 * g + 2 * i + 1], __uint_as_float(r[8 * g + 2 * i]),
                   __uint_as_float(r[8 * g + 2 * i + 1]), row_scale, row_scale, t.x, t.y);
          }
        }
        if (c + kParts < nch) {
          if (kLdAhead) tmem_ld32(tbase + 32 * (c + kParts), r);
          load_bias(p, n + 32 * kParts, bq);
        }
        if (p.pos) {
          const size_t poff = size_t(row % p.pos_rows) * size_t(p.N) + size_t(n);
#pragma unroll
          for (int g = 0; g < 4; ++g)
            if (g < ngroups) {
              float bb[8];
              load8h(p.pos + poff + 8 * g, bb);
#pragma unroll
              for (int i = 0; i < 8; ++i) v[8 * g + i] += bb[i];
            }
        }
        if (p.act == SV_ACT_GELU_TANH) {
#pragma unroll
          for (int i = 0; i < 16; ++i) gelu_tanh_x2(v[2 * i], v[2 * i + 1]);
        }
        if (p.has_res) {
          if (!__all_sync(0xffffffffu, mbar_wait<kSleepEpi>(rbar + 8 * kb, uint32_t(q / C::kEpiRing) & 1u, abort_flag, p.err))) {
            ok = false;
            break;
          }
          const uint8_t* rrow = blk + lane * 64;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const uint4 u = *reinterpret_cast<const uint4*>(rrow + 16 * (g ^ ((lane >> 1) & 3)));
            add8h(u, v + 8 * g);
          }
          __syncwarp();  // every lane has read its residual row before the block is overwritten
        }
        if (kParts == 2 && p.ln_part) {  // two-lane sums: (even, odd) columns
          if (c == part) st_x0 = v[0];
#pragma unroll
          for (int g = 0; g < 4; ++g)
            if (g < ngroups) {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                float d0, d1;
                add_x2(d0, d1, v[8 * g + 2 * i], v[8 * g + 2 * i + 1], -st_x0, -st_x0);
                add_x2(st_s1, st_s1b, st_s1, st_s1b, d0, d1);
                fma_x2(st_s2, st_s2b, d0, d1, d0, d1, st_s2, st_s2b);
              }
            }
        }
        if (p.blk) {  // head-blocked layout for attention: 16-byte stores, consecutive rows contiguous
          if (row < p.M) {
            const int D = p.blk_H * 72;
            const int bimg = row / p.blk_T, t = row - bimg * p.blk_T;
            const size_t rowoff = (size_t(bimg) * p.blk_H * p.blk_tiles + (t >> 7)) * 18432 + (t & 127) * 16;
            const size_t which_stride = size_t(p.blk_B) * p.blk_H * p.blk_tiles * 18432;
#pragma unroll
            for (int g = 0; g < 4; ++g)
              if (g < ngroups) {
                const int col = p.blk_col0 + n + 8 * g;
                const int which = col >= 2 * D ? 2 : (col >= D ? 1 : 0);
                const int rem = col - which * D;
                const int h = (rem * 58255) >> 22;  // rem / 72, exact for rem < 4096
                const int cg = (rem - h * 72) >> 3;
                uint8_t* dst = p.blk + which * which_stride + rowoff + size_t(h) * p.blk_tiles * 18432;
                if (p.blk_qk8 && which < 2) {
                  // E4M3 Q / K: column group cg is half of the 16-column group cg / 2;
                  // the head's last group (columns 64..71) also writes the zero pad 72..79
                  uint2 w8;
                  __nv_fp8x2_storage_t* qq = reinterpret_cast<__nv_fp8x2_storage_t*>(&w8);
#pragma unroll
                  for (int i = 0; i < 4; ++i)
                    qq[i] = __nv_cvt_float2_to_fp8x2(make_float2(16.0f * v[8 * g + 2 * i], 16.0f * v[8 * g + 2 * i + 1]),
                                                     __NV_SATFINITE, __NV_E4M3);
                  uint8_t* d8 = dst + (cg >> 1) * 2048 + (cg & 1) * 8;
                  if (cg == 8)
                    *reinterpret_cast<uint4*>(d8) = make_uint4(w8.x, w8.y, 0u, 0u);
                  else
                    *reinterpret_cast<uint2*>(d8) = w8;
                  continue;
                }
                uint4 w;
                __half2* hh = reinterpret_cast<__half2*>(&w);
#pragma unroll
                for (int i = 0; i < 4; ++i) hh[i] = __floats2half2_rn(v[8 * g + 2 * i], v[8 * g + 2 * i + 1]);
                *reinterpret_cast<uint4*>(dst + cg * 2048) = w;
              }
          }
          continue;
        }
        if (!p.has_res) {  // the store that last read this block (kEpiRing chunks ago) is done
          if (lane == 0) bulk_wait_read<C::kEpiRing - 1>();
          __syncwarp();
        }
        if (!p.out_e4m3) {
          uint8_t* orow = blk + lane * 64;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint4 w;
            __half2* h = reinterpret_cast<__half2*>(&w);
#pragma unroll
            for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(v[8 * g + 2 * i], v[8 * g + 2 * i + 1]);
            *reinterpret_cast<uint4*>(orow + 16 * (g ^ ((lane >> 1) & 3))) = w;
          }
        } else {
          uint8_t* orow = blk + lane * 32;
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            uint4 w;
            __nv_fp8x2_storage_t* qq = reinterpret_cast<__nv_fp8x2_storage_t*>(&w);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              qq[i] = __nv_cvt_float2_to_fp8x2(make_float2(16.0f * v[16 * g + 2 * i], 16.0f * v[16 * g + 2 * i + 1]),
                                               __NV_SATFINITE, __NV_E4M3);
            *reinterpret_cast<uint4*>(orow + 16 * (g ^ ((lane >> 2) & 1))) = w;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmC, smem_u32(blk), n, row0);
          bulk_commit();
        }
      }
      // (mean, M2) of this row's columns of the tile, one entry per warp of the quarter
      // (two: the statistics are written by the F16 kernels only)
      if (kParts == 2 && p.ln_part && ok && row < p.M && part < nch) {
        const int w = min(BN, p.N - n0);
        int cols = 0;  // this warp's columns of the tile
        for (int c = part; c < nch; c += kParts) cols += min(32, w - 32 * c);
        const float s1 = st_s1 + st_s1b, m1 = s1 / float(cols);
        p.ln_part[(size_t(row) * p.n_tiles + nt) * 2 + part] =
            make_float2(st_x0 + m1, fmaxf(st_s2 + st_s2b - s1 * m1, 0.0f));
      }
      tc_fence_before();
      if (PAIR)
        mbar_arrive_cluster(tempty_lead0 + 8 * acc);  // the leader's MMA waits for both CTAs
      else
        mbar_arrive(bar_tempty + 8 * acc);
    }
    tmem_ld_wait();  // a load of the next chunk may be in flight after an abort
    if (lane == 0) {
      bulk_wait_all();  // every store has read shared memory and written global memory
      for (int k = 0; k < C::kEpiRing; ++k)
        if (res_issued & (1u << k)) mbar_wait_bounded(rbar + 8 * k, (res_par >> k) & 1u, p.err);
    }
    __syncwarp();
  }
  __syncthreads();
  if (PAIR) cluster_sync();  // the leader's MMAs write this CTA's TMEM: no release before they finish
  if (warp == 1) {
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else
      tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// Split-K reduction and epilogue. One warp per (row, 256-column tile), eight
// consecutive columns per lane (lane / 4 = the 32-column chunk): the splits' partial
// sums are added in split order (the result does not depend on the schedule), then
// scale, bias, positions, tanh-GELU, residual and the F16 / E4M3 store as in the GEMM
// epilogue, and the same per-half row statistics (chunks h, h + 2, ... of the tile,
// merged across lanes) for the next LayerNorm.
struct ReduceParams {
  const float* ws;
  int k_splits, n_main, n_split;  // split tiles: tile items n_main .. n_main + n_split - 1
  int row_units, rows_per;  // 128-row tiles or 256-row pairs, and their rows (128 / 256)
  int n_tiles, n_full, tail_last;
  int M, N;
  float scale;
  const __half* bias;
  const __half* pos;
  int pos_rows;
  const __half* res;
  int act, out_e4m3;
  void* out;
  float2* ln_part;
  // ROWSTATS: the whole row's LayerNorm statistics instead of ln_part (every tile split):
  // ln_r[row] = 1 / sqrt(var + eps), ln_aug[row, 0..15] = (-mean_hi, -mean_hi, -mean_lo, 0, ...)
  float* ln_r;
  __half* ln_aug;
  float eps;
};

// ROWSTATS: one block per row, warp w = column tile w (N <= 8 * 256), every tile split.
template <bool ROWSTATS>
__global__ void __launch_bounds__(256) gemm_splitk_reduce_kernel(const ReduceParams q) {
  pdl_launch_dependents();
  pdl_wait();  // the partial sums come from the GEMM launched just before
  const int lane = threadIdx.x & 31;
  int qt, r, row, nt;
  if (ROWSTATS) {
    row = int(blockIdx.x);
    nt = int(threadIdx.x >> 5);
    const int mu = row / q.rows_per;
    r = row - mu * q.rows_per;
    qt = tile_index(mu, nt, q.row_units, q.n_tiles, q.n_full, q.tail_last) - q.n_main;
  } else {
    const long wid = (long(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;  // (split tile, row of it)
    qt = int(wid / q.rows_per);
    r = int(wid - long(qt) * q.rows_per);
    if (qt >= q.n_split) return;  // whole warps
    int mu;
    tile_pos(q.n_main + qt, q.row_units, q.n_tiles, q.n_full, q.tail_last, mu, nt);
    row = mu * q.rows_per + r;
    if (row >= q.M) return;  // whole warps
  }
  const int col = nt * 256 + 8 * lane;
  const bool live = col < q.N;  // N is a multiple of 16: all eight columns exist
  // this row's sums of K range s: workspace row (qt * k_splits + s) * rows_per + r
  const float* wsr = q.ws + (size_t(qt) * q.k_splits * q.rows_per + r) * 256 + 8 * lane;
  const size_t s_stride = size_t(q.rows_per) * 256;
  float v[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
  if (live) {
    float4 a[2 * 8];
    const int ns = q.k_splits < 8 ? q.k_splits : 8;
#pragma unroll
    for (int s = 0; s < 8; ++s)
      if (s < ns) {
        const float4* src = reinterpret_cast<const float4*>(wsr + s * s_stride);
        a[2 * s] = __ldg(src);
        a[2 * s + 1] = __ldg(src + 1);
      }
#pragma unroll
    for (int s = 0; s < 8; ++s)
      if (s < ns) {
        v[0] += a[2 * s].x, v[1] += a[2 * s].y, v[2] += a[2 * s].z, v[3] += a[2 * s].w;
        v[4] += a[2 * s + 1].x, v[5] += a[2 * s + 1].y, v[6] += a[2 * s + 1].z, v[7] += a[2 * s + 1].w;
      }
    for (int s = 8; s < q.k_splits; ++s) {
      const float4* src = reinterpret_cast<const float4*>(wsr + s * s_stride);
      const float4 x = __ldg(src), y = __ldg(src + 1);
      v[0] += x.x, v[1] += x.y, v[2] += x.z, v[3] += x.w, v[4] += y.x, v[5] += y.y, v[6] += y.z, v[7] += y.w;
    }
    float b[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
    if (q.bias) load8h(q.bias + col, b);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = fmaf(v[i], q.scale, b[i]);
    if (q.pos) {
      float pp[8];
      load8h(q.pos + size_t(row % q.pos_rows) * size_t(q.N) + size_t(col), pp);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] += pp[i];
    }
    if (q.act == SV_ACT_GELU_TANH) {
#pragma unroll
      for (int i = 0; i < 4; ++i) gelu_tanh_x2(v[2 * i], v[2 * i + 1]);
    }
    const size_t off = size_t(row) * q.N + col;
    if (q.res) add8h(__ldg(reinterpret_cast<const uint4*>(q.res + off)), v);
    if (!q.out_e4m3) {
      uint4 w;
      __half2* h = reinterpret_cast<__half2*>(&w);
#pragma unroll
      for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
      *reinterpret_cast<uint4*>(static_cast<__half*>(q.out) + off) = w;
    } else {
      uint2 w;
      __nv_fp8x2_storage_t* c8 = reinterpret_cast<__nv_fp8x2_storage_t*>(&w);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        c8[i] = __nv_cvt_float2_to_fp8x2(make_float2(16.0f * v[2 * i], 16.0f * v[2 * i + 1]), __NV_SATFINITE,
                                         __NV_E4M3);
      *reinterpret_cast<uint2*>(static_cast<uint8_t*>(q.out) + off) = w;
    }
  }
  if (ROWSTATS || q.ln_part) {  // (mean, M2): this lane's columns, its chunk, then the chunks of each parity
    float n = 0.0f, mean = 0.0f, m2 = 0.0f;
    if (live) {
      float sum = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) sum += v[i];
      mean = sum * 0.125f;
#pragma unroll
      for (int i = 0; i < 8; ++i) m2 = fmaf(v[i] - mean, v[i] - mean, m2);
      n = 8.0f;
    }
#pragma unroll
    for (int o = 1; o <= 16; o <<= 1) {
      if (!ROWSTATS && o == 4) continue;  // lane bit 2 is the chunk's parity: the halves stay apart
      const float nb = __shfl_xor_sync(0xffffffffu, n, o), mb = __shfl_xor_sync(0xffffffffu, mean, o),
                  m2b = __shfl_xor_sync(0xffffffffu, m2, o);
      chan_merge(n, mean, m2, nb, mb, m2b);
    }
    if (!ROWSTATS) {
      if ((lane == 0 || lane == 4) && n > 0.0f)
        q.ln_part[(size_t(row) * q.n_tiles + nt) * 2 + (lane >> 2)] = make_float2(mean, m2);
    } else {  // the row's tiles merged by its first thread, then 1/std and the -mean block
      __shared__ float3 tile_st[8];
      if (lane == 0) tile_st[nt] = make_float3(n, mean, m2);
      __syncthreads();
      if (threadIdx.x == 0) {
        float rn = 0.0f, rm = 0.0f, rm2 = 0.0f;
        for (int t = 0; t < q.n_tiles; ++t) chan_merge(rn, rm, rm2, tile_st[t].x, tile_st[t].y, tile_st[t].z);
        q.ln_r[row] = rsqrtf(rm2 / float(q.N) + q.eps);
        const __half hi = __float2half_rn(-rm);
        const __half lo = __float2half_rn(-rm - __half2float(hi));
        uint4 w;
        __half2* h = reinterpret_cast<__half2*>(&w);
        h[0] = __halves2half2(hi, hi);
        h[1] = __halves2half2(lo, __float2half_rn(0.0f));
        h[2] = h[3] = __float2half2_rn(0.0f);
        uint4* dst = reinterpret_cast<uint4*>(q.ln_aug + size_t(row) * 16);
        dst[0] = w;
        dst[1] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
}

template <int BN, bool FP8, bool PAIR, int ATOMS = 1, int SPLIT = 0, int EPI = (FP8 && PAIR) ? 12 : 8>
sv_status launch_bn(const GemmOperands& g, const Params& prm, cudaStream_t s) {
  using C = Cfg<BN, PAIR, ATOMS, EPI>;
  auto kern = gemm_tc_kernel<BN, FP8, PAIR, ATOMS, SPLIT, EPI>;
  // the attribute is per device: set it once on each device the kernel runs on
  static unsigned long long attr_set = 0;
  int dev = 0;
  cudaError_t de = cudaGetDevice(&dev);
  if (de != cudaSuccess) return cuda_fail(de, "cudaGetDevice(gemm)");
  const unsigned long long bit = (dev >= 0 && dev < kMaxAttrDevices) ? 1ull << dev : 0ull;
  if (!(attr_set & bit) || !bit) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(gemm)");
    attr_set |= bit;
  }
  const int tile_items = PAIR ? ((prm.m_tiles + 1) / 2) * prm.n_tiles : prm.m_tiles * prm.n_tiles;
  const int n_main = SPLIT == 1 ? 0 : prm.n_main;
  const int items = SPLIT ? n_main + (tile_items - n_main) * prm.k_splits : tile_items;
  const int slots = PAIR ? num_sms() / 2 : num_sms();  // one CTA (PAIR: one two-CTA cluster) per SM (pair)
  const int units = items < slots ? items : slots;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.gridDim = dim3(unsigned(PAIR ? 2 * units : units), 1, 1);
  cfg.blockDim = dim3(gemm_threads<EPI>(), 1, 1);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  // programmatic stream serialization: the prologue (barriers, TMEM, tensor-map
  // prefetch) may overlap the previous kernel's tail; the kernel waits before any
  // global access
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (PAIR) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  const CUtensorMap& tr = g.has_res ? g.tr : g.tc;
  const CUtensorMap& twt = (PAIR && g.tail_n) ? g.tw_tail : g.tw;
  // split K: the workspace map takes the place of the (unused) folded-LayerNorm A block
  const CUtensorMap& taa = SPLIT ? g.tws : (prm.ln_aug ? g.ta_aug : g.ta);
  const CUtensorMap& twa = prm.ln_aug ? g.tw_aug : g.tw;
  const CUtensorMap& twat = (prm.ln_aug && PAIR && g.tail_n) ? g.tw_aug_tail : twa;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, g.ta, g.tw, twt, g.tc, tr, taa, twa, twat, prm);
  if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
  return SV_OK;
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  }
  return fn;
}

}  // namespace

sv_status make_tmap(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* ptr, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle sw) {
  EncodeFn fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return SV_ERR_CUDA;
  }
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) gs[i] = strides_bytes[i];
  }
  CUresult r = fn(m, dt, cuuint32_t(rank), const_cast<void*>(ptr), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d): rank %d dims0 %llu dims1 %llu box %u x %u", int(r), rank,
              (unsigned long long)dims[0], (unsigned long long)(rank > 1 ? dims[1] : 0), box[0],
              rank > 1 ? box[1] : 0);
    return SV_ERR_INVALID_ARG;
  }
  return SV_OK;
}

sv_status gemm_operand_map(CUtensorMap* m, const void* ptr, int rows, int K, int fp8, int box_rows) {
  const uint64_t dims[2] = {uint64_t(K), uint64_t(rows)};
  const uint64_t strides[1] = {uint64_t(K) * (fp8 ? 1u : 2u)};
  const uint32_t box[2] = {uint32_t(fp8 ? kSwzBytes : kSwzBytes / 2), uint32_t(box_rows)};
  return make_tmap(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, ptr, dims, strides,
                   box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Output-tile width: estimated time = waves x per-tile time, with the per-tile
// time proportional to BN / (sustained TFLOP/s of that width). The rates are the
// ones measured on GB300 for 23,328-row GEMMs with the copies and epilogue
// running (TFLOP/s at 256 / 192 / 128 / 64 columns: about 1780 / 1480 / 1000 /
// 600): wide tiles win whenever there are enough of them to fill the SMs.
int gemm_pick_bn(int M, int N, int K, bool pair, double* t_best, int sms) {
  const int cand[4] = {256, 192, 128, 64};
  const double rate[4] = {1780.0, 1480.0, 1000.0, 600.0};
  if (sms <= 0) sms = 148;
  int best = 256;
  double best_t = 1e30;
  const int mt = (M + kBM - 1) / kBM;
  for (int i = 0; i < 4; ++i) {
    const int bn = cand[i];
    const long tiles = long(pair ? 2 * ((mt + 1) / 2) : mt) * ((N + bn - 1) / bn);
    const long waves = (tiles + sms - 1) / sms;
    const double t = double(waves) * bn / rate[i] * double(K);
    if (t < best_t * 0.999) {
      best_t = t;
      best = bn;
    }
  }
  if (t_best) *t_best = best_t;
  return best;
}

namespace {

// Split K. At small M a long-K GEMM's tiles fill few SMs, each streaming all of K.
// Splitting K into ranges gives 256-wide tiles on most SMs, plus a reduction kernel
// whose cost does not shrink with the main loop. In gemm_pick_bn's time units (E4M3
// main loops at half the F16 time) the reduction costs about 125, from measured times
// (us per call, unsplit -> split): F16 729 x 1152 x 4304 24.0 -> 16.3 (5 ranges),
// 1458 rows 25.3 -> 23.0 (2), 32 rows 22.5 -> 11.2 (8); E4M3 32 rows 12.9 -> 10.4 (8),
// while E4M3 729 rows (14.1 vs 14.4 split) and 1458 rows (15.8 vs 19.6) stay whole.
// Returns the number of K ranges (1: no split); sets *bn and *mc for the split layout.
int pick_splits(int M, int N, int K, int fp8, bool allow_pair, int max_splits, double t_unsplit, int* bn,
                int* mc, int sms) {
  constexpr double kReduceCost = 125.0;
  if (max_splits < 2 || K < 2048) return 1;
  const int mt = (M + kBM - 1) / kBM;
  const bool pair = allow_pair && mt >= 2 && sms >= 2;
  const int w = 256;
  const int items = (pair ? (mt + 1) / 2 : mt) * ((N + w - 1) / w);
  const int slots = pair ? sms / 2 : sms;
  const int k_blocks = (K + (fp8 ? kSwzBytes : kSwzBytes / 2) - 1) / (fp8 ? kSwzBytes : kSwzBytes / 2);
  int splits = slots / items;
  if (splits > max_splits) splits = max_splits;
  const int min_blocks = fp8 ? 4 : 8;  // at least 512 K elements a range
  if (splits > k_blocks / min_blocks) splits = k_blocks / min_blocks;
  if (splits < 2) return 1;
  const double f = fp8 ? 0.5 : 1.0;  // main-loop time relative to F16
  const double t_split = f * double(w) / 1780.0 * double(K) / splits + kReduceCost;
  if (t_split > 0.8 * f * t_unsplit) return 1;
  *bn = w;
  *mc = pair ? 1 : 0;
  return splits;
}

// Split the tiles of a short last wave. When a long-K GEMM's tiles fill all CTAs
// (pairs) for some waves and then only a few of them, the last round runs those few
// tiles at whole K while the rest wait (the 23,328 x 1152 x 4304 MLP-down projection:
// 460 pair tiles on 76 pairs, 4 in the seventh round). Their K is split over the idle
// pairs instead and the reduction finishes them. Measured on that shape: 161.1 -> 152.1
// us with F16 operands (the whole step at 32 images 0.9% faster), a round of one narrow
// tile (128 columns, 93,312 rows) no gain, and E4M3 99.2 -> 102.2 us (its main loop is
// short against the epilogue); so F16 only, and only when the round shortens by more than
// three reductions (gemm_pick_bn's time units, as pick_splits).
void pick_tail_split(GemmOperands* g, int k_blocks, int sms) {
  constexpr double kReduceCost = 125.0;
  if (g->fp8 || g->K < 2048 || g->bn != 256 || g->atoms != 1) return;
  const int mt = (g->M + kBM - 1) / kBM, units = g->mc ? (mt + 1) / 2 : mt;
  const int n_tiles = (g->N + g->bn - 1) / g->bn, n_full = g->tail_n ? n_tiles - 1 : n_tiles;
  const int items = units * n_tiles, slots = g->mc ? sms / 2 : sms;
  const int rem = items % slots;
  if (items < slots || rem == 0 || rem * 8 > slots) return;
  int splits = slots / rem;
  if (splits > 8) splits = 8;
  if (splits > k_blocks / 8) splits = k_blocks / 8;
  if (splits < 2) return;
  int width = 0;  // the widest tile of the last round
  for (int it = items - rem; it < items; ++it) {
    int mu, nt;
    tile_pos(it, units, n_tiles, n_full, g->tail_last, mu, nt);
    const int w = (nt == n_full && g->tail_n) ? g->tail_n : g->bn;
    width = w > width ? w : width;
  }
  const double t_tile = double(width) / 1780.0 * double(g->K);
  if (t_tile * (1.0 - 1.0 / splits) <= 3.0 * kReduceCost) return;
  g->k_splits = splits;
  g->n_main = items - rem;
}

// Tile, pairing, stage and split choices for an M x N x K GEMM on `sms` SMs (no tensor maps).
void gemm_choose(GemmOperands* g, int M, int N, int K, int fp8, bool allow_pair, int max_splits, int sms) {
  if (sms <= 0) sms = 148;
  g->M = M;
  g->N = N;
  g->K = K;
  g->fp8 = fp8;
  g->has_aug = 0;
  // CTA pairs (256-row tiles, half the W traffic per SM, deeper pipelines) for K >= 1024
  // or wide N (every encoder GEMM but the patch embedding). A single CTA's 128 x 256 tile
  // moves 96 KB through shared memory per 64-wide K block (TMA writes and MMA reads of A
  // and W), more than shared memory delivers in the block's 512 tensor cycles; a pair
  // halves the W part. Measured on the 27-layer encoder: about 2% faster on the MLP and
  // QKV GEMMs, and with two swizzle rows of K per stage 1% per step faster on the
  // 1152 x 1152 output projection (batch 32 and 128).
  g->mc = allow_pair && (M + kBM - 1) / kBM >= 2 && sms >= 2 && (K >= 1024 || N >= 2048);
  double t_unsplit = 0.0;
  g->bn = gemm_pick_bn(M, N, K, g->mc, &t_unsplit, sms);
  if (g->mc && g->bn > kPairMaxBn) g->bn = kPairMaxBn;
  g->k_splits = pick_splits(M, N, K, fp8, allow_pair, max_splits, t_unsplit, &g->bn, &g->mc, sms);
  // two swizzle rows of K per stage for 256-wide F16 CTA-pair tiles over a short K that
  // they divide (see Cfg). Not for E4M3: over K = 1152 half of the last stage would be
  // empty, and with the E4M3 pairs' wider epilogue only two 64 KB stages would fit.
  g->atoms = (!fp8 && g->mc && g->bn == 256 && K <= 2048 && K % (2 * kSwzBytes / 2) == 0 && g->k_splits == 1) ? 2 : 1;
  g->kb_split = 0;
  g->n_main = 0;  // with a small-M split every tile is split

  // A narrower last column tile (N % bn columns) runs MMAs of its own width, rounded
  // up to 16 columns (32 for a CTA pair, whose CTAs hold half of the W rows each).
  const int rem = N % g->bn;
  const int gran = g->mc ? 32 : 16;
  const int tail = (rem + gran - 1) / gran * gran;
  g->tail_n = (rem != 0 && tail < g->bn) ? tail : 0;
  g->tail_last = 0;
  if (g->tail_n) {
    // Narrow tiles last when that shortens the busiest CTA's (pair's) share of the
    // round-robin tile schedule by 5% or more, and A is small enough (<= 64 MB) to be
    // read again from L2 rather than DRAM by the narrow tiles. (Measured on the
    // encoder's GEMMs: a 3% shorter schedule did not pay for the second pass over A.)
    const int mu = g->mc ? ((M + kBM - 1) / kBM + 1) / 2 : (M + kBM - 1) / kBM;
    const int nt_all = (N + g->bn - 1) / g->bn, nf = nt_all - 1;
    const int units = g->mc ? sms / 2 : sms;
    const long items = long(mu) * nt_all;
    auto makespan = [&](bool tail_last) {
      long worst = 0;
      for (int c = 0; c < units && c < items; ++c) {
        long t = 0;
        for (long it = c; it < items; it += units) {
          const bool narrow = tail_last ? it >= long(mu) * nf : (it % nt_all) == nf;
          t += narrow ? g->tail_n : g->bn;
        }
        worst = t > worst ? t : worst;
      }
      return worst;
    };
    const double a_bytes = double(M) * K * (fp8 ? 1 : 2);
    if (units > 0 && a_bytes <= 64e6 && makespan(true) * 20 <= makespan(false) * 19) g->tail_last = 1;
  }
  const int bk = (fp8 ? kSwzBytes : kSwzBytes / 2) * g->atoms;
  const int k_blocks = (K + bk - 1) / bk;
  if (g->k_splits == 1 && max_splits > 1) pick_tail_split(g, k_blocks, sms);
  if (g->k_splits > 1) {  // equal ranges of whole stages; no range is empty
    g->kb_split = (k_blocks + g->k_splits - 1) / g->k_splits;
    g->k_splits = (k_blocks + g->kb_split - 1) / g->kb_split;
  }
}

}  // namespace

size_t gemm_splitk_ws_bytes(const GemmOperands& g) {
  if (g.k_splits <= 1) return 0;
  const int mt = (g.M + kBM - 1) / kBM, units = g.mc ? (mt + 1) / 2 : mt;
  const int n_split = units * ((g.N + g.bn - 1) / g.bn) - g.n_main;
  return size_t(n_split) * g.k_splits * (g.mc ? 2 : 1) * size_t(kBM) * g.bn * sizeof(float);
}

size_t gemm_splitk_ws_bytes_for(int M, int N, int K, int fp8, int max_splits) {
  GemmOperands g;
  gemm_choose(&g, M, N, K, fp8, true, max_splits, num_sms());
  return gemm_splitk_ws_bytes(g);
}

sv_status gemm_prepare(GemmOperands* g, const void* A, const void* W, int M, int N, int K, int fp8,
                       bool allow_pair, int max_splits) {
  gemm_choose(g, M, N, K, fp8, allow_pair, max_splits, num_sms());
  sv_status st = gemm_operand_map(&g->ta, A, M, K, fp8, kBM);
  if (st != SV_OK) return st;
  st = gemm_operand_map(&g->tw, W, N, K, fp8, g->mc ? g->bn / 2 : g->bn);
  if (st != SV_OK) return st;
  if (g->mc && g->tail_n) return gemm_operand_map(&g->tw_tail, W, N, K, fp8, g->tail_n / 2);
  return SV_OK;
}

// Output (and residual) maps of a [M, N] row-major matrix in 32 x 32 blocks:
// F16 with 64-byte rows and the 64-byte swizzle, E4M3 with 32-byte rows and
// the 32-byte swizzle (the layout the epilogue writes in shared memory).
sv_status gemm_output_map(CUtensorMap* m, const void* ptr, int M, int N, int e4m3) {
  const uint64_t dims[2] = {uint64_t(N), uint64_t(M)};
  const uint64_t strides[1] = {uint64_t(N) * (e4m3 ? 1u : 2u)};
  const uint32_t box[2] = {32, 32};
  return make_tmap(m, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, ptr, dims, strides,
                   box, e4m3 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B);
}

// The folded LayerNorm's extra K block: [rows, 16] F16 tiles with 32-byte rows in
// the 32-byte swizzle (the layout the MMA descriptor names).
sv_status gemm_aug_map(CUtensorMap* m, const void* ptr, int rows, int box_rows) {
  const uint64_t dims[2] = {16, uint64_t(rows)};
  const uint64_t strides[1] = {32};
  const uint32_t box[2] = {16, uint32_t(box_rows)};
  return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_32B);
}

sv_status gemm_bind_epilogue(GemmOperands* g, const GemmEpi& e) {
  if (e.ln_r && e.ln_aug_a && e.ln_aug_w && !g->fp8) {
    sv_status st = gemm_aug_map(&g->ta_aug, e.ln_aug_a, g->M, kBM);
    if (st == SV_OK) st = gemm_aug_map(&g->tw_aug, e.ln_aug_w, g->N, g->mc ? g->bn / 2 : g->bn);
    if (st == SV_OK && g->mc && g->tail_n) st = gemm_aug_map(&g->tw_aug_tail, e.ln_aug_w, g->N, g->tail_n / 2);
    if (st != SV_OK) return st;
    g->has_aug = 1;
  }
  sv_status st = gemm_output_map(&g->tc, e.out, g->M, g->N, e.out_e4m3);
  if (st != SV_OK) return st;
  g->has_res = e.residual != nullptr;
  g->out = e.out;
  g->out_e4m3 = e.out_e4m3;
  g->res = e.residual;
  g->ws = nullptr;
  if (g->k_splits > 1 && e.ws) {  // split K: [rows, BN] F32 (Params), 32 x 32 blocks, 128-byte swizzle
    const uint64_t rows = gemm_splitk_ws_bytes(*g) / (sizeof(float) * size_t(g->bn));
    const uint64_t dims[2] = {uint64_t(g->bn), rows};
    const uint64_t strides[1] = {uint64_t(g->bn) * 4u};
    const uint32_t box[2] = {32, 32};
    st = make_tmap(&g->tws, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, e.ws, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != SV_OK) return st;
    g->ws = e.ws;
  }
  if (g->has_res) return gemm_output_map(&g->tr, e.residual, g->M, g->N, 0);
  return SV_OK;
}

namespace {

sv_status launch_main(const GemmOperands& g, const Params& p, cudaStream_t s, bool split) {
  if (split) {  // split K: 256-wide tiles, one swizzle row of K per stage (gemm_choose)
    const int key = (g.bn == 256 && g.atoms == 1) ? (g.fp8 ? 1 : 0) | (g.mc ? 2 : 0) | (g.n_main ? 4 : 0) : -1;
    switch (key) {
      case 0: return launch_bn<256, false, false, 1, 1>(g, p, s);
      case 1: return launch_bn<256, true, false, 1, 1>(g, p, s);
      case 2: return launch_bn<256, false, true, 1, 1>(g, p, s);
      case 3: return launch_bn<256, true, true, 1, 1>(g, p, s);
      case 4: return launch_bn<256, false, false, 1, 2>(g, p, s);  // a split last round (F16 only)
      case 6: return launch_bn<256, false, true, 1, 2>(g, p, s);
      default: set_error("gemm: no split-K kernel for this configuration"); return SV_ERR_UNSUPPORTED;
    }
  }
  const int key = g.bn | (g.fp8 ? 1 : 0) | (g.mc ? 2 : 0) | (g.atoms == 2 ? 4 : 0);
  switch (key) {
    case 256: return launch_bn<256, false, false>(g, p, s);
    case 257: return launch_bn<256, true, false>(g, p, s);
    case 258: return launch_bn<256, false, true>(g, p, s);
    case 259: return launch_bn<256, true, true>(g, p, s);
    case 262: return launch_bn<256, false, true, 2>(g, p, s);
    case 192: return launch_bn<192, false, false>(g, p, s);
    case 193: return launch_bn<192, true, false>(g, p, s);
    case 194:  // twelve epilogue warps unless the GEMM keeps LayerNorm statistics
      return p.ln_part ? launch_bn<192, false, true>(g, p, s) : launch_bn<192, false, true, 1, 0, 12>(g, p, s);
    case 195: return launch_bn<192, true, true>(g, p, s);
    case 128: return launch_bn<128, false, false>(g, p, s);
    case 129: return launch_bn<128, true, false>(g, p, s);
    case 130: return launch_bn<128, false, true>(g, p, s);
    case 131: return launch_bn<128, true, true>(g, p, s);
    case 64: return launch_bn<64, false, false>(g, p, s);
    case 65: return launch_bn<64, true, false>(g, p, s);
    case 66: return launch_bn<64, false, true>(g, p, s);
    case 67: return launch_bn<64, true, true>(g, p, s);
    default: set_error("gemm: no kernel for tile width %d", g.bn); return SV_ERR_UNSUPPORTED;
  }
}

}  // namespace

sv_status gemm_launch(const GemmOperands& g, const GemmEpi& e, cudaStream_t s, int part) {
  if (e.out != g.out || e.out_e4m3 != g.out_e4m3 || e.residual != g.res) {
    set_error("gemm: epilogue buffers differ from the ones the tensor maps were built for");
    return SV_ERR_INVALID_ARG;
  }
  const bool split = g.k_splits > 1;
  Params p;
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.m_tiles = (g.M + kBM - 1) / kBM;
  p.n_tiles = (g.N + g.bn - 1) / g.bn;
  p.tail_n = g.tail_n;
  p.n_full = g.tail_n ? p.n_tiles - 1 : p.n_tiles;
  p.tail_last = g.tail_last;
  const int bk = (g.fp8 ? kSwzBytes : kSwzBytes / 2) * g.atoms;
  p.k_blocks = (g.K + bk - 1) / bk;
  p.bias = e.bias;
  p.pos = e.pos;
  p.pos_rows = e.pos_rows > 0 ? e.pos_rows : 1;
  p.has_res = e.residual != nullptr;
  p.out = e.out;
  p.blk = static_cast<uint8_t*>(e.blk_out);
  p.blk_T = e.blk_T;
  p.blk_H = e.blk_H;
  p.blk_B = e.blk_B;
  p.blk_col0 = e.blk_col0;
  p.blk_qk8 = e.blk_qk8;
  p.ln_part = e.ln_part;
  // (E4M3 pair kernels run three epilogue warps per lane quarter, which keep no statistics:
  // only a GEMM whose every tile is split, and so reduced, can give them)
  if (e.ln_part && (e.blk_out || 2 * p.n_tiles > kMaxLnTiles || (g.fp8 && g.mc && (!split || g.n_main > 0)))) {
    set_error("gemm: row statistics need a row-major output of at most %d column tiles (and not E4M3 operands "
              "with CTA pairs)", kMaxLnTiles / 2);
    return SV_ERR_INVALID_ARG;
  }
  p.blk_tiles = (e.blk_T + 127) / 128;
  p.act = e.act;
  p.out_e4m3 = e.out_e4m3;
  p.scale = e.scale;
  p.ln_r = e.ln_r;
  p.ln_aug = e.ln_r != nullptr;
  if (e.ln_r && (!e.ln_aug_a || !e.ln_aug_w || e.pos || g.fp8 || !g.has_aug)) {
    set_error("gemm: a folded LayerNorm needs its extra K block and F16 operands");
    return SV_ERR_INVALID_ARG;
  }
  p.err = dev_err();
  p.k_splits = split ? g.k_splits : 1;
  p.kb_split = split ? g.kb_split : 0;
  p.n_main = split ? g.n_main : 0;
  if (!split) return part == 1 ? SV_OK : launch_main(g, p, s, false);
  if (!e.ws || e.ws != g.ws || e.ln_r || e.blk_out || g.bn != 256) {
    set_error("gemm: a split-K GEMM needs the partial-sum workspace its maps were built for and a row-major "
              "output without a folded LayerNorm");
    return SV_ERR_INVALID_ARG;
  }
  if ((e.ln_r_out || e.ln_aug_out) && (!e.ln_r_out || !e.ln_aug_out || e.ln_part || g.n_main || p.n_tiles > 8)) {
    set_error("gemm: whole-row LayerNorm statistics need every tile split, at most 8 column tiles, and no "
              "per-tile statistics");
    return SV_ERR_INVALID_ARG;
  }
  if (part != 1) {  // whole tiles with their epilogue, and the split tiles' K ranges' raw sums
    sv_status st = launch_main(g, p, s, true);
    if (st != SV_OK || part == 0) return st;
  }
  // the split tiles: their ranges' sums added up and the epilogue
  const int units = g.mc ? (p.m_tiles + 1) / 2 : p.m_tiles;
  ReduceParams q;
  q.ws = e.ws;
  q.k_splits = g.k_splits;
  q.n_main = g.n_main;
  q.n_split = units * p.n_tiles - g.n_main;
  q.row_units = units;
  q.rows_per = g.mc ? 2 * kBM : kBM;
  q.n_tiles = p.n_tiles;
  q.n_full = p.n_full;
  q.tail_last = p.tail_last;
  q.M = g.M;
  q.N = g.N;
  q.scale = e.scale;
  q.bias = e.bias;
  q.pos = e.pos;
  q.pos_rows = p.pos_rows;
  q.res = e.residual;
  q.act = e.act;
  q.out_e4m3 = e.out_e4m3;
  q.out = e.out;
  q.ln_part = e.ln_part;
  q.ln_r = e.ln_r_out;
  q.ln_aug = e.ln_aug_out;
  q.eps = e.ln_eps;
  cudaError_t ce;
  if (e.ln_r_out) {  // one block per row, a warp per column tile
    ce = launch_pdl(gemm_splitk_reduce_kernel<true>, dim3(unsigned(g.M)), dim3(unsigned(32 * p.n_tiles)), 0, s, q);
  } else {
    const long warps = long(q.n_split) * q.rows_per;
    ce = launch_pdl(gemm_splitk_reduce_kernel<false>, dim3(unsigned((warps + 7) / 8)), dim3(256), 0, s, q);
  }
  if (ce != cudaSuccess) return cuda_fail(ce, "gemm split-K reduction launch");
  return SV_OK;
}

}  // namespace sv

// The tile, pairing, stage and split choices for an M x N x K GEMM on `sms` SMs, as
// gemm_prepare makes them with max_splits (a host-only computation, for tests).
extern "C" sv_status sv_debug_gemm_plan(int M, int N, int K, int gemm_dtype, int sms, int max_splits, int* out,
                                        size_t* ws_bytes) {
  if (M < 1 || N < 16 || K < 16 || N % 16 || K % 16 || (gemm_dtype != 0 && gemm_dtype != 1) || sms < 1 ||
      max_splits < 1 || !out) {
    sv::set_error("sv_debug_gemm_plan: bad arguments");
    return SV_ERR_INVALID_ARG;
  }
  sv::GemmOperands g;
  sv::gemm_choose(&g, M, N, K, gemm_dtype, true, max_splits, sms);
  const int v[8] = {g.bn, g.mc, g.atoms, g.tail_n, g.tail_last, g.k_splits, g.kb_split, g.n_main};
  for (int i = 0; i < 8; ++i) out[i] = v[i];
  if (ws_bytes) *ws_bytes = sv::gemm_splitk_ws_bytes(g);
  return SV_OK;
}
