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
// FP8 score products ("FP8 attention and resident image/embedding transfers",
// Projected attention: the QK product on E4M3 operands at scale 2^-4, both
// operands written quantised by their producer): Q and K blocks hold E4M3(16 x)
// in 16-value groups (10 KB a tile), S = Q K^T runs as three kind::f8f6f4 MMAs
// of K = 32 (72 columns padded to 96) and the softmax scale absorbs the 2^-8;
// P V stays F16 (P reaches 2^15, beyond E4M3's range).
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
// Persistent CTAs (one per SM) walk work items of (256 queries as two 128-row
// tiles, head, image); 320 threads:
//   warp 0      bulk copies: Q (both tiles) of the next item into a staging buffer,
//               K and V tiles of 128 keys into 3 + 3 stages, each with its own release;
//   warp 1      the MMA issuer, in the order S_0(0), S_1(0), then per key tile t:
//               O_0 += P_0(t) V_t, S_0(t+1), O_1 += P_1(t) V_t, S_1(t+1), where
//               S_w = Q_w K^T (M 128, N 128) and O_w += P_w V (M 128, N 80). Q_w and
//               P_w are read from tensor memory, only K and V from shared memory. The
//               MMAs of one thread run in issue order, so S_w(t+1) overwrites P_w(t)
//               only after the P V product has read it, and the completion of S_w(t+1)
//               also means that O_w holds the sum up to tile t. One issuer for both
//               groups staggers them: group 1's products run while group 0 computes
//               its softmax, and the other way round;
//   warps 2..5  softmax group 0, warps 6..9 softmax group 1: one thread per query
//               row reads its S row from TMEM, writes P = 2^(scale s - m) as F16
//               pairs back over the first 64 columns of S, and rescales O in TMEM
//               only when the row maximum grows by more than 2^15; the softmax
//               denominator comes out of the P V product (a column of ones in V's
//               pad group). On an item's last tile the group also moves the next
//               item's Q rows from the staging buffer into TMEM; an item's output rows
//               are written from registers at the start of the group's next item.
// Shared-memory traffic per key tile is then the K and V copies and their reads by
// the tensor core: an N = 80 or N = 128 product with both operands in shared memory
// needs about as many bytes per cycle as shared memory delivers.
//
// Small grids: when every 128-query tile can have a CTA of its own in the first round
// (one image of 729 tokens and 16 heads: 96 tiles, against 48 two-tile items), a
// second kernel (attention_slots_kernel) takes items of one tile, 320 threads:
//   warp 0      bulk copies: Q of an item into one of two buffers, K and V tiles into
//               4 + 3 stages;
//   warp 1      the MMA issuer: S(t) = Q K_t^T (Q and K from shared memory) into one of
//               three score slots in tensor memory, O += P(t) V_t (P from the slot), in
//               the order S(0), S(1), S(2), then per key tile t: P(t) V_t, S(t+3), so the
//               scores run three tiles ahead of the softmax; issue order keeps S(t+3) from
//               overwriting P(t) before the P V product has read it;
//   warps 2..9  the softmax, two warps per TMEM lane quarter, one for keys 0..63 and one
//               for keys 64..127 of each tile, the row maximum combined through shared
//               memory; P over the first 32 columns of each half's S, O rescaled per half.
// Tensor memory holds the three score slots (3 x 128 columns) and O (80). On a full grid
// this kernel is slower than the two-tile one: the row-maximum exchange between its two
// warps sits on every tile's path.

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
// E4M3 Q / K tiles (FP8 score products): 5 groups of 16 values in memory (72 columns and
// 8 zero bytes), 6 in shared memory (96 columns: three MMA K steps of 32)
constexpr int kGroups8 = 5;
constexpr int kOpBytes8 = 6 * kGroupBytes;
constexpr int kThreads = 320;
constexpr int kBarBytes = 384;  // barriers, TMEM address slot, abort flag

// Shared memory map (offsets from the 1024-aligned base) for QB query staging buffers
// (of two tiles each), KS key stages and VS value stages; QK8: E4M3 Q and K tiles.
template <int QB, int KS, int VS, bool QK8>
struct Smem {
  static constexpr int kQKOp = QK8 ? kOpBytes8 : kOpBytes;  // one Q or K tile
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * QB * kQKOp;
  static constexpr int kOffV = kOffK + KS * kQKOp;
  static constexpr int kOffBar = kOffV + VS * kOpBytes;
  static constexpr int kBytes = 1024 + kOffBar + kBarBytes;
  static_assert(kBytes <= 232448, "shared memory budget");
  static_assert(QB >= 1 && QB <= 2 && KS >= 2 && KS <= 4 && VS >= 2 && VS <= 4, "buffer counts");
};

// TMEM columns: S_w at 128 w (P_w, 64 columns of F16 pairs, over its first half), O_w
// at 256 + 80 w, Q_w at 416 + 48 w (40 columns of F16 pairs, or 24 of E4M3 quads).
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
  kBarQFull = 0,    // +buffer
  kBarQEmpty = 2,   // +buffer: every softmax thread has moved its Q row into TMEM
  kBarKFull = 4,    // +stage
  kBarKEmpty = 8,   // +stage
  kBarVFull = 12,   // +stage
  kBarVEmpty = 16,  // +stage
  kBarSFull = 20,   // +group: S_w(t) has finished (and with it O_w += P_w(t-1) V_{t-1})
  kBarPFull = 22,   // +group: the group has written P_w(t) (and any O rescale, and on an
                    //   item's last tile the next item's Q) to TMEM
  kBarQtFull = 24,  // +group: the first item's Q rows are in TMEM
  kBarDrain = 26,
  kNumBars = 27
};
static_assert(8 * kNumBars + 8 <= kBarBytes, "barrier area");

// The reference maximum of a row (log2 units) is raised only when a tile's
// maximum exceeds it by more than this: P <= 2^15 stays finite in F16 (whose
// relative precision does not depend on the magnitude), and O is rescaled rarely.
constexpr float kSlack = 15.0f;

// Zeros for the rows of a partial V tile past the last token.
__device__ __align__(128) uint8_t g_zero_rows[kGroupBytes];

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

// Copies the existing rows of the first `groups` column groups of one operand tile;
// returns the bytes it will deliver.
__device__ __forceinline__ uint32_t copy_tile(uint32_t dst, const uint8_t* src, int rows, uint32_t bar,
                                              int groups) {
  if (rows == kTile) {
    bulk_copy(dst, src, uint32_t(groups * kGroupBytes), bar);
    return uint32_t(groups * kGroupBytes);
  }
  for (int g = 0; g < groups; ++g) bulk_copy(dst + g * kGroupBytes, src + g * kGroupBytes, rows * 16, bar);
  return uint32_t(groups * rows * 16);
}

// As copy_tile, and the rows past the last token are filled with zeros (a V tile:
// its masked keys have P = 0, and 0 times a zero row stays 0 whatever the buffer
// held before).
__device__ __forceinline__ uint32_t copy_tile_zero_tail(uint32_t dst, const uint8_t* src, int rows, uint32_t bar) {
  if (rows == kTile) {
    bulk_copy(dst, src, kBlockBytes, bar);
    return kBlockBytes;
  }
  for (int g = 0; g < kGroups; ++g) {
    bulk_copy(dst + g * kGroupBytes, src + g * kGroupBytes, rows * 16, bar);
    bulk_copy(dst + g * kGroupBytes + rows * 16, g_zero_rows, (kTile - rows) * 16, bar);
  }
  return kBlockBytes;
}

__device__ __forceinline__ uint32_t tile_bytes(int rows, int groups) {
  return uint32_t(groups * (rows == kTile ? kGroupBytes : rows * 16));
}

// Work item -> (query block, head, image), the query block being a pair of 128-row
// tiles or one tile; the query blocks of one (image, head) are consecutive items, so
// CTAs running at the same time share K and V in L2.
struct Item {
  int q, h, b;
};
__device__ __forceinline__ Item item_of(int it, int nq, int H) {
  Item r;
  r.q = it % nq;
  const int bh = it / nq;
  r.h = bh % H;
  r.b = bh / H;
  return r;
}

// Persistent: one CTA per SM walks the items blockIdx.x, blockIdx.x + gridDim.x, ...
// The K / V stream and the softmax pipeline run on across item boundaries; the next
// item's Q arrives in the staging buffer while the current item runs.
template <int QB, int KS, int VS, bool QK8>
// 10 warps: three share each of two SM sub-partitions, so a thread may hold at most
// 16384 / (3 x 32) registers, rounded down to the allocation granule.
__global__ void __maxnreg__(168) attention_kernel(const Params p) {
  using L = Smem<QB, KS, VS, QK8>;
  constexpr int kQKOp = L::kQKOp, kQKGroups = QK8 ? kGroups8 : kGroups;
  constexpr int kOffQ = L::kOffQ, kOffK = L::kOffK, kOffV = L::kOffV, kOffBar = L::kOffBar;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kOffBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto bar = [&](int i) { return bar0 + 8u * uint32_t(i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.T;
  const int nkv = (T + kTile - 1) / kTile;
  const int nq = (T + 2 * kTile - 1) / (2 * kTile);
  const int items = nq * p.H * p.B;
  const int n_my = int(blockIdx.x) < items ? (items - 1 - int(blockIdx.x)) / int(gridDim.x) + 1 : 0;
  const int total = n_my * nkv;  // kv tiles this CTA walks, over all its items
  // operand block of (which, image, head, tile)
  auto block = [&](int which, int b, int h, int tile) {
    return p.blocked + (((size_t(which) * p.B + b) * p.H + h) * p.tiles + tile) * size_t(kBlockBytes);
  };

  // Zero every operand buffer (Q, K and V tiles including their pad column group),
  // except V's pad group, whose first column is 1: P V then carries the row sum
  // of P (the softmax denominator, from the same F16 P) in output column 72.
  for (int i = threadIdx.x; i < kOffBar / 16; i += kThreads) {
    const int off = i * 16;
    const bool v_pad = off >= kOffV && ((off - kOffV) % kOpBytes) >= kGroups * kGroupBytes;
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(v_pad ? 0x3C00u : 0u, 0, 0, 0);
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    for (int s = 0; s < QB; ++s) {
      mbar_init(bar(kBarQFull + s), 1);
      mbar_init(bar(kBarQEmpty + s), 256);  // every softmax thread
    }
    for (int s = 0; s < KS; ++s) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarKEmpty + s), 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarVEmpty + s), 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(bar(kBarSFull + w), 1);
      mbar_init(bar(kBarPFull + w), 128);  // every softmax thread of the group arrives
      mbar_init(bar(kBarQtFull + w), 128);
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
  pdl_launch_dependents();
  pdl_wait();  // Q, K, V are written by the previous kernel

  if (warp == 0) {
    if (lane == 0) {
      // copies in flight per full barrier (bit b: Q buffer b, 4 + K stage, 8 + V stage) and their phase bit
      uint32_t issued = 0, issued_phase = 0;
      auto note = [&](int bit, uint32_t ph) {
        issued |= 1u << bit;
        issued_phase = (issued_phase & ~(1u << bit)) | (ph << bit);
      };
      bool ok = true;
      for (int n = 0; n < n_my && ok; ++n) {
        const Item I = item_of(int(blockIdx.x) + n * int(gridDim.x), nq, p.H);
        const int qb = n % QB;
        const uint32_t qph = (n / QB) & 1;
        if (!mbar_wait(bar(kBarQEmpty + qb), qph ^ 1, abort_flag, p.err)) break;
        const int qr0 = tile_rows(T, 2 * I.q), qr1 = tile_rows(T, 2 * I.q + 1);
        mbar_arrive_expect_tx(bar(kBarQFull + qb),
                              tile_bytes(qr0, kQKGroups) + (qr1 ? tile_bytes(qr1, kQKGroups) : 0));
        copy_tile(sbase + kOffQ + (2 * qb) * kQKOp, block(0, I.b, I.h, 2 * I.q), qr0, bar(kBarQFull + qb),
                  kQKGroups);
        if (qr1)
          copy_tile(sbase + kOffQ + (2 * qb + 1) * kQKOp, block(0, I.b, I.h, 2 * I.q + 1), qr1,
                    bar(kBarQFull + qb), kQKGroups);
        note(qb, qph);
        for (int j = 0; j < nkv; ++j) {
          const int t = n * nkv + j, ks = t % KS, vs = t % VS;
          const uint32_t kph = (t / KS) & 1, vph = (t / VS) & 1;
          const int rows = tile_rows(T, j);
          if (!mbar_wait(bar(kBarKEmpty + ks), kph ^ 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(kBarKFull + ks), tile_bytes(rows, kQKGroups));
          copy_tile(sbase + kOffK + ks * kQKOp, block(1, I.b, I.h, j), rows, bar(kBarKFull + ks), kQKGroups);
          note(4 + ks, kph);
          if (!mbar_wait(bar(kBarVEmpty + vs), vph ^ 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(kBarVFull + vs), kBlockBytes);
          copy_tile_zero_tail(sbase + kOffV + vs * kOpBytes, block(2, I.b, I.h, j), rows, bar(kBarVFull + vs));
          note(8 + vs, vph);
        }
      }
      // every copy this thread issued lands before the CTA can exit
      for (int i = 0; i < 12; ++i) {
        const int fb = i < 4 ? kBarQFull + i : (i < 8 ? kBarKFull + i - 4 : kBarVFull + i - 8);
        if (issued & (1u << i)) mbar_wait_bounded(bar(fb), (issued_phase >> i) & 1, p.err);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // The MMA issuer. Tile t = item t / nkv, key tile t % nkv. After the last tile one
      // more commit on each group's S barrier tells the group that its O is final.
      // S = Q K^T with A (Q) in TMEM and B (K) K-major in shared memory (F16, or E4M3
      // with the same type code 0 under kind::f8f6f4); O = P V with A (P) in TMEM and B
      // (V) MN-major in shared memory.
      constexpr uint32_t idesc_s = make_idesc(128, 128, 0, false);
      constexpr uint32_t idesc_o = make_idesc(128, 80, 0, true);
      auto issue_s = [&](int w, int t) {
        const uint32_t s_tm = tmem + uint32_t(128 * w), q_tm = tmem + uint32_t(416 + 48 * w);
        const uint32_t ka = sbase + kOffK + (t % KS) * kQKOp;
        if (QK8) {
#pragma unroll
          for (int kk = 0; kk < 3; ++kk)  // K = 96 in steps of 32 (two 16-byte column groups)
            mma_f8_ts(s_tm, q_tm + uint32_t(8 * kk), make_sdesc(ka + kk * 2 * kGroupBytes, kGroupBytes, 128, 0),
                      idesc_s, kk > 0);
        } else {
#pragma unroll
          for (int kk = 0; kk < 5; ++kk)  // K = 80 in steps of 16 (two column groups)
            mma_f16_ts(s_tm, q_tm + uint32_t(8 * kk), make_sdesc(ka + kk * 2 * kGroupBytes, kGroupBytes, 128, 0),
                       idesc_s, kk > 0);
        }
        tc_commit(bar(kBarSFull + w));
      };
      auto issue_pv = [&](int w, int t) {
        const uint32_t s_tm = tmem + uint32_t(128 * w), o_tm = tmem + uint32_t(256 + 80 * w);
        const uint32_t va = sbase + kOffV + (t % VS) * kOpBytes;
        const int j = t % nkv;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // K = 128 keys in steps of 16 (8 TMEM columns of P each)
          mma_f16_ts(o_tm, s_tm + uint32_t(8 * kk), make_sdesc(va + kk * 256, 128, kGroupBytes, 0), idesc_o,
                     (j | kk) > 0);
      };
      bool ok = total > 0;
      if (ok) {
        ok = mbar_wait(bar(kBarKFull), 0, abort_flag, p.err);
        for (int w = 0; w < 2 && ok; ++w) {
          ok = mbar_wait(bar(kBarQtFull + w), 0, abort_flag, p.err);
          if (ok) {
            tc_fence_after();
            issue_s(w, 0);
          }
        }
        if (ok) tc_commit(bar(kBarKEmpty));
      }
      for (int t = 0; ok && t < total; ++t) {
        for (int w = 0; w < 2 && ok; ++w) {
          ok = mbar_wait(bar(kBarPFull + w), t & 1, abort_flag, p.err) &&
               (w == 1 || mbar_wait(bar(kBarVFull + t % VS), (t / VS) & 1, abort_flag, p.err));
          if (!ok) break;
          tc_fence_after();
          issue_pv(w, t);
          if (w == 1) tc_commit(bar(kBarVEmpty + t % VS));
          if (t + 1 < total) {
            const int u = t + 1;
            if (w == 0 && !(ok = mbar_wait(bar(kBarKFull + u % KS), (u / KS) & 1, abort_flag, p.err))) break;
            tc_fence_after();
            issue_s(w, u);
            if (w == 1) tc_commit(bar(kBarKEmpty + u % KS));
          } else {
            tc_commit(bar(kBarSFull + w));  // O_w final
          }
        }
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
    const uint32_t o_tm = tmem + uint32_t(256 + w * 80) + lane_off;
    const uint32_t q_tm = tmem + uint32_t(416 + w * 48) + lane_off;
    const float sl2 = QK8 ? p.scale_log2 * (1.0f / 256.0f) : p.scale_log2;  // E4M3 operands hold 16 q, 16 k
    const int D = p.H * kDh;
    // Q row r of the group's tile of item n: from the staging buffer into TMEM (F16
    // pairs, 40 columns with the zero pad; or E4M3 quads, 24 columns), then the buffer
    // is released to the copy warp.
    auto stage_q = [&](int n) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarQFull + n % QB), (n / QB) & 1, abort_flag, p.err)))
        return false;
      const uint8_t* qs = smem + kOffQ + (2 * (n % QB) + w) * kQKOp + r * 16;
      if (QK8) {
        uint32_t q[16], z[8];
#pragma unroll
        for (int g = 0; g < 4; ++g) *reinterpret_cast<uint4*>(&q[4 * g]) = *reinterpret_cast<const uint4*>(qs + g * kGroupBytes);
        const uint4 last = *reinterpret_cast<const uint4*>(qs + 4 * kGroupBytes);
        z[0] = last.x, z[1] = last.y, z[2] = last.z, z[3] = last.w;
        z[4] = z[5] = z[6] = z[7] = 0u;
        tmem_st16(q_tm, q);
        tmem_st8(q_tm + 16, z);
      } else {
        uint32_t q[32], z[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) *reinterpret_cast<uint4*>(&q[4 * g]) = *reinterpret_cast<const uint4*>(qs + g * kGroupBytes);
        const uint4 last = *reinterpret_cast<const uint4*>(qs + 8 * kGroupBytes);
        z[0] = last.x, z[1] = last.y, z[2] = last.z, z[3] = last.w;
        z[4] = z[5] = z[6] = z[7] = 0u;
        tmem_st32(q_tm, q);
        tmem_st8(q_tm + 32, z);
      }
      mbar_arrive(bar(kBarQEmpty + n % QB));
      return true;
    };
    // Output rows of item n, once its last P V has finished: O (with its row sum in
    // column 72) read from TMEM, scaled by 1 / row sum, stored as F16 (16-byte stores)
    // or E4M3 codes of 16 x (8-byte stores); rows past the image's last token are not stored.
    auto write_item = [&](int n) {
      const Item I = item_of(int(blockIdx.x) + n * int(gridDim.x), nq, p.H);
      const int tq = (2 * I.q + w) * kTile + r;
      uint32_t o[5][16];
#pragma unroll
      for (int c = 0; c < 5; ++c) tmem_ld16(o_tm + 16 * c, o[c]);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 5; ++c)
#pragma unroll
        for (int i = 0; i < 16; ++i) asm volatile("" : "+r"(o[c][i]));  // no use before the wait
      if (tq >= T) return;
      const float inv = 1.0f / __uint_as_float(o[4][8]);  // column 72: the row sum
      const size_t row = size_t(I.b) * size_t(T) + size_t(tq);
#pragma unroll
      for (int g = 0; g < kGroups; ++g) {  // output columns 8 g .. 8 g + 7
        const uint32_t* v = &o[g >> 1][8 * (g & 1)];
        if (!p.out_e4m3) {
          uint4 wv;
          __half2* hw = reinterpret_cast<__half2*>(&wv);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float a, b;
            mul_x2(a, b, __uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]), inv, inv);
            hw[i] = __floats2half2_rn(a, b);
          }
          *reinterpret_cast<uint4*>(static_cast<__half*>(p.out) + row * D + I.h * kDh + 8 * g) = wv;
        } else {
          uint2 wv;
          __nv_fp8x2_storage_t* q = reinterpret_cast<__nv_fp8x2_storage_t*>(&wv);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            q[i] = __nv_cvt_float2_to_fp8x2(make_float2(16.0f * __uint_as_float(v[2 * i]) * inv,
                                                        16.0f * __uint_as_float(v[2 * i + 1]) * inv),
                                            __NV_SATFINITE, __NV_E4M3);
          *reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.out) + row * D + I.h * kDh + 8 * g) = wv;
        }
      }
    };
    bool ok = true;
    if (total > 0) {  // the first item's Q
      ok = stage_q(0);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(kBarQtFull + w));
    }
    // Reference maximum (log2 units) of this row's P tiles and of the O accumulator
    // in TMEM; the softmax denominator accumulates in O's column 72.
    float m = -INFINITY;
    for (int t = 0; t < total && ok; ++t) {
      const int n = t / nkv, j = t - n * nkv;
      // S(t) has finished, and with it every P V product of the group before it
      if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarSFull + w), t & 1, abort_flag, p.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (j == 0) {
        if (n > 0) write_item(n - 1);  // O of the previous item is final
        m = -INFINITY;
      }
      // the whole S row in registers (four loads in flight)
      uint32_t sv[4][32];
      tmem_ld32(s_tm, sv[0]);
      tmem_ld32(s_tm + 32, sv[1]);
      tmem_ld32(s_tm + 64, sv[2]);
      tmem_ld32(s_tm + 96, sv[3]);
      tmem_ld_wait(sv[0]);
      reg_fence(sv[1]);
      reg_fence(sv[2]);
      reg_fence(sv[3]);
      const int valid = T - j * kTile;  // keys of this tile that exist (>= 1)
      if (valid < kTile) {              // keys past the last token: -inf, so P = 0 exactly
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * c + i >= valid) sv[c][i] = 0xff800000u;
      }
      // row maximum: eight independent chains, then combined
      float mq[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mq[k] = fmaxf(__uint_as_float(sv[k >> 1][(k & 1) * 16]), __uint_as_float(sv[k >> 1][(k & 1) * 16 + 1]));
#pragma unroll
      for (int k = 0; k < 8; ++k)
#pragma unroll
        for (int i = 2; i < 16; i += 2)
          mq[k] = fmax3(mq[k], __uint_as_float(sv[k >> 1][(k & 1) * 16 + i]),
                        __uint_as_float(sv[k >> 1][(k & 1) * 16 + i + 1]));
      const float mx = fmaxf(fmaxf(fmax3(mq[0], mq[1], mq[2]), fmax3(mq[3], mq[4], mq[5])), fmaxf(mq[6], mq[7]));
      const float m_tile = mx * sl2;
      const bool raise = m_tile > m + kSlack;  // always on an item's first tile
      const float m_new = raise ? m_tile : m;
      if (j > 0 && __any_sync(0xffffffffu, raise)) {
        // O (and its row sum) *= 2^(m - m_new), 1 for kept rows; O holds P V up to
        // tile t - 1, which finished before S(t) did
        const float f = ex2(m - m_new);
#pragma unroll 1
        for (int c = 0; c < 10; ++c) {  // 80 columns, 8 at a time (few live registers)
          uint32_t e[8];
          tmem_ld8(o_tm + 8 * c, e);
          tmem_ld_wait();
          asm volatile("" : "+r"(e[0]), "+r"(e[1]), "+r"(e[2]), "+r"(e[3]), "+r"(e[4]), "+r"(e[5]), "+r"(e[6]),
                       "+r"(e[7]));
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float a, b;
            mul_x2(a, b, __uint_as_float(e[2 * i]), __uint_as_float(e[2 * i + 1]), f, f);
            e[2 * i] = __float_as_uint(a);
            e[2 * i + 1] = __float_as_uint(b);
          }
          tmem_st8(o_tm + 8 * c, e);
        }
      }
      m = m_new;
      // P = 2^(scale log2(e) s - m) as F16 pairs (key 2 i in the lower half of column i)
      // over the first 64 columns of S
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint32_t* s2 = &sv[2 * c + (i >> 4)][2 * (i & 15)];
          float x0, x1;  // scale log2(e) s - m for two keys in one two-lane FMA
          fma_x2(x0, x1, __uint_as_float(s2[0]), __uint_as_float(s2[1]), sl2, sl2, -m, -m);
          const __half2 h = __floats2half2_rn(ex2(x0), ex2(x1));
          pk[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        tmem_st32(s_tm + 32 * c, pk);
      }
      // the item's last S product has finished: the next item's Q may replace Q_w
      if (j == nkv - 1 && n + 1 < n_my && !stage_q(n + 1)) {
        ok = false;
        break;
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(kBarPFull + w));
    }
    // the last item's output rows, once the final P V has finished
    if (ok && total > 0 && __all_sync(0xffffffffu, mbar_wait(bar(kBarSFull + w), total & 1, abort_flag, p.err))) {
      tc_fence_after();
      write_item(n_my - 1);
    }
    tmem_ld_wait();
    tmem_st_wait();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Three score slots, one 128-query tile per item: for grids that one round of
// two-tile items would leave mostly idle (one image: 48 items of 256 queries,
// 96 of 128).
namespace slots {

constexpr int kSlots = 3;       // score tiles in tensor memory
constexpr int kRedBytes = 2 * 2 * kTile * 4;  // partial row maxima: [tile parity][key half][row]

// Shared memory map (offsets from the 1024-aligned base) for QB query buffers, KS key
// stages and VS value stages; QK8: E4M3 Q and K tiles.
template <int QB, int KS, int VS, bool QK8>
struct Smem {
  static constexpr int kQKOp = QK8 ? kOpBytes8 : kOpBytes;  // one Q or K tile
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + QB * kQKOp;
  static constexpr int kOffV = kOffK + KS * kQKOp;
  static constexpr int kOffBar = kOffV + VS * kOpBytes;
  static constexpr int kOffRed = kOffBar + kBarBytes;
  static constexpr int kBytes = 1024 + kOffRed + kRedBytes;
  static_assert(kBytes <= 232448, "shared memory budget");
  static_assert(QB >= 1 && QB <= 4 && KS >= 2 && KS <= 4 && VS >= 2 && VS <= 4, "buffer counts");
};

// TMEM columns: score slot k at 128 k (P of keys 64 h .. 64 h + 63 over columns
// 128 k + 64 h .. + 31 as F16 pairs, key 2 i in the lower half of column i), O at 384.
constexpr uint32_t kTmemO = kSlots * kTile;

// Barrier indices (8 bytes each).
enum {
  kBarQFull = 0,    // +buffer
  kBarQEmpty = 2,   // +buffer: the item's last S product has finished reading Q
  kBarKFull = 4,    // +stage
  kBarKEmpty = 8,   // +stage
  kBarVFull = 12,   // +stage
  kBarVEmpty = 16,  // +stage
  kBarSFull = 20,   // +slot: S of the slot's tile has finished
  kBarPFull = 23,   // +slot: every softmax thread has written P (and any O rescale) to TMEM
  kBarPDone = 26,   // +tile parity: O += P(t) V_t has finished
  kBarODone = 28,   // the CTA's last P V product has finished
  kBarDrain = 29,
  kBarX = 30,       // +2 quarter + tile parity: both halves' row maxima are in shared memory
  kNumBars = 38
};
static_assert(8 * kNumBars + 8 <= kBarBytes, "barrier area");

// Persistent: one CTA per SM walks the items (one 128-query tile of one head and
// image each) blockIdx.x, blockIdx.x + gridDim.x, ...; the K / V stream and the score
// products run on across item boundaries, and the next item's Q arrives in the other
// Q buffer while the current item runs.
template <int QB, int KS, int VS, bool QK8>
// 10 warps: three share each of two SM sub-partitions, so a thread may hold at most
// 16384 / (3 x 32) registers, rounded down to the allocation granule.
__global__ void __maxnreg__(168) attention_slots_kernel(const Params p) {
  using L = Smem<QB, KS, VS, QK8>;
  constexpr int kQKOp = L::kQKOp, kQKGroups = QK8 ? kGroups8 : kGroups;
  constexpr int kOffQ = L::kOffQ, kOffK = L::kOffK, kOffV = L::kOffV, kOffBar = L::kOffBar, kOffRed = L::kOffRed;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kOffBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto bar = [&](int i) { return bar0 + 8u * uint32_t(i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.T;
  const int nkv = (T + kTile - 1) / kTile;
  const int nq = nkv;  // query tiles of an image
  const int items = nq * p.H * p.B;
  const int n_my = int(blockIdx.x) < items ? (items - 1 - int(blockIdx.x)) / int(gridDim.x) + 1 : 0;
  const int total = n_my * nkv;  // kv tiles this CTA walks, over all its items
  // operand block of (which, image, head, tile)
  auto block = [&](int which, int b, int h, int tile) {
    return p.blocked + (((size_t(which) * p.B + b) * p.H + h) * p.tiles + tile) * size_t(kBlockBytes);
  };

  // Zero every operand buffer (Q, K and V tiles including their pad column group),
  // except V's pad group, whose first column is 1: P V then carries the row sum
  // of P (the softmax denominator, from the same F16 P) in output column 72.
  for (int i = threadIdx.x; i < kOffBar / 16; i += kThreads) {
    const int off = i * 16;
    const bool v_pad = off >= kOffV && ((off - kOffV) % kOpBytes) >= kGroups * kGroupBytes;
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(v_pad ? 0x3C00u : 0u, 0, 0, 0);
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    for (int s = 0; s < QB; ++s) {
      mbar_init(bar(kBarQFull + s), 1);
      mbar_init(bar(kBarQEmpty + s), 1);
    }
    for (int s = 0; s < KS; ++s) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarKEmpty + s), 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarVEmpty + s), 1);
    }
    for (int k = 0; k < kSlots; ++k) {
      mbar_init(bar(kBarSFull + k), 1);
      mbar_init(bar(kBarPFull + k), 256);  // every softmax thread arrives
    }
    mbar_init(bar(kBarPDone), 1);
    mbar_init(bar(kBarPDone + 1), 1);
    mbar_init(bar(kBarODone), 1);
    mbar_init(bar(kBarDrain), 1);
    for (int x = 0; x < 8; ++x) mbar_init(bar(kBarX + x), 64);  // both warps of a lane quarter
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
  pdl_launch_dependents();
  pdl_wait();  // Q, K, V are written by the previous kernel

  if (warp == 0) {
    if (lane == 0) {
      // copies in flight per full barrier (bit b: Q buffer b, 4 + K stage, 8 + V stage) and their phase bit
      uint32_t issued = 0, issued_phase = 0;
      auto note = [&](int bit, uint32_t ph) {
        issued |= 1u << bit;
        issued_phase = (issued_phase & ~(1u << bit)) | (ph << bit);
      };
      bool ok = true;
      for (int n = 0; n < n_my && ok; ++n) {
        const Item I = item_of(int(blockIdx.x) + n * int(gridDim.x), nq, p.H);
        const int qb = n % QB;
        const uint32_t qph = (n / QB) & 1;
        if (!mbar_wait(bar(kBarQEmpty + qb), qph ^ 1, abort_flag, p.err)) break;
        const int qr = tile_rows(T, I.q);
        mbar_arrive_expect_tx(bar(kBarQFull + qb), tile_bytes(qr, kQKGroups));
        copy_tile(sbase + kOffQ + qb * kQKOp, block(0, I.b, I.h, I.q), qr, bar(kBarQFull + qb), kQKGroups);
        note(qb, qph);
        for (int j = 0; j < nkv; ++j) {
          const int t = n * nkv + j, ks = t % KS, vs = t % VS;
          const uint32_t kph = (t / KS) & 1, vph = (t / VS) & 1;
          const int rows = tile_rows(T, j);
          if (!mbar_wait(bar(kBarKEmpty + ks), kph ^ 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(kBarKFull + ks), tile_bytes(rows, kQKGroups));
          copy_tile(sbase + kOffK + ks * kQKOp, block(1, I.b, I.h, j), rows, bar(kBarKFull + ks), kQKGroups);
          note(4 + ks, kph);
          if (!mbar_wait(bar(kBarVEmpty + vs), vph ^ 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(kBarVFull + vs), kBlockBytes);
          copy_tile_zero_tail(sbase + kOffV + vs * kOpBytes, block(2, I.b, I.h, j), rows, bar(kBarVFull + vs));
          note(8 + vs, vph);
        }
      }
      // every copy this thread issued lands before the CTA can exit
      for (int i = 0; i < 12; ++i) {
        const int fb = i < 4 ? kBarQFull + i : (i < 8 ? kBarKFull + i - 4 : kBarVFull + i - 8);
        if (issued & (1u << i)) mbar_wait_bounded(bar(fb), (issued_phase >> i) & 1, p.err);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // The MMA issuer. Tile t = item t / nkv, key tile t % nkv, its scores in slot t % 3.
      // S = Q K^T with A (Q) and B (K) K-major in shared memory (F16, or E4M3 with the
      // same type code 0 under kind::f8f6f4); O = P V with A (P) in TMEM and B (V)
      // MN-major in shared memory. Order: S(0), S(1), S(2), then per tile t: P(t) V_t,
      // S(t+3). The MMAs of one thread run in issue order, so S(t+3) overwrites slot
      // t % 3 only after P(t) V_t has read P from it, and the completion of S(t+3)
      // implies that of every P V product up to tile t.
      constexpr uint32_t idesc_s = make_idesc(128, 128, 0, false);
      constexpr uint32_t idesc_o = make_idesc(128, 80, 0, true);
      // K tile u (and, for an item's first tile, the item's Q) in shared memory
      auto operands_s = [&](int u) {
        const int n = u / nkv;
        return (u % nkv != 0 || mbar_wait(bar(kBarQFull + n % QB), (n / QB) & 1, abort_flag, p.err)) &&
               mbar_wait(bar(kBarKFull + u % KS), (u / KS) & 1, abort_flag, p.err);
      };
      auto issue_s = [&](int u) {
        const uint32_t s_tm = tmem + uint32_t(kTile * (u % kSlots));
        const uint32_t qa = sbase + kOffQ + ((u / nkv) % QB) * kQKOp;
        const uint32_t ka = sbase + kOffK + (u % KS) * kQKOp;
        if (QK8) {
#pragma unroll
          for (int kk = 0; kk < 3; ++kk)  // K = 96 in steps of 32 (two 16-byte column groups)
            mma_f8(s_tm, make_sdesc(qa + kk * 2 * kGroupBytes, kGroupBytes, 128, 0),
                   make_sdesc(ka + kk * 2 * kGroupBytes, kGroupBytes, 128, 0), idesc_s, kk > 0);
        } else {
#pragma unroll
          for (int kk = 0; kk < 5; ++kk)  // K = 80 in steps of 16 (two column groups)
            mma_f16(s_tm, make_sdesc(qa + kk * 2 * kGroupBytes, kGroupBytes, 128, 0),
                    make_sdesc(ka + kk * 2 * kGroupBytes, kGroupBytes, 128, 0), idesc_s, kk > 0);
        }
        tc_commit(bar(kBarSFull + u % kSlots));
        tc_commit(bar(kBarKEmpty + u % KS));
        if (u % nkv == nkv - 1) tc_commit(bar(kBarQEmpty + (u / nkv) % QB));  // the item's Q is read
      };
      // P of keys 64 h .. 64 h + 63 sits in slot columns 64 h .. 64 h + 31 (F16 pairs)
      auto issue_pv = [&](int t) {
        const uint32_t p_tm = tmem + uint32_t(kTile * (t % kSlots)), o_tm = tmem + kTmemO;
        const uint32_t va = sbase + kOffV + (t % VS) * kOpBytes;
        const int j = t % nkv;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // K = 128 keys in steps of 16
          mma_f16_ts(o_tm, p_tm + uint32_t(64 * (kk >> 2) + 8 * (kk & 3)),
                     make_sdesc(va + kk * 256, 128, kGroupBytes, 0), idesc_o, (j | kk) > 0);
        tc_commit(bar(kBarPDone + (t & 1)));
        tc_commit(bar(kBarVEmpty + t % VS));
        if (t == total - 1) tc_commit(bar(kBarODone));
      };
      bool ok = true;
      for (int u = 0; u < kSlots && u < total && ok; ++u) {
        if ((ok = operands_s(u))) {
          tc_fence_after();
          issue_s(u);
        }
      }
      for (int t = 0; ok && t < total; ++t) {
        if (!(ok = mbar_wait(bar(kBarPFull + t % kSlots), (t / kSlots) & 1, abort_flag, p.err) &&
                   mbar_wait(bar(kBarVFull + t % VS), (t / VS) & 1, abort_flag, p.err)))
          break;
        tc_fence_after();
        issue_pv(t);
        const int u = t + kSlots;
        if (u < total) {
          if (!(ok = operands_s(u))) break;
          tc_fence_after();
          issue_s(u);
        }
      }
      tc_commit(bar(kBarDrain));
      mbar_wait_bounded(bar(kBarDrain), 0, p.err);
    }
  } else {
    const int sub = warp & 3;          // TMEM lane quarter
    const int hf = (warp - 2) >> 2;    // key half of a tile: keys 64 hf .. 64 hf + 63
    const int r = sub * 32 + lane;     // query row within the tile == TMEM lane
    const uint32_t lane_off = uint32_t(sub * 32) << 16;
    const uint32_t o_tm = tmem + kTmemO + lane_off;
    float* red = reinterpret_cast<float*>(smem + kOffRed);  // [tile parity][half][row] partial maxima
    const float sl2 = QK8 ? p.scale_log2 * (1.0f / 256.0f) : p.scale_log2;  // E4M3 operands hold 16 q, 16 k
    const int D = p.H * kDh;
    // waits until P(u) V_u has finished: completion u / 2 of the barrier of u's parity.
    // The completion of S(t) implies that of P(t-3) V, so a wait at tile t for u = t - 1
    // finds that barrier at most one completion short.
    auto wait_pv = [&](int u) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarPDone + (u & 1)), (u >> 1) & 1, abort_flag, p.err)))
        return false;
      tc_fence_after();
      return true;
    };
    // Output rows of item n once its last P V has finished: this half's 40 columns of O
    // (half 0: columns 0..39, half 1: 40..79, with the row sum in column 72), scaled by
    // 1 / row sum, stored as F16 (16-byte stores) or E4M3 codes of 16 x (8-byte stores);
    // rows past the image's last token are not stored.
    auto write_item = [&](int n) {
      const Item I = item_of(int(blockIdx.x) + n * int(gridDim.x), nq, p.H);
      const int tq = I.q * kTile + r;
      uint32_t o[5][8], rs[8];
#pragma unroll
      for (int c = 0; c < 5; ++c) tmem_ld8(o_tm + uint32_t(40 * hf + 8 * c), o[c]);
      tmem_ld8(o_tm + 72, rs);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 5; ++c)
#pragma unroll
        for (int i = 0; i < 8; ++i) asm volatile("" : "+r"(o[c][i]));  // no use before the wait
      asm volatile("" : "+r"(rs[0]));
      if (tq >= T) return;
      const float inv = 1.0f / __uint_as_float(rs[0]);  // column 72: the row sum
      const size_t row = size_t(I.b) * size_t(T) + size_t(tq);
#pragma unroll
      for (int c = 0; c < 5; ++c) {  // output columns 40 hf + 8 c .. + 7
        const int g = 5 * hf + c;
        if (g >= kGroups) break;
        const uint32_t* v = o[c];
        if (!p.out_e4m3) {
          uint4 wv;
          __half2* hw = reinterpret_cast<__half2*>(&wv);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float a, b;
            mul_x2(a, b, __uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]), inv, inv);
            hw[i] = __floats2half2_rn(a, b);
          }
          *reinterpret_cast<uint4*>(static_cast<__half*>(p.out) + row * D + I.h * kDh + 8 * g) = wv;
        } else {
          uint2 wv;
          __nv_fp8x2_storage_t* q = reinterpret_cast<__nv_fp8x2_storage_t*>(&wv);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            q[i] = __nv_cvt_float2_to_fp8x2(make_float2(16.0f * __uint_as_float(v[2 * i]) * inv,
                                                        16.0f * __uint_as_float(v[2 * i + 1]) * inv),
                                            __NV_SATFINITE, __NV_E4M3);
          *reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.out) + row * D + I.h * kDh + 8 * g) = wv;
        }
      }
    };
    bool ok = true;
    // Reference maximum (log2 units) of this row's P tiles and of the O accumulator
    // in TMEM; the softmax denominator accumulates in O's column 72.
    float m = -INFINITY;
    for (int t = 0; t < total && ok; ++t) {
      const int n = t / nkv, j = t - n * nkv, slot = t % kSlots;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarSFull + slot), (t / kSlots) & 1, abort_flag, p.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (j == 0) m = -INFINITY;
      const uint32_t s_tm = tmem + uint32_t(kTile * slot + 64 * hf) + lane_off;
      // this half of the S row in registers (two loads in flight)
      uint32_t sv[2][32];
      tmem_ld32(s_tm, sv[0]);
      tmem_ld32(s_tm + 32, sv[1]);
      tmem_ld_wait(sv[0]);
      reg_fence(sv[1]);
      const int valid = T - j * kTile - 64 * hf;  // keys of this half that exist (may be <= 0)
      if (valid < 64) {                           // keys past the last token: -inf, so P = 0 exactly
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * c + i >= valid) sv[c][i] = 0xff800000u;
      }
      // row maximum of this half: four independent chains, then combined
      float mq[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        mq[k] = fmaxf(__uint_as_float(sv[k >> 1][(k & 1) * 16]), __uint_as_float(sv[k >> 1][(k & 1) * 16 + 1]));
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int i = 2; i < 16; i += 2)
          mq[k] = fmax3(mq[k], __uint_as_float(sv[k >> 1][(k & 1) * 16 + i]),
                        __uint_as_float(sv[k >> 1][(k & 1) * 16 + i + 1]));
      const float mh = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
      // and of the whole row, through the other half's warp (same lanes, other keys): both
      // arrive on their quarter's barrier for this tile parity. The buffers alternate by
      // tile, and a buffer is rewritten only after both warps have passed the next tile's
      // barrier
      float* rb = red + (t & 1) * 2 * kTile;
      rb[hf * kTile + r] = mh;
      const int xb = kBarX + 2 * sub + (t & 1);
      mbar_arrive(bar(xb));
      if (!__all_sync(0xffffffffu, mbar_wait(bar(xb), (t >> 1) & 1, abort_flag, p.err))) {
        ok = false;
        break;
      }
      const float mx = fmaxf(mh, rb[(1 - hf) * kTile + r]);
      const float m_tile = mx * sl2;
      const bool raise = m_tile > m + kSlack;  // always on an item's first tile
      const float m_new = raise ? m_tile : m;
      if (j > 0 && __any_sync(0xffffffffu, raise)) {
        // this half's 40 columns of O (and the row sum) *= 2^(m - m_new), 1 for kept
        // rows, once O holds P V up to tile t - 1
        if (!wait_pv(t - 1)) {
          ok = false;
          break;
        }
        const float f = ex2(m - m_new);
#pragma unroll 1
        for (int c = 0; c < 5; ++c) {
          uint32_t e[8];
          tmem_ld8(o_tm + uint32_t(40 * hf + 8 * c), e);
          tmem_ld_wait();
          asm volatile("" : "+r"(e[0]), "+r"(e[1]), "+r"(e[2]), "+r"(e[3]), "+r"(e[4]), "+r"(e[5]), "+r"(e[6]),
                       "+r"(e[7]));
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float a, b;
            mul_x2(a, b, __uint_as_float(e[2 * i]), __uint_as_float(e[2 * i + 1]), f, f);
            e[2 * i] = __float_as_uint(a);
            e[2 * i + 1] = __float_as_uint(b);
          }
          tmem_st8(o_tm + uint32_t(40 * hf + 8 * c), e);
        }
      }
      m = m_new;
      // P = 2^(scale log2(e) s - m) as F16 pairs (key 2 i of the half in the lower half
      // of column i) over the first 32 columns of this half's S
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const uint32_t* s2 = &sv[i >> 4][2 * (i & 15)];
        float x0, x1;  // scale log2(e) s - m for two keys in one two-lane FMA
        fma_x2(x0, x1, __uint_as_float(s2[0]), __uint_as_float(s2[1]), sl2, sl2, -m, -m);
        const __half2 h = __floats2half2_rn(ex2(x0), ex2(x1));
        pk[i] = *reinterpret_cast<const uint32_t*>(&h);
      }
      // an item's first tile: O of the previous item is final once its last P V has
      // finished, and is read before this tile's P V starts the item's sum anew
      if (j == 0 && n > 0) {
        if (!wait_pv(t - 1)) {
          ok = false;
          break;
        }
        write_item(n - 1);
      }
      tmem_st32(s_tm, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(kBarPFull + slot));
    }
    // the last item's output rows, once the final P V has finished
    if (ok && total > 0 && __all_sync(0xffffffffu, mbar_wait(bar(kBarODone), 0, abort_flag, p.err))) {
      tc_fence_after();
      write_item(n_my - 1);
    }
    tmem_ld_wait();
    tmem_st_wait();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace slots

// One 16-byte group of 8 values (column group cg of head h, token t of image b) into
// the head-blocked layout; qk8: Q and K as E4M3(16 x), 8 bytes per group (the head's
// last group also writes the zero pad of its 16-value group).
__device__ __forceinline__ void store_blocked(uint8_t* blk, int which, int bimg, int h, int t, int cg, const uint4& u,
                                              int qk8, int B, int H, int tiles) {
  const size_t idx = ((size_t(which) * B + bimg) * H + h) * tiles + (t >> 7);
  uint8_t* dst = blk + idx * kBlockBytes + (t & 127) * 16;
  if (qk8 && which < 2) {
    const __half2* hv = reinterpret_cast<const __half2*>(&u);
    uint2 w8;
    __nv_fp8x2_storage_t* q = reinterpret_cast<__nv_fp8x2_storage_t*>(&w8);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(hv[i]);
      q[i] = __nv_cvt_float2_to_fp8x2(make_float2(16.0f * f.x, 16.0f * f.y), __NV_SATFINITE, __NV_E4M3);
    }
    uint8_t* d8 = dst + (cg >> 1) * kGroupBytes + (cg & 1) * 8;
    if (cg == kGroups - 1)
      *reinterpret_cast<uint4*>(d8) = make_uint4(w8.x, w8.y, 0u, 0u);
    else
      *reinterpret_cast<uint2*>(d8) = w8;
    return;
  }
  *reinterpret_cast<uint4*>(dst + cg * kGroupBytes) = u;
}

// Row-major [B, T, 3 D] -> head-blocked; one thread per 16-byte group of 8 values.
__global__ void repack_kernel(const __half* __restrict__ qkv, uint8_t* __restrict__ blk, int B, int T, int H,
                              int tiles, int qk8) {
  const int D = H * kDh;
  const long i = long(blockIdx.x) * blockDim.x + threadIdx.x;
  const long per_row = 3L * D / 8;
  if (i >= long(B) * T * per_row) return;
  const long m = i / per_row;
  const int col = int(i - m * per_row) * 8;
  const int bimg = int(m / T), t = int(m - long(bimg) * T);
  const int which = col / D, rem = col - which * D, h = rem / kDh, cg = (rem - h * kDh) >> 3;
  const uint4 u = *reinterpret_cast<const uint4*>(qkv + m * 3 * D + col);
  store_blocked(blk, which, bimg, h, t, cg, u, qk8, B, H, tiles);
}

// Per-head q, k, v [B, H, T, stride] (the first 72 values of a row) -> head-blocked;
// one thread per 16-byte group of 8 values.
__global__ void repack_heads_kernel(const __half* __restrict__ q, const __half* __restrict__ k,
                                    const __half* __restrict__ v, uint8_t* __restrict__ blk, int B, int T, int H,
                                    int stride, int tiles, int qk8) {
  const long i = long(blockIdx.x) * blockDim.x + threadIdx.x;
  const long per_which = long(B) * H * T * kGroups;
  if (i >= 3 * per_which) return;
  const int which = int(i / per_which);
  long r = i - which * per_which;
  const int cg = int(r % kGroups);
  r /= kGroups;  // ((b H + h) T + t)
  const int t = int(r % T);
  const long bh = r / T;
  const int h = int(bh % H), bimg = int(bh / H);
  const __half* src = which == 0 ? q : (which == 1 ? k : v);
  const uint4 u = *reinterpret_cast<const uint4*>(src + r * stride + cg * 8);
  store_blocked(blk, which, bimg, h, t, cg, u, qk8, B, H, tiles);
}

// Head-blocked F16 Q, K, V -> row-major [B, T, 3 D]; one thread per 16-byte group.
__global__ void unpack_kernel(const uint8_t* __restrict__ blk, __half* __restrict__ qkv, int B, int T, int H,
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
  *reinterpret_cast<uint4*>(qkv + m * 3 * D + col) =
      *reinterpret_cast<const uint4*>(blk + idx * kBlockBytes + (t & 127) * 16 + cg * kGroupBytes);
}

// Buffer configurations launched. Two-tile items: one Q staging buffer (both tiles of
// an item; the next item's queries arrive in it during the current item) and 3 + 3 K / V
// stages. Three score slots: two Q buffers (the next item's queries arrive in one while
// the current item reads the other), 4 K stages (the score products run three tiles
// ahead) and 3 V stages.
template <int QB, int KS, int VS, bool QK8, bool SLOTS>
sv_status attention_launch_cfg(const Params& p, int grid, cudaStream_t s) {
  void (*kern)(const Params);
  int bytes;
  if constexpr (SLOTS) {
    kern = slots::attention_slots_kernel<QB, KS, VS, QK8>;
    bytes = slots::Smem<QB, KS, VS, QK8>::kBytes;
  } else {
    kern = attention_kernel<QB, KS, VS, QK8>;
    bytes = Smem<QB, KS, VS, QK8>::kBytes;
  }
  // the attribute is per device: set it once on each device the kernel runs on
  static unsigned long long attr_set = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice(attention)");
  const unsigned long long bit = (dev >= 0 && dev < kMaxAttrDevices) ? 1ull << dev : 0ull;
  if (!(attr_set & bit) || !bit) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attention)");
    attr_set |= bit;
  }
  e = launch_pdl(kern, dim3(unsigned(grid)), dim3(kThreads), size_t(bytes), s, p);
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return SV_OK;
}

// Which kernel runs: 0 chooses by size, 1 forces two-tile items, 2 three score slots
// (set by sv_debug_attention_kernel).
int g_attention_choice = 0;

// Three score slots (2) when every one-tile item runs in the first round of the grid:
// the grid is then under-filled by two-tile items, and one-tile items use twice the SMs
// (one image of 729 tokens and 16 heads: 96 items instead of 48). Otherwise two-tile
// items (1), whose two softmax groups share each CTA's products.
int attention_kernel_for(int B, int T, int H, int sms) {
  if (g_attention_choice) return g_attention_choice;
  const long items1 = long((T + kTile - 1) / kTile) * H * B;
  return items1 <= sms ? 2 : 1;
}

int attention_grid_for(int kernel, int B, int T, int H, int sms) {
  const long per_head = kernel == 2 ? (T + kTile - 1) / kTile : (T + 2 * kTile - 1) / (2 * kTile);
  const long items = per_head * H * B;
  return int(items < sms ? items : sms);
}

}  // namespace

size_t attention_blocked_bytes(int B, int T, int H) {
  return size_t(3) * B * H * ((T + kTile - 1) / kTile) * size_t(kBlockBytes);
}

sv_status attention_repack_launch(const __half* qkv, void* blocked, int B, int T, int H, int qk8, cudaStream_t s) {
  const long n = long(B) * T * (3L * H * kDh / 8);
  repack_kernel<<<unsigned((n + 255) / 256), 256, 0, s>>>(qkv, static_cast<uint8_t*>(blocked), B, T, H,
                                                           (T + kTile - 1) / kTile, qk8);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SV_OK : cuda_fail(e, "attention repack launch");
}

sv_status attention_repack_heads_launch(const __half* q, const __half* k, const __half* v, void* blocked, int B,
                                        int T, int H, int stride, int qk8, cudaStream_t s) {
  const long n = 3L * B * H * T * kGroups;
  repack_heads_kernel<<<unsigned((n + 255) / 256), 256, 0, s>>>(q, k, v, static_cast<uint8_t*>(blocked), B, T, H,
                                                                 stride, (T + kTile - 1) / kTile, qk8);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SV_OK : cuda_fail(e, "attention repack (per head) launch");
}

sv_status attention_unpack_launch(const void* blocked, __half* qkv, int B, int T, int H, cudaStream_t s) {
  const long n = long(B) * T * (3L * H * kDh / 8);
  unpack_kernel<<<unsigned((n + 255) / 256), 256, 0, s>>>(static_cast<const uint8_t*>(blocked), qkv, B, T, H,
                                                          (T + kTile - 1) / kTile);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SV_OK : cuda_fail(e, "attention unpack launch");
}

sv_status attention_launch(const void* blocked, void* o, int B, int T, int H, float scale, int out_e4m3, int qk8,
                           cudaStream_t s) {
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
  const int sms = num_sms() > 0 ? num_sms() : 1;
  const int kernel = attention_kernel_for(B, T, H, sms);
  const int grid = attention_grid_for(kernel, B, T, H, sms);
  if (kernel == 2) {
    if (qk8) return attention_launch_cfg<2, 4, 3, true, true>(p, grid, s);
    return attention_launch_cfg<2, 4, 3, false, true>(p, grid, s);
  }
  if (qk8) return attention_launch_cfg<1, 3, 3, true, false>(p, grid, s);
  return attention_launch_cfg<1, 3, 3, false, false>(p, grid, s);
}

}  // namespace sv

// Forces the attention kernel of later launches (tests): 0 by size, 1 two-tile items,
// 2 three score slots.
extern "C" sv_status sv_debug_attention_kernel(int choice) {
  if (choice < 0 || choice > 2) {
    sv::set_error("sv_debug_attention_kernel: choice must be 0, 1 or 2");
    return SV_ERR_INVALID_ARG;
  }
  sv::g_attention_choice = choice;
  return SV_OK;
}

// The kernel (1: two-tile items, 2: three score slots) and grid an attention launch of
// these sizes takes on a GPU with `sms` SMs under the current choice (host only).
extern "C" sv_status sv_debug_attention_plan(int B, int T, int H, int sms, int* kernel, int* grid) {
  if (B < 1 || T < 1 || H < 1 || sms < 1 || !kernel || !grid) {
    sv::set_error("sv_debug_attention_plan: bad arguments");
    return SV_ERR_INVALID_ARG;
  }
  *kernel = sv::attention_kernel_for(B, T, H, sms);
  *grid = sv::attention_grid_for(*kernel, B, T, H, sms);
  return SV_OK;
}
