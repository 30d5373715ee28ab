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
// tiles, head, image); 352 threads:
//   warp 0      bulk copies: Q (both tiles) per item, then K and V tiles of 128
//               keys into 3 + 3 stages, each with its own release;
//   warps 1, 2  MMA issuers, one per softmax group w: S_w = Q_w K_j^T
//               (M 128, N 128) into TMEM, then O_w += P_w V_j (M 128, N 80) in
//               two 64-key halves, O_w kept in TMEM for the whole item;
//   warps 3..6  softmax group 0, warps 7..10 softmax group 1: one thread per
//               query row reads its S row from TMEM once (S is then free for the
//               next product), writes P (F16) to shared memory, and rescales O
//               in TMEM only when the row maximum grows by more than 2^15; the
//               softmax denominator comes out of the P V product (a column of
//               ones in V's pad group). An item's output rows are staged in shared
//               memory and written by a TMA store during the next item.

#include <cuda_fp8.h>

#include <cstring>

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
constexpr int kPBytes = 16 * kGroupBytes;    // 128 keys of probabilities
constexpr int kThreads = 352;
constexpr int kBarBytes = 384;  // barriers, TMEM address slot, abort flag

// Shared memory map (offsets from the 1024-aligned base) for QB query buffers
// (of two tiles each), KS key stages and VS value stages; QK8: E4M3 Q and K tiles.
template <int QB, int KS, int VS, bool QK8>
struct Smem {
  static constexpr int kQKOp = QK8 ? kOpBytes8 : kOpBytes;  // one Q or K tile
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * QB * kQKOp;
  static constexpr int kOffV = kOffK + KS * kQKOp;
  static constexpr int kOffP = kOffV + VS * kOpBytes;  // one buffer per softmax group
  static constexpr int kOffBar = kOffP + 2 * kPBytes;
  static constexpr int kBytes = 1024 + kOffBar + kBarBytes;
  static_assert(kBytes <= 232448, "shared memory budget");
  static_assert(QB >= 1 && QB <= 2 && KS >= 2 && KS <= 4 && VS >= 2 && VS <= 4, "buffer counts");
};

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
  kBarQFull = 0,    // +buffer
  kBarQEmpty = 2,   // +buffer: both groups' last S product of the item has finished
  kBarKFull = 4,    // +stage
  kBarKEmpty = 8,   // +stage
  kBarVFull = 12,   // +stage
  kBarVEmpty = 16,  // +stage
  kBarSFull = 20,   // +group
  kBarSEmpty = 22,  // +group: the group has read S into registers
  kBarPFull = 24,   // +2 group + half: that half of the group's P tile is written
  kBarPEmpty = 28,  // +2 group + half: O += P V of that half has finished
  kBarOFull = 32,   // +group: O += P V of the group's latest tile has finished
  kBarOEmpty = 34,  // +group: the group has read the item's final O
  kBarDrain = 36,   // +group
  kBarStage = 38,   // +group: every warp's output store has read its staging rows
  kNumBars = 40
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

// Work item -> (query pair, head, image); the query pairs of one (image, head)
// are consecutive items, so CTAs running at the same time share K and V in L2.
struct Item {
  int qp, h, b;
};
__device__ __forceinline__ Item item_of(int it, int nq, int H) {
  Item r;
  r.qp = it % nq;
  const int bh = it / nq;
  r.h = bh % H;
  r.b = bh / H;
  return r;
}

// Persistent: one CTA per SM walks the items blockIdx.x, blockIdx.x + gridDim.x, ...
// The K / V stream and the softmax pipeline run on across item boundaries; Q is
// double buffered so the next item's queries arrive during the current item.
template <int QB, int KS, int VS, bool QK8>
// 11 warps: three share each of three SM sub-partitions, so a thread may hold at most
// 16384 / (3 x 32) registers, rounded down to the allocation granule.
__global__ void __maxnreg__(168) attention_kernel(const __grid_constant__ CUtensorMap tm_out, const Params p) {
  using L = Smem<QB, KS, VS, QK8>;
  constexpr int kQKOp = L::kQKOp, kQKGroups = QK8 ? kGroups8 : kGroups;
  constexpr int kOffQ = L::kOffQ, kOffK = L::kOffK, kOffV = L::kOffV, kOffP = L::kOffP, kOffBar = L::kOffBar;
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
  for (int i = threadIdx.x; i < kOffP / 16; i += kThreads) {
    const int off = i * 16;
    const bool v_pad = off >= kOffV && ((off - kOffV) % kOpBytes) >= kGroups * kGroupBytes;
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(v_pad ? 0x3C00u : 0u, 0, 0, 0);
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    for (int s = 0; s < QB; ++s) {
      mbar_init(bar(kBarQFull + s), 1);
      mbar_init(bar(kBarQEmpty + s), 2);  // one release per group
    }
    for (int s = 0; s < KS; ++s) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarKEmpty + s), 2);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarVEmpty + s), 2);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(bar(kBarSFull + w), 1);
      mbar_init(bar(kBarSEmpty + w), 128);  // every softmax thread of the group arrives
      for (int h = 0; h < 2; ++h) {
        mbar_init(bar(kBarPFull + 2 * w + h), 128);
        mbar_init(bar(kBarPEmpty + 2 * w + h), 1);
      }
      mbar_init(bar(kBarOFull + w), 1);
      mbar_init(bar(kBarOEmpty + w), 128);
    }
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarDrain + 1), 1);
    mbar_init(bar(kBarStage), 4);  // one arrival per warp of the group
    mbar_init(bar(kBarStage + 1), 4);
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
        const int qr0 = tile_rows(T, 2 * I.qp), qr1 = tile_rows(T, 2 * I.qp + 1);
        mbar_arrive_expect_tx(bar(kBarQFull + qb),
                              tile_bytes(qr0, kQKGroups) + (qr1 ? tile_bytes(qr1, kQKGroups) : 0));
        copy_tile(sbase + kOffQ + (2 * qb) * kQKOp, block(0, I.b, I.h, 2 * I.qp), qr0, bar(kBarQFull + qb),
                  kQKGroups);
        if (qr1)
          copy_tile(sbase + kOffQ + (2 * qb + 1) * kQKOp, block(0, I.b, I.h, 2 * I.qp + 1), qr1,
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
  } else if (warp <= 2) {
    if (lane == 0) {
      // MMA issuer of softmax group w = warp - 1, in the group's own order: S(0); then per
      // tile t (item t / nkv, key tile t % nkv): S(t+1) once K_{t+1} (and, on an item's
      // first tile, its Q) is in and the group has read S(t) from TMEM; O += P V for
      // each 64-key half of P(t) once that half is written, V_t is in and (an item's
      // first tile) the group has read the previous item's O.
      const int w = warp - 1;
      // S = Q K^T, both K-major (F16, or E4M3 with the same type code 0 under kind::f8f6f4)
      constexpr uint32_t idesc_s = make_idesc(128, 128, 0, false);
      constexpr uint32_t idesc_o = make_idesc(128, 80, 0, true);    // O = P V, V MN-major
      auto issue_s = [&](int t) -> bool {
        const int n = t / nkv, j = t - n * nkv;
        if (!mbar_wait(bar(kBarKFull + t % KS), (t / KS) & 1, abort_flag, p.err)) return false;
        if (!mbar_wait(bar(kBarSEmpty + w), (t & 1) ^ 1, abort_flag, p.err)) return false;
        if (j == 0 && !mbar_wait(bar(kBarQFull + n % QB), (n / QB) & 1, abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t qa = sbase + kOffQ + (2 * (n % QB) + w) * kQKOp, ka = sbase + kOffK + (t % KS) * kQKOp;
        if (QK8) {
#pragma unroll
          for (int kk = 0; kk < 3; ++kk)  // K = 96 in steps of 32 (two 16-byte column groups)
            mma_f8(tmem + uint32_t(w * 128), make_sdesc(qa + kk * 2 * kGroupBytes, kGroupBytes, 128, 0),
                   make_sdesc(ka + kk * 2 * kGroupBytes, kGroupBytes, 128, 0), idesc_s, kk > 0);
        } else {
#pragma unroll
          for (int kk = 0; kk < 5; ++kk)  // K = 80 in steps of 16 (two column groups)
            mma_f16(tmem + uint32_t(w * 128), make_sdesc(qa + kk * 2 * kGroupBytes, kGroupBytes, 128, 0),
                    make_sdesc(ka + kk * 2 * kGroupBytes, kGroupBytes, 128, 0), idesc_s, kk > 0);
        }
        tc_commit(bar(kBarSFull + w));
        tc_commit(bar(kBarKEmpty + t % KS));
        if (j == nkv - 1) tc_commit(bar(kBarQEmpty + n % QB));
        return true;
      };
      auto issue_pv = [&](int u, int half) -> bool {
        const int n = u / nkv, j = u - n * nkv;
        if (!mbar_wait(bar(kBarPFull + 2 * w + half), u & 1, abort_flag, p.err)) return false;
        if (!mbar_wait(bar(kBarVFull + u % VS), (u / VS) & 1, abort_flag, p.err)) return false;
        if (j == 0 && half == 0 && n > 0 && !mbar_wait(bar(kBarOEmpty + w), (n - 1) & 1, abort_flag, p.err))
          return false;
        tc_fence_after();
        const uint32_t pa = sbase + kOffP + w * kPBytes + half * (kPBytes / 2),
                       va = sbase + kOffV + (u % VS) * kOpBytes + half * 4 * 256;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // K = 64 keys in steps of 16
          mma_f16(tmem + uint32_t(256 + w * 128), make_sdesc(pa + kk * 2 * kGroupBytes, kGroupBytes, 128, 0),
                  make_sdesc(va + kk * 256, 128, kGroupBytes, 0), idesc_o, (j | half | kk) > 0);
        tc_commit(bar(kBarPEmpty + 2 * w + half));
        if (half) {
          tc_commit(bar(kBarOFull + w));
          tc_commit(bar(kBarVEmpty + u % VS));
        }
        return true;
      };
      bool ok = total == 0 || issue_s(0);
      for (int t = 0; ok && t < total; ++t)
        ok = (t + 1 >= total || issue_s(t + 1)) && issue_pv(t, 0) && issue_pv(t, 1);
      tc_commit(bar(kBarDrain + w));
      mbar_wait_bounded(bar(kBarDrain + w), 0, p.err);
    }
  } else {
    const int w = (warp - 3) >> 2;  // softmax group
    const int sub = warp & 3;       // TMEM lane quarter
    const int r = sub * 32 + lane;  // query row within the group's tile == TMEM lane
    const uint32_t lane_off = uint32_t(sub * 32) << 16;
    const uint32_t s_tm = tmem + uint32_t(w * 128) + lane_off;
    const uint32_t o_tm = tmem + uint32_t(256 + w * 128) + lane_off;
    uint8_t* pbuf = smem + kOffP + w * kPBytes;
    const float sl2 = QK8 ? p.scale_log2 * (1.0f / 256.0f) : p.scale_log2;  // E4M3 operands hold 16 q, 16 k
    const int D = p.H * kDh;
    // An item's output rows, at the end of its last tile (the S row is no longer held,
    // so all 80 columns of O are read at once): the final O (with its row sum in column
    // 72) of the group's query tile, read from TMEM once its last P V has finished,
    // scaled by 1 / row sum. F16 rows are staged as this warp's 32 x 72 block in the
    // group's P buffer (free once that P V has finished) and written by one TMA store
    // that clips the rows past the image's last token; E4M3 rows are stored directly.
    auto finish_item = [&](int n, int tl) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarOFull + w), tl & 1, abort_flag, p.err))) return false;
      tc_fence_after();
      const Item I = item_of(int(blockIdx.x) + n * int(gridDim.x), nq, p.H);
      const int tq0 = (2 * I.qp + w) * kTile + sub * 32;  // first query row of this warp
      const int tq = tq0 + lane;
      uint8_t* stg = pbuf + sub * (32 * kDh * 2) + lane * (kDh * 2);
      uint8_t* dst8 = static_cast<uint8_t*>(p.out) + (size_t(I.b) * size_t(T) + size_t(tq)) * size_t(D) + size_t(I.h) * kDh;
      uint32_t o[5][16];
#pragma unroll
      for (int c = 0; c < 5; ++c) tmem_ld16(o_tm + 16 * c, o[c]);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 5; ++c)
#pragma unroll
        for (int i = 0; i < 16; ++i) asm volatile("" : "+r"(o[c][i]));  // no use before the wait
      const float inv = 1.0f / __uint_as_float(o[4][8]);  // column 72: the row sum
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
          *reinterpret_cast<uint4*>(stg + 16 * g) = wv;
        } else if (tq < T) {
          uint2 wv;
          __nv_fp8x2_storage_t* q = reinterpret_cast<__nv_fp8x2_storage_t*>(&wv);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            q[i] = __nv_cvt_float2_to_fp8x2(make_float2(16.0f * __uint_as_float(v[2 * i]) * inv,
                                                        16.0f * __uint_as_float(v[2 * i + 1]) * inv),
                                            __NV_SATFINITE, __NV_E4M3);
          *reinterpret_cast<uint2*>(dst8 + 8 * g) = wv;
        }
      }
      tc_fence_before();
      mbar_arrive(bar(kBarOEmpty + w));  // the next item's first P V may overwrite O
      if (!p.out_e4m3) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && tq0 < T) {
          tma_store_3d(&tm_out, smem_u32(pbuf + sub * (32 * kDh * 2)), I.h * kDh, tq0, I.b);
          bulk_commit();
        }
      }
      return true;
    };
    // Reference maximum (log2 units) of this row's P tiles and of the O accumulator
    // in TMEM; the softmax denominator accumulates in O's column 72.
    float m = -INFINITY;
    bool ok = true;
    bool pend = false;  // the previous item's output rows were staged at the end of its last tile
    int staged = 0;     // items whose output went through the staging rows

    for (int t = 0; t < total && ok; ++t) {
      const int n = t / nkv, j = t - n * nkv;
      if (j == 0) m = -INFINITY;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarSFull + w), t & 1, abort_flag, p.err))) {
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
      // The previous item's staged output: its store must read the staging rows before
      // this tile's P overwrites them.
      bool wait_stage = false;
      if (pend) {
        pend = false;
        if (!p.out_e4m3) {
          wait_stage = true;
          if (lane == 0) bulk_wait_read<0>();  // this warp's store has read its staging rows
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBarStage + w));
        }
      }
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
      for (int k = 0; k < 8; ++k) mq[k] = fmaxf(__uint_as_float(sv[k >> 1][(k & 1) * 16]), __uint_as_float(sv[k >> 1][(k & 1) * 16 + 1]));
#pragma unroll
      for (int k = 0; k < 8; ++k)
#pragma unroll
        for (int i = 2; i < 16; i += 2)
          mq[k] = fmax3(mq[k], __uint_as_float(sv[k >> 1][(k & 1) * 16 + i]), __uint_as_float(sv[k >> 1][(k & 1) * 16 + i + 1]));
      const float mx = fmaxf(fmaxf(fmax3(mq[0], mq[1], mq[2]), fmax3(mq[3], mq[4], mq[5])), fmaxf(mq[6], mq[7]));
      const float m_tile = mx * sl2;
      const bool raise = m_tile > m + kSlack;  // always on an item's first tile
      const float m_new = raise ? m_tile : m;
      if (j > 0 && __any_sync(0xffffffffu, raise)) {
        // O (and its row sum) *= 2^(m - m_new), 1 for kept rows, once O += P(t-1) V has finished
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarOFull + w), (t - 1) & 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
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
        tmem_st_wait();
      }
      m = m_new;
      // every warp of the group has finished reading the staging rows (they alias P)
      if (wait_stage && !__all_sync(0xffffffffu, mbar_wait(bar(kBarStage + w), staged & 1, abort_flag, p.err))) {
        ok = false;
        break;
      }
      staged += wait_stage ? 1 : 0;
      // P = 2^(scale log2(e) s - m) as F16, in two halves of 64 keys; a half's buffer
      // is free once O += P V of the same half of the previous tile has finished
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarPEmpty + 2 * w + half), (t & 1) ^ 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        uint8_t* ph = pbuf + half * (kPBytes / 2);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint4 wv;
            __half2* hw = reinterpret_cast<__half2*>(&wv);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              float x0, x1;  // scale log2(e) s - m for two keys in one two-lane FMA
              fma_x2(x0, x1, __uint_as_float(sv[2 * half + cc][8 * g + 2 * i]),
                     __uint_as_float(sv[2 * half + cc][8 * g + 2 * i + 1]), sl2, sl2, -m, -m);
              hw[i] = __floats2half2_rn(ex2(x0), ex2(x1));
            }
            *reinterpret_cast<uint4*>(ph + (4 * cc + g) * kGroupBytes + r * 16) = wv;
          }
        }
        tc_fence_before();
        fence_proxy_async_smem();  // P (generic-proxy stores) visible to the tensor core
        mbar_arrive(bar(kBarPFull + 2 * w + half));
      }
      if (!ok) break;

      if (j == nkv - 1) {  // the item's output rows, once its last P V has finished
        if (!finish_item(n, t)) {
          ok = false;
          break;
        }
        pend = true;
      }
    }
    if (lane == 0) bulk_wait_all();  // output stores have read shared memory before the CTA exits
    tmem_ld_wait();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Row-major [B, T, 3 D] -> head-blocked; one thread per 16-byte group of 8 values.
// qk8: Q and K as E4M3(16 x), 8 bytes per group (the head's last group also writes the
// zero pad of its 16-value group).
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
  const size_t idx = ((size_t(which) * B + bimg) * H + h) * tiles + (t >> 7);
  const uint4 u = *reinterpret_cast<const uint4*>(qkv + m * 3 * D + col);
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

// Buffer configuration launched: one Q buffer (both tiles of an item) and 3 + 3 K / V
// stages. Two Q buffers with 2 + 2 stages, or one with 4 K + 2 V stages, fill the same
// shared memory and measured slower at 16 heads x 729 tokens (B = 32: 137 us against
// 139 and 139 us).
template <int QB, int KS, int VS, bool QK8>
sv_status attention_launch_cfg(const CUtensorMap& tmo, const Params& p, int grid, cudaStream_t s) {
  static bool attr_set = false;
  using L = Smem<QB, KS, VS, QK8>;
  auto kern = attention_kernel<QB, KS, VS, QK8>;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attention)");
    attr_set = true;
  }
  cudaError_t e = launch_pdl(kern, dim3(unsigned(grid)), dim3(kThreads), L::kBytes, s, tmo, p);
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return SV_OK;
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
  const int items = ((T + 2 * kTile - 1) / (2 * kTile)) * H * B;
  const int sms = num_sms() > 0 ? num_sms() : 1;
  const int grid = items < sms ? items : sms;
  // F16 output rows are written by TMA stores of 32 x 72 blocks: [B][T][D] as a 3-D
  // tensor, so a block's rows past an image's last token are clipped.
  CUtensorMap tmo;
  memset(&tmo, 0, sizeof(tmo));
  if (!out_e4m3) {
    const uint64_t dims[3] = {uint64_t(H) * kDh, uint64_t(T), uint64_t(B)};
    const uint64_t strides[2] = {uint64_t(H) * kDh * 2, uint64_t(T) * H * kDh * 2};
    const uint32_t box[3] = {uint32_t(kDh), 32, 1};
    sv_status st = make_tmap(&tmo, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, o, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != SV_OK) return st;
  }
  if (qk8) return attention_launch_cfg<1, 3, 3, true>(tmo, p, grid, s);
  return attention_launch_cfg<1, 3, 3, false>(tmo, p, grid, s);
}

}  // namespace sv
