// fwd.cu -- tcgen05 forward of cartridge attention (sm_103a).
//
// A work item is two 128-row query tiles, A and B, that stream the same
// keys: in fixed-layout training with an even group size, the same query
// tile of two heads of one kv group (both see exactly the same key tiles);
// otherwise in training, consecutive row tiles of one (sequence, head); in
// decode mode, the two halves of a kv head's stacked decode rows.  Training
// CTAs are persistent (one per SM) and follow a static plan (fixed layout)
// or take items heaviest first from a counter; a decode CTA runs one item.  Both tiles of an item walk the key tiles
// of concat(cartridge rows, real tokens) -- first every cartridge tile (all
// visible), then the real-token tiles up to their diagonal (end-aligned
// causal mask: real key j is visible from query i iff j <= i; Cartridges
// guide, "Semantics", attention bullet) -- so every K/V tile is staged once
// for both.  The two tiles are independent softmax streams: while one
// warpgroup turns its S into P, the tensor pipe runs the other tile's
// products, and the exp work of one tile overlaps the MMAs of the other.
//
// Roles (320 threads):
//   warps 0-3  softmax of tile A, warps 4-7 softmax of tile B.  Thread t owns
//              row t of its tile (TMEM lane t) and reads the whole 128-key S
//              row, so row maxima and sums need no exchange.  O is rescaled
//              in TMEM only when the running maximum grows by more than 2^8
//              (lazy rescaling, log2 domain).  P (bf16 pairs) goes back into
//              TMEM over the first 64 columns of the tile's S.  Training
//              queries arrive rotated (the prep kernel applies RoPE); in
//              decode mode the group rotates the raw queries of row (b, hh)
//              at p + len[b] in shared memory.  The epilogue stages O in a
//              4 KB slice per warp of its own.
//   warp 8     TMA producer: takes the next item, then both Q tiles of the
//              item (once the previous item's S MMAs have read Q), then K
//              and V tiles into two separate 2-stage rings that run on
//              across items.
//   warp 9     MMA issuer (one thread).  Per key tile t:
//                PV_A(t), S_A(t+1) = Q_A K(t+1)^T, PV_B(t), S_B(t+1).
//              One CTA's MMAs run in issue order, so the commit that
//              publishes S_X(t+1) also certifies that PV_X(t) has finished
//              reading P_X(t) and writing O_X.
// TMEM (512 columns): S_A 0-127, S_B 128-255, O_A at 256, O_B at 384.
//
// Variants (one kernel instance each, see FwdMode):
//   packed segments  a sequence's tiles start at its first packed row and
//                    its own length bounds the tiles, the causal mask and
//                    the stores (a store that would cross into the next
//                    segment goes row by row);
//   sliding window   a CTA starts at the first key tile its tile A's first
//                    row can see, and each row masks the keys before its
//                    window (a row that has seen no visible key yet keeps
//                    P = 0); in decode mode the CTA starts at the earliest
//                    window among its conversations.
#include <algorithm>
#include <climits>
#include <cstring>
#include <map>
#include <mutex>
#include <queue>
#include <tuple>
#include <vector>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.cuh"
#include "ptx.cuh"

namespace cart {
namespace {

struct FwdParams {
  int n_rows, Hq_map, G, n_qblocks, p, n_real, cart_tiles_per_split, n_qtiles, n_pairs;
  float scale_log2;
  void* out;
  float* lse;
  int out_f32;
  int decode;
  int tma_out;          // training bf16 output: warps store their rows with mO32
  int tma_dec;          // decode f32 partials: warps store 32 x 32 blocks with mO32
  uint32_t* status;
  // training: work items and the counter CTAs take them from (zeroed by the
  // prep kernel that runs before the forward)
  int n_items;
  // fixed-layout training with an even group size: an item's tile B is the
  // same query tile of the next head (same kv head, same keys) instead of
  // the next query tile of the same head
  int cross;
  int* sched;
  // decode mode: raw query rows r = b*G + hh, rotated here at p + len[b]
  const int* dec_len;
  int dec_B, dec_G, dec_rows;
  int dec_s;  // span: rows of one conversation's s queries are consecutive
  // training, packed layout (SeqRows): segment table and packed token count
  const int* cu;
  int total;
  // sliding window in keys (0: none): the query at position P sees keys at
  // positions P - window + 1 .. P (cartridge row j at position j)
  int window;
  float2 turns[kMaxHeadDim / 2];
};

constexpr int kFwdThreads = 320;

#ifdef CART_TEST_HOOKS
// Test-hook build only: while nonzero, the MMA warp of the first CTA
// withholds its commit to tile B's O-done barrier, whose one waiter is tile
// B's epilogue: that bounded wait runs out, the CTA unwinds through its
// abort path and the status word gets the epilogue bit alone.
__device__ int g_test_skip_arrival;
#endif

template <int D>
struct FwdSmem {
  static constexpr int kTileBytes = kTile * D * 2;  // one 128-row Q, K or V tile (bf16)
  static constexpr int kQ = 0;                      // Q_A, Q_B
  static constexpr int kK = kQ + 2 * kTileBytes;    // K ring, 2 stages
  static constexpr int kV = kK + 2 * kTileBytes;    // V ring, 2 stages
  static constexpr int kStage = kV + 2 * kTileBytes;  // output staging, 4 KB per softmax warp
  static constexpr int kBar = kStage + 8 * 4096;   // barriers, TMEM slot
  static constexpr int kItems = kBar + 256;         // two item slots
  static constexpr int kBytes = kItems + 128;
  static constexpr int kAlloc = kBytes + 1024;      // slack for 1024-B alignment
};

enum FwdBar {
  kQFull = 0,  // TMA: both Q tiles landed
  kQReady0,    // decode, softmax group x: its Q tile is rotated; 128 arrivals
  kQReady1,
  kQEmpty0,    // the item's last S MMA of tile x has read Q_x (MMA commit)
  kQEmpty1,
  kItemFull0,  // the producer published the next item in slot s
  kItemFull1,
  kItemEmpty0, // the MMA warp and the 8 softmax warps have read slot s
  kItemEmpty1,
  kKFull0,
  kKFull1,
  kKEmpty0,
  kKEmpty1,
  kVFull0,
  kVFull1,
  kVEmpty0,
  kVEmpty1,
  kSFull0,  // S of tile x is in TMEM (MMA commit)
  kSFull1,
  kPFull0,  // P of tile x is in TMEM (128 arrivals)
  kPFull1,
  kODone0,  // the last PV of tile x has completed
  kODone1,
  kDrain,
  kNumBars
};
static_assert(kNumBars * 8 + 8 <= 256, "barrier area");

// RoPE of one Q row held in a 128-byte-swizzled tile, in place.
// cs(j0, c) fills c[0..31] with the (cos, sin) of pairs j0..j0+31.
// Rotate-half pairs (c, c + D/2): for D = 128 chunk j of the first 64-wide
// block pairs with chunk j of the second block; for D = 64 chunk j pairs
// with chunk j + 4.  Work goes by 32 pairs: all their angles first, then all
// loads of the row's chunks, then the rotations and stores, so that the
// latencies of each batch overlap.
template <int D, class CS>
__device__ __forceinline__ void rotate_q_row(uint8_t* sQ, uint32_t row, CS cs) {
  const uint32_t base = smem_u32(sQ);
#pragma unroll
  for (int half = 0; half < D / 64; ++half) {
    float2 c[32];
    cs(32 * half, c);
    uint4 av[4], bv[4];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int j = 4 * half + jj;
      const uint32_t o0 = sw128_offset(row, j);
      const uint32_t o1 = D == 128 ? 16384u + sw128_offset(row, j) : sw128_offset(row, j + 4);
      av[jj] = lds_u4(base + o0);
      bv[jj] = lds_u4(base + o1);
    }
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int j = 4 * half + jj;
      const uint32_t o0 = sw128_offset(row, j);
      const uint32_t o1 = D == 128 ? 16384u + sw128_offset(row, j) : sw128_offset(row, j + 4);
      const uint32_t pa[4] = {av[jj].x, av[jj].y, av[jj].z, av[jj].w};
      const uint32_t pb[4] = {bv[jj].x, bv[jj].y, bv[jj].z, bv[jj].w};
      uint32_t ya[4], yb[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = bf16x2_to_float2(pa[e]);
        const float2 fb = bf16x2_to_float2(pb[e]);
        float y0a, y1a, y0b, y1b;
        rope_pair(fa.x, fb.x, c[8 * jj + 2 * e], y0a, y1a);
        rope_pair(fa.y, fb.y, c[8 * jj + 2 * e + 1], y0b, y1b);
        ya[e] = pack_bf16x2(y0a, y0b);
        yb[e] = pack_bf16x2(y1a, y1b);
      }
      sts_u4(base + o0, make_uint4(ya[0], ya[1], ya[2], ya[3]));
      sts_u4(base + o1, make_uint4(yb[0], yb[1], yb[2], yb[3]));
    }
  }
}

enum FwdMode { kFwdTrain = 0, kFwdGeneral = 1, kFwdDecode = 2 };

// One work item: two query tiles A and B that see the same keys, and the key
// tiles they walk -- cartridge tiles [ct_lo, ct_lo + n_ct), then real tiles
// from rt_lo up to each tile's diagonal.  T_x tiles for tile x (0: no work).
struct FwdItem {
  int head, qb, pair, kvh, split;
  int xh;       // tile B: the same rows of head + 1 (pair = their query tile)
  int seq_len;  // rows of the query block (decode: the stacked rows)
  SeqRows sq;   // training: where the query block's rows sit
  int n_ct, ct_lo, rt_lo, T_A, T_B, T;
  bool hasB;
};

// An item as the producer publishes it in a shared-memory slot (w < 0: no
// more items).  The other roles read each field where they use it (volatile
// loads), so that no item field stays in registers across the softmax loop.
struct ItemSlot {
  int w, head, qb, pair, split, seq_len, row0, blk, g0, n_ct, ct_lo, rt_lo, T_A, T_B, T, xh;
};
static_assert(sizeof(ItemSlot) == 64, "item slot");

// Tile counts of a pair of query tiles under the causal mask and the window.
__device__ __forceinline__ void item_tiles(const FwdParams& a, FwdItem& I, int window,
                                           bool decode) {
  const int n_qtiles = decode ? a.n_qtiles : (I.seq_len + kTile - 1) / kTile;
  I.T_A = I.T_B = I.T = I.n_ct = 0;
  I.rt_lo = 0;
  I.hasB = false;
  if (I.xh) {  // two heads, query tile I.pair: the same keys for both
    I.n_ct = (a.p + kTile - 1) / kTile;
    I.ct_lo = 0;
    I.hasB = true;
    I.T_A = I.T_B = I.T = I.n_ct + min(I.pair + 1, n_qtiles);
    return;
  }
  if (2 * I.pair >= n_qtiles) return;  // a packed segment shorter than the longest
  I.hasB = 2 * I.pair + 1 < n_qtiles;
  const int n_ct_all = (a.p + kTile - 1) / kTile;
  int ct_hi = n_ct_all, n_rt_A = 0, n_rt_B = 0;
  if (decode) {
    ct_hi = min((I.split + 1) * a.cart_tiles_per_split, n_ct_all);
  } else {
    I.ct_lo = 0;
    n_rt_A = min(2 * I.pair + 1, n_qtiles);
    n_rt_B = I.hasB ? min(2 * I.pair + 2, n_qtiles) : 0;
    if (window > 0) {
      // the first key any row of tile A sees: position p + q0A - window + 1
      const int lo = a.p + 2 * I.pair * kTile - window + 1;
      if (lo > 0) {
        I.ct_lo = min(lo / kTile, n_ct_all);
        I.rt_lo = lo > a.p ? (lo - a.p) / kTile : 0;
      }
    }
  }
  I.n_ct = max(ct_hi - I.ct_lo, 0);
  I.T_A = I.n_ct + n_rt_A - I.rt_lo;
  I.T_B = I.hasB ? I.n_ct + n_rt_B - I.rt_lo : 0;
  I.T = max(I.T_A, I.T_B);
}

// Training work item w: items are numbered heaviest first (the query tile,
// or pair of tiles, falls as w grows; every item of a sequence sees all
// cartridge tiles and the later ones more real tiles), so CTAs that take the
// next free item form a longest-first schedule.  Cross items (may_cross and
// a.cross): (query tile, sequence, head pair); else (pair, sequence, head).
__device__ __forceinline__ FwdItem train_item(const FwdParams& a, int w, const int* cu,
                                              int window, bool may_cross) {
  FwdItem I;
  I.xh = may_cross && a.cross;
  if (a.cross) {  // (query tile, sequence, head pair), query tile falling
    const int hb = (a.Hq_map / 2) * a.n_qblocks;
    I.pair = a.n_qtiles - 1 - w / hb;
    const int rem = w % hb;
    I.head = 2 * (rem % (a.Hq_map / 2));
    I.qb = rem / (a.Hq_map / 2);
  } else {
    const int hb = a.Hq_map * a.n_qblocks;
    I.pair = a.n_pairs - 1 - w / hb;
    const int rem = w % hb;
    I.head = rem % a.Hq_map;
    I.qb = rem / a.Hq_map;
  }
  I.kvh = I.head / a.G;
  I.split = 0;
  I.sq = seq_rows(cu, a.total, a.n_rows, I.qb);
  I.seq_len = I.sq.len;
  item_tiles(a, I, window, false);
  return I;
}

// Only the fixed-layout instance carries a full static schedule (WorkPlan).
template <int kMode>
using PlanOf = WorkPlan<kMode == kFwdTrain ? kPlanItems : 1>;

// kMode: kFwdTrain (training, fixed [B, n] layout, no window, bf16 output),
// kFwdGeneral (training with packed segments, a sliding window or an f32
// output) or kFwdDecode
// (the decode cartridge pass); each mode compiles only its own code.
//
// Training CTAs are persistent (one per SM): the producer lane takes the
// next item from a counter that the prep kernel zeroed, publishes it in a
// two-slot ring, and every role walks the same item sequence with barrier
// phases that carry across items.  TMEM is allocated once.  Q of the next
// item is loaded as soon as the last S MMA of the current one has read its
// Q tile, and the output is staged in a region of its own, so that the next
// item's first products overlap the current item's last softmax and its
// epilogue.  A decode CTA runs its one item (blockIdx) the same way.
template <int D, int kMode>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mKc,
               const __grid_constant__ CUtensorMap mVc, const __grid_constant__ CUtensorMap mK,
               const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mO32,
               const FwdParams a, const __grid_constant__ PlanOf<kMode> plan) {
  using L = FwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBar + kNumBars * 8);
  ItemSlot* items = reinterpret_cast<ItemSlot*>(smem + L::kItems);
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr bool kDecode = kMode == kFwdDecode;
  // packed training layout: the segment table (a constant null otherwise)
  const int* const cu = kMode == kFwdGeneral ? a.cu : nullptr;
  const int window = kMode == kFwdTrain ? 0 : a.window;

  // ---- decode: this CTA's one item (its window bound needs the block) ----
  FwdItem dec{};
  if (kDecode) {
    dec.head = blockIdx.x;
    dec.qb = 0;
    dec.pair = blockIdx.y;
    dec.kvh = dec.head;
    dec.split = blockIdx.z;
    dec.seq_len = a.n_rows;
    dec.sq = SeqRows{0, 0, 0, a.n_rows};
    const int n_ct_all = (a.p + kTile - 1) / kTile;
    dec.ct_lo = dec.split * a.cart_tiles_per_split;
    if (window > 0) {
      // skip the tiles before every row's window: the earliest first key of
      // the CTA's rows is that of a t = 0 row (conversation b's rows are
      // (b*s + t)*G + hh), position p + len[b] - window + 1
      __shared__ int s_lo;
      if (threadIdx.x == 0) s_lo = INT_MAX;
      __syncthreads();
      const int r_lo = 2 * dec.pair * kTile, r_hi = min(r_lo + 2 * kTile, a.n_rows);
      const int b_lo = (r_lo / a.dec_G) / a.dec_s;
      const int b_hi = min(((r_hi - 1) / a.dec_G) / a.dec_s, a.dec_B / a.dec_s - 1);
      const int lmax = a.dec_rows - a.dec_s;
      for (int bb = b_lo + static_cast<int>(threadIdx.x); bb <= b_hi; bb += blockDim.x) {
        int len = __ldg(a.dec_len + bb);
        len = len < 0 ? 0 : (len > lmax ? lmax : len);
        atomicMin(&s_lo, a.p + len - window + 1);
      }
      __syncthreads();
      const int lo = s_lo;
      const int ct_hi = min(dec.ct_lo + a.cart_tiles_per_split, n_ct_all);
      if (lo > 0) dec.ct_lo = max(dec.ct_lo, min(lo / kTile, ct_hi));  // none left: T = 0
    }
    item_tiles(a, dec, window, true);
  }

  if (threadIdx.x == 0) {
    // decode mode: let the dependent private pass start right away (it waits
    // for this grid before it reads what this grid writes)
    if (kDecode) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    abort_flag = 0;
    mbar_init(&bars[kQFull], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kQReady0 + s], 128);
      mbar_init(&bars[kQEmpty0 + s], 1);
      mbar_init(&bars[kKFull0 + s], 1);
      mbar_init(&bars[kKEmpty0 + s], 1);
      mbar_init(&bars[kVFull0 + s], 1);
      mbar_init(&bars[kVEmpty0 + s], 1);
      mbar_init(&bars[kSFull0 + s], 1);
      mbar_init(&bars[kPFull0 + s], 128);
      mbar_init(&bars[kODone0 + s], 1);
      mbar_init(&bars[kItemFull0 + s], 1);
      mbar_init(&bars[kItemEmpty0 + s], 9);  // the MMA warp and the 8 softmax warps
    }
    mbar_init(&bars[kDrain], 1);
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t abort_s = smem_u32(&abort_flag);
  // (training launches are programmatic dependents of the prep kernel: the
  // set-up above overlaps its end; no global access before this)
  pdl_wait();

  if (warp == 8) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mKc);
      tma_prefetch_desc(&mVc);
      tma_prefetch_desc(&mK);
      tma_prefetch_desc(&mV);
      // the next item: decode has one; training takes the counter's next
      // the next item: decode has one; training follows its static plan
      // if it has one, else takes the counter's next
      auto fetch = [&](int k) -> int {
        if (kDecode) return k == 0 ? 0 : -1;
        if (kMode == kFwdTrain && plan.n > 0) {
          const int o = plan.off[blockIdx.x] + k;
          return o < plan.off[blockIdx.x + 1] ? static_cast<int>(plan.items[o]) : -1;
        }
        const int w = atomicAdd(a.sched, 1);
        return w < a.n_items ? w : -1;
      };
      int g = 0;           // K / V tiles issued, over all items
      int nq = 0;          // Q loads issued (items with work)
      int k_issued = 0, v_issued = 0;
      bool ok = true;
      int w = fetch(0);
      for (int it = 0; ok; ++it) {
        const int sl = it & 1;
        if (it >= 2) {
          ok = mbar_wait(&bars[kItemEmpty0 + sl], ((it >> 1) - 1) & 1, abort_s, a.status,
                         kDevErrTimeoutTma);
          if (!ok) break;
        }
        FwdItem I{};
        if (w >= 0) I = kDecode ? dec : train_item(a, w, cu, window, kMode == kFwdTrain);
        ItemSlot& o = items[sl];
        o.w = w;
        o.head = I.head;
        o.qb = I.qb;
        o.pair = I.pair;
        o.split = I.split;
        o.seq_len = I.seq_len;
        o.row0 = I.sq.row0;
        o.blk = I.sq.blk;
        o.g0 = I.sq.g0;
        o.n_ct = I.n_ct;
        o.ct_lo = I.ct_lo;
        o.rt_lo = I.rt_lo;
        o.T_A = I.T_A;
        o.T_B = I.T_B;
        o.T = I.T;
        o.xh = I.xh;
        mbar_arrive(&bars[kItemFull0 + sl]);  // (release: the slot is visible to the waiters)
        if (w < 0) break;
        const int w_next = fetch(it + 1);
        if (I.T > 0) {
          // Q of this item once every S MMA of the previous one has read Q
          if (nq >= 1) {
            ok = mbar_wait(&bars[kQEmpty0], (nq - 1) & 1, abort_s, a.status, kDevErrTimeoutTma) &&
                 mbar_wait(&bars[kQEmpty1], (nq - 1) & 1, abort_s, a.status, kDevErrTimeoutTma);
            if (!ok) break;
          }
          // tile B: the next 128 rows, or (cross) the same rows of head + 1
          const int q0A = (I.xh ? I.pair : 2 * I.pair) * kTile;
          const int q0B = I.xh ? q0A : q0A + kTile;
          mbar_arrive_expect_tx(&bars[kQFull], 2 * L::kTileBytes);
#pragma unroll
          for (int h = 0; h < D / 64; ++h) {
            // tile B of a lone last tile reads rows past the end: zero fill
            if (kDecode) {  // (d, G, Hkv, B) map, 128/G conversations per box
              tma_load_4d(smem + L::kQ + h * 16384, &mQ, &bars[kQFull], h * 64, 0, I.kvh,
                          q0A / a.dec_G);
              tma_load_4d(smem + L::kQ + L::kTileBytes + h * 16384, &mQ, &bars[kQFull], h * 64,
                          0, I.kvh, (q0A + kTile) / a.dec_G);
            } else {
              tma_load_4d(smem + L::kQ + h * 16384, &mQ, &bars[kQFull], h * 64, I.head,
                          I.sq.row0 + q0A, I.sq.blk);
              tma_load_4d(smem + L::kQ + L::kTileBytes + h * 16384, &mQ, &bars[kQFull], h * 64,
                          I.head + I.xh, I.sq.row0 + q0B, I.sq.blk);
            }
          }
          ++nq;
          for (int t = 0; t < I.T && ok; ++t, ++g) {
            const int s = g & 1;
            const bool cart = t < I.n_ct;
            const int row0 =
                cart ? (I.ct_lo + t) * kTile : I.sq.row0 + (I.rt_lo + t - I.n_ct) * kTile;
            const CUtensorMap* mk = cart ? &mKc : &mK;
            const CUtensorMap* mv = cart ? &mVc : &mV;
            const int blk = cart ? 0 : I.sq.blk;
            if (g >= 2) {
              ok = mbar_wait(&bars[kKEmpty0 + s], ((g >> 1) - 1) & 1, abort_s, a.status,
                             kDevErrTimeoutTma);
              if (!ok) break;
            }
            uint8_t* sK = smem + L::kK + s * L::kTileBytes;
            mbar_arrive_expect_tx(&bars[kKFull0 + s], L::kTileBytes);
#pragma unroll
            for (int h = 0; h < D / 64; ++h)
              tma_load_4d(sK + h * 16384, mk, &bars[kKFull0 + s], h * 64, I.kvh, row0, blk);
            k_issued = g + 1;
            if (g >= 2) {
              ok = mbar_wait(&bars[kVEmpty0 + s], ((g >> 1) - 1) & 1, abort_s, a.status,
                             kDevErrTimeoutTma);
              if (!ok) break;
            }
            uint8_t* sV = smem + L::kV + s * L::kTileBytes;
            mbar_arrive_expect_tx(&bars[kVFull0 + s], L::kTileBytes);
#pragma unroll
            for (int h = 0; h < D / 64; ++h)
              tma_load_4d(sV + h * 16384, mv, &bars[kVFull0 + s], h * 64, I.kvh, row0, blk);
            v_issued = g + 1;
          }
        }
        w = w_next;
      }
      // training: every load of this CTA is issued; the next launch on the
      // stream (which waits for this grid before it touches memory) may
      // start setting up
      if (!kDecode) pdl_release();
      if (!ok) {
        // Give the copies still in flight (the last Q load, the last two K
        // and V tiles) a bounded chance to land before the CTA releases its
        // shared memory.
        if (nq > 0) mbar_wait(&bars[kQFull], (nq - 1) & 1, 0u, nullptr, 0);
        for (int t = max(k_issued - 2, 0); t < k_issued; ++t)
          mbar_wait(&bars[kKFull0 + (t & 1)], (t >> 1) & 1, 0u, nullptr, 0);
        for (int t = max(v_issued - 2, 0); t < v_issued; ++t)
          mbar_wait(&bars[kVFull0 + (t & 1)], (t >> 1) & 1, 0u, nullptr, 0);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ----------------------------------------------------------------- MMA --
    // The whole warp runs this loop (warp-uniform descriptors); one elected
    // lane issues each MMA and commit.
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu,
                        mbar_wait(bar, parity, abort_s, a.status, kDevErrTimeoutMma));
    };
    const uint32_t idS = idesc_bf16(128, 128, false, false);
    const uint32_t idPV = idesc_bf16(128, D, false, true);
    // Base descriptors, computed once; each MMA adds an offset.
    const uint64_t dQ0 = sdesc_sw128(smem_u32(smem + L::kQ), 16u, 1024u);
    const uint64_t dQ1 = desc_add(dQ0, L::kTileBytes);
    const uint64_t dK0 = sdesc_sw128(smem_u32(smem + L::kK), 16u, 1024u);
    const uint64_t dK1 = desc_add(dK0, L::kTileBytes);
    const uint64_t dV0 = sdesc_sw128(smem_u32(smem + L::kV), 16384u, 1024u);
    const uint64_t dV1 = desc_add(dV0, L::kTileBytes);
    // S_x = Q_x K^T from ring slot s (K-major operands; K step k of 16 at
    // byte offset (k/4)*16384 + (k%4)*32 within the two 64-wide blocks)
    auto issue_qk = [&](int x, int s) {
      const uint64_t dq = x ? dQ1 : dQ0;
      const uint64_t dk = s ? dK1 : dK0;
      const uint32_t ts = tmem + x * 128;
      umma_bf16_ss_w(ts, dq, dk, idS, 0u);
#pragma unroll
      for (int k = 1; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
        umma_bf16_ss_w(ts, desc_add(dq, off), desc_add(dk, off), idS, 1u);
      }
      umma_commit_w(&bars[kSFull0 + x]);
    };
    // O_x (+)= P_x V from ring slot s: P from TMEM (K step k of 16 keys = 8
    // packed columns at 8k), V MN-major (16 rows = 2048 B per K step).
    auto issue_pv = [&](int x, int s, bool acc) {
      const uint64_t dv = s ? dV1 : dV0;
      const uint32_t tp = tmem + x * 128;
      const uint32_t to = tmem + 256 + x * 128;
      umma_bf16_ts_w(to, tp, dv, idPV, acc ? 1u : 0u);
#pragma unroll
      for (int k = 1; k < kTile / 16; ++k)
        umma_bf16_ts_w(to, tp + k * 8, desc_add(dv, k * 2048), idPV, 1u);
    };
    int g = 0;             // K / V tiles consumed, over all items
    int nq = 0;            // Q loads consumed
    int nP0 = 0, nP1 = 0;  // P tiles of A / B consumed, over all items
    bool ok = true;
    for (int it = 0; ok && (!kDecode || it < 1); ++it) {
      ok = wait(&bars[kItemFull0 + (it & 1)], (it >> 1) & 1);
      if (!ok) break;
      const ItemSlot& sI = items[it & 1];
      const int w = vld(sI.w);
      const int TA = vld(sI.T_A), TB = vld(sI.T_B), T = vld(sI.T);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kItemEmpty0 + (it & 1)]);  // read all it needs
      if (w < 0) break;
      if (T == 0) continue;
      ok = kDecode ? wait(&bars[kQReady0], 0) : wait(&bars[kQFull], nq & 1);
      ok = ok && wait(&bars[kKFull0 + (g & 1)], (g >> 1) & 1);
      if (ok) {
        tc_fence_after();
        issue_qk(0, g & 1);
        if (TA == 1) umma_commit_w(&bars[kQEmpty0]);
      }
      if (ok && TB > 0) {
        if (kDecode) ok = wait(&bars[kQReady1], 0);
        if (ok) {
          tc_fence_after();
          issue_qk(1, g & 1);
          if (TB == 1) umma_commit_w(&bars[kQEmpty1]);
        }
      }
      if (ok && TB == 0) umma_commit_w(&bars[kQEmpty1]);  // no MMA reads Q_B
      if (ok) umma_commit_w(&bars[kKEmpty0 + (g & 1)]);
      for (int t = 0; t < T && ok; ++t) {
        const int gt = g + t, s = gt & 1;
        ok = wait(&bars[kVFull0 + s], (gt >> 1) & 1);
        if (!ok) break;
        const bool next = t + 1 < T;
        if (t < TA) {
          ok = wait(&bars[kPFull0], (nP0 + t) & 1);
          if (!ok) break;
          tc_fence_after();
          issue_pv(0, s, t > 0);
          if (t == TA - 1) umma_commit_w(&bars[kODone0]);
        }
        if (next) {
          ok = wait(&bars[kKFull0 + (s ^ 1)], ((gt + 1) >> 1) & 1);
          if (!ok) break;
          tc_fence_after();
          if (t + 1 < TA) {
            issue_qk(0, s ^ 1);
            if (t + 1 == TA - 1) umma_commit_w(&bars[kQEmpty0]);
          }
        }
        if (t < TB) {
          ok = wait(&bars[kPFull1], (nP1 + t) & 1);
          if (!ok) break;
          tc_fence_after();
          issue_pv(1, s, t > 0);
#ifdef CART_TEST_HOOKS
          if (t == TB - 1 && !(blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 &&
                               *reinterpret_cast<volatile int*>(&g_test_skip_arrival)))
#else
          if (t == TB - 1)
#endif
            umma_commit_w(&bars[kODone1]);
          if (t + 1 < TB) {
            issue_qk(1, s ^ 1);
            if (t + 1 == TB - 1) umma_commit_w(&bars[kQEmpty1]);
          }
        }
        umma_commit_w(&bars[kVEmpty0 + s]);
        if (next) umma_commit_w(&bars[kKEmpty0 + (s ^ 1)]);
      }
      g += T;
      ++nq;
      nP0 += TA;
      nP1 += TB;
    }
    // Drain: every MMA issued above completes before the CTA tears down.
    umma_commit_w(&bars[kDrain]);
    mbar_wait(&bars[kDrain], 0, 0u, nullptr, 0);
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax --
    const int x = warp >> 2;  // 0: tile A, 1: tile B
    const int row = threadIdx.x & 127;  // == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + x * 128 + lane_off;
    const uint32_t tO = tmem + 256 + x * 128 + lane_off;
    // this warp's output staging slice (32 rows x 128 bytes)
    uint8_t* const stg = smem + L::kStage + warp * 4096;
    int nS = 0;  // S tiles of this tile x consumed, over all items
    int nO = 0;  // items of tile x finished
    bool ok = true;
    // (a decode CTA has one item: the loop ends without reading the end mark)
    for (int it = 0; ok && (!kDecode || it < 1); ++it) {
      ok = mbar_wait(&bars[kItemFull0 + (it & 1)], (it >> 1) & 1, abort_s, a.status,
                     kDevErrTimeoutSoftmax);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      // the slot is released once the item's epilogue is done with it
      const ItemSlot& sI = items[it & 1];
      if (vld(sI.w) < 0) break;
      const int Tx = x ? vld(sI.T_B) : vld(sI.T_A);
      if (Tx == 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kItemEmpty0 + (it & 1)]);
        continue;
      }
      // query row within its block (cross items: the pair's tile, head + x)
      const int i = ((kMode == kFwdTrain && vld(sI.xh)) ? vld(sI.pair) : 2 * vld(sI.pair) + x) *
                        kTile + row;
      const int seq_len = vld(sI.seq_len);
      float m = -INFINITY, l = 0.f;
      // decode: position of the row's first visible key (window > 0)
      int key_lo_dec = 0;
      if (kDecode) {
        // row i = (b*s + t)*G + hh of this kv head: query t of conversation
        // b's span at position p + len[b] + t.  The length, the position and
        // the angles of the first 32 pairs come before the Q tile lands.
        const int vb = i / a.dec_G;
        const bool live = vb < a.dec_B;
        int pos = 0;
        float2 c0[32];
        if (live) {
          int len = __ldg(a.dec_len + vb / a.dec_s);
          const int lmax = a.dec_rows - a.dec_s;
          len = len < 0 ? 0 : (len > lmax ? lmax : len);
          pos = a.p + len + vb % a.dec_s;
          if (window > 0) key_lo_dec = pos - window + 1;
#pragma unroll
          for (int q = 0; q < 32; ++q) c0[q] = rope_cs_turns_fast(a.turns[q], pos);
        }
        ok = mbar_wait(&bars[kQFull], 0, abort_s, a.status, kDevErrTimeoutSoftmax);
        ok = __all_sync(0xffffffffu, ok);
        if (ok && live) {
          rotate_q_row<D>(smem + L::kQ + x * L::kTileBytes, static_cast<uint32_t>(row),
                          [&](int j0, float2* c) {
#pragma unroll
                            for (int q = 0; q < 32; ++q)
                              c[q] = j0 == 0 ? c0[q] : rope_cs_turns_fast(a.turns[j0 + q], pos);
                          });
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars[kQReady0 + x]);
        if (!ok) break;
      }
      const int i_cap = min(i, seq_len - 1);  // decode: no real keys, unused
      // the item's key tiles (kept in registers for the tile loop)
      const int n_ct = vld(sI.n_ct), ct_lo = vld(sI.ct_lo), rt_lo = vld(sI.rt_lo);
      for (int t = 0; t < Tx && ok; ++t) {
        ok = mbar_wait(&bars[kSFull0 + x], (nS + t) & 1, abort_s, a.status,
                       kDevErrTimeoutSoftmax);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        uint32_t r[4][32];
        tmem_ld32(tS, r[0]);
        tmem_ld32(tS + 32, r[1]);
        tmem_ld32(tS + 64, r[2]);
        tmem_ld32(tS + 96, r[3]);
        tmem_ld_wait();
        tmem_reg_fence(r[0]);
        tmem_reg_fence(r[1]);
        tmem_reg_fence(r[2]);
        tmem_reg_fence(r[3]);
        // number of visible keys of this tile (leading columns)
        // and the first one (sliding window); key positions of this tile
        // start at kpos0
        const int kpos0 =
            t < n_ct ? (ct_lo + t) * kTile : a.p + (rt_lo + t - n_ct) * kTile;
        int valid = t < n_ct ? a.p - kpos0 : i_cap - (kpos0 - a.p) + 1;
        valid = max(0, min(valid, kTile));
        int first = 0;
        if (window > 0) {
          const int key_lo = kDecode ? key_lo_dec : a.p + i - window + 1;
          first = max(0, min(key_lo - kpos0, kTile));
        }
        if (__any_sync(0xffffffffu, valid < kTile || first > 0)) {
#pragma unroll
          for (int c = 0; c < kTile; ++c)
            if (c >= valid || c < first) r[c >> 5][c & 31] = __float_as_uint(-INFINITY);
        }
        // row maximum of the raw scores (scale_log2 > 0), 4 independent
        // chains of three-input maxima
        float mx[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float v = fmax3(__uint_as_float(r[q][0]), __uint_as_float(r[q][1]),
                          __uint_as_float(r[q][2]));
#pragma unroll
          for (int c = 3; c < 31; c += 2)
            v = fmax3(v, __uint_as_float(r[q][c]), __uint_as_float(r[q][c + 1]));
          mx[q] = fmaxf(v, __uint_as_float(r[q][31]));
        }
        const float rmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * a.scale_log2;
        // Lazy rescaling: keep the stale max unless the new one exceeds it
        // by more than 8 (P values then stay below 2^8, safe in bf16 / f32).
        float alpha = 1.f;
        bool rescale = false;
        if (rmax > m + 8.f) {
          alpha = exp2_approx(m - rmax);  // exp2(-inf) = 0 on the first tile
          m = rmax;
          rescale = t > 0;
        }
        // P = 2^(S * scale * log2(e) - m), two keys per packed two-lane op
        const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
        // (a row that has seen no visible key yet keeps m = -inf: P = 0)
        const float mr = (kMode != kFwdTrain && m == -INFINITY) ? 0.f : m;
        const float2 nm2 = make_float2(-mr, -mr);
        float2 rs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float2 x0 = __ffma2_rn(u2f2(r[q][2 * c], r[q][2 * c + 1]), sc2, nm2);
            const float2 p01 = make_float2(exp2_approx(x0.x), exp2_approx(x0.y));
            rs[c & 3] = __fadd2_rn(rs[c & 3], p01);
            pk[c] = pack_bf16x2(p01.x, p01.y);
          }
          // keys 32q .. 32q + 31 -> packed columns 16q .. 16q + 15 (S of
          // the whole row is already in registers)
          tmem_st16(tS + 16 * q, pk);
        }
        const float2 rs01 = __fadd2_rn(rs[0], rs[1]), rs23 = __fadd2_rn(rs[2], rs[3]);
        l = l * alpha + ((rs01.x + rs01.y) + (rs23.x + rs23.y));
        if (__any_sync(0xffffffffu, rescale)) {
          // PV(t-1) has completed: the commit that published S(t) follows it.
#pragma unroll
          for (int blk = 0; blk < D / 32; ++blk) {
            uint32_t o[32];
            tmem_ld32(tO + blk * 32, o);
            tmem_ld_wait();
            tmem_reg_fence(o);
            const float2 al2 = make_float2(alpha, alpha);
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              const float2 v = __fmul2_rn(u2f2(o[c], o[c + 1]), al2);
              o[c] = __float_as_uint(v.x);
              o[c + 1] = __float_as_uint(v.y);
            }
            tmem_st32(tO + blk * 32, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars[kPFull0 + x]);
      }
      nS += Tx;
      // ---------------------------------------------------------- epilogue --
      if (ok) {
        ok = mbar_wait(&bars[kODone0 + x], nO & 1, abort_s, a.status, kDevErrTimeoutEpilogue);
        ok = __all_sync(0xffffffffu, ok);
      }
      ++nO;
      if (!ok) break;
      tc_fence_after();
      // (once this thread has read O from TMEM, the next item's first PV may
      // overwrite it: its P-ready arrival for that item comes later)
      // a decode split may hold none of a windowed row's keys: O = 0
      const float inv_l = (kMode == kFwdTrain || l > 0.f) ? 1.f / l : 0.f;
      const bool row_ok = i < seq_len;
      const bool f32 = kDecode || a.out_f32;
      const int head =
          vld(sI.head) + ((kMode == kFwdTrain && vld(sI.xh)) ? x : 0), split = vld(sI.split);
      const SeqRows sq = {vld(sI.row0), vld(sI.blk), vld(sI.g0), seq_len};
      const int wr0 =
          ((kMode == kFwdTrain && vld(sI.xh)) ? vld(sI.pair) : 2 * vld(sI.pair) + x) * kTile +
          (warp & 3) * 32;
      // a packed segment's last rows: a TMA store of the warp's 32 rows would
      // run into the next segment, so those warps store row by row
      // (the fixed-layout training instance always has a bf16 output map)
      const bool use_tma =
          kMode == kFwdTrain ||
          (a.tma_out && (!cu || wr0 + 32 <= sq.len || sq.row0 + sq.len == a.total));
      if (use_tma) {
        // bf16 output by TMA, 64 columns at a time: every thread writes its
        // row into the warp's slice in the 128-byte-swizzled layout of the
        // output map's 64 x 32 box, then lane 0 stores the box (rows past n
        // are clipped by the map) and waits until the slice has been read.
        const uint32_t base = smem_u32(stg);
        // every column block of O in flight at once, one wait
        uint32_t ob[D / 32][32];
#pragma unroll
        for (int blk = 0; blk < D / 32; ++blk) tmem_ld32(tO + blk * 32, ob[blk]);
        tmem_ld_wait();
#pragma unroll
        for (int blk = 0; blk < D / 32; ++blk) tmem_reg_fence(ob[blk]);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t* o = ob[2 * h + (k >> 2)] + 8 * (k & 3);
            sts_u4(base + sw128_offset(static_cast<uint32_t>(lane), static_cast<uint32_t>(k)),
                   make_uint4(pack_bf16x2(__uint_as_float(o[0]) * inv_l, __uint_as_float(o[1]) * inv_l),
                              pack_bf16x2(__uint_as_float(o[2]) * inv_l, __uint_as_float(o[3]) * inv_l),
                              pack_bf16x2(__uint_as_float(o[4]) * inv_l, __uint_as_float(o[5]) * inv_l),
                              pack_bf16x2(__uint_as_float(o[6]) * inv_l, __uint_as_float(o[7]) * inv_l)));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_4d(&mO32, stg, h * 64, head, sq.row0 + wr0, sq.blk);
            bulk_commit_group();
            bulk_wait_read_all();
          }
          __syncwarp();
        }
      } else {
        // Each warp turns its 32 rows x 32 columns at a time around through
        // its slice, so that global stores cover whole 32-byte sectors:
        // 16-byte granule k of staged row r sits at r*128 + (k ^ (r & 7))*16.
        // O is read one 32-column block at a time (few registers live).
        const int gpr = f32 ? 8 : 4;  // 16-byte granules per row and 32 columns
#pragma unroll 1
        for (int blk = 0; blk < D / 32; ++blk) {
          uint32_t o[32];
          tmem_ld32(tO + blk * 32, o);
          tmem_ld_wait();
          tmem_reg_fence(o);
          uint8_t* my = stg + lane * 128;
          if (f32) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              *reinterpret_cast<float4*>(my + ((k ^ (lane & 7)) << 4)) = make_float4(
                  __uint_as_float(o[4 * k]) * inv_l, __uint_as_float(o[4 * k + 1]) * inv_l,
                  __uint_as_float(o[4 * k + 2]) * inv_l, __uint_as_float(o[4 * k + 3]) * inv_l);
          } else {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              *reinterpret_cast<uint4*>(my + ((k ^ (lane & 7)) << 4)) = make_uint4(
                  pack_bf16x2(__uint_as_float(o[8 * k]) * inv_l, __uint_as_float(o[8 * k + 1]) * inv_l),
                  pack_bf16x2(__uint_as_float(o[8 * k + 2]) * inv_l, __uint_as_float(o[8 * k + 3]) * inv_l),
                  pack_bf16x2(__uint_as_float(o[8 * k + 4]) * inv_l, __uint_as_float(o[8 * k + 5]) * inv_l),
                  pack_bf16x2(__uint_as_float(o[8 * k + 6]) * inv_l, __uint_as_float(o[8 * k + 7]) * inv_l));
          }
          __syncwarp();
          if (kDecode && a.tma_dec) {
            // the staged 32 x 32 f32 block is the 128-byte-swizzled layout
            // of the partials map's box: one bulk store (rows past R are
            // clipped)
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_4d(&mO32, stg, blk * 32, wr0, head, split);
              bulk_commit_group();
              bulk_wait_read_all();  // the slice is staged again for the next block
            }
            __syncwarp();
            continue;
          }
          for (int st = 0; st < gpr; ++st) {
            const int gi = st * 32 + lane;
            const int r = gi / gpr, k = gi % gpr;
            const int grow = wr0 + r;
            if (grow < sq.len) {
              const uint4 v = *reinterpret_cast<const uint4*>(stg + r * 128 + ((k ^ (r & 7)) << 4));
              long long off;  // element offset of the row
              if (kDecode)
                off = ((static_cast<long long>(split) * a.Hq_map + head) * a.n_rows + grow) * D;
              else
                off = ((static_cast<long long>(sq.g0) + grow) * a.Hq_map + head) * D;
              if (f32)
                *reinterpret_cast<uint4*>(static_cast<float*>(a.out) + off + blk * 32 + k * 4) = v;
              else
                *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + off + blk * 32 +
                                          k * 8) = v;
            }
          }
          __syncwarp();
        }
      }
      if (row_ok) {
        const float lse2 = m + __log2f(l);
        if (kDecode)
          a.lse[(static_cast<long long>(split) * a.Hq_map + head) * a.n_rows + i] = lse2;
        else
          a.lse[lse_index(cu, a.total, a.n_rows, a.Hq_map, vld(sI.qb), head, sq, i)] =
              lse2 * 0.69314718055994531f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kItemEmpty0 + (it & 1)]);
    }
    if (lane == 0) bulk_wait_all();  // this warp's stores are done before exit
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, 512);
}

// The static schedule for `grid` persistent CTAs and the fixed-layout items
// (numbering of train_item): an item costs its tiles (one unit = one 128-key
// tile for one query tile) plus 2.5 for its start and end.  Cached per
// geometry (its host cost is milliseconds).
const std::vector<uint16_t>& fwd_plan(int n_pairs, int hb, int n_ct, int n_qtiles, int grid,
                                      bool cross, std::vector<uint16_t>* off_out) {
  constexpr double kItemCost = 2.5;
  struct Plan {
    std::vector<uint16_t> items, off;
  };
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int, int, bool>, Plan> cache;
  std::lock_guard<std::mutex> lk(mu);
  const auto key = std::make_tuple(n_pairs, hb, n_ct, n_qtiles, grid, cross);
  auto it = cache.find(key);
  if (it == cache.end()) {
    // cross items: hb counts (sequence, head pair) and an item's two tiles
    // are query tile t of both heads
    const int n = (cross ? n_qtiles : n_pairs) * hb;
    std::vector<double> cost(n);
    for (int w = 0; w < n; ++w) {
      if (cross) {
        const int t = n_qtiles - 1 - w / hb;
        cost[w] = 2 * (n_ct + t + 1) + kItemCost;
        continue;
      }
      const int pr = n_pairs - 1 - w / hb;
      const bool hasB = 2 * pr + 1 < n_qtiles;
      const int rA = std::min(2 * pr + 1, n_qtiles);
      const int rB = hasB ? std::min(2 * pr + 2, n_qtiles) : 0;
      cost[w] = (hasB ? 2 : 1) * n_ct + rA + rB + kItemCost;
    }
    Plan pl;
    build_work_plan(cost, grid, &pl.items, &pl.off);
    it = cache.emplace(key, std::move(pl)).first;
  }
  *off_out = it->second.off;
  return it->second.items;
}

template <int D, int kMode>
cudaError_t launch_fwd_mode(const FwdLaunch& a, const FwdParams& p, dim3 grid,
                            const PlanOf<kMode>& plan, cudaStream_t st) {
  using L = FwdSmem<D>;
  cudaError_t e = set_smem_once<fwd_kernel<D, kMode>>(L::kAlloc);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kFwdThreads, 1, 1);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, fwd_kernel<D, kMode>, *a.mQ, *a.mKc, *a.mVc, *a.mK, *a.mV,
                            (p.tma_out || p.tma_dec) ? *a.mO32 : *a.mQ, p, plan);
}

template <int D>
cudaError_t launch_fwd_d(const FwdLaunch& a, cudaStream_t st) {
  using L = FwdSmem<D>;
  static_assert(L::kAlloc <= 232448, "shared memory budget");
  // kFwdTrain: fixed layout, no window, bf16 output stored by TMA
  const bool general = !a.decode && (a.cu || a.window > 0 || a.out_f32 || !a.mO32);
  FwdParams p{};
  p.n_rows = a.n_rows;
  p.Hq_map = a.Hq_map;
  p.G = a.G;
  p.n_qblocks = a.n_qblocks;
  p.p = a.p;
  p.n_real = a.n_real;
  p.cart_tiles_per_split = a.cart_tiles_per_split;
  p.n_qtiles = (a.n_rows + kTile - 1) / kTile;
  p.n_pairs = (p.n_qtiles + 1) / 2;
  p.scale_log2 = a.scale_log2;
  p.out = a.out;
  p.lse = a.lse;
  p.out_f32 = a.out_f32 ? 1 : 0;
  p.decode = a.decode ? 1 : 0;
  p.tma_out = (!a.decode && !a.out_f32 && a.mO32) ? 1 : 0;
  p.tma_dec = (a.decode && a.mO32) ? 1 : 0;
  p.status = device_status_ptr();
  // fixed-layout training with an even group size pairs heads, not tiles
  p.cross = (!a.decode && !general && a.G % 2 == 0) ? 1 : 0;
  p.n_items = p.cross ? p.n_qtiles * (a.Hq_map / 2) * a.n_qblocks
                      : p.n_pairs * a.Hq_map * a.n_qblocks;
  p.sched = a.sched;
  if (a.decode) {
    p.dec_len = a.dec_len;
    p.dec_B = a.dec_B;
    p.dec_G = a.dec_G;
    p.dec_rows = a.dec_rows;
    p.dec_s = a.dec_s;
    for (int j = 0; j < kMaxHeadDim / 2; ++j) p.turns[j] = a.freqs->turns[j];
  } else {
    p.cu = a.cu;
    p.total = a.total;
  }
  p.window = a.window;
  if (a.decode) {
    PlanOf<kFwdDecode> none{};
    return launch_fwd_mode<D, kFwdDecode>(a, p, dim3(a.Hq_map, p.n_pairs, a.n_splits), none, st);
  }
  // persistent: one CTA per SM, none idle from the start
  const int nsm = sm_count();
  if (nsm < 1) return cudaErrorInvalidValue;
  const int g = p.n_items < nsm ? p.n_items : nsm;
  TraceScope tr("fwd", st);
  if (general) {
    PlanOf<kFwdGeneral> none{};
    return launch_fwd_mode<D, kFwdGeneral>(a, p, dim3(g, 1, 1), none, st);
  }
  static thread_local PlanOf<kFwdTrain> plan;
  plan.n = 0;
  if (p.n_items <= kPlanItems && g <= kPlanCtas) {
    std::vector<uint16_t> off;
    const std::vector<uint16_t>& items =
        fwd_plan(p.n_pairs, (p.cross ? a.Hq_map / 2 : a.Hq_map) * a.n_qblocks,
                 (a.p + kTile - 1) / kTile, p.n_qtiles, g, p.cross != 0, &off);
    plan.n = static_cast<int>(items.size());
    std::memcpy(plan.off, off.data(), off.size() * sizeof(uint16_t));
    std::memcpy(plan.items, items.data(), items.size() * sizeof(uint16_t));
  }
  return launch_fwd_mode<D, kFwdTrain>(a, p, dim3(g, 1, 1), plan, st);
}

}  // namespace

cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t st) {
  if (!a.decode && !a.sched) return cudaErrorInvalidValue;
  if (a.decode && (!a.dec_len || !a.freqs || a.dec_G < 1 || kTile % a.dec_G != 0 ||
                   a.dec_s < 1 || a.dec_B % a.dec_s != 0))
    return cudaErrorInvalidValue;
  if (a.d == 128) return launch_fwd_d<128>(a, st);
  if (a.d == 64) return launch_fwd_d<64>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace cart

#ifdef CART_TEST_HOOKS
// Test-hook build only: sets the flag above (0 or 1) on the current device.
extern "C" CART_API int cart_test_skip_arrival(int on) {
  return cudaMemcpyToSymbol(cart::g_test_skip_arrival, &on, sizeof on) == cudaSuccess
             ? CART_OK
             : CART_ERR_CUDA;
}
#endif
