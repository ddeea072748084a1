// bwd.cu -- tcgen05 backward of cartridge attention (sm_103a).
//
// Gradients of sum(dO * O) for O = softmax(scale * q~ K~^T + mask) V with
// K~ = concat(cartridge rows, RoPE(real keys)), end-aligned causal mask.
// (Cartridges guide, "Semantics": the f32-KV backward routes gradients
// through the concat into the trainable rows; row 0 is the frozen sink.)
//
// With the forward's log-sum-exp per query row, P = exp(scale*S - lse) and
// D_i = sum_c dO_ic O_ic, the softmax backward is dS = P (dP - D) with
// dP = dO V^T.  Two kernels, no atomics, deterministic:
//
//  dkdv_kernel  one CTA per 128-row key tile.  A cartridge tile is seen by
//               every query of every sequence, so its CTA loops over all
//               (sequence, head of the group, 128-row query tile) and sums the
//               batch inside its TMEM accumulators: the cartridge gradient
//               needs no cross-CTA reduction.  A real-token tile loops over
//               the heads of the group and the query tiles at or after it.
//               Per step: S^T = K Q^T, dP^T = V dO^T (TMEM, double buffered),
//               P^T, dS^T (bf16, shared memory), dV += P^T dO, dK += dS^T Q.
//               Epilogue: cartridge rows (f32, frozen rows = 0) or
//               real rows (dK rotated back by R(p+j)^T).
//  dq_kernel    persistent, one 128-row query tile per work item: S = Q K^T,
//               dP = dO V^T, dS = P (dP - D) -> TMEM, dQ += dS K over
//               128-key steps; epilogue rotates back by R(p+i)^T.
// Both kernels have a second instance (kGeneral) for packed segments and /
// or a sliding window: sequences located through the segment table, key
// tiles limited to the query tiles' windows and query tiles to the key
// tiles' windows, per-row / per-key window bounds in the masks, and exact
// zeros for cartridge tiles no query reaches.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <type_traits>
#include <vector>

#include "internal.cuh"
#include "ptx.cuh"

namespace cart {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
  int B, n, Hq, Hkv, G, p, frozen_prefix, n_ct, n_rt, n_qtiles;
  float scale, scale_log2;
  const float* nlse2;  // [B, Hq, npad] -lse * log2(e) (-inf past n)
  const float* nDvec;  // [B, Hq, npad] -D (0 past n)
  int npad;
  void* dq;
  void* dk;
  void* dv;
  int out_f32;
  float* dkc;
  float* dvc;
  int accumulate;
  const float2* table;
  uint32_t* status;
  // dQ: work items (query tiles of every head and sequence) and the counter
  // CTAs take them from (zeroed by the prep launch before the backward)
  int n_items;
  int* sched;
  // RoPE angle of pair c at position x, in turns: x * (turns[c].x + turns[c].y)
  float2 turns[kMaxHeadDim / 2];
  // cartridge rows frozen besides those < frozen_prefix (composed parts' sinks)
  int n_frozen;
  int frozen_rows[CART_MAX_FROZEN_ROWS];
  // packed layout (SeqRows): segment table and packed token count
  const int* cu;
  int total;
  // sliding window in keys (0: none): the query at position P sees keys at
  // positions P - window + 1 .. P (cartridge row j at position j)
  int window;
};

// Query tiles (of any sequence) that can see a key at position kmax or
// before under the window: queries i <= kmax - p + window - 1.
__device__ __forceinline__ int window_qtiles(const BwdParams& a, int window, int kmax) {
  if (window <= 0) return 1 << 30;
  const int i_max = kmax - a.p + window - 1;
  return i_max < 0 ? 0 : i_max / kTile + 1;
}

// 128-row query tiles of sequence b (cu: the packed table, or null).
__device__ __forceinline__ int seq_qtiles(const BwdParams& a, const int* cu, int b) {
  return cu ? (seq_rows(cu, a.total, a.n, b).len + kTile - 1) / kTile : a.n_qtiles;
}

// Cartridge row j gets no gradient: below frozen_prefix, or listed.
__device__ __forceinline__ bool row_frozen(const BwdParams& a, int j) {
  bool f = j < a.frozen_prefix;
  for (int i = 0; i < a.n_frozen; ++i) f |= a.frozen_rows[i] == j;
  return f;
}

__device__ __forceinline__ void store_row_out(void* base, long long off, const float* x, int n,
                                              bool f32) {
  if (f32) {
    float4* d4 = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
    for (int c = 0; c < n / 4; ++c)
      d4[c] = make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]);
  } else {
    uint4* d4 = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + off);
    for (int c = 0; c < n / 8; ++c)
      d4[c] = make_uint4(pack_bf16x2(x[8 * c], x[8 * c + 1]), pack_bf16x2(x[8 * c + 2], x[8 * c + 3]),
                         pack_bf16x2(x[8 * c + 4], x[8 * c + 5]),
                         pack_bf16x2(x[8 * c + 6], x[8 * c + 7]));
  }
}

// =========================================================== dK / dV ======
// Threads: warps 0-15 are four P^T / dS^T warpgroups that share every
// 128-query step, warpgroup w taking queries [32w, 32w + 32) (thread t of a
// group owns key row t = TMEM lane t); warp 16 is the TMA producer, warp 17
// issues the MMAs.  Every MMA has N = 128.
// TMEM (512 columns): S^T at 0, dP^T at 128 (f32), dV at 256, dK at 384.
// A warpgroup loads its 32 S^T columns, forms P^T and writes it packed as
// bf16 pairs over the first 16 of them (P phase); it later loads its 32 dP^T
// columns and writes dS^T the same way over the first 16 of those (dS
// phase).  dV and dK read P^T / dS^T as their A operand straight from TMEM
// (K step k of 16 queries at column (k/2)*32 + (k%2)*8 of the region).
// MMA order per step u:
//   dV(u) [after the P phase], S^T(u+1), dK(u) [after the dS phase], dP^T(u+1)
// so that dV(u) and S^T(u+1) run during the dS phase and dK(u), dP^T(u+1)
// during the next P phase; S^T(u+1) overwrites P^T(u) after dV(u) has read
// it, dP^T(u+1) overwrites dS^T(u) after dK(u) (one CTA's MMAs run in issue
// order).
// Q and dO have rings of their own: a Q slot is released by dK(u), a dO
// slot by dV(u).  Q gets three slots, so a Q tile is copied while two full
// steps of MMAs run; dO gets two (its first reader, dP^T, comes later in the
// step).  The step's -lse2 entries travel with Q, its -D entries with dO.
// The layout fills the 227 KB limit, so it relies on the dynamic shared
// memory starting 1024-byte aligned (checked at entry; no static shared
// variables).
constexpr int kDkdvThreads = 576;
constexpr int kDkdvQSlots = 3, kDkdvDoSlots = 2;

template <int D>
struct DkdvSmem {
  static constexpr int kTileBytes = kTile * D * 2;           // 128-row bf16 tile
  static constexpr int kK = 0;                                // resident K
  static constexpr int kV = kK + kTileBytes;                  // resident V
  static constexpr int kQ0 = kV + kTileBytes;                 // Q ring
  static constexpr int kDo0 = kQ0 + kDkdvQSlots * kTileBytes;  // dO ring
  static constexpr int kVecL = kDo0 + kDkdvDoSlots * kTileBytes;  // -lse2 [128] per Q slot
  static constexpr int kVecD = kVecL + kDkdvQSlots * 512;         // -D [128] per dO slot
  static constexpr int kBar = kVecD + kDkdvDoSlots * 512;
  static constexpr int kBytes = kBar + 256;
  static constexpr int kAlloc = kBytes;
  static_assert(kAlloc <= 232448, "dK/dV shared memory above the 227 KB limit");
};

enum DkdvBar { kResFull = 0, kQFull0, kQEmpty0 = kQFull0 + kDkdvQSlots,
               kDoFull0 = kQEmpty0 + kDkdvQSlots, kDoEmpty0 = kDoFull0 + kDkdvDoSlots,
               kStFull = kDoEmpty0 + kDkdvDoSlots, kPtFull, kDpTFull, kDsFull, kAccDone,
               kDkdvDrain, kDkdvBars };
// barrier area: the barriers, the TMEM address, the abort word, and the
// query tile of the step in each Q slot (read by the masks under a window)
static_assert(kDkdvBars * 8 + 16 + 4 * kDkdvQSlots <= 256, "dK/dV barrier area");

// The steps of a key tile in order: a cartridge tile sees every (sequence,
// head of the group, 128-row query tile), sequence-major; real tile rt of a
// sequence sees the heads of the group and query tiles rt.. (the causal
// diagonal and after).  Under a sliding window only the first qcap query
// tiles of a sequence can reach the key tile.  The query tile runs fastest,
// then the head.  (Packed and / or windowed instances; the fixed layout
// without a window maps a step to its tile in closed form.)
struct DkdvCursor {
  int b, hh, qt;
  int nq;         // query tiles of sequence b that see the key tile
  int qcap;       // query tiles the window lets see the key tile
  int row0, blk;  // sequence b on the maps' token axis
  __device__ __forceinline__ void load_seq(const BwdParams& a, const int* cu) {
    const SeqRows r = seq_rows(cu, a.total, a.n, b);
    nq = min(cu ? (r.len + kTile - 1) / kTile : a.n_qtiles, qcap);
    row0 = r.row0;
    blk = r.blk;
  }
  __device__ __forceinline__ void start(const BwdParams& a, const int* cu, bool cart, int b_real,
                                        int rt, int cap) {
    qcap = cap;
    b = cart ? 0 : b_real;
    hh = 0;
    qt = cart ? 0 : rt;
    load_seq(a, cu);
    if (cart) skip_empty(a, cu);
  }
  // (cartridge tiles) move past sequences without tokens
  __device__ __forceinline__ void skip_empty(const BwdParams& a, const int* cu) {
    while (nq == 0 && b + 1 < a.B) {
      ++b;
      load_seq(a, cu);
    }
  }
  __device__ __forceinline__ void next(const BwdParams& a, const int* cu, bool cart, int rt) {
    if (++qt < nq) return;
    qt = cart ? 0 : rt;
    if (++hh < a.G || !cart) return;
    hh = 0;
    if (b + 1 < a.B) {
      ++b;
      load_seq(a, cu);
      skip_empty(a, cu);
    }
  }
};

__device__ __forceinline__ void write_cart_row(float* dst, const float* x, int n, bool frozen,
                                               int accumulate) {
  float4* d4 = reinterpret_cast<float4*>(dst);
  for (int c = 0; c < n / 4; ++c) {
    float4 v = make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]);
    if (frozen) {
      v = make_float4(0.f, 0.f, 0.f, 0.f);
    } else if (accumulate) {
      const float4 o = d4[c];
      v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
    }
    d4[c] = v;
  }
}

template <int D, bool kGeneral>
__global__ void __launch_bounds__(kDkdvThreads, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mdO,
                const __grid_constant__ CUtensorMap mKc, const __grid_constant__ CUtensorMap mVc,
                const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
                const BwdParams a) {
  using L = DkdvSmem<D>;
  constexpr int SQ = kDkdvQSlots, SD = kDkdvDoSlots;
  extern __shared__ __align__(1024) uint8_t dkdv_smem[];
  uint8_t* smem = dkdv_smem;
  if (smem_u32(smem) & 1023u) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0 && a.status) atomicOr(a.status, kDevErrSmemLayout);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBar + kDkdvBars * 8);
  int* abort_flag = reinterpret_cast<int*>(smem + L::kBar + kDkdvBars * 8 + 8);
  int* step_qt = reinterpret_cast<int*>(smem + L::kBar + kDkdvBars * 8 + 16);  // [SQ]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int* const cu = kGeneral ? a.cu : nullptr;  // packed segment table
  const int window = kGeneral ? a.window : 0;

  // ---- work item: cartridge tiles first (heaviest), then real tiles ----
  int blk = blockIdx.x;
  bool cart;
  int g, tile, b_real = 0;
  if (blk < a.n_ct * a.Hkv) {
    cart = true;
    tile = blk / a.Hkv;
    g = blk % a.Hkv;
  } else {
    cart = false;
    blk -= a.n_ct * a.Hkv;
    tile = blk / (a.Hkv * a.B);
    const int rem = blk % (a.Hkv * a.B);
    b_real = rem / a.Hkv;
    g = rem % a.Hkv;
  }
  // query tiles the window lets see this key tile (its last key position)
  const int qcap = window_qtiles(
      a, window, cart ? min(tile * kTile + kTile - 1, a.p - 1) : a.p + tile * kTile + kTile - 1);
  int U;
  if (!kGeneral) {
    U = cart ? a.B * a.G * a.n_qtiles : a.G * max(a.n_qtiles - tile, 0);
  } else if (cart) {  // every sequence's query tiles
    int tiles = 0;
    for (int b = 0; b < a.B; ++b) tiles += min(seq_qtiles(a, cu, b), qcap);
    U = a.G * tiles;
  } else {
    U = a.G * max(min(seq_qtiles(a, cu, b_real), qcap) - tile, 0);
  }
  if (kGeneral && U == 0) {
    // no query sees the tile: a packed segment shorter than the longest, or
    // cartridge rows before every query's window (gradient 0); the fixed
    // layout without a window always has steps
    if (cart) {
      for (int e = threadIdx.x; e < kTile * (D / 4); e += blockDim.x) {
        const int j = tile * kTile + e / (D / 4);
        if (j >= a.p) continue;
        const float zero[4] = {0.f, 0.f, 0.f, 0.f};
        const long long off = (static_cast<long long>(j) * a.Hkv + g) * D + (e % (D / 4)) * 4;
        write_cart_row(a.dkc + off, zero, 4, row_frozen(a, j), a.accumulate);
        write_cart_row(a.dvc + off, zero, 4, row_frozen(a, j), a.accumulate);
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(&bars[kResFull], 1);
    for (int s = 0; s < SQ; ++s) {
      mbar_init(&bars[kQFull0 + s], 1);
      mbar_init(&bars[kQEmpty0 + s], 1);
    }
    for (int s = 0; s < SD; ++s) {
      mbar_init(&bars[kDoFull0 + s], 1);
      mbar_init(&bars[kDoEmpty0 + s], 1);
    }
    mbar_init(&bars[kStFull], 1);
    mbar_init(&bars[kPtFull], 512);
    mbar_init(&bars[kDpTFull], 1);
    mbar_init(&bars[kDsFull], 512);
    mbar_init(&bars[kAccDone], 1);
    mbar_init(&bars[kDkdvDrain], 1);
    fence_mbar_init();
  }
  if (warp == 17) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tST = tmem, tDP = tmem + 128, tDV = tmem + 256, tDK = tmem + 384;
  const uint32_t abort_s = smem_u32(abort_flag);
  uint8_t* sK = smem + L::kK;
  uint8_t* sV = smem + L::kV;
  float* vecL = reinterpret_cast<float*>(smem + L::kVecL);
  float* vecD = reinterpret_cast<float*>(smem + L::kVecD);

  if (warp == 16) {
    // ------------------------------------------------------------ producer --
    // One lane: per step the Q tile with the step's 128 entries of -lse2,
    // then the dO tile with its 128 entries of -D (TMA for the tiles, plain
    // bulk copies from the padded row vectors), each pair completing on its
    // ring slot's full barrier.
    if (lane == 0 && U > 0) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mdO);
      mbar_arrive_expect_tx(&bars[kResFull], 2 * L::kTileBytes);
#pragma unroll
      for (int h = 0; h < D / 64; ++h) {
        if (cart) {
          tma_load_4d(sK + h * 16384, &mKc, &bars[kResFull], h * 64, g, tile * kTile, 0);
          tma_load_4d(sV + h * 16384, &mVc, &bars[kResFull], h * 64, g, tile * kTile, 0);
        } else {
          const SeqRows r = seq_rows(cu, a.total, a.n, b_real);
          tma_load_4d(sK + h * 16384, &mK, &bars[kResFull], h * 64, g, r.row0 + tile * kTile,
                      r.blk);
          tma_load_4d(sV + h * 16384, &mV, &bars[kResFull], h * 64, g, r.row0 + tile * kTile,
                      r.blk);
        }
      }
      int issued_q = 0, issued_do = 0;
      bool ok = true;
      DkdvCursor it;
      if (kGeneral) it.start(a, cu, cart, b_real, tile, qcap);
      for (int u = 0; u < U; ++u) {
        const int sq = u % SQ, sd = u % SD;
        if (kGeneral) {
          if (u > 0) it.next(a, cu, cart, tile);
        } else {  // fixed layout: every sequence has n_qtiles query tiles
          const int nq = cart ? a.n_qtiles : a.n_qtiles - tile;
          const int per_b = a.G * nq;
          it.b = cart ? u / per_b : b_real;
          it.hh = (u % per_b) / nq;
          it.qt = (cart ? 0 : tile) + u % nq;
          it.row0 = 0;
          it.blk = it.b;
        }
        const int h = g * a.G + it.hh;
        uint8_t* sQ = smem + L::kQ0 + sq * L::kTileBytes;
        uint8_t* sdO = smem + L::kDo0 + sd * L::kTileBytes;
        const long long vo = (static_cast<long long>(it.b) * a.Hq + h) * a.npad + it.qt * kTile;
        if (u >= SQ) {
          ok = mbar_wait(&bars[kQEmpty0 + sq], ((u / SQ) - 1) & 1, abort_s, a.status,
                         kDevErrTimeoutTma);
          if (!ok) break;
        }
        if (kGeneral) step_qt[sq] = it.qt;  // published by the arrive below
        mbar_arrive_expect_tx(&bars[kQFull0 + sq], L::kTileBytes + 512);
#pragma unroll
        for (int hc = 0; hc < D / 64; ++hc)
          tma_load_4d(sQ + hc * 16384, &mQ, &bars[kQFull0 + sq], hc * 64, h,
                      it.row0 + it.qt * kTile, it.blk);
        bulk_load(vecL + sq * 128, a.nlse2 + vo, 512, &bars[kQFull0 + sq]);
        issued_q = u + 1;
        if (u >= SD) {
          ok = mbar_wait(&bars[kDoEmpty0 + sd], ((u / SD) - 1) & 1, abort_s, a.status,
                         kDevErrTimeoutTma);
          if (!ok) break;
        }
        mbar_arrive_expect_tx(&bars[kDoFull0 + sd], L::kTileBytes + 512);
#pragma unroll
        for (int hc = 0; hc < D / 64; ++hc)
          tma_load_4d(sdO + hc * 16384, &mdO, &bars[kDoFull0 + sd], hc * 64, h,
                      it.row0 + it.qt * kTile, it.blk);
        bulk_load(vecD + sd * 128, a.nDvec + vo, 512, &bars[kDoFull0 + sd]);
        issued_do = u + 1;
      }
      if (!ok) {
        // let the copies in flight land before the CTA exits
        mbar_wait(&bars[kResFull], 0, 0u, nullptr, 0);
        for (int u = max(issued_q - SQ, 0); u < issued_q; ++u)
          mbar_wait(&bars[kQFull0 + u % SQ], (u / SQ) & 1, 0u, nullptr, 0);
        for (int u = max(issued_do - SD, 0); u < issued_do; ++u)
          mbar_wait(&bars[kDoFull0 + u % SD], (u / SD) & 1, 0u, nullptr, 0);
      }
    }
    __syncwarp();
  } else if (warp == 17) {
    // ----------------------------------------------------------------- MMA --
    // The whole warp runs this loop (warp-uniform descriptors); one elected
    // lane issues each MMA and commit.
    if (U > 0) {
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu,
                          mbar_wait(bar, parity, abort_s, a.status, kDevErrTimeoutMma));
      };
      const uint32_t idST = idesc_bf16(128, 128, false, false);
      const uint32_t idACC = idesc_bf16(128, D, false, true);
      const uint64_t dK0 = sdesc_sw128(smem_u32(sK), 16u, 1024u);
      const uint64_t dV0 = sdesc_sw128(smem_u32(sV), 16u, 1024u);
      // Q and dO ring slots as K-major (S^T, dP^T) and MN-major (dK, dV)
      const uint64_t dQk0 = sdesc_sw128(smem_u32(smem + L::kQ0), 16u, 1024u);
      const uint64_t dQm0 = sdesc_sw128(smem_u32(smem + L::kQ0), 16384u, 1024u);
      const uint64_t dOk0 = sdesc_sw128(smem_u32(smem + L::kDo0), 16u, 1024u);
      const uint64_t dOm0 = sdesc_sw128(smem_u32(smem + L::kDo0), 16384u, 1024u);
      // C (f32, TMEM) = A (128 rows) * B^T (128 rows), both K-major over d
      auto issue_nt = [&](uint32_t c, uint64_t da, uint64_t db) {
        umma_bf16_ss_w(c, da, db, idST, 0u);
#pragma unroll
        for (int k = 1; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
          umma_bf16_ss_w(c, desc_add(da, off), desc_add(db, off), idST, 1u);
        }
      };
      // S^T = K Q^T from Q slot `slot`, or dP^T = V dO^T from dO slot `slot`
      auto issue_st_dpt = [&](int slot, bool st) {
        if (st) {
          issue_nt(tST, dK0, desc_add(dQk0, slot * L::kTileBytes));
          umma_commit_w(&bars[kStFull]);
        } else {
          issue_nt(tDP, dV0, desc_add(dOk0, slot * L::kTileBytes));
          umma_commit_w(&bars[kDpTFull]);
        }
      };
      bool ok = wait(&bars[kResFull], 0) &&
                wait(&bars[kQFull0], 0);
      if (ok) {
        tc_fence_after();
        issue_st_dpt(0, true);
        ok = wait(&bars[kDoFull0], 0);
        tc_fence_after();
        if (ok) issue_st_dpt(0, false);
      }
      // ring slots and phases advance incrementally (no division per step)
      int sq = 0, sd = 0, sq1 = 1 % SQ, sd1 = 1 % SD;
      uint32_t ph1q = SQ == 1 ? 1u : 0u, ph1d = SD == 1 ? 1u : 0u;  // phases of slot u+1
      for (int u = 0; u < U && ok; ++u) {
        const bool next = u + 1 < U;
        const uint32_t first = u > 0 ? 1u : 0u;
        // dV += P^T dO: A = P^T from TMEM (over S^T), B = the step's dO tile
        // as an MN-major operand (16 rows = 2048 B per K step)
        ok = wait(&bars[kPtFull], u & 1);
        if (!ok) break;
        tc_fence_after();
        const uint64_t ddo = desc_add(dOm0, sd * L::kTileBytes);
        umma_bf16_ts_w(tDV, tST, ddo, idACC, first);
#pragma unroll
        for (int k = 1; k < kTile / 16; ++k)
          umma_bf16_ts_w(tDV, tST + (k >> 1) * 32 + (k & 1) * 8, desc_add(ddo, k * 2048), idACC,
                         1u);
        umma_commit_w(&bars[kDoEmpty0 + sd]);
        if (next) {  // S^T(u+1) over P^T(u), after dV(u) in issue order
          ok = wait(&bars[kQFull0 + sq1], ph1q);
          if (!ok) break;
          tc_fence_after();
          issue_st_dpt(sq1, true);
        }
        // dK += dS^T Q: A = dS^T from TMEM (over dP^T), B = the Q tile
        ok = wait(&bars[kDsFull], u & 1);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dq = desc_add(dQm0, sq * L::kTileBytes);
        umma_bf16_ts_w(tDK, tDP, dq, idACC, first);
#pragma unroll
        for (int k = 1; k < kTile / 16; ++k)
          umma_bf16_ts_w(tDK, tDP + (k >> 1) * 32 + (k & 1) * 8, desc_add(dq, k * 2048), idACC,
                         1u);
        umma_commit_w(&bars[kQEmpty0 + sq]);
        if (next) {  // dP^T(u+1) over dS^T(u), after dK(u) in issue order
          ok = wait(&bars[kDoFull0 + sd1], ph1d);
          if (!ok) break;
          tc_fence_after();
          issue_st_dpt(sd1, false);
        }
        sq = sq1;
        sd = sd1;
        if (++sq1 == SQ) sq1 = 0, ph1q ^= 1u;
        if (++sd1 == SD) sd1 = 0, ph1d ^= 1u;
      }
      if (ok) umma_commit_w(&bars[kAccDone]);
      umma_commit_w(&bars[kDkdvDrain]);
      mbar_wait(&bars[kDkdvDrain], 0, 0u, nullptr, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------- P^T / dS^T warpgroups 0-3 --
    const int wg = warp >> 2;
    const int row = threadIdx.x & 127;  // key row within the tile == TMEM lane
    const int j = tile * kTile + row;
    // real tiles: the sequence's query tiles (those the window allows) and
    // tokens; the last query that sees this key under the window
    const int nq_real = cart ? 0 : min(seq_qtiles(a, cu, b_real), qcap);
    const int i_hi = window > 0 ? (cart ? j : a.p + j) - a.p + window - 1 : 1 << 30;
    const bool key_ok = cart ? (j < a.p) : (j < (cu ? seq_rows(cu, a.total, a.n, b_real).len : a.n));
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    bool ok = true;
    // ring slots, their phases and (real tiles) the query tile of step u,
    // advanced incrementally: no integer division in the per-step path
    int sq = 0, sd = 0, qt = tile;
    uint32_t phq = 0, phd = 0;
    for (int u = 0; u < U && ok; ++u) {
      ok = mbar_wait(&bars[kStFull], u & 1, abort_s, a.status, kDevErrTimeoutSoftmax);
      // the step's -lse2 entries landed with Q (kQFull already complete: the
      // MMAs behind kStFull waited for it); waiting makes them visible
      if (ok) ok = mbar_wait(&bars[kQFull0 + sq], phq, abort_s, a.status, kDevErrTimeoutSoftmax);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tst = tST + wg * 32 + lane_off;
      const uint32_t tdp = tDP + wg * 32 + lane_off;
      // this group's columns c (query qt*128 + wg*32 + c) are invisible
      // for c < qlim: none for a cartridge key, query < key for a real key,
      // all for rows past the end of the keys
      const int qlim = !key_ok ? 32 : (cart ? 0 : max(0, min(32, j - qt * kTile - wg * 32)));
      // ... and for c >= qhi (past the key's window)
      // (a cartridge tile's steps run over every sequence's query tiles: the
      // producer leaves the step's tile next to its Q slot)
      const int qt_u = (window > 0 && cart) ? *reinterpret_cast<volatile int*>(step_qt + sq) : qt;
      const int qhi = window > 0 ? max(0, min(32, i_hi - qt_u * kTile - wg * 32 + 1)) : 32;
      const uint32_t lse_s = smem_u32(vecL + sq * 128 + wg * 32);
      const uint32_t dv_s = smem_u32(vecD + sd * 128 + wg * 32);
      uint32_t r[32];
      tmem_ld32(tst, r);
      tmem_ld_wait();
      tmem_reg_fence(r);
      // P^T = 2^(S^T * scale * log2(e) - lse2) (f32, kept in p for dS^T)
      // while dP^T is still being computed; two queries per packed op
      const bool masked = __any_sync(0xffffffffu, qlim > 0 || qhi < 32);
      const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
      float2 p[16];
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 l4 = lds128(lse_s + c4 * 16);  // -lse2 of 4 queries
        const float2 x0 = __ffma2_rn(u2f2(r[4 * c4], r[4 * c4 + 1]), sc2, make_float2(l4.x, l4.y));
        const float2 x1 =
            __ffma2_rn(u2f2(r[4 * c4 + 2], r[4 * c4 + 3]), sc2, make_float2(l4.z, l4.w));
        p[2 * c4] = make_float2(exp2_approx(x0.x), exp2_approx(x0.y));
        p[2 * c4 + 1] = make_float2(exp2_approx(x1.x), exp2_approx(x1.y));
      }
      if (masked) {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          p[c].x = (2 * c >= qlim && 2 * c < qhi) ? p[c].x : 0.f;
          p[c].y = (2 * c + 1 >= qlim && 2 * c + 1 < qhi) ? p[c].y : 0.f;
        }
      }
      {
        // P^T packed over the first 16 of this group's S^T columns (read)
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) pk[c] = pack_bf16x2(p[c].x, p[c].y);
        tmem_st16(tst, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars[kPtFull]);
      }
      ok = mbar_wait(&bars[kDpTFull], u & 1, abort_s, a.status, kDevErrTimeoutSoftmax);
      // the step's -D entries landed with dO (kDoFull already complete: the
      // MMAs behind kDpTFull waited for it); waiting makes them visible
      if (ok) ok = mbar_wait(&bars[kDoFull0 + sd], phd, abort_s, a.status, kDevErrTimeoutSoftmax);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t dr[32], pd[16];
      tmem_ld32(tdp, dr);
      tmem_ld_wait();
      tmem_reg_fence(dr);
      // dS^T = P^T * (dP^T - D)
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 d4 = lds128(dv_s + c4 * 16);  // -D of 4 queries
        const float2 ds0 =
            __fmul2_rn(p[2 * c4], __fadd2_rn(u2f2(dr[4 * c4], dr[4 * c4 + 1]), make_float2(d4.x, d4.y)));
        const float2 ds1 = __fmul2_rn(
            p[2 * c4 + 1], __fadd2_rn(u2f2(dr[4 * c4 + 2], dr[4 * c4 + 3]), make_float2(d4.z, d4.w)));
        pd[2 * c4] = pack_bf16x2(ds0.x, ds0.y);
        pd[2 * c4 + 1] = pack_bf16x2(ds1.x, ds1.y);
      }
      // dS^T packed over the first 16 of this group's dP^T columns (read)
      tmem_st16(tdp, pd);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars[kDsFull]);
      if (++sq == SQ) sq = 0, phq ^= 1u;
      if (++sd == SD) sd = 0, phd ^= 1u;
      if (++qt == nq_real) qt = tile;  // real tiles: query tiles tile..nq_real-1
    }
    // ------------------------------------------------------------ epilogue --
    // warpgroups 0 and 1 write the two halves of dV; 2 and 3 take the RoPE
    // pairs [w2*D/4, (w2+1)*D/4) of dK with their partners D/2 further on
    if (ok) {
      ok = mbar_wait(&bars[kAccDone], 0, abort_s, a.status, kDevErrTimeoutEpilogue);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      constexpr int HW = D / 2, QP = D / 4;
      if (wg < 2) {
        float x[HW];
#pragma unroll
        for (int c = 0; c < HW / 16; ++c) {
          uint32_t rr[16];
          tmem_ld16(tDV + lane_off + wg * HW + c * 16, rr);
          tmem_ld_wait();
          tmem_reg_fence16(rr);
#pragma unroll
          for (int e = 0; e < 16; ++e) x[c * 16 + e] = __uint_as_float(rr[e]);
        }
        if (key_ok) {
          if (cart)
            write_cart_row(a.dvc + (static_cast<long long>(j) * a.Hkv + g) * D + wg * HW, x, HW,
                           row_frozen(a, j), a.accumulate);
          else
            store_row_out(a.dv,
                          ((static_cast<long long>(seq_rows(cu, a.total, a.n, b_real).g0) + j) *
                               a.Hkv + g) * D + wg * HW,
                          x, HW, a.out_f32 != 0);
        }
      } else {
        const int w2 = wg - 2;
        float lo[QP], hi[QP];
#pragma unroll
        for (int c = 0; c < QP / 16; ++c) {
          uint32_t rr[16];
          tmem_ld16(tDK + lane_off + w2 * QP + c * 16, rr);
          tmem_ld_wait();
          tmem_reg_fence16(rr);
#pragma unroll
          for (int e = 0; e < 16; ++e) lo[c * 16 + e] = __uint_as_float(rr[e]) * a.scale;
          tmem_ld16(tDK + lane_off + D / 2 + w2 * QP + c * 16, rr);
          tmem_ld_wait();
          tmem_reg_fence16(rr);
#pragma unroll
          for (int e = 0; e < 16; ++e) hi[c * 16 + e] = __uint_as_float(rr[e]) * a.scale;
        }
        if (key_ok) {
          if (cart) {
            float* dst = a.dkc + (static_cast<long long>(j) * a.Hkv + g) * D;
            const bool frozen = row_frozen(a, j);
            write_cart_row(dst + w2 * QP, lo, QP, frozen, a.accumulate);
            write_cart_row(dst + D / 2 + w2 * QP, hi, QP, frozen, a.accumulate);
          } else {
            // inverse rotation at position p + j; (cos, sin) computed here:
            // one row of table per thread would be gathered uncoalesced
#pragma unroll
            for (int e = 0; e < QP; ++e) {
              const float2 cs = rope_cs_turns_fast(a.turns[w2 * QP + e], a.p + j);
              const float x0 = lo[e], x1 = hi[e];
              lo[e] = x0 * cs.x + x1 * cs.y;
              hi[e] = x1 * cs.x - x0 * cs.y;
            }
            const long long off =
                ((static_cast<long long>(seq_rows(cu, a.total, a.n, b_real).g0) + j) * a.Hkv +
                 g) * D;
            store_row_out(a.dk, off + w2 * QP, lo, QP, a.out_f32 != 0);
            store_row_out(a.dk, off + D / 2 + w2 * QP, hi, QP, a.out_f32 != 0);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 17) tmem_dealloc(tmem, 512);
}

// ================================================================ dQ ======
// Persistent: one CTA per SM takes work items -- 128-row query tiles of one
// (head, sequence), heaviest first -- from a counter that the prep launch
// zeroes; the producer publishes each item in a two-slot shared-memory ring.
// Q and dO of an item are resident in shared memory; the next item's Q loads
// once the current item's last S MMA has read Q, its dO once the last dP MMA
// has read dO.  Keys stream in 128-row steps (every MMA has N = 128).
// TMEM: S double buffered at x*128 (x = step & 1, steps counted over all
// items), dP at 256, dQ at 384.  Both warpgroups work on every step,
// warpgroup w on keys [64w, 64w + 64) (thread = query row = TMEM lane).  A
// warpgroup reads its S and dP columns, releases dP at once (so dP of the
// next step can be computed while it works), then overwrites the first 32 of
// its 64 S columns with dS = P (dP - D) packed as bf16 pairs; dQ += dS K
// reads dS from TMEM as its A operand (K step k of 16 keys at column
// (k/4)*64 + (k%4)*8), K entering as an MN-major operand.  MMA order per
// step t:
//   S(t+1), dP(t+1) [after dP(t) is released], dQ(t) [after dS(t)].
// K has a 3-stage ring (read by S and dQ), V a 2-stage ring (read by dP);
// both run on across items.  The epilogue rotates dQ back and stores each
// thread's row straight from registers (no staging, so the next item's Q and
// dO are not held up); the next item's first dQ MMA, which overwrites the
// accumulator, follows that item's first dS, which the softmax warps write
// only after their epilogue has read dQ out.
// Threads: warps 0-7 the two warpgroups, warp 8 TMA, warp 9 MMA.
constexpr int kDqThreads = 320;
constexpr int kDqKStages = 3;
constexpr int kDqVStages = 2;

template <int D>
struct DqSmem {
  static constexpr int kTileBytes = kTile * D * 2;  // one 128-row bf16 tile
  static constexpr int kQ = 0;
  static constexpr int kdO = kQ + kTileBytes;
  static constexpr int kK = kdO + kTileBytes;                 // K ring
  static constexpr int kV = kK + kDqKStages * kTileBytes;     // V ring
  static constexpr int kBar = kV + kDqVStages * kTileBytes;   // barriers, TMEM slot, abort word
  static constexpr int kItems = kBar + 256;                   // two item slots
  static constexpr int kBytes = kItems + 128;
  static constexpr int kAlloc = kBytes;  // dynamic shared memory starts 1024-aligned
};

enum DqBar {
  kQFull = 0,
  kQEmpty,                           // the item's last S MMA has read Q
  kdOFull,
  kdOEmpty,                          // the item's last dP MMA has read dO
  kKFull0,
  kKEmpty0 = kKFull0 + kDqKStages,
  kVFull0 = kKEmpty0 + kDqKStages,
  kVEmpty0 = kVFull0 + kDqVStages,
  kSdFull0 = kVEmpty0 + kDqVStages,  // S of buffer x computed
  kDpFull = kSdFull0 + 2,            // dP computed
  kDpFree,                           // both groups read dP (256 arrivals)
  kDsdFull0,                         // dS of buffer x written (256 arrivals)
  kDqDone = kDsdFull0 + 2,           // the item's last dQ MMA has completed
  kDqDrain,
  kDqItemFull0,                      // the producer published the next item in slot s
  kDqItemEmpty0 = kDqItemFull0 + 2,  // the MMA warp and the 8 softmax warps are done with slot s
  kDqBars = kDqItemEmpty0 + 2
};
static_assert(kDqBars * 8 + 8 <= 256, "dQ barrier area");

// One dQ work item: query tile qt of (head h, sequence b) and its key tiles
// -- cartridge tiles [ct_lo, ct_lo + n_ct), then real tiles [rt_lo, rt_hi).
struct DqItem {
  int h, b, q0, kvh, seq_len, n_ct, ct_lo, rt_lo, T;
  SeqRows sr;
};

// As published in a shared-memory slot (w < 0: no more items); the roles
// read each field where they use it.
struct DqSlot {
  int w, h, b, q0, seq_len, row0, blk, g0, n_ct, ct_lo, rt_lo, T, pad[4];
};
static_assert(sizeof(DqSlot) == 64, "dQ item slot");

// Item w: tiles are numbered heaviest first (the query tile index falls as w
// grows: later tiles see more real keys).
__device__ __forceinline__ DqItem dq_item(const BwdParams& a, int w, const int* cu, int window) {
  DqItem I;
  const int hb = a.Hq * a.B;
  const int z = w / hb, rem = w % hb;
  I.h = rem % a.Hq;
  I.b = rem / a.Hq;
  const int qt = a.n_qtiles - 1 - z;
  I.sr = seq_rows(cu, a.total, a.n, I.b);
  I.seq_len = cu ? I.sr.len : a.n;
  I.kvh = I.h / a.G;
  I.q0 = qt * kTile;
  I.n_ct = I.ct_lo = I.rt_lo = I.T = 0;
  if (I.q0 >= I.seq_len) return I;  // a segment shorter than the longest
  const int n_ct_all = (a.p + kTile - 1) / kTile;
  const int last_q = min(I.q0 + kTile, I.seq_len) - 1;  // last real query of the tile
  const int rt_hi = last_q / kTile + 1;                  // real key steps up to the diagonal
  if (window > 0) {
    // the first key any row of the tile sees: position p + q0 - window + 1
    const int lo = a.p + I.q0 - window + 1;
    if (lo > 0) {
      I.ct_lo = min(lo / kTile, n_ct_all);
      I.rt_lo = lo > a.p ? (lo - a.p) / kTile : 0;
    }
  }
  I.n_ct = n_ct_all - I.ct_lo;
  I.T = I.n_ct + rt_hi - I.rt_lo;
  return I;
}

// The fixed-layout instance takes a static schedule of its items (WorkPlan);
// the packed / windowed one takes items from the counter.
template <bool kGeneral>
using DqPlanOf = WorkPlan<kGeneral ? 1 : kPlanItems>;

template <int D, bool kGeneral>
__global__ void __launch_bounds__(kDqThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mdO,
              const __grid_constant__ CUtensorMap mKc, const __grid_constant__ CUtensorMap mVc,
              const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
              const BwdParams a, const __grid_constant__ DqPlanOf<kGeneral> plan) {
  using L = DqSmem<D>;
  constexpr int SK = kDqKStages, SV = kDqVStages;
  extern __shared__ __align__(1024) uint8_t dq_smem[];
  uint8_t* smem = dq_smem;
  if (smem_u32(smem) & 1023u) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0 && a.status) atomicOr(a.status, kDevErrSmemLayout);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBar + kDqBars * 8);
  int* abort_flag = reinterpret_cast<int*>(smem + L::kBar + kDqBars * 8 + 4);
  DqSlot* items = reinterpret_cast<DqSlot*>(smem + L::kItems);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int* const cu = kGeneral ? a.cu : nullptr;  // packed segment table
  const int window = kGeneral ? a.window : 0;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(&bars[kQFull], 1);
    mbar_init(&bars[kQEmpty], 1);
    mbar_init(&bars[kdOFull], 1);
    mbar_init(&bars[kdOEmpty], 1);
    for (int s = 0; s < SK; ++s) {
      mbar_init(&bars[kKFull0 + s], 1);
      mbar_init(&bars[kKEmpty0 + s], 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(&bars[kVFull0 + s], 1);
      mbar_init(&bars[kVEmpty0 + s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars[kSdFull0 + x], 1);
      mbar_init(&bars[kDsdFull0 + x], 256);
      mbar_init(&bars[kDqItemFull0 + x], 1);
      mbar_init(&bars[kDqItemEmpty0 + x], 9);  // the MMA warp and the 8 softmax warps
    }
    mbar_init(&bars[kDpFull], 1);
    mbar_init(&bars[kDpFree], 256);
    mbar_init(&bars[kDqDone], 1);
    mbar_init(&bars[kDqDrain], 1);
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
  const uint32_t tS0 = tmem, tDP = tmem + 256, tDQ = tmem + 384;
  const uint32_t abort_s = smem_u32(abort_flag);
  uint8_t* sQ = smem + L::kQ;
  uint8_t* sdO = smem + L::kdO;

  if (warp == 8) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mdO);
      tma_prefetch_desc(&mKc);
      tma_prefetch_desc(&mVc);
      tma_prefetch_desc(&mK);
      tma_prefetch_desc(&mV);
      // the next item: the static plan's if there is one, else the counter's
      auto fetch = [&](int k) -> int {
        if (!kGeneral && plan.n > 0) {
          const int o = plan.off[blockIdx.x] + k;
          return o < plan.off[blockIdx.x + 1] ? static_cast<int>(plan.items[o]) : -1;
        }
        const int w = atomicAdd(a.sched, 1);
        return w < a.n_items ? w : -1;
      };
      int g = 0;   // K / V tiles issued, over all items
      int nq = 0;  // Q / dO loads issued (items with work)
      int k_issued = 0, v_issued = 0;
      bool ok = true;
      int w = fetch(0);
      for (int it = 0; ok; ++it) {
        const int sl = it & 1;
        if (it >= 2) {
          ok = mbar_wait(&bars[kDqItemEmpty0 + sl], ((it >> 1) - 1) & 1, abort_s, a.status,
                         kDevErrTimeoutTma);
          if (!ok) break;
        }
        DqItem I{};
        if (w >= 0) I = dq_item(a, w, cu, window);
        DqSlot& o = items[sl];
        o.w = w;
        o.h = I.h;
        o.b = I.b;
        o.q0 = I.q0;
        o.seq_len = I.seq_len;
        o.row0 = I.sr.row0;
        o.blk = I.sr.blk;
        o.g0 = I.sr.g0;
        o.n_ct = I.n_ct;
        o.ct_lo = I.ct_lo;
        o.rt_lo = I.rt_lo;
        o.T = I.T;
        mbar_arrive(&bars[kDqItemFull0 + sl]);  // (release: the slot is visible to the waiters)
        if (w < 0) break;
        const int w_next = fetch(it + 1);
        if (I.T > 0) {
          // Q and dO of this item once the previous item's last S / dP MMA
          // has read them
          if (nq >= 1) {
            ok = mbar_wait(&bars[kQEmpty], (nq - 1) & 1, abort_s, a.status, kDevErrTimeoutTma);
            if (!ok) break;
          }
          mbar_arrive_expect_tx(&bars[kQFull], L::kTileBytes);
#pragma unroll
          for (int hc = 0; hc < D / 64; ++hc)
            tma_load_4d(sQ + hc * 16384, &mQ, &bars[kQFull], hc * 64, I.h, I.sr.row0 + I.q0,
                        I.sr.blk);
          if (nq >= 1) {
            ok = mbar_wait(&bars[kdOEmpty], (nq - 1) & 1, abort_s, a.status, kDevErrTimeoutTma);
            if (!ok) break;
          }
          mbar_arrive_expect_tx(&bars[kdOFull], L::kTileBytes);
#pragma unroll
          for (int hc = 0; hc < D / 64; ++hc)
            tma_load_4d(sdO + hc * 16384, &mdO, &bars[kdOFull], hc * 64, I.h, I.sr.row0 + I.q0,
                        I.sr.blk);
          ++nq;
          for (int t = 0; t < I.T && ok; ++t, ++g) {
            const bool cart = t < I.n_ct;
            const int row0 =
                cart ? (I.ct_lo + t) * kTile : I.sr.row0 + (I.rt_lo + t - I.n_ct) * kTile;
            const int blk = cart ? 0 : I.sr.blk;
            const int sk = g % SK, sv = g % SV;
            if (g >= SK) {
              ok = mbar_wait(&bars[kKEmpty0 + sk], ((g / SK) - 1) & 1, abort_s, a.status,
                             kDevErrTimeoutTma);
              if (!ok) break;
            }
            uint8_t* sK = smem + L::kK + sk * L::kTileBytes;
            mbar_arrive_expect_tx(&bars[kKFull0 + sk], L::kTileBytes);
#pragma unroll
            for (int hc = 0; hc < D / 64; ++hc)
              tma_load_4d(sK + hc * 16384, cart ? &mKc : &mK, &bars[kKFull0 + sk], hc * 64, I.kvh,
                          row0, blk);
            k_issued = g + 1;
            if (g >= SV) {
              ok = mbar_wait(&bars[kVEmpty0 + sv], ((g / SV) - 1) & 1, abort_s, a.status,
                             kDevErrTimeoutTma);
              if (!ok) break;
            }
            uint8_t* sV = smem + L::kV + sv * L::kTileBytes;
            mbar_arrive_expect_tx(&bars[kVFull0 + sv], L::kTileBytes);
#pragma unroll
            for (int hc = 0; hc < D / 64; ++hc)
              tma_load_4d(sV + hc * 16384, cart ? &mVc : &mV, &bars[kVFull0 + sv], hc * 64, I.kvh,
                          row0, blk);
            v_issued = g + 1;
          }
        }
        w = w_next;
      }
      if (!ok) {
        // Give the copies still in flight (the last Q and dO loads, the last
        // K and V tiles) a bounded chance to land before the CTA releases
        // its shared memory.
        if (nq > 0) {
          mbar_wait(&bars[kQFull], (nq - 1) & 1, 0u, nullptr, 0);
          mbar_wait(&bars[kdOFull], (nq - 1) & 1, 0u, nullptr, 0);
        }
        for (int t = max(k_issued - SK, 0); t < k_issued; ++t)
          mbar_wait(&bars[kKFull0 + t % SK], (t / SK) & 1, 0u, nullptr, 0);
        for (int t = max(v_issued - SV, 0); t < v_issued; ++t)
          mbar_wait(&bars[kVFull0 + t % SV], (t / SV) & 1, 0u, nullptr, 0);
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
    const uint32_t idDQ = idesc_bf16(128, D, false, true);
    const uint64_t dQd = sdesc_sw128(smem_u32(sQ), 16u, 1024u);
    const uint64_t dOd = sdesc_sw128(smem_u32(sdO), 16u, 1024u);
    const uint64_t dKk0 = sdesc_sw128(smem_u32(smem + L::kK), 16u, 1024u);      // K-major
    const uint64_t dKm0 = sdesc_sw128(smem_u32(smem + L::kK), 16384u, 1024u);   // MN-major
    const uint64_t dVk0 = sdesc_sw128(smem_u32(smem + L::kV), 16u, 1024u);
    // C (f32, TMEM) = A (128 rows) * B^T (128 rows), both K-major over d
    auto issue_nt = [&](uint32_t c, uint64_t da, uint64_t db) {
      umma_bf16_ss_w(c, da, db, idS, 0u);
#pragma unroll
      for (int k = 1; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
        umma_bf16_ss_w(c, desc_add(da, off), desc_add(db, off), idS, 1u);
      }
    };
    int g = 0;   // K / V tiles consumed, over all items
    int gs = 0;  // steps, over all items (S buffer, dP and dS phases)
    int nq = 0;  // Q / dO loads consumed
    bool ok = true;
    for (int it = 0; ok; ++it) {
      ok = wait(&bars[kDqItemFull0 + (it & 1)], (it >> 1) & 1);
      if (!ok) break;
      const DqSlot& sI = items[it & 1];
      const int w = vld(sI.w), T = vld(sI.T);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kDqItemEmpty0 + (it & 1)]);  // read all it needs
      if (w < 0) break;
      if (T == 0) continue;
      // first step: S into buffer gs & 1, dP once dP of the previous step
      // (the previous item's last) has been read
      ok = wait(&bars[kQFull], nq & 1) && wait(&bars[kKFull0 + g % SK], (g / SK) & 1);
      if (ok) {
        tc_fence_after();
        issue_nt(tS0 + (gs & 1) * 128, dQd, desc_add(dKk0, (g % SK) * L::kTileBytes));
        umma_commit_w(&bars[kSdFull0 + (gs & 1)]);
        if (T == 1) umma_commit_w(&bars[kQEmpty]);
        ok = wait(&bars[kdOFull], nq & 1) && (gs == 0 || wait(&bars[kDpFree], (gs - 1) & 1)) &&
             wait(&bars[kVFull0 + g % SV], (g / SV) & 1);
      }
      if (ok) {
        tc_fence_after();
        issue_nt(tDP, dOd, desc_add(dVk0, (g % SV) * L::kTileBytes));
        umma_commit_w(&bars[kDpFull]);
        umma_commit_w(&bars[kVEmpty0 + g % SV]);
        if (T == 1) umma_commit_w(&bars[kdOEmpty]);
      }
      for (int t = 0; t < T && ok; ++t) {
        const int G = gs + t, x = G & 1;
        if (t + 1 < T) {
          const int gk = g + t + 1, sk = gk % SK, sv = gk % SV;
          ok = wait(&bars[kKFull0 + sk], (gk / SK) & 1);
          if (!ok) break;
          tc_fence_after();
          // buffer x^1 last held dS(G-1), read by dQ(G-1) issued earlier
          // (one CTA's MMAs run in issue order)
          issue_nt(tS0 + (x ^ 1) * 128, dQd, desc_add(dKk0, sk * L::kTileBytes));
          umma_commit_w(&bars[kSdFull0 + (x ^ 1)]);
          if (t + 1 == T - 1) umma_commit_w(&bars[kQEmpty]);
          ok = wait(&bars[kDpFree], G & 1) && wait(&bars[kVFull0 + sv], (gk / SV) & 1);
          if (!ok) break;
          tc_fence_after();
          issue_nt(tDP, dOd, desc_add(dVk0, sv * L::kTileBytes));
          umma_commit_w(&bars[kDpFull]);
          umma_commit_w(&bars[kVEmpty0 + sv]);
          if (t + 1 == T - 1) umma_commit_w(&bars[kdOEmpty]);
        }
        ok = wait(&bars[kDsdFull0 + x], (G >> 1) & 1);
        if (!ok) break;
        tc_fence_after();
        const int sk = (g + t) % SK;
        const uint64_t dkm = desc_add(dKm0, sk * L::kTileBytes);
        const uint32_t ds = tS0 + x * 128;
        umma_bf16_ts_w(tDQ, ds, dkm, idDQ, t > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 1; k < kTile / 16; ++k)
          umma_bf16_ts_w(tDQ, ds + (k >> 2) * 64 + (k & 3) * 8, desc_add(dkm, k * 2048), idDQ, 1u);
        umma_commit_w(&bars[kKEmpty0 + sk]);
      }
      if (ok) umma_commit_w(&bars[kDqDone]);
      g += T;
      gs += T;
      ++nq;
    }
    // Drain: every MMA issued above completes before the CTA tears down.
    umma_commit_w(&bars[kDqDrain]);
    mbar_wait(&bars[kDqDrain], 0, 0u, nullptr, 0);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ dS / dQ --
    const int wg = warp >> 2;
    const int row = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
    int gs = 0;  // steps, over all items
    int nd = 0;  // items finished
    bool ok = true;
    for (int it = 0; ok; ++it) {
      ok = mbar_wait(&bars[kDqItemFull0 + (it & 1)], (it >> 1) & 1, abort_s, a.status,
                     kDevErrTimeoutSoftmax);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      // the slot is released once the item's epilogue is done with it
      const DqSlot& sI = items[it & 1];
      if (vld(sI.w) < 0) break;
      const int T = vld(sI.T);
      if (T == 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kDqItemEmpty0 + (it & 1)]);
        continue;
      }
      const int h = vld(sI.h), b = vld(sI.b);
      const int i = vld(sI.q0) + row;
      const int seq_len = vld(sI.seq_len);
      const int n_ct = vld(sI.n_ct), ct_lo = vld(sI.ct_lo), rt_lo = vld(sI.rt_lo);
      // padded vectors: rows past n read -lse2 = -inf (P = 0) and -D = 0
      const long long vidx = (static_cast<long long>(b) * a.Hq + h) * a.npad + i;
      const float nl = __ldg(a.nlse2 + vidx), ndv = __ldg(a.nDvec + vidx);
      const float2 nl2 = make_float2(nl, nl), nd2 = make_float2(ndv, ndv);
      const int i_cap = min(i, seq_len - 1);
      for (int t = 0; t < T && ok; ++t) {
        const int G = gs + t, x = G & 1;
        ok = mbar_wait(&bars[kSdFull0 + x], (G >> 1) & 1, abort_s, a.status,
                       kDevErrTimeoutSoftmax) &&
             mbar_wait(&bars[kDpFull], G & 1, abort_s, a.status, kDevErrTimeoutSoftmax);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        // visible keys of this group's 64 (leading columns)
        // (key positions of this group's 64 columns start at kpos0)
        const int kpos0 =
            (t < n_ct ? (ct_lo + t) * kTile : a.p + (rt_lo + t - n_ct) * kTile) + wg * 64;
        int valid = t < n_ct ? a.p - kpos0 : i_cap - (kpos0 - a.p) + 1;
        valid = max(0, min(valid, 64));
        // ... and the first one under the window
        const int first = window > 0 ? max(0, min(a.p + i - window + 1 - kpos0, 64)) : 0;
        const uint32_t ts = tS0 + x * 128 + wg * 64 + lane_off;
        const uint32_t tdp = tDP + wg * 64 + lane_off;
        uint32_t sa[32], sb[32], da[32], db[32];
        tmem_ld32(ts, sa);
        tmem_ld32(ts + 32, sb);
        tmem_ld32(tdp, da);
        tmem_ld32(tdp + 32, db);
        tmem_ld_wait();
        tmem_reg_fence(sa);
        tmem_reg_fence(sb);
        tmem_reg_fence(da);
        tmem_reg_fence(db);
        tc_fence_before();
        mbar_arrive(&bars[kDpFree]);
        uint32_t pk[32];
        auto compute = [&](auto masked) {
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            // two keys per packed two-lane op: P = 2^(S*scale*log2(e) - lse2),
            // dS = P * (dP - D)
            const float2 sv = c < 32 ? u2f2(sa[c], sa[c + 1]) : u2f2(sb[c - 32], sb[c - 31]);
            const float2 dv = c < 32 ? u2f2(da[c], da[c + 1]) : u2f2(db[c - 32], db[c - 31]);
            const float2 xe = __ffma2_rn(sv, sc2, nl2);
            float2 pe = make_float2(exp2_approx(xe.x), exp2_approx(xe.y));
            if (decltype(masked)::value) {
              pe.x = (c < valid && c >= first) ? pe.x : 0.f;
              pe.y = (c + 1 < valid && c + 1 >= first) ? pe.y : 0.f;
            }
            const float2 ds = __fmul2_rn(pe, __fadd2_rn(dv, nd2));
            pk[c / 2] = pack_bf16x2(ds.x, ds.y);
          }
        };
        if (__any_sync(0xffffffffu, valid < 64 || first > 0))
          compute(std::true_type{});
        else
          compute(std::false_type{});
        // dS over the first 32 of this group's S columns (already read)
        tmem_st32(ts, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars[kDsdFull0 + x]);
      }
      gs += T;
      // ---------------------------------------------------------- epilogue --
      if (ok) {
        ok = mbar_wait(&bars[kDqDone], nd & 1, abort_s, a.status, kDevErrTimeoutEpilogue);
        ok = __all_sync(0xffffffffu, ok);
      }
      ++nd;
      if (!ok) break;
      tc_fence_after();
      // warpgroup wg finishes the rotation pairs j in [wg*D/4, wg*D/4 + D/4)
      // and their partners j + D/2
      constexpr int Q = D / 4;
      float lo[Q], hi[Q];
      const uint32_t base = tDQ + lane_off + wg * Q;
#pragma unroll
      for (int c = 0; c < Q / 16; ++c) {
        // columns [wg*Q + 16c, +16) and their partners D/2 further on
        uint32_t r[16];
        tmem_ld16(base + c * 16, r);
        tmem_ld_wait();
        tmem_reg_fence16(r);
#pragma unroll
        for (int e = 0; e < 16; ++e) lo[c * 16 + e] = __uint_as_float(r[e]) * a.scale;
        tmem_ld16(base + D / 2 + c * 16, r);
        tmem_ld_wait();
        tmem_reg_fence16(r);
#pragma unroll
        for (int e = 0; e < 16; ++e) hi[c * 16 + e] = __uint_as_float(r[e]) * a.scale;
      }
      if (i < seq_len) {
        // inverse rotation at position p + i; (cos, sin) computed here: one
        // row of table per thread would be gathered uncoalesced
#pragma unroll
        for (int e = 0; e < Q; ++e) {
          const float2 cs = rope_cs_turns_fast(a.turns[wg * Q + e], a.p + i);
          const float x0 = lo[e], x1 = hi[e];
          lo[e] = x0 * cs.x + x1 * cs.y;
          hi[e] = x1 * cs.x - x0 * cs.y;
        }
        // this thread's row, straight from registers (whole 16-byte pieces)
        const long long off = ((static_cast<long long>(vld(sI.g0)) + i) * a.Hq + h) * D;
        store_row_out(a.dq, off + wg * Q, lo, Q, a.out_f32 != 0);
        store_row_out(a.dq, off + D / 2 + wg * Q, hi, Q, a.out_f32 != 0);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kDqItemEmpty0 + (it & 1)]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, 512);
}

// The static schedule of the fixed-layout dQ items (numbering of dq_item):
// an item costs its key steps plus 2 for its start and end.  Cached per
// geometry.
const std::vector<uint16_t>& dq_plan(const BwdParams& p, int grid, std::vector<uint16_t>* off_out) {
  constexpr double kItemCost = 2.0;
  struct Plan {
    std::vector<uint16_t> items, off;
  };
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int, int>, Plan> cache;
  std::lock_guard<std::mutex> lk(mu);
  const auto key = std::make_tuple(p.Hq * p.B, p.n_qtiles, p.n_ct, p.n, grid);
  auto it = cache.find(key);
  if (it == cache.end()) {
    const int hb = p.Hq * p.B, n = hb * p.n_qtiles;
    std::vector<double> cost(n);
    for (int w = 0; w < n; ++w) {
      const int qt = p.n_qtiles - 1 - w / hb;
      const int last_q = std::min(qt * kTile + kTile, p.n) - 1;
      cost[w] = p.n_ct + last_q / kTile + 1 + kItemCost;
    }
    Plan pl;
    build_work_plan(cost, grid, &pl.items, &pl.off);
    it = cache.emplace(key, std::move(pl)).first;
  }
  *off_out = it->second.off;
  return it->second.items;
}

template <int D>
cudaError_t launch_bwd_d(const BwdLaunch& l, cudaStream_t st_dkdv, cudaStream_t st_dq) {
  static_assert(DkdvSmem<D>::kAlloc <= 232448, "dkdv shared memory budget");
  static_assert(DqSmem<D>::kAlloc <= 232448, "dq shared memory budget");
  BwdParams p{};
  p.B = l.B;
  p.n = l.n;
  p.Hq = l.Hq;
  p.Hkv = l.Hkv;
  p.G = l.Hq / l.Hkv;
  p.p = l.p;
  p.frozen_prefix = l.frozen_prefix;
  p.n_frozen = l.n_frozen;
  for (int i = 0; i < l.n_frozen; ++i) p.frozen_rows[i] = l.frozen_rows[i];
  p.n_ct = (l.p + kTile - 1) / kTile;
  p.n_rt = (l.n + kTile - 1) / kTile;
  p.n_qtiles = p.n_rt;
  p.scale = l.scale;
  p.scale_log2 = l.scale * kLog2e;
  p.nlse2 = l.nlse2;
  p.nDvec = l.nDvec;
  p.npad = l.npad;
  p.dq = l.dq;
  p.dk = l.dk;
  p.dv = l.dv;
  p.out_f32 = l.out_f32 ? 1 : 0;
  p.dkc = l.dkc;
  p.dvc = l.dvc;
  p.accumulate = l.accumulate;
  p.table = l.table;
  p.cu = l.cu;
  p.total = l.total;
  p.window = l.window;
  for (int c = 0; c < D / 2; ++c) p.turns[c] = l.freqs->turns[c];
  p.status = device_status_ptr();
  const bool general = l.cu != nullptr || l.window > 0;
  cudaError_t e = general ? set_smem_once<dkdv_kernel<D, true>>(DkdvSmem<D>::kAlloc)
                         : set_smem_once<dkdv_kernel<D, false>>(DkdvSmem<D>::kAlloc);
  if (e != cudaSuccess) return e;
  e = general ? set_smem_once<dq_kernel<D, true>>(DqSmem<D>::kAlloc)
             : set_smem_once<dq_kernel<D, false>>(DqSmem<D>::kAlloc);
  if (e != cudaSuccess) return e;
  const int n_blocks = p.n_ct * p.Hkv + p.n_rt * p.Hkv * p.B;
  if (n_blocks > 0) {
    TraceScope tr("bwd_dkdv", st_dkdv);
    auto* kern = general ? dkdv_kernel<D, true> : dkdv_kernel<D, false>;
    kern<<<n_blocks, kDkdvThreads, DkdvSmem<D>::kAlloc, st_dkdv>>>(*l.mQ, *l.mdO, *l.mKc, *l.mVc,
                                                                   *l.mK, *l.mV, p);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  TraceScope tr("bwd_dq", st_dq);
  // persistent: one CTA per SM, none idle from the start
  p.n_items = p.Hq * p.B * p.n_qtiles;
  p.sched = l.sched;
  const int nsm = sm_count();
  if (nsm < 1 || !l.sched) return cudaErrorInvalidValue;
  const int grid = p.n_items < nsm ? p.n_items : nsm;
  if (general) {
    DqPlanOf<true> none{};
    dq_kernel<D, true><<<grid, kDqThreads, DqSmem<D>::kAlloc, st_dq>>>(
        *l.mQ, *l.mdO, *l.mKc, *l.mVc, *l.mK, *l.mV, p, none);
    return cudaGetLastError();
  }
  static thread_local DqPlanOf<false> plan;
  plan.n = 0;
  if (p.n_items <= kPlanItems && grid <= kPlanCtas) {
    std::vector<uint16_t> off;
    const std::vector<uint16_t>& items = dq_plan(p, grid, &off);
    plan.n = static_cast<int>(items.size());
    std::memcpy(plan.off, off.data(), off.size() * sizeof(uint16_t));
    std::memcpy(plan.items, items.data(), items.size() * sizeof(uint16_t));
  }
  dq_kernel<D, false><<<grid, kDqThreads, DqSmem<D>::kAlloc, st_dq>>>(
      *l.mQ, *l.mdO, *l.mKc, *l.mVc, *l.mK, *l.mV, p, plan);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdLaunch& l, cudaStream_t st_dkdv, cudaStream_t st_dq) {
  if (l.d == 128) return launch_bwd_d<128>(l, st_dkdv, st_dq);
  if (l.d == 64) return launch_bwd_d<64>(l, st_dkdv, st_dq);
  return cudaErrorInvalidValue;
}

}  // namespace cart
