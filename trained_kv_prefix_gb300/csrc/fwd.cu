// fwd.cu -- tcgen05 forward of cartridge attention (sm_103a).
//
// One CTA owns a 128-row query tile of one (sequence, head) and walks the key
// tiles of concat(cartridge rows, real tokens): first every cartridge tile
// (all visible), then the real-token tiles up to the diagonal (end-aligned
// causal mask: key j of the real part is visible from query i iff j <= i).
// (Cartridges guide, "Semantics", attention bullet.)
//
// Roles (320 threads):
//   warps 0-7  two softmax warpgroups.  Thread t of a group owns query row t
//              (TMEM lane t); warpgroup w handles key columns [64w, 64w+64)
//              of every 128-key tile.  The row maximum is exchanged between
//              the two groups through shared memory; each keeps its own
//              partial row sum and rescales its own half of O in TMEM when
//              the maximum grows by more than 2^8 (lazy rescaling, log2
//              domain).  P (bf16 pairs) is written back into TMEM over the
//              group's own S columns.
//   warp 8     TMA producer: Q tile once, then K/V tiles into a 2-stage ring.
//   warp 9     MMA issuer (one thread): S = Q K^T into a double-buffered S
//              (columns 0-127 / 128-255) and O += P V with P read from TMEM
//              as the A operand (columns 256.. hold O).
//
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.cuh"
#include "ptx.cuh"

namespace cart {
namespace {

struct FwdParams {
  int n_rows, Hq_map, G, p, n_real, cart_tiles_per_split, n_qtiles;
  float scale_log2;
  void* out;
  float* lse;
  int out_f32;
  int decode;
  uint32_t* status;
};

constexpr int kFwdThreads = 320;

// NS = K/V stages in shared memory: 2 for training; 1 in decode mode, where
// the cartridge pass runs next to the private pass and leaves it room.
template <int D, int NS>
struct FwdSmem {
  static constexpr int kTileBytes = kTile * D * 2;      // one Q, K or V tile (bf16)
  static constexpr int kStages = NS;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  // row maxima [2 tile buffers][2 groups][128] then row sums [2 groups][128], f32
  static constexpr int kRed = kV + kStages * kTileBytes;
  static constexpr int kBar = kRed + 3 * 256 * 4;
  static constexpr int kBytes = kBar + 128;             // barriers + TMEM slot
  static constexpr int kAlloc = kBytes + 1024;          // slack for 1024-B alignment
};

// kRedFull0/1: both softmax groups published a tile's row maxima; kLFull:
// both published their row sums.  (mbarriers rather than a named barrier, so
// that every wait stays bounded.)
enum FwdBar { kQFull = 0, kKVFull0, kKVFull1, kKVEmpty0, kKVEmpty1, kSFull0, kSFull1, kPFull0,
              kPFull1, kODone, kRedFull0, kRedFull1, kLFull, kDrain, kNumBars };

template <int D, int NS>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mKc,
               const __grid_constant__ CUtensorMap mVc, const __grid_constant__ CUtensorMap mK,
               const __grid_constant__ CUtensorMap mV, const FwdParams a) {
  using L = FwdSmem<D, NS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBar + kNumBars * 8);
  float* red = reinterpret_cast<float*>(smem + L::kRed);
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item ----
  int head, qb, qt, kvh, split;
  if (!a.decode) {
    head = blockIdx.x;
    qb = blockIdx.y;
    qt = a.n_qtiles - 1 - static_cast<int>(blockIdx.z);  // heaviest tiles first
    kvh = head / a.G;
    split = 0;
  } else {
    head = blockIdx.x;
    qb = 0;
    qt = blockIdx.y;
    kvh = head;
    split = blockIdx.z;
  }
  const int q0 = qt * kTile;
  const int n_ct_all = (a.p + kTile - 1) / kTile;
  int ct_lo = 0, ct_hi = n_ct_all, n_rt = 0;
  if (a.decode) {
    ct_lo = split * a.cart_tiles_per_split;
    ct_hi = min(ct_lo + a.cart_tiles_per_split, n_ct_all);
  } else {
    n_rt = min(qt + 1, (a.n_real + kTile - 1) / kTile);
  }
  const int n_ct = max(ct_hi - ct_lo, 0);
  const int T = n_ct + n_rt;

  if (threadIdx.x == 0) {
    // decode mode: let the dependent private pass start right away (it only
    // waits for this grid where it reads the cartridge partials)
    if (a.decode) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    abort_flag = 0;
    mbar_init(&bars[kQFull], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kKVFull0 + s], 1);
      mbar_init(&bars[kKVEmpty0 + s], 1);
      mbar_init(&bars[kSFull0 + s], 1);
      mbar_init(&bars[kPFull0 + s], 256);
      mbar_init(&bars[kRedFull0 + s], 256);
    }
    mbar_init(&bars[kLFull], 256);
    mbar_init(&bars[kODone], 1);
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
  const uint32_t tS0 = tmem;        // S buffers at columns 0 and 128
  const uint32_t tO = tmem + 256;
  volatile int* abort_p = &abort_flag;
  uint8_t* sQ = smem + L::kQ;

  if (warp == 8) {
    // ------------------------------------------------------------ producer --
    if (lane == 0 && T > 0) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mKc);
      tma_prefetch_desc(&mVc);
      tma_prefetch_desc(&mK);
      tma_prefetch_desc(&mV);
      mbar_arrive_expect_tx(&bars[kQFull], L::kTileBytes);
#pragma unroll
      for (int h = 0; h < D / 64; ++h)
        tma_load_4d(sQ + h * 16384, &mQ, &bars[kQFull], h * 64, head, q0, qb);
      int issued = 0;
      bool ok = true;
      for (int t = 0; t < T; ++t) {
        const int s = t % NS;
        if (t >= NS) {
          ok = mbar_wait(&bars[kKVEmpty0 + s], ((t / NS) - 1) & 1, abort_p, a.status,
                         kDevErrTimeoutTma);
          if (!ok) break;
        }
        uint8_t* sK = smem + L::kK + s * L::kTileBytes;
        uint8_t* sV = smem + L::kV + s * L::kTileBytes;
        mbar_arrive_expect_tx(&bars[kKVFull0 + s], 2 * L::kTileBytes);
        if (t < n_ct) {
          const int row0 = (ct_lo + t) * kTile;
#pragma unroll
          for (int h = 0; h < D / 64; ++h) {
            tma_load_4d(sK + h * 16384, &mKc, &bars[kKVFull0 + s], h * 64, kvh, row0, 0);
            tma_load_4d(sV + h * 16384, &mVc, &bars[kKVFull0 + s], h * 64, kvh, row0, 0);
          }
        } else {
          const int row0 = (t - n_ct) * kTile;
#pragma unroll
          for (int h = 0; h < D / 64; ++h) {
            tma_load_4d(sK + h * 16384, &mK, &bars[kKVFull0 + s], h * 64, kvh, row0, qb);
            tma_load_4d(sV + h * 16384, &mV, &bars[kKVFull0 + s], h * 64, kvh, row0, qb);
          }
        }
        issued = t + 1;
      }
      if (!ok) {
        // Give the copies already in flight a bounded chance to land before
        // the CTA releases its shared memory.
        int dummy = 0;
        mbar_wait(&bars[kQFull], 0, &dummy, nullptr, 0);
        for (int t = max(issued - NS, 0); t < issued; ++t)
          mbar_wait(&bars[kKVFull0 + t % NS], (t / NS) & 1, &dummy, nullptr, 0);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ----------------------------------------------------------------- MMA --
    if (lane == 0 && T > 0) {
      const uint32_t idS = idesc_bf16(128, 128, false, false);
      const uint32_t idPV = idesc_bf16(128, D, false, true);
      // Base descriptors, computed once; each MMA adds a compile-time offset.
      const uint64_t dQ0 = sdesc_sw128(smem_u32(sQ), 16u, 1024u);
      const uint64_t dKs0 = sdesc_sw128(smem_u32(smem + L::kK), 16u, 1024u);
      const uint64_t dVs0 = sdesc_sw128(smem_u32(smem + L::kV), 16384u, 1024u);
      const uint64_t dKs1 = desc_add(dKs0, L::kTileBytes);
      const uint64_t dVs1 = desc_add(dVs0, L::kTileBytes);
      bool ok = mbar_wait(&bars[kQFull], 0, abort_p, a.status, kDevErrTimeoutMma);
      // O += P V for tile t: P from TMEM buffer t&1 (K step k of 16 keys at
      // column (k/4)*64 + (k%4)*8: warpgroup w packed keys 64w.. at 64w),
      // V MN-major (16 rows = 2048 B per K step).
      auto issue_pv = [&](int t) {
        const int sp = t % NS;           // smem stage of V
        const uint64_t dv = sp ? dVs1 : dVs0;
        const uint32_t tp = tS0 + (t & 1) * 128;  // TMEM buffer holding P
        umma_bf16_ts(tO, tp, dv, idPV, t > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 1; k < kTile / 16; ++k)
          umma_bf16_ts(tO, tp + (k >> 2) * 64 + (k & 3) * 8, desc_add(dv, k * 2048), idPV, 1u);
        umma_commit(&bars[kODone]);
        umma_commit(&bars[kKVEmpty0 + sp]);
      };
      for (int t = 0; t < T && ok; ++t) {
        const int ks = t % NS, s = t & 1;
        ok = mbar_wait(&bars[kKVFull0 + ks], (t / NS) & 1, abort_p, a.status, kDevErrTimeoutMma);
        if (!ok) break;
        tc_fence_after();
        // S buffer s last held P of tile t-2, read by the PV MMA issued
        // before this point (one CTA's MMAs run in issue order).
        const uint64_t dk = ks ? dKs1 : dKs0;
        const uint32_t ts = tS0 + s * 128;
        umma_bf16_ss(ts, dQ0, dk, idS, 0u);
#pragma unroll
        for (int k = 1; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
          umma_bf16_ss(ts, desc_add(dQ0, off), desc_add(dk, off), idS, 1u);
        }
        umma_commit(&bars[kSFull0 + s]);
        if constexpr (NS == 1) {
          // one K/V slot: PV(t) must free it before tile t+1 can load
          ok = mbar_wait(&bars[kPFull0 + s], (t >> 1) & 1, abort_p, a.status, kDevErrTimeoutMma);
          if (!ok) break;
          tc_fence_after();
          issue_pv(t);
        } else if (t > 0) {
          ok = mbar_wait(&bars[kPFull0 + (s ^ 1)], ((t - 1) >> 1) & 1, abort_p, a.status,
                         kDevErrTimeoutMma);
          if (!ok) break;
          tc_fence_after();
          issue_pv(t - 1);
        }
      }
      if (NS > 1 && ok) {
        ok = mbar_wait(&bars[kPFull0 + ((T - 1) & 1)], ((T - 1) >> 1) & 1, abort_p, a.status,
                       kDevErrTimeoutMma);
        if (ok) {
          tc_fence_after();
          issue_pv(T - 1);
        }
      }
      // Drain: every MMA issued above completes before the CTA tears down.
      umma_commit(&bars[kDrain]);
      int dummy = 0;
      mbar_wait(&bars[kDrain], 0, &dummy, nullptr, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax --
    const int wg = warp >> 2;
    const int row = threadIdx.x & 127;  // == TMEM lane
    const int i = q0 + row;             // query row within its block
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    float m = -INFINITY, l = 0.f;
    bool ok = T > 0;
    for (int t = 0; t < T && ok; ++t) {
      const int x = t & 1;
      ok = mbar_wait(&bars[kSFull0 + x], (t >> 1) & 1, abort_p, a.status, kDevErrTimeoutSoftmax);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t ts = tS0 + x * 128 + wg * 64 + lane_off;
      uint32_t r0[32], r1[32];
      tmem_ld32(ts, r0);
      tmem_ld32(ts + 32, r1);
      tmem_ld_wait();
      tmem_reg_fence(r0);
      tmem_reg_fence(r1);
      // number of visible columns of this group's 64 (leading columns)
      int valid;
      if (t < n_ct) {
        valid = a.p - (ct_lo + t) * kTile - wg * 64;
      } else {
        const int col0 = (t - n_ct) * kTile + wg * 64;
        valid = min(i, a.n_real - 1) - col0 + 1;
      }
      valid = max(0, min(valid, 64));
      float s[64];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        s[c] = __uint_as_float(r0[c]) * a.scale_log2;
        s[32 + c] = __uint_as_float(r1[c]) * a.scale_log2;
      }
      if (__any_sync(0xffffffffu, valid < 64)) {
#pragma unroll
        for (int c = 0; c < 64; ++c) s[c] = c < valid ? s[c] : -INFINITY;
      }
      // row maximum of this group's columns (4 independent chains), then of
      // the whole tile through shared memory
      float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
      for (int c = 4; c < 64; c += 4) {
        mx0 = fmaxf(mx0, s[c]);
        mx1 = fmaxf(mx1, s[c + 1]);
        mx2 = fmaxf(mx2, s[c + 2]);
        mx3 = fmaxf(mx3, s[c + 3]);
      }
      float rmax = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
      // Slot reuse is safe: the other group read this buffer two tiles ago,
      // before it arrived on the other buffer's barrier, which this group has
      // waited for since.
      float* redt = red + x * 256;
      redt[wg * 128 + row] = rmax;
      mbar_arrive(&bars[kRedFull0 + x]);
      ok = mbar_wait(&bars[kRedFull0 + x], (t >> 1) & 1, abort_p, a.status, kDevErrTimeoutSoftmax);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      rmax = fmaxf(rmax, redt[(wg ^ 1) * 128 + row]);
      // Lazy rescaling: keep the stale max unless the new one exceeds it by
      // more than 8 (P values then stay below 2^8, safe in bf16 / f32).
      float alpha = 1.f;
      bool rescale = false;
      if (rmax > m + 8.f) {
        alpha = exp2_approx(m - rmax);  // exp2(-inf) = 0 on the first tile
        m = rmax;
        rescale = t > 0;
      }
      float rs0 = 0.f, rs1 = 0.f;
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = exp2_approx(s[2 * c] - m);
        const float p1 = exp2_approx(s[2 * c + 1] - m);
        rs0 += p0;
        rs1 += p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      // P over the first 32 columns of this group's S half (already read)
      tmem_st32(ts, pk);
      l = l * alpha + (rs0 + rs1);
      if (t > 0) {
        ok = mbar_wait(&bars[kODone], (t - 1) & 1, abort_p, a.status, kDevErrTimeoutSoftmax);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, rescale)) {
          // this group's half of the O columns
#pragma unroll
          for (int blk = 0; blk < D / 64; ++blk) {
            uint32_t o[32];
            const uint32_t addr = tO + lane_off + wg * (D / 2) + blk * 32;
            tmem_ld32(addr, o);
            tmem_ld_wait();
            tmem_reg_fence(o);
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tmem_st32(addr, o);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars[kPFull0 + x]);
    }
    // ------------------------------------------------------------ epilogue --
    if (ok) {
      ok = mbar_wait(&bars[kODone], (T - 1) & 1, abort_p, a.status, kDevErrTimeoutEpilogue);
      ok = __all_sync(0xffffffffu, ok);
    }
    // combine the two groups' row sums (own smem slots, own barrier)
    float l_all = l;
    if (ok) {
      red[512 + wg * 128 + row] = l;
      mbar_arrive(&bars[kLFull]);
      ok = mbar_wait(&bars[kLFull], 0, abort_p, a.status, kDevErrTimeoutEpilogue);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) l_all = l + red[512 + (wg ^ 1) * 128 + row];
    }
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l_all;
      const bool row_ok = i < a.n_rows;
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk) {
        uint32_t o[32];
        const int col = wg * (D / 2) + blk * 32;
        tmem_ld32(tO + lane_off + col, o);
        tmem_ld_wait();
        tmem_reg_fence(o);
        if (row_ok) {
          if (a.decode || a.out_f32) {
            float* dst;
            if (a.decode)
              dst = static_cast<float*>(a.out) +
                    ((static_cast<long long>(split) * a.Hq_map + head) * a.n_rows + i) * D;
            else
              dst = static_cast<float*>(a.out) +
                    ((static_cast<long long>(qb) * a.n_rows + i) * a.Hq_map + head) * D;
            float4* d4 = reinterpret_cast<float4*>(dst + col);
#pragma unroll
            for (int c = 0; c < 8; ++c)
              d4[c] = make_float4(__uint_as_float(o[4 * c]) * inv_l,
                                  __uint_as_float(o[4 * c + 1]) * inv_l,
                                  __uint_as_float(o[4 * c + 2]) * inv_l,
                                  __uint_as_float(o[4 * c + 3]) * inv_l);
          } else {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) +
                                 ((static_cast<long long>(qb) * a.n_rows + i) * a.Hq_map + head) * D;
            uint4* d4 = reinterpret_cast<uint4*>(dst + col);
#pragma unroll
            for (int c = 0; c < 4; ++c)
              d4[c] = make_uint4(
                  pack_bf16x2(__uint_as_float(o[8 * c]) * inv_l, __uint_as_float(o[8 * c + 1]) * inv_l),
                  pack_bf16x2(__uint_as_float(o[8 * c + 2]) * inv_l, __uint_as_float(o[8 * c + 3]) * inv_l),
                  pack_bf16x2(__uint_as_float(o[8 * c + 4]) * inv_l, __uint_as_float(o[8 * c + 5]) * inv_l),
                  pack_bf16x2(__uint_as_float(o[8 * c + 6]) * inv_l, __uint_as_float(o[8 * c + 7]) * inv_l));
          }
        }
      }
      if (row_ok && wg == 0) {
        const float lse2 = m + __log2f(l_all);
        if (a.decode)
          a.lse[(static_cast<long long>(split) * a.Hq_map + head) * a.n_rows + i] = lse2;
        else
          a.lse[(static_cast<long long>(qb) * a.Hq_map + head) * a.n_rows + i] =
              lse2 * 0.69314718055994531f;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, 512);
}

template <int D, int NS>
cudaError_t launch_fwd_d(const FwdLaunch& a, cudaStream_t st) {
  using L = FwdSmem<D, NS>;
  static_assert(L::kAlloc <= 232448, "shared memory budget");
  cudaError_t e = set_smem_once<fwd_kernel<D, NS>>(L::kAlloc);
  if (e != cudaSuccess) return e;
  FwdParams p{};
  p.n_rows = a.n_rows;
  p.Hq_map = a.Hq_map;
  p.G = a.G;
  p.p = a.p;
  p.n_real = a.n_real;
  p.cart_tiles_per_split = a.cart_tiles_per_split;
  p.n_qtiles = (a.n_rows + kTile - 1) / kTile;
  p.scale_log2 = a.scale_log2;
  p.out = a.out;
  p.lse = a.lse;
  p.out_f32 = a.out_f32 ? 1 : 0;
  p.decode = a.decode ? 1 : 0;
  p.status = device_status_ptr();
  dim3 grid;
  if (!a.decode)
    grid = dim3(a.Hq_map, a.n_qblocks, p.n_qtiles);
  else
    grid = dim3(a.Hq_map, p.n_qtiles, a.n_splits);
  TraceScope tr(a.decode ? "decode_cartridge" : "fwd", st);
  fwd_kernel<D, NS><<<grid, kFwdThreads, L::kAlloc, st>>>(*a.mQ, *a.mKc, *a.mVc, *a.mK, *a.mV, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t st) {
  if (a.decode) {
    if (a.d == 128) return launch_fwd_d<128, 1>(a, st);
    if (a.d == 64) return launch_fwd_d<64, 1>(a, st);
  } else {
    if (a.d == 128) return launch_fwd_d<128, 2>(a, st);
    if (a.d == 64) return launch_fwd_d<64, 2>(a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace cart
