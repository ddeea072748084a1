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
//               (sequence, head of the group, 64-row query tile) and sums the
//               batch inside its TMEM accumulators: the cartridge gradient
//               needs no cross-CTA reduction.  A real-token tile loops over
//               the heads of the group and the query tiles at or after it.
//               Per step: S^T = K Q^T, dP^T = V dO^T (TMEM, double buffered),
//               P^T, dS^T (bf16, shared memory), dV += P^T dO, dK += dS^T Q.
//               Epilogue: cartridge rows (f32, rows < frozen_prefix = 0) or
//               real rows (dK rotated back by R(p+j)^T).
//  dq_kernel    one CTA per 128-row query tile (like the forward): S = Q K^T,
//               dP = dO V^T, dS = P (dP - D) -> shared memory, dQ += dS K;
//               epilogue rotates back by R(p+i)^T.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.cuh"
#include "ptx.cuh"

namespace cart {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
  int B, n, Hq, Hkv, G, p, frozen_prefix, nq64, n_ct, n_rt, n_qtiles;
  float scale, scale_log2;
  const float* lse;
  const float* Dvec;
  void* dq;
  void* dk;
  void* dv;
  int out_f32;
  float* dkc;
  float* dvc;
  int accumulate;
  const float2* table;
  uint32_t* status;
};

// K-major operand descriptor: `k` is the 16-element K step; atom columns
// (64 elements of K) are `atom_stride` bytes apart (= rows * 128 B).
__device__ __forceinline__ uint64_t kdesc(uint32_t base, int k, uint32_t atom_stride) {
  return sdesc_sw128(base + static_cast<uint32_t>(k >> 2) * atom_stride +
                         static_cast<uint32_t>(k & 3) * 32u,
                     16u, 1024u);
}
// MN-major operand descriptor: `k` steps 16 rows along K (2 x 1024 B groups);
// 64-wide M/N blocks are `block_stride` bytes apart.
__device__ __forceinline__ uint64_t mndesc(uint32_t base, int k, uint32_t block_stride) {
  return sdesc_sw128(base + static_cast<uint32_t>(k) * 2048u, block_stride, 1024u);
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
template <int D>
struct DkdvSmem {
  static constexpr int kStages = 2;
  static constexpr int kKV = kTile * D * 2;        // resident K or V tile
  static constexpr int kQT = 64 * D * 2;           // 64-row Q or dO tile
  static constexpr int kK = 0;
  static constexpr int kV = kK + kKV;
  static constexpr int kStage0 = kV + kKV;         // stage s: Q at +0, dO at +kQT
  static constexpr int kPT = kStage0 + kStages * 2 * kQT;
  static constexpr int kDST = kPT + kTile * 64 * 2;
  static constexpr int kVec = kDST + kTile * 64 * 2;  // stage s: lse2[64], D[64]
  static constexpr int kBar = kVec + kStages * 512;
  static constexpr int kBytes = kBar + 256;
  static constexpr int kAlloc = kBytes + 1024;
};

enum DkdvBar { kResFull = 0, kQdoFull0, kQdoFull1, kQdoEmpty0, kQdoEmpty1, kStFull0, kStFull1,
               kStFree0, kStFree1, kDsFull, kDsFree, kAccDone, kDkdvDrain, kDkdvBars };

struct DkdvItem {
  int b, hh, qt;
};

__device__ __forceinline__ DkdvItem dkdv_item(const BwdParams& a, bool cart, int b_real, int rt,
                                              int u) {
  DkdvItem it;
  if (cart) {
    const int per_b = a.G * a.nq64;
    it.b = u / per_b;
    const int rem = u % per_b;
    it.hh = rem / a.nq64;
    it.qt = rem % a.nq64;
  } else {
    const int nq = a.nq64 - 2 * rt;
    it.b = b_real;
    it.hh = u / nq;
    it.qt = 2 * rt + u % nq;
  }
  return it;
}

template <int D>
__global__ void __launch_bounds__(192, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap mQ64, const __grid_constant__ CUtensorMap mdO64,
                const __grid_constant__ CUtensorMap mKc, const __grid_constant__ CUtensorMap mVc,
                const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
                const BwdParams a) {
  using L = DkdvSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBar + kDkdvBars * 8);
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

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
  const int U = cart ? a.B * a.G * a.nq64 : a.G * max(a.nq64 - 2 * tile, 0);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bars[kResFull], 1);
    mbar_init(&bars[kQdoFull0], 32);
    mbar_init(&bars[kQdoFull1], 32);
    mbar_init(&bars[kQdoEmpty0], 1);
    mbar_init(&bars[kQdoEmpty1], 1);
    mbar_init(&bars[kStFull0], 1);
    mbar_init(&bars[kStFull1], 1);
    mbar_init(&bars[kStFree0], 128);
    mbar_init(&bars[kStFree1], 128);
    mbar_init(&bars[kDsFull], 128);
    mbar_init(&bars[kDsFree], 1);
    mbar_init(&bars[kAccDone], 1);
    mbar_init(&bars[kDkdvDrain], 1);
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tST0 = tmem, tDP0 = tmem + 128, tDV = tmem + 256, tDK = tmem + 384;
  volatile int* abort_p = &abort_flag;
  uint8_t* sK = smem + L::kK;
  uint8_t* sV = smem + L::kV;
  uint8_t* sPT = smem + L::kPT;
  uint8_t* sDST = smem + L::kDST;
  float* vec = reinterpret_cast<float*>(smem + L::kVec);

  if (warp == 4) {
    // ------------------------------------------------------------ producer --
    bool ok = U > 0;
    if (ok && lane == 0) {
      tma_prefetch_desc(&mQ64);
      tma_prefetch_desc(&mdO64);
      mbar_arrive_expect_tx(&bars[kResFull], 2 * L::kKV);
#pragma unroll
      for (int h = 0; h < D / 64; ++h) {
        if (cart) {
          tma_load_4d(sK + h * 16384, &mKc, &bars[kResFull], h * 64, g, tile * kTile, 0);
          tma_load_4d(sV + h * 16384, &mVc, &bars[kResFull], h * 64, g, tile * kTile, 0);
        } else {
          tma_load_4d(sK + h * 16384, &mK, &bars[kResFull], h * 64, g, tile * kTile, b_real);
          tma_load_4d(sV + h * 16384, &mV, &bars[kResFull], h * 64, g, tile * kTile, b_real);
        }
      }
    }
    int issued = 0;
    for (int u = 0; u < U && ok; ++u) {
      const int s = u % L::kStages;
      if (u >= L::kStages) {
        ok = mbar_wait(&bars[kQdoEmpty0 + s], ((u / L::kStages) - 1) & 1, abort_p, a.status,
                       kDevErrTimeoutTma);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      const DkdvItem it = dkdv_item(a, cart, b_real, tile, u);
      const int h = g * a.G + it.hh;
      float* lse2 = vec + s * 128;
      float* dv = lse2 + 64;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int c = lane + 32 * r;
        const int q = it.qt * 64 + c;
        float l2 = INFINITY, dd = 0.f;
        if (q < a.n) {
          const long long idx = (static_cast<long long>(it.b) * a.Hq + h) * a.n + q;
          l2 = __ldg(a.lse + idx) * kLog2e;
          dd = __ldg(a.Dvec + idx);
        }
        lse2[c] = l2;
        dv[c] = dd;
      }
      if (lane == 0) {
        uint8_t* sQ = smem + L::kStage0 + s * 2 * L::kQT;
        uint8_t* sdO = sQ + L::kQT;
        mbar_arrive_expect_tx(&bars[kQdoFull0 + s], 2 * L::kQT);
#pragma unroll
        for (int hc = 0; hc < D / 64; ++hc) {
          tma_load_4d(sQ + hc * 8192, &mQ64, &bars[kQdoFull0 + s], hc * 64, h, it.qt * 64, it.b);
          tma_load_4d(sdO + hc * 8192, &mdO64, &bars[kQdoFull0 + s], hc * 64, h, it.qt * 64,
                      it.b);
        }
      } else {
        mbar_arrive(&bars[kQdoFull0 + s]);
      }
      issued = u + 1;
    }
    if (!ok && lane == 0 && U > 0) {
      int dummy = 0;
      mbar_wait(&bars[kResFull], 0, &dummy, nullptr, 0);
      for (int u = max(issued - L::kStages, 0); u < issued; ++u)
        mbar_wait(&bars[kQdoFull0 + u % L::kStages], (u / L::kStages) & 1, &dummy, nullptr, 0);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ----------------------------------------------------------------- MMA --
    if (lane == 0 && U > 0) {
      const uint32_t idST = idesc_bf16(128, 64, false, false);
      const uint32_t idACC = idesc_bf16(128, D, false, true);
      const uint32_t k_base = smem_u32(sK), v_base = smem_u32(sV);
      const uint32_t pt_base = smem_u32(sPT), dst_base = smem_u32(sDST);
      bool ok = mbar_wait(&bars[kResFull], 0, abort_p, a.status, kDevErrTimeoutMma);
      auto issue_acc = [&](int u) {
        const int s = u % L::kStages;
        const uint32_t q_base = smem_u32(smem + L::kStage0 + s * 2 * L::kQT);
        const uint32_t do_base = q_base + L::kQT;
#pragma unroll
        for (int k = 0; k < 4; ++k)  // 64 queries = 4 K steps
          umma_bf16_ss(tDV, kdesc(pt_base, k, 16384u), mndesc(do_base, k, 8192u), idACC,
                       (u > 0 || k > 0) ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_bf16_ss(tDK, kdesc(dst_base, k, 16384u), mndesc(q_base, k, 8192u), idACC,
                       (u > 0 || k > 0) ? 1u : 0u);
        umma_commit(&bars[kDsFree]);
        umma_commit(&bars[kQdoEmpty0 + s]);
      };
      for (int u = 0; u < U && ok; ++u) {
        const int s = u % L::kStages, x = u & 1;
        ok = mbar_wait(&bars[kQdoFull0 + s], (u / L::kStages) & 1, abort_p, a.status,
                       kDevErrTimeoutMma);
        if (!ok) break;
        if (u >= 2) {
          ok = mbar_wait(&bars[kStFree0 + x], ((u >> 1) - 1) & 1, abort_p, a.status,
                         kDevErrTimeoutMma);
          if (!ok) break;
        }
        tc_fence_after();
        const uint32_t q_base = smem_u32(smem + L::kStage0 + s * 2 * L::kQT);
        const uint32_t do_base = q_base + L::kQT;
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          umma_bf16_ss(tST0 + x * 64, kdesc(k_base, k, 16384u), kdesc(q_base, k, 8192u), idST,
                       k > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          umma_bf16_ss(tDP0 + x * 64, kdesc(v_base, k, 16384u), kdesc(do_base, k, 8192u), idST,
                       k > 0 ? 1u : 0u);
        umma_commit(&bars[kStFull0 + x]);
        if (u > 0) {
          ok = mbar_wait(&bars[kDsFull], (u - 1) & 1, abort_p, a.status, kDevErrTimeoutMma);
          if (!ok) break;
          tc_fence_after();
          issue_acc(u - 1);
        }
      }
      if (ok) {
        ok = mbar_wait(&bars[kDsFull], (U - 1) & 1, abort_p, a.status, kDevErrTimeoutMma);
        if (ok) {
          tc_fence_after();
          issue_acc(U - 1);
          umma_commit(&bars[kAccDone]);
        }
      }
      umma_commit(&bars[kDkdvDrain]);
      int dummy = 0;
      mbar_wait(&bars[kDkdvDrain], 0, &dummy, nullptr, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ P^T / dS^T warpgroup --
    const int row = threadIdx.x;  // key row within the tile == TMEM lane
    const int j = tile * kTile + row;
    const bool key_ok = cart ? (j < a.p) : (j < a.n);
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    bool ok = U > 0;
    for (int u = 0; u < U && ok; ++u) {
      const int s = u % L::kStages, x = u & 1;
      const DkdvItem it = dkdv_item(a, cart, b_real, tile, u);
      ok = mbar_wait(&bars[kStFull0 + x], (u >> 1) & 1, abort_p, a.status, kDevErrTimeoutSoftmax);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      // acquire the lse / D vectors the producer lanes published with kQdoFull
      // (already complete: the MMAs behind kStFull waited for it)
      ok = mbar_wait(&bars[kQdoFull0 + s], (u / L::kStages) & 1, abort_p, a.status,
                     kDevErrTimeoutSoftmax);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t s0[32], s1[32], d0[32], d1[32];
      tmem_ld32(tST0 + x * 64 + lane_off, s0);
      tmem_ld32(tST0 + x * 64 + lane_off + 32, s1);
      tmem_ld32(tDP0 + x * 64 + lane_off, d0);
      tmem_ld32(tDP0 + x * 64 + lane_off + 32, d1);
      tmem_ld_wait();
      tmem_reg_fence(s0);
      tmem_reg_fence(s1);
      tmem_reg_fence(d0);
      tmem_reg_fence(d1);
      tc_fence_before();
      mbar_arrive(&bars[kStFree0 + x]);
      const float* lse2 = vec + s * 128;
      const float* dvv = lse2 + 64;
      // query q = qt*64 + c sees key j: cartridge always; real iff j <= q
      int qlim = cart ? 64 : (j - it.qt * 64);  // columns c < qlim are masked for real keys
      uint32_t pk[32], dk[32];
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        float pv[2], dsv[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int cc = c + e;
          const float sv = __uint_as_float(cc < 32 ? s0[cc] : s1[cc - 32]);
          const float dp = __uint_as_float(cc < 32 ? d0[cc] : d1[cc - 32]);
          const bool vis = key_ok && (cart || cc >= qlim);
          const float pe = vis ? exp2_approx(sv * a.scale_log2 - lse2[cc]) : 0.f;
          pv[e] = pe;
          dsv[e] = pe * (dp - dvv[cc]);
        }
        pk[c / 2] = pack_bf16x2(pv[0], pv[1]);
        dk[c / 2] = pack_bf16x2(dsv[0], dsv[1]);
      }
      if (u > 0) {
        ok = mbar_wait(&bars[kDsFree], (u - 1) & 1, abort_p, a.status, kDevErrTimeoutSoftmax);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
#pragma unroll
      for (int c16 = 0; c16 < 8; ++c16) {
        *reinterpret_cast<uint4*>(sPT + sw128_offset(row, c16)) =
            make_uint4(pk[4 * c16], pk[4 * c16 + 1], pk[4 * c16 + 2], pk[4 * c16 + 3]);
        *reinterpret_cast<uint4*>(sDST + sw128_offset(row, c16)) =
            make_uint4(dk[4 * c16], dk[4 * c16 + 1], dk[4 * c16 + 2], dk[4 * c16 + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars[kDsFull]);
    }
    // ------------------------------------------------------------ epilogue --
    if (ok) {
      ok = mbar_wait(&bars[kAccDone], 0, abort_p, a.status, kDevErrTimeoutEpilogue);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      float kv[D];
      // dV row
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tDV + lane_off + c * 32, r);
        tmem_ld_wait();
        tmem_reg_fence(r);
#pragma unroll
        for (int e = 0; e < 32; ++e) kv[c * 32 + e] = __uint_as_float(r[e]);
      }
      if (key_ok) {
        if (cart) {
          float* dst = a.dvc + (static_cast<long long>(j) * a.Hkv + g) * D;
          float4* d4 = reinterpret_cast<float4*>(dst);
          const bool frozen = j < a.frozen_prefix;
          for (int c = 0; c < D / 4; ++c) {
            float4 v = make_float4(kv[4 * c], kv[4 * c + 1], kv[4 * c + 2], kv[4 * c + 3]);
            if (frozen) {
              v = make_float4(0.f, 0.f, 0.f, 0.f);
            } else if (a.accumulate) {
              const float4 o = d4[c];
              v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
            }
            d4[c] = v;
          }
        } else {
          store_row_out(a.dv, ((static_cast<long long>(b_real) * a.n + j) * a.Hkv + g) * D, kv, D,
                        a.out_f32 != 0);
        }
      }
      // dK row (scaled), rotated back for real keys
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tDK + lane_off + c * 32, r);
        tmem_ld_wait();
        tmem_reg_fence(r);
#pragma unroll
        for (int e = 0; e < 32; ++e) kv[c * 32 + e] = __uint_as_float(r[e]) * a.scale;
      }
      if (key_ok) {
        if (cart) {
          float* dst = a.dkc + (static_cast<long long>(j) * a.Hkv + g) * D;
          float4* d4 = reinterpret_cast<float4*>(dst);
          const bool frozen = j < a.frozen_prefix;
          for (int c = 0; c < D / 4; ++c) {
            float4 v = make_float4(kv[4 * c], kv[4 * c + 1], kv[4 * c + 2], kv[4 * c + 3]);
            if (frozen) {
              v = make_float4(0.f, 0.f, 0.f, 0.f);
            } else if (a.accumulate) {
              const float4 o = d4[c];
              v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
            }
            d4[c] = v;
          }
        } else {
          const float2* tb = a.table + static_cast<long long>(j) * (D / 2);
#pragma unroll
          for (int e = 0; e < D / 2; ++e) {
            const float2 cs = __ldg(tb + e);
            const float x0 = kv[e], x1 = kv[e + D / 2];
            kv[e] = x0 * cs.x + x1 * cs.y;
            kv[e + D / 2] = x1 * cs.x - x0 * cs.y;
          }
          store_row_out(a.dk, ((static_cast<long long>(b_real) * a.n + j) * a.Hkv + g) * D, kv, D,
                        a.out_f32 != 0);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, 512);
}

// ================================================================ dQ ======
template <int D>
struct DqSmem {
  static constexpr int kStages = 2;
  static constexpr int kT = kTile * D * 2;
  static constexpr int kQ = 0;
  static constexpr int kdO = kQ + kT;
  static constexpr int kK = kdO + kT;
  static constexpr int kV = kK + kStages * kT;
  static constexpr int kDS = kV + kStages * kT;
  static constexpr int kBar = kDS + kTile * kTile * 2;
  static constexpr int kBytes = kBar + 128;
  static constexpr int kAlloc = kBytes + 1024;
};

enum DqBar { kQdFull = 0, kKvFull0, kKvFull1, kKvEmpty0, kKvEmpty1, kSdFull, kSdFree, kDsdFull,
             kDqDone, kDqDrain, kDqBars };

template <int D>
__global__ void __launch_bounds__(192, 1)
    dq_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mdO,
              const __grid_constant__ CUtensorMap mKc, const __grid_constant__ CUtensorMap mVc,
              const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
              const BwdParams a) {
  using L = DqSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBar + kDqBars * 8);
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int h = blockIdx.x, b = blockIdx.y;
  const int qt = a.n_qtiles - 1 - static_cast<int>(blockIdx.z);
  const int kvh = h / a.G;
  const int q0 = qt * kTile;
  const int n_ct = a.n_ct;
  const int n_rt = min(qt + 1, a.n_rt);
  const int T = n_ct + n_rt;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bars[kQdFull], 1);
    mbar_init(&bars[kKvFull0], 1);
    mbar_init(&bars[kKvFull1], 1);
    mbar_init(&bars[kKvEmpty0], 1);
    mbar_init(&bars[kKvEmpty1], 1);
    mbar_init(&bars[kSdFull], 1);
    mbar_init(&bars[kSdFree], 128);
    mbar_init(&bars[kDsdFull], 128);
    mbar_init(&bars[kDqDone], 1);
    mbar_init(&bars[kDqDrain], 1);
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tDP = tmem + 128, tDQ = tmem + 256;
  volatile int* abort_p = &abort_flag;
  uint8_t* sQ = smem + L::kQ;
  uint8_t* sdO = smem + L::kdO;
  uint8_t* sDS = smem + L::kDS;

  if (warp == 4) {
    if (lane == 0 && T > 0) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mdO);
      mbar_arrive_expect_tx(&bars[kQdFull], 2 * L::kT);
#pragma unroll
      for (int hc = 0; hc < D / 64; ++hc) {
        tma_load_4d(sQ + hc * 16384, &mQ, &bars[kQdFull], hc * 64, h, q0, b);
        tma_load_4d(sdO + hc * 16384, &mdO, &bars[kQdFull], hc * 64, h, q0, b);
      }
      int issued = 0;
      bool ok = true;
      for (int t = 0; t < T; ++t) {
        const int s = t & 1;
        if (t >= 2) {
          ok = mbar_wait(&bars[kKvEmpty0 + s], ((t >> 1) - 1) & 1, abort_p, a.status,
                         kDevErrTimeoutTma);
          if (!ok) break;
        }
        uint8_t* sK = smem + L::kK + s * L::kT;
        uint8_t* sV = smem + L::kV + s * L::kT;
        mbar_arrive_expect_tx(&bars[kKvFull0 + s], 2 * L::kT);
#pragma unroll
        for (int hc = 0; hc < D / 64; ++hc) {
          if (t < n_ct) {
            tma_load_4d(sK + hc * 16384, &mKc, &bars[kKvFull0 + s], hc * 64, kvh, t * kTile, 0);
            tma_load_4d(sV + hc * 16384, &mVc, &bars[kKvFull0 + s], hc * 64, kvh, t * kTile, 0);
          } else {
            tma_load_4d(sK + hc * 16384, &mK, &bars[kKvFull0 + s], hc * 64, kvh,
                        (t - n_ct) * kTile, b);
            tma_load_4d(sV + hc * 16384, &mV, &bars[kKvFull0 + s], hc * 64, kvh,
                        (t - n_ct) * kTile, b);
          }
        }
        issued = t + 1;
      }
      if (!ok) {
        int dummy = 0;
        mbar_wait(&bars[kQdFull], 0, &dummy, nullptr, 0);
        for (int t = max(issued - 2, 0); t < issued; ++t)
          mbar_wait(&bars[kKvFull0 + (t & 1)], (t >> 1) & 1, &dummy, nullptr, 0);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    if (lane == 0 && T > 0) {
      const uint32_t idS = idesc_bf16(128, 128, false, false);
      const uint32_t idDQ = idesc_bf16(128, D, false, true);
      const uint32_t q_base = smem_u32(sQ), do_base = smem_u32(sdO), ds_base = smem_u32(sDS);
      bool ok = mbar_wait(&bars[kQdFull], 0, abort_p, a.status, kDevErrTimeoutMma);
      auto issue_dq = [&](int t) {
        const int sp = t & 1;
        const uint32_t k_base = smem_u32(smem + L::kK + sp * L::kT);
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k)
          umma_bf16_ss(tDQ, kdesc(ds_base, k, 16384u), mndesc(k_base, k, 16384u), idDQ,
                       (t > 0 || k > 0) ? 1u : 0u);
        umma_commit(&bars[kDqDone]);
        umma_commit(&bars[kKvEmpty0 + sp]);
      };
      for (int t = 0; t < T && ok; ++t) {
        const int s = t & 1;
        ok = mbar_wait(&bars[kKvFull0 + s], (t >> 1) & 1, abort_p, a.status, kDevErrTimeoutMma);
        if (!ok) break;
        if (t > 0) {
          ok = mbar_wait(&bars[kSdFree], (t - 1) & 1, abort_p, a.status, kDevErrTimeoutMma);
          if (!ok) break;
        }
        tc_fence_after();
        const uint32_t k_base = smem_u32(smem + L::kK + s * L::kT);
        const uint32_t v_base = smem_u32(smem + L::kV + s * L::kT);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          umma_bf16_ss(tS, kdesc(q_base, k, 16384u), kdesc(k_base, k, 16384u), idS,
                       k > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          umma_bf16_ss(tDP, kdesc(do_base, k, 16384u), kdesc(v_base, k, 16384u), idS,
                       k > 0 ? 1u : 0u);
        umma_commit(&bars[kSdFull]);
        if (t > 0) {
          ok = mbar_wait(&bars[kDsdFull], (t - 1) & 1, abort_p, a.status, kDevErrTimeoutMma);
          if (!ok) break;
          tc_fence_after();
          issue_dq(t - 1);
        }
      }
      if (ok) {
        ok = mbar_wait(&bars[kDsdFull], (T - 1) & 1, abort_p, a.status, kDevErrTimeoutMma);
        if (ok) {
          tc_fence_after();
          issue_dq(T - 1);
        }
      }
      umma_commit(&bars[kDqDrain]);
      int dummy = 0;
      mbar_wait(&bars[kDqDrain], 0, &dummy, nullptr, 0);
    }
    __syncwarp();
  } else {
    const int row = threadIdx.x;
    const int i = q0 + row;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    float lse2 = INFINITY, Di = 0.f;
    if (i < a.n) {
      const long long idx = (static_cast<long long>(b) * a.Hq + h) * a.n + i;
      lse2 = __ldg(a.lse + idx) * kLog2e;
      Di = __ldg(a.Dvec + idx);
    }
    bool ok = T > 0;
    for (int t = 0; t < T && ok; ++t) {
      ok = mbar_wait(&bars[kSdFull], t & 1, abort_p, a.status, kDevErrTimeoutSoftmax);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      int valid;
      if (t < n_ct) {
        valid = min(kTile, a.p - t * kTile);
      } else {
        const int col0 = (t - n_ct) * kTile;
        valid = max(0, min(min(i, a.n - 1) - col0 + 1, kTile));
      }
      uint32_t pk[64];
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        uint32_t sr[32], dr[32];
        tmem_ld32(tS + lane_off + blk * 32, sr);
        tmem_ld32(tDP + lane_off + blk * 32, dr);
        tmem_ld_wait();
        tmem_reg_fence(sr);
        tmem_reg_fence(dr);
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float ds[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int cc = blk * 32 + c + e;
            const float pe = (cc < valid)
                                 ? exp2_approx(__uint_as_float(sr[c + e]) * a.scale_log2 - lse2)
                                 : 0.f;
            ds[e] = pe * (__uint_as_float(dr[c + e]) - Di);
          }
          pk[blk * 16 + c / 2] = pack_bf16x2(ds[0], ds[1]);
        }
      }
      tc_fence_before();
      mbar_arrive(&bars[kSdFree]);
      if (t > 0) {
        ok = mbar_wait(&bars[kDqDone], (t - 1) & 1, abort_p, a.status, kDevErrTimeoutSoftmax);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
#pragma unroll
      for (int c16 = 0; c16 < 16; ++c16)
        *reinterpret_cast<uint4*>(sDS + (c16 >> 3) * 16384 + sw128_offset(row, c16 & 7)) =
            make_uint4(pk[4 * c16], pk[4 * c16 + 1], pk[4 * c16 + 2], pk[4 * c16 + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars[kDsdFull]);
    }
    if (ok) {
      ok = mbar_wait(&bars[kDqDone], (T - 1) & 1, abort_p, a.status, kDevErrTimeoutEpilogue);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      float x[D];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tDQ + lane_off + c * 32, r);
        tmem_ld_wait();
        tmem_reg_fence(r);
#pragma unroll
        for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(r[e]) * a.scale;
      }
      if (i < a.n) {
        const float2* tb = a.table + static_cast<long long>(i) * (D / 2);
#pragma unroll
        for (int e = 0; e < D / 2; ++e) {
          const float2 cs = __ldg(tb + e);
          const float x0 = x[e], x1 = x[e + D / 2];
          x[e] = x0 * cs.x + x1 * cs.y;
          x[e + D / 2] = x1 * cs.x - x0 * cs.y;
        }
        store_row_out(a.dq, ((static_cast<long long>(b) * a.n + i) * a.Hq + h) * D, x, D,
                      a.out_f32 != 0);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, 512);
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
  p.nq64 = (l.n + 63) / 64;
  p.n_ct = (l.p + kTile - 1) / kTile;
  p.n_rt = (l.n + kTile - 1) / kTile;
  p.n_qtiles = p.n_rt;
  p.scale = l.scale;
  p.scale_log2 = l.scale * kLog2e;
  p.lse = l.lse;
  p.Dvec = l.Dvec;
  p.dq = l.dq;
  p.dk = l.dk;
  p.dv = l.dv;
  p.out_f32 = l.out_f32 ? 1 : 0;
  p.dkc = l.dkc;
  p.dvc = l.dvc;
  p.accumulate = l.accumulate;
  p.table = l.table;
  p.status = device_status_ptr();
  cudaError_t e = cudaFuncSetAttribute(dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       DkdvSmem<D>::kAlloc);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           DqSmem<D>::kAlloc);
  if (e != cudaSuccess) return e;
  const int n_blocks = p.n_ct * p.Hkv + p.n_rt * p.Hkv * p.B;
  if (n_blocks > 0) {
    TraceScope tr("bwd_dkdv", st_dkdv);
    dkdv_kernel<D><<<n_blocks, 192, DkdvSmem<D>::kAlloc, st_dkdv>>>(
        *l.mQ64, *l.mdO64, *l.mKc, *l.mVc, *l.mK, *l.mV, p);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  TraceScope tr("bwd_dq", st_dq);
  dq_kernel<D><<<dim3(p.Hq, p.B, p.n_qtiles), 192, DqSmem<D>::kAlloc, st_dq>>>(
      *l.mQ, *l.mdO, *l.mKc, *l.mVc, *l.mK, *l.mV, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdLaunch& l, cudaStream_t st_dkdv, cudaStream_t st_dq) {
  if (l.d == 128) return launch_bwd_d<128>(l, st_dkdv, st_dq);
  if (l.d == 64) return launch_bwd_d<64>(l, st_dkdv, st_dq);
  return cudaErrorInvalidValue;
}

}  // namespace cart
