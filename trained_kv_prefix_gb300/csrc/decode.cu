// decode.cu -- q_seq = 1 decode of B conversations behind one shared cartridge.
// (Cartridges guide, "Semantics", serving bullet: decoding continues at
// position p with the training-time layout.)
//
// Work split:
//   prep      rotates every query at position p + len[b] (fp64 angle
//             reduction once per conversation) and lays the rotated queries
//             out per kv head as [B*G rows, Hkv, d], so that the cartridge
//             part runs as ONE tensor-core problem per kv head (rows of all
//             conversations batched into M) -- see fwd.cu; zeroes the
//             arrival counters.
//   private   split-KV over each conversation's own rows 0..len[b]: TMA-staged
//             chunks, mma.sync for the two small products, the new token's
//             rotation and append fused in.  Bound by HBM.  Launched as the
//             programmatic dependent of the cartridge pass, so the two run
//             together; the last CTA of each (conversation, kv head) waits
//             for the cartridge grid and merges all parts with their
//             log-sum-exps.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.cuh"
#include "ptx.cuh"

namespace cart {
namespace {

__device__ __forceinline__ int clamp_len(const int* len, int b, int rows) {
  int L = __ldg(len + b);
  return L < 0 ? 0 : (L >= rows ? rows - 1 : L);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float2 t = __bfloat1622float2(p[e]);
    f[2 * e] = t.x;
    f[2 * e + 1] = t.y;
  }
}

// ---------------------------------------------------------------- prep ----
// Rotated queries for the cartridge pass, laid out per kv head as
// [B*G rows, Hkv, d] (row r = b*G + hh).  grid: B blocks; block: 128 threads.
__global__ void __launch_bounds__(128) decode_prep_kernel(DecodeLaunch a, const RopeFreqs f) {
  __shared__ float2 cs[kMaxHeadDim / 2];
  const int b = blockIdx.x;
  const int L = clamp_len(a.len, b, a.rows);
  const int d = a.d, half = d / 2, G = a.Hq / a.Hkv;
  if (threadIdx.x < half) {
    const double ang = static_cast<double>(a.p + L) * f.inv_freq[threadIdx.x];
    const double k = rint(ang * 0.15915494309189535);
    double r = fma(-k, 6.283185307179586232, ang);
    r = fma(-k, 2.4492935982947064e-16, r);
    const float rh = static_cast<float>(r);
    const float rl = static_cast<float>(r - static_cast<double>(rh));
    float s, c;
    sincosf(rh, &s, &c);
    cs[threadIdx.x] = make_float2(c - s * rl, s + c * rl);
  }
  __syncthreads();
  if (threadIdx.x < a.Hkv) a.counters[b * a.Hkv + threadIdx.x] = 0;
  if (a.p == 0) return;
  const int chunks = half / 8;  // 8 pair indices per task
  const int tasks = a.Hq * chunks;
  for (int t = threadIdx.x; t < tasks; t += blockDim.x) {
    const int h = t / chunks, j0 = (t % chunks) * 8;
    const int g = h / G, hh = h % G;
    const __nv_bfloat16* src = a.q + (static_cast<long long>(b) * a.Hq + h) * d;
    __nv_bfloat16* dst = a.q_rot + (static_cast<long long>(b * G + hh) * a.Hkv + g) * d;
    float x0[8], x1[8], y0[8], y1[8];
    bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(src + j0)), x0);
    bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(src + j0 + half)), x1);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float2 c = cs[j0 + e];
      y0[e] = x0[e] * c.x - x1[e] * c.y;
      y1[e] = x1[e] * c.x + x0[e] * c.y;
    }
    *reinterpret_cast<uint4*>(dst + j0) =
        make_uint4(pack_bf16x2(y0[0], y0[1]), pack_bf16x2(y0[2], y0[3]),
                   pack_bf16x2(y0[4], y0[5]), pack_bf16x2(y0[6], y0[7]));
    *reinterpret_cast<uint4*>(dst + j0 + half) =
        make_uint4(pack_bf16x2(y1[0], y1[1]), pack_bf16x2(y1[2], y1[3]),
                   pack_bf16x2(y1[4], y1[5]), pack_bf16x2(y1[6], y1[7]));
  }
}

constexpr int kPrivCH = kDecodeChunk;
constexpr int kPrivMT = kPrivCH / 64;  // m16 key tiles per warp

// ------------------------------------------------------------- combine ----
// One warp merges the parts of one (conversation b, query head h); lane owns
// d/32 dims.  All log-sum-exps are in the log2 domain.  Part p < S is
// cartridge split p (normalised output, lse); part S + c is private chunk c
// (unnormalised acc against m, sum l).  Partials written by other CTAs are
// read through L2 (ld.global.cg).
__device__ __forceinline__ void combine_head_warp(const DecodeLaunch& a, int b, int h, int lane) {
  const int G = a.Hq / a.Hkv, g = h / G, hh = h % G;
  const int d = a.d;
  const int R = a.B * G, r = b * G + hh;
  const int L = clamp_len(a.len, b, a.rows);
  const int n_chunks = (a.rows + kPrivCH - 1) / kPrivCH;
  const int S = a.n_cart_splits;
  const int np = S + L / kPrivCH + 1;
  const long long pbase = ((static_cast<long long>(b) * a.Hkv + g) * n_chunks) * G + hh;
  auto part_lw = [&](int p, float* scale_m, float* lsum) {
    if (p < S) {
      *scale_m = __ldcg(a.cart_lse + (static_cast<long long>(p) * a.Hkv + g) * R + r);
      *lsum = 1.f;
      return *scale_m;
    }
    const long long pi = pbase + static_cast<long long>(p - S) * G;
    *scale_m = __ldcg(a.priv_ml + pi * 2);
    *lsum = __ldcg(a.priv_ml + pi * 2 + 1);
    return *scale_m + __log2f(*lsum);
  };
  float M = -INFINITY;
  for (int p = lane; p < np; p += 32) {
    float sm, ls;
    M = fmaxf(M, part_lw(p, &sm, &ls));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float num[4] = {0.f, 0.f, 0.f, 0.f};
  float den = 0.f;
  const int per_lane = d / 32;  // 4 or 2
  for (int p0 = 0; p0 < np; p0 += 32) {
    float w = 0.f, dn = 0.f;
    if (p0 + lane < np) {
      float sm, ls;
      part_lw(p0 + lane, &sm, &ls);
      w = exp2_approx(sm - M);   // scales the stored row
      dn = w * ls;
    }
    const int cnt = min(32, np - p0);
    // eight parts per round: all eight rows are requested before any is used
    for (int j0 = 0; j0 < cnt; j0 += 8) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int p = p0 + j0 + u;
        v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j0 + u < cnt) {
          const float* src = p < S
              ? a.cart_part + ((static_cast<long long>(p) * a.Hkv + g) * R + r) * d
              : a.priv_part + (pbase + static_cast<long long>(p - S) * G) * d;
          if (per_lane == 4) {
            v[u] = __ldcg(reinterpret_cast<const float4*>(src) + lane);
          } else {
            const float2 t2 = __ldcg(reinterpret_cast<const float2*>(src) + lane);
            v[u] = make_float4(t2.x, t2.y, 0.f, 0.f);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = min(j0 + u, 31);
        const float wj = (j0 + u < cnt) ? __shfl_sync(0xffffffffu, w, j) : 0.f;
        const float dj = __shfl_sync(0xffffffffu, dn, j);
        if (j0 + u < cnt) den += dj;
        num[0] = fmaf(wj, v[u].x, num[0]);
        num[1] = fmaf(wj, v[u].y, num[1]);
        num[2] = fmaf(wj, v[u].z, num[2]);
        num[3] = fmaf(wj, v[u].w, num[3]);
      }
    }
  }
  const float inv = 1.f / den;
  __nv_bfloat16* out = a.o + (static_cast<long long>(b) * a.Hq + h) * d + lane * per_lane;
  if (per_lane == 4) {
    *reinterpret_cast<uint2*>(out) = make_uint2(pack_bf16x2(num[0] * inv, num[1] * inv),
                                                pack_bf16x2(num[2] * inv, num[3] * inv));
  } else {
    *reinterpret_cast<uint32_t*>(out) = pack_bf16x2(num[0] * inv, num[1] * inv);
  }
}

// ------------------------------------------------------------- private ----
// grid: (Hkv, chunks, B); block: 128 threads (4 warps).  Keys of the chunk:
// private rows [c*CH, min((c+1)*CH, len+1)).
//   * 16-byte cp.async copies stage the chunk's K and V rows in shared memory
//     (128-byte swizzled layout, only the 16-row groups the chunk covers).
//   * Meanwhile the block rotates the group's G queries at position p+len
//     (one fp64-reduced cos/sin per frequency, shared through shared memory)
//     straight into mma.sync B fragments (queries padded to 8 columns).
//   * The block whose chunk holds row len rotates the new key, writes it and
//     the new value into the cache and patches its shared-memory copy.
//   * S^T = K Q^T with mma.sync m16n8k16 (keys as M: warp w owns keys
//     32w..32w+31), softmax statistics per query across the block, P (bf16)
//     through shared memory, O^T = V^T P^T with V^T fragments read by
//     ldmatrix.trans (warp w owns output dims 32w..32w+31).
// Output per query head: unnormalised acc[d] against the chunk's own max m
// (log2 domain) and its sum l.

template <int D>
struct PrivSmem {
  static constexpr int kHalf = kPrivCH * 128;          // 64 dims x 128 rows (bf16)
  static constexpr int kK = 0;
  static constexpr int kV = kK + (D / 64) * kHalf;
  static constexpr int kP = kV + (D / 64) * kHalf;     // bf16 [8 queries][CH + 8]
  static constexpr int kPStride = kPrivCH + 8;         // padded row: conflict-free B loads
  static constexpr int kCS = kP + 8 * kPStride * 2;    // float2 [D/2]
  static constexpr int kRed = kCS + (D / 2) * 8;       // f32 [2][4 warps][8]
  static constexpr int kBytes = kRed + 2 * 4 * 8 * 4;
  static constexpr int kAlloc = kBytes + 1024;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Address of the 16-byte chunk holding dims [8*dc, 8*dc + 8) of row `row` in a
// TMA-written tile (two 64-dim halves, 128-byte swizzle).
__device__ __forceinline__ uint32_t tile_chunk(uint32_t base, int row, int dc) {
  return base + (dc >> 3) * (kPrivCH * 128) + row * 128 + ((((dc & 7) ^ (row & 7))) << 4);
}

__device__ __forceinline__ float2 rope_cs(const RopeFreqs& f, int j, int pos) {
  const double ang = static_cast<double>(pos) * f.inv_freq[j];
  const double k = rint(ang * 0.15915494309189535);
  double r = fma(-k, 6.283185307179586232, ang);
  r = fma(-k, 2.4492935982947064e-16, r);
  const float rh = static_cast<float>(r);
  const float rl = static_cast<float>(r - static_cast<double>(rh));
  float s, c;
  sincosf(rh, &s, &c);
  return make_float2(c - s * rl, s + c * rl);
}

template <int D, int G>
__global__ void __launch_bounds__(128) decode_private_kernel(DecodeLaunch a, const RopeFreqs f,
                                                             float scale_log2) {
  using L = PrivSmem<D>;
  constexpr int CH = kPrivCH;
  constexpr int HALF = D / 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __nv_bfloat16* sP = reinterpret_cast<__nv_bfloat16*>(smem + L::kP);
  float2* scs = reinterpret_cast<float2*>(smem + L::kCS);
  float* sred = reinterpret_cast<float*>(smem + L::kRed);

  // kv head fastest: the CTAs reading the interleaved head slices of the
  // same cache rows run together (DRAM row locality)
  const int g = blockIdx.x, c = blockIdx.y, b = blockIdx.z;
  const int Lb = clamp_len(a.len, b, a.rows);
  const int k0 = c * CH;
  if (k0 > Lb) return;  // whole chunk beyond this conversation's rows
  const int kn = min(CH, Lb + 1 - k0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, tig = lane & 3;
  const int pos = a.p + Lb;
  const uint32_t sK = smem_u32(smem + L::kK), sV = smem_u32(smem + L::kV);

  // Stage the chunk's rows 0..16*ceil(kn/16) of K and V with 16-byte
  // cp.async copies into the 128-byte-swizzled layout (rows >= kn of the last
  // 16-row group are zero-filled, so P = 0 never meets stale data).
  const int kgroups = (kn + 15) / 16;
  {
    constexpr int kPieces = D / 8;  // 16-byte pieces per row
    const long long rstride = static_cast<long long>(a.Hkv) * D;
    const __nv_bfloat16* kg = a.k_cache + (static_cast<long long>(b) * a.rows + k0) * rstride + g * D;
    const __nv_bfloat16* vg = a.v_cache + (static_cast<long long>(b) * a.rows + k0) * rstride + g * D;
    const uint32_t sKb = smem_u32(smem + L::kK), sVb = smem_u32(smem + L::kV);
    for (int t = tid; t < kgroups * 16 * kPieces; t += 128) {
      const int rr = t / kPieces, dc = t % kPieces;
      const uint32_t so = tile_chunk(0, rr, dc);
      const int src_bytes = rr < kn ? 16 : 0;
      const long long go = static_cast<long long>(min(rr, kn - 1)) * rstride + dc * 8;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sKb + so),
                   "l"(kg + go), "r"(src_bytes) : "memory");
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sVb + so),
                   "l"(vg + go), "r"(src_bytes) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  if (tid < HALF) scs[tid] = rope_cs(f, tid, pos);
  __syncthreads();

  // ---- rotated queries as B fragments: bq[k][0] = q[g8][16k + 2tig, +1],
  // bq[k][1] = q[g8][16k + 8 + 2tig, +1]; rows g8 >= G are zero padding
  uint32_t bq[D / 16][2];
  {
    float qv[D / 16][4];
    if (g8 < G) {
      const __nv_bfloat16* qrow = a.q + (static_cast<long long>(b) * a.Hq + g * G + g8) * D;
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const __nv_bfloat162 v =
              *reinterpret_cast<const __nv_bfloat162*>(qrow + 16 * k + 8 * hf + 2 * tig);
          const float2 fv = __bfloat1622float2(v);
          qv[k][2 * hf] = fv.x;
          qv[k][2 * hf + 1] = fv.y;
        }
    } else {
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
#pragma unroll
        for (int e = 0; e < 4; ++e) qv[k][e] = 0.f;
    }
    // rotate-half: element j < D/2 pairs with j + D/2, i.e. K step k with
    // step k + D/32 and the same offsets
#pragma unroll
    for (int k = 0; k < D / 32; ++k)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = 16 * k + 8 * (e >> 1) + 2 * tig + (e & 1);
        const float2 cs = scs[j];
        const float x0 = qv[k][e], x1 = qv[k + D / 32][e];
        qv[k][e] = x0 * cs.x - x1 * cs.y;
        qv[k + D / 32][e] = x1 * cs.x + x0 * cs.y;
      }
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      bq[k][0] = pack_bf16x2(qv[k][0], qv[k][1]);
      bq[k][1] = pack_bf16x2(qv[k][2], qv[k][3]);
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();

  // ---- the new token: rotated key and value into the cache row len and
  // into this block's shared copy (its chunk holds that row)
  if (Lb - k0 < CH) {
    const int rr = Lb - k0;
    const long long crow = ((static_cast<long long>(b) * a.rows + Lb) * a.Hkv + g) * D;
    const long long nrow = (static_cast<long long>(b) * a.Hkv + g) * D;
    for (int j = tid; j < HALF; j += 128) {
      const float x0 = __bfloat162float(a.k_new[nrow + j]);
      const float x1 = __bfloat162float(a.k_new[nrow + j + HALF]);
      const float2 cs = scs[j];
      const __nv_bfloat16 y0 = __float2bfloat16_rn(x0 * cs.x - x1 * cs.y);
      const __nv_bfloat16 y1 = __float2bfloat16_rn(x1 * cs.x + x0 * cs.y);
      a.k_cache[crow + j] = y0;
      a.k_cache[crow + j + HALF] = y1;
      const int j1 = j + HALF;
      *reinterpret_cast<__nv_bfloat16*>(smem + L::kK + (tile_chunk(0, rr, j >> 3)) + (j & 7) * 2) = y0;
      *reinterpret_cast<__nv_bfloat16*>(smem + L::kK + (tile_chunk(0, rr, j1 >> 3)) + (j1 & 7) * 2) = y1;
    }
    for (int j = tid; j < D; j += 128) {
      const __nv_bfloat16 v = a.v_new[nrow + j];
      a.v_cache[crow + j] = v;
      *reinterpret_cast<__nv_bfloat16*>(smem + L::kV + (tile_chunk(0, rr, j >> 3)) + (j & 7) * 2) = v;
    }
    __syncthreads();
  }

  // ---- S^T = K Q^T for this warp's keys (MT m16 tiles)
  constexpr int MT = kPrivMT;
  float sacc[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) sacc[mt][e] = 0.f;
    // lane -> row address: matrices (rows 0-7,k lo), (rows 8-15,k lo),
    // (rows 0-7,k hi), (rows 8-15,k hi)
    const int row = warp * 16 * MT + mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      uint32_t af[4];
      ldsm_x4(tile_chunk(sK, row, 2 * k + (lane >> 4)), af);
      mma_bf16_16816(sacc[mt], af, bq[k][0], bq[k][1]);
    }
  }
  // thread holds keys r0 = warp*32 + mt*16 + g8 (+8) and queries 2tig, 2tig+1
  float mq[2], lq[2];
#pragma unroll
  for (int qq = 0; qq < 2; ++qq) {
    float mx = -INFINITY;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int key = warp * 16 * MT + mt * 16 + g8 + 8 * hf;
        float sv = sacc[mt][2 * hf + qq] * scale_log2;
        sv = key < kn ? sv : -INFINITY;
        sacc[mt][2 * hf + qq] = sv;
        mx = fmaxf(mx, sv);
      }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    mq[qq] = mx;
  }
  if (g8 == 0) {
    sred[warp * 8 + 2 * tig] = mq[0];
    sred[warp * 8 + 2 * tig + 1] = mq[1];
  }
  __syncthreads();
#pragma unroll
  for (int qq = 0; qq < 2; ++qq) {
    const int q = 2 * tig + qq;
    mq[qq] = fmaxf(fmaxf(sred[q], sred[8 + q]), fmaxf(sred[16 + q], sred[24 + q]));
    float sum = 0.f;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int key = warp * 16 * MT + mt * 16 + g8 + 8 * hf;
        const float pv = exp2_approx(sacc[mt][2 * hf + qq] - mq[qq]);  // 0 for masked keys
        sum += pv;
        sP[q * L::kPStride + key] = __float2bfloat16_rn(pv);
      }
    sum += __shfl_xor_sync(0xffffffffu, sum, 4);
    sum += __shfl_xor_sync(0xffffffffu, sum, 8);
    sum += __shfl_xor_sync(0xffffffffu, sum, 16);
    lq[qq] = sum;
  }
  if (g8 == 0) {
    sred[32 + warp * 8 + 2 * tig] = lq[0];
    sred[32 + warp * 8 + 2 * tig + 1] = lq[1];
  }
  __syncthreads();
  const int n_chunks = (a.rows + CH - 1) / CH;
  const long long part_idx = ((static_cast<long long>(b) * a.Hkv + g) * n_chunks + c) * G;
  if (warp == 0 && g8 == 0) {
#pragma unroll
    for (int qq = 0; qq < 2; ++qq) {
      const int q = 2 * tig + qq;
      if (q < G) {
        const float lsum = (sred[32 + q] + sred[40 + q]) + (sred[48 + q] + sred[56 + q]);
        a.priv_ml[(part_idx + q) * 2 + 0] = mq[qq];
        a.priv_ml[(part_idx + q) * 2 + 1] = lsum;
      }
    }
  }

  // ---- O^T = V^T P^T: warp w owns dims 32w..32w+31 (two m16 tiles)
  constexpr int kDimTiles = D / 16;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int dt = warp * 2 + i;
    if (dt >= kDimTiles) break;
    float oacc[4] = {0.f, 0.f, 0.f, 0.f};
    // lane -> stored row (key) and dim chunk for the transposed matrices:
    // m0 (dims lo, keys lo), m1 (dims hi, keys lo), m2 (dims lo, keys hi),
    // m3 (dims hi, keys hi)
    const int dchunk = 2 * dt + ((lane >> 3) & 1);
    const int krow = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
    for (int k = 0; k < CH / 16; ++k) {
      if (k >= kgroups) break;  // uniform across the block
      uint32_t af[4];
      ldsm_x4_t(tile_chunk(sV, 16 * k + krow, dchunk), af);
      const uint32_t b0 =
          *reinterpret_cast<const uint32_t*>(sP + g8 * L::kPStride + 16 * k + 2 * tig);
      const uint32_t b1 =
          *reinterpret_cast<const uint32_t*>(sP + g8 * L::kPStride + 16 * k + 8 + 2 * tig);
      mma_bf16_16816(oacc, af, b0, b1);
    }
    // oacc: dims 16dt + g8 (+8), queries 2tig, 2tig+1
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        const int q = 2 * tig + qq;
        if (q < G) a.priv_part[(part_idx + q) * D + 16 * dt + g8 + 8 * hf] = oacc[2 * hf + qq];
      }
  }

  // ---- the last private CTA of (b, g) merges every part of its G heads
  __shared__ int s_last;
  __threadfence();  // this CTA's partials are visible before it is counted
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(a.counters + b * a.Hkv + g, 1);
    s_last = prev == Lb / CH;  // used chunks of this conversation = Lb/CH + 1
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // the cartridge partials come from the grid this one depends on
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int hh = warp; hh < G; hh += 4) combine_head_warp(a, b, g * G + hh, lane);
  if (tid == 0) a.counters[b * a.Hkv + g] = 0;
}

template <int D, int G>
cudaError_t launch_private_dg(const DecodeLaunch& a, const RopeFreqs& f, bool dependent,
                              cudaStream_t st) {
  using L = PrivSmem<D>;
  cudaError_t e = set_smem_once<decode_private_kernel<D, G>>(L::kAlloc);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.Hkv, (a.rows + kPrivCH - 1) / kPrivCH, a.B);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  const float scale_log2 = a.scale * 1.4426950408889634f;
  TraceScope tr("decode_private", st);
  return cudaLaunchKernelEx(&cfg, decode_private_kernel<D, G>, a, f, scale_log2);
}

}  // namespace

cudaError_t launch_decode(const DecodeLaunch& a, const RopeFreqs& f, cudaStream_t st) {
  const int G = a.Hq / a.Hkv;
  if (a.chunk != kPrivCH) return cudaErrorInvalidValue;
  {
    TraceScope tr("decode_prep", st);
    decode_prep_kernel<<<a.B, 128, 0, st>>>(a, f);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.p > 0) {
    CUtensorMap mQ, mKc, mVc;
    if (!make_bf16_rows_map(&mQ, a.q_rot, 1, a.B * G, a.Hkv, a.d, 128) ||
        !make_bf16_rows_map(&mKc, a.kc, 1, a.p, a.Hkv, a.d, 128) ||
        !make_bf16_rows_map(&mVc, a.vc, 1, a.p, a.Hkv, a.d, 128))
      return cudaErrorInvalidValue;
    FwdLaunch l{};
    l.mQ = &mQ;
    l.mKc = &mKc;
    l.mVc = &mVc;
    l.mK = &mKc;  // no real-token tiles in decode mode
    l.mV = &mVc;
    l.d = a.d;
    l.n_rows = a.B * G;
    l.n_qblocks = 1;
    l.Hq_map = a.Hkv;
    l.G = 1;
    l.p = a.p;
    l.n_real = 0;
    l.cart_tiles_per_split = a.cart_tiles_per_split;
    l.n_splits = a.n_cart_splits;
    l.scale_log2 = a.scale * 1.4426950408889634f;
    l.out = const_cast<float*>(a.cart_part);
    l.out_f32 = true;
    l.lse = const_cast<float*>(a.cart_lse);
    l.decode = true;
    e = launch_fwd(l, st);
    if (e != cudaSuccess) return e;
  }
  const bool dep = a.p > 0;
  if (a.d == 128) {
    switch (G) {
      case 1: return launch_private_dg<128, 1>(a, f, dep, st);
      case 2: return launch_private_dg<128, 2>(a, f, dep, st);
      case 4: return launch_private_dg<128, 4>(a, f, dep, st);
      case 8: return launch_private_dg<128, 8>(a, f, dep, st);
    }
  } else if (a.d == 64) {
    switch (G) {
      case 1: return launch_private_dg<64, 1>(a, f, dep, st);
      case 2: return launch_private_dg<64, 2>(a, f, dep, st);
      case 4: return launch_private_dg<64, 4>(a, f, dep, st);
      case 8: return launch_private_dg<64, 8>(a, f, dep, st);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace cart
