// decode.cu -- decode of B conversations behind one shared cartridge: one new
// token per conversation (q_seq = 1), or a span of s new tokens per
// conversation checked in one step (span verification: token t at position
// p + len[b] + t sees the cartridge and private rows 0 .. len[b] + t;
// Cartridges guide, "Batched self-study (measured)", the --spec-b bullet).
// (Cartridges guide, "Semantics", serving bullet: decoding continues at
// position p with the training-time layout.)
//
// Work split (three kernels chained by programmatic dependent launch):
//   cartridge the forward kernel in decode mode (fwd.cu): the B*s*G query
//             rows of each kv head, rotated in shared memory at their
//             positions, run as ONE tensor-core problem per kv head against
//             the shared rows, split into a few key ranges; writes
//             normalised partial outputs and log-sum-exps.  Launched first,
//             on a few SMs.
//   private   fixed units of up to kDecodeUnit private rows of one
//             (conversation, kv head) per CTA: TMA-staged 64-row chunks,
//             mma.sync for the two small products over the s*G query
//             columns, online softmax, the new tokens' rotation and append
//             fused in; writes normalised partial outputs and log-sum-exps.
//             Bound by HBM; fills the GPU next to the cartridge pass.
//   merge     combines the cartridge and private parts of every
//             (conversation, span position, query head) with their
//             log-sum-exps into o.
// With a sliding window the cartridge pass starts at the earliest window of
// its conversations, the private pass skips units and chunks before a
// conversation's window, and the merge reads only the parts inside its
// row's window.
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


// ------------------------------------------------------------- private ----
// grid: (Hkv, B, max_units); block: 128 threads (4 warps).  CTA (g, b, u)
// owns private rows [u*U, min((u+1)*U, len+s)) of kv head g of conversation
// b (U = kDecodeUnit; CTAs past the end of a conversation exit at once) and
// streams them through a ring of 64-row chunk buffers (kPrivStagesFor):
//   * Thread 0 stages a chunk's K and V rows in shared memory by TMA (one
//     (64, 1, 64, 1) box per 64-dim half, 128-byte swizzled, completing on
//     the slot's mbarrier) as soon as the slot is free; staged V
//     rows past the unit's end are zeroed after they land (the cache may
//     hold anything there, and 0 * a non-finite value is not 0).
//   * The block rotates the s*G query columns c = t*G + hh (t the span
//     position, at p + len + t) straight into mma.sync B fragments, 8
//     columns per tile, padded with zero columns.  With s = 1 every column
//     shares one position: its cos/sin (all-f32 turn reduction, hardware
//     sine / cosine) are evaluated once and shared through shared memory.
//   * The CTA whose unit holds a new row len + t writes token t's rotated
//     key and its value into that cache row and patches its staged copy.
//   * Per chunk: S^T = K Q^T with mma.sync m16n8k16 (keys as M: warp w owns
//     keys 16w..16w+15), the causal mask of span columns (key row <= len +
//     t), online softmax per column across the block, P (bf16) through
//     shared memory, O^T += V^T P^T with V^T fragments read by
//     ldmatrix.trans (warp w owns output dims 16*dt.. of its tiles), O kept
//     in registers and rescaled when a column's running maximum grows.
//   * Output: the unit's normalised O and its log2-domain log-sum-exp per
//     column (O = 0, lse = -inf for a column that saw none of its rows).
constexpr int kPrivCH = kDecodeChunk;  // keys per chunk
// Chunk buffers per CTA.  One for up to 16 query columns: each chunk is
// copied once the previous one is done, and the copies of one CTA overlap
// the compute of the others (about six CTAs fit per SM this way; two buffers
// per CTA leave room for three and measured 9 % slower on the serving step).
// Two for 24-32 columns, whose registers already limit an SM to three CTAs.
template <int QN>
constexpr int kPrivStagesFor = QN >= 3 ? 2 : 1;

template <int D, int QN>
struct PrivSmem {
  static constexpr int kPrivStages = kPrivStagesFor<QN>;
  static constexpr int kHalf = kPrivCH * 128;          // 64 dims x CH rows (bf16)
  static constexpr int kTile = (D / 64) * kHalf;       // one K or V chunk
  static constexpr int kStage = 2 * kTile;             // K then V
  static constexpr int kP = kPrivStages * kStage;      // bf16 [8*QN query columns][CH + 8]
  static constexpr int kPStride = kPrivCH + 8;         // padded row: conflict-free B loads
  static constexpr int kCS = kP + 8 * QN * kPStride * 2;  // float2 [D/2]: a new key's angles
  static constexpr int kRed = kCS + (D / 2) * 8;       // f32 [2][4 warps][8*QN]
  static constexpr int kBar = kRed + 2 * 4 * 8 * QN * 4;  // full[stages], abort word
  static constexpr int kBytes = kBar + kPrivStages * 8 + 16;
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
// staged chunk: 64-dim halves of CH rows, each the 128-byte-swizzled layout a
// (64, 1, CH, 1) TMA box of the cache map writes.
__device__ __forceinline__ uint32_t tile_chunk(uint32_t base, int row, int dc) {
  return base + (dc >> 3) * (kPrivCH * 128) + row * 128 + ((((dc & 7) ^ (row & 7))) << 4);
}

// kG = 0: a span of query positions per conversation, G from the launch;
// kG > 0: the single-token step with G = kG, compiled without the
// per-column causal mask.
template <int D, int QN, int kG>
__global__ void __launch_bounds__(128) decode_private_kernel(
    const __grid_constant__ CUtensorMap mKs, const __grid_constant__ CUtensorMap mVs,
    const __grid_constant__ CUtensorMap mKt, const __grid_constant__ CUtensorMap mVt,
    DecodeLaunch a, const RopeFreqs f, float scale_log2) {
  using L = PrivSmem<D, QN>;
  constexpr int kPrivStages = L::kPrivStages;
  constexpr int CH = kPrivCH;
  constexpr int HALF = D / 2;
  static_assert(CH == 64, "four warps own 16 keys each");
  constexpr bool kSpan = kG == 0;
  const int G = kSpan ? a.Hq / a.Hkv : kG, S = kSpan ? a.span : 1;
  const int QC = G * S;  // query columns c = t*G + hh
  const int g = blockIdx.x, b = blockIdx.y, u = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, tig = lane & 3;
  // the query words first: their global latency overlaps the length load,
  // the staging and the angles below.  Thread column j*8 + g8 of tile j;
  // columns >= QC are zero padding.
  uint32_t qraw[QN][D / 16][2];
  if constexpr (!kSpan) {  // one column per query head, G known here
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
        a.q + (static_cast<long long>(b) * a.Hq + g * kG + (g8 < kG ? g8 : 0)) * D);
#pragma unroll
    for (int k = 0; k < D / 16; ++k)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
        qraw[0][k][hf] = g8 < kG ? __ldg(qrow + 8 * k + 4 * hf + tig) : 0u;
  } else {
#pragma unroll
    for (int j = 0; j < QN; ++j) {
      const int c = j * 8 + g8;
      const int cc = c < QC ? c : 0;
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          a.q + ((static_cast<long long>(b) * S + cc / G) * a.Hq + g * G + cc % G) * D);
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
          qraw[j][k][hf] = c < QC ? __ldg(qrow + 8 * k + 4 * hf + tig) : 0u;
    }
  }
  const int Lb = clamp_len(a.len, b, a.rows - S + 1);  // new rows Lb .. Lb + S - 1
  const int k_lo = u * kDecodeUnit;
  // sliding window: column t sees private rows Lb + t - window + 1 .. Lb + t;
  // lo0 is the first row any column sees, u_lo its unit
  const int W = a.window;
  const int lo0 = W > 0 ? Lb - W + 1 : 0;
  const int u_lo = lo0 > 0 ? lo0 / kDecodeUnit : 0;
  if (k_lo > Lb + S - 1 || u < u_lo) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    return;  // past the end of this conversation's rows, or before its window
  }
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __nv_bfloat16* sP = reinterpret_cast<__nv_bfloat16*>(smem + L::kP);
  float2* scs = reinterpret_cast<float2*>(smem + L::kCS);
  float* sred = reinterpret_cast<float*>(smem + L::kRed);
  const int nk = min(kDecodeUnit, Lb + S - k_lo);  // keys of this unit
  const int nc = (nk + CH - 1) / CH;               // chunks
  const int c0 = lo0 > k_lo ? (lo0 - k_lo) / CH : 0;  // first chunk in the window
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBar);
  int* abort_flag = reinterpret_cast<int*>(full + kPrivStages);
  const uint32_t abort_s = smem_u32(abort_flag);
  if (tid == 0) {
    *abort_flag = 0;
    for (int s2 = 0; s2 < kPrivStages; ++s2) mbar_init(&full[s2], 1);
    fence_mbar_init();
  }

  // Stage chunk c into ring slot (c - c0) % kPrivStages (thread 0): the K and
  // V rows of the chunk by TMA, one 64-row box per 64-dim half, or for the
  // unit's last, partial chunk 16-row boxes up to its last row (rows past the
  // cache's end read as zero; rows past the unit's end are whatever the
  // cache holds).  A 16-row box lands where the 64-row box would put those
  // rows: the 128-byte swizzle repeats every 8 rows.
  auto stage = [&](int c) {
    if (tid != 0) return;
    const int sl = (c - c0) % kPrivStages;
    uint8_t* sK = smem + sl * L::kStage;
    const int row = k_lo + c * CH;
    const int kn_c = min(CH, nk - c * CH);
    if (kn_c == CH) {
      mbar_arrive_expect_tx(&full[sl], L::kStage);
#pragma unroll
      for (int h = 0; h < D / 64; ++h) {
        tma_load_4d(sK + h * L::kHalf, &mKs, &full[sl], h * 64, g, row, b);
        tma_load_4d(sK + L::kTile + h * L::kHalf, &mVs, &full[sl], h * 64, g, row, b);
      }
    } else {
      const int nb = (kn_c + 15) / 16;
      mbar_arrive_expect_tx(&full[sl], nb * 16 * 128 * (D / 64) * 2);
      for (int q = 0; q < nb; ++q)
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          tma_load_4d(sK + h * L::kHalf + q * 2048, &mKt, &full[sl], h * 64, g, row + 16 * q, b);
          tma_load_4d(sK + L::kTile + h * L::kHalf + q * 2048, &mVt, &full[sl], h * 64, g,
                      row + 16 * q, b);
        }
    }
  };
  for (int c = c0; c < c0 + kPrivStages && c < nc; ++c) stage(c);
  // one position for every column when S = 1: its angles once, shared
  if (S == 1 && tid < HALF) scs[tid] = rope_cs_turns_fast(f.turns[tid], a.p + Lb);
  __syncthreads();

  // ---- rotated queries as B fragments: bq[j][k][0] = q[col][16k + 2tig, +1],
  // bq[j][k][1] = q[col][16k + 8 + 2tig, +1] for col = j*8 + g8, rotated at
  // position p + Lb + t (t = col / G)
  uint32_t bq[QN][D / 16][2];
  auto rotate_queries = [&](auto angles) {
#pragma unroll
    for (int j = 0; j < QN; ++j) {
      const int c = j * 8 + g8;
      const int pos = a.p + Lb + (c < QC ? c / G : 0);
      float qv[D / 16][4];
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const float2 fv = bf16x2_to_float2(qraw[j][k][hf]);  // zero for padding columns
          qv[k][2 * hf] = fv.x;
          qv[k][2 * hf + 1] = fv.y;
        }
      // rotate-half: element e < D/2 pairs with e + D/2, i.e. K step k with
      // step k + D/32 and the same offsets
#pragma unroll
      for (int k = 0; k < D / 32; ++k)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int jp = 16 * k + 8 * (e >> 1) + 2 * tig + (e & 1);
          float y0, y1;
          rope_pair(qv[k][e], qv[k + D / 32][e], angles(jp, pos), y0, y1);
          qv[k][e] = y0;
          qv[k + D / 32][e] = y1;
        }
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        bq[j][k][0] = pack_bf16x2(qv[k][0], qv[k][1]);
        bq[j][k][1] = pack_bf16x2(qv[k][2], qv[k][3]);
      }
    }
  };
  if (S == 1)
    rotate_queries([&](int jp, int) { return scs[jp]; });
  else  // positions differ across columns: each thread its own angles
    rotate_queries([&](int jp, int pos) { return rope_cs_turns_fast(f.turns[jp], pos); });
  // last private row each of this thread's columns j*8 + 2tig + qq sees
  int qlast[QN][2];
#pragma unroll
  for (int j = 0; j < QN; ++j)
#pragma unroll
    for (int qq = 0; qq < 2; ++qq) {
      const int c = j * 8 + 2 * tig + qq;
      qlast[j][qq] = Lb + (c < QC ? c / G : S - 1);
    }

  // running statistics of this thread's columns j*8 + 2tig + qq, and its O^T
  // fragments: dims 16*dt + g8 (+8) for the warp's dim tiles dt
  constexpr int kTilesPerWarp = D / 64;  // 2 (D = 128) or 1 (D = 64)
  float mrun[QN][2], lrun[QN][2];
  float oacc[kTilesPerWarp][QN][4];
#pragma unroll
  for (int j = 0; j < QN; ++j) {
    mrun[j][0] = mrun[j][1] = -INFINITY;
    lrun[j][0] = lrun[j][1] = 0.f;
#pragma unroll
    for (int i = 0; i < kTilesPerWarp; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) oacc[i][j][e] = 0.f;
  }

  for (int c = c0; c < nc; ++c) {
    // chunk c has landed when its slot's phase completes
    const int cr = c - c0;
    const bool ok = mbar_wait(&full[cr % kPrivStages], (cr / kPrivStages) & 1, abort_s, a.status,
                              kDevErrTimeoutTma);
    if (__syncthreads_or(!ok)) break;
    const int k0 = c * CH;
    const int kn = min(CH, nk - k0);
    uint8_t* sKp = smem + (cr % kPrivStages) * L::kStage;
    const uint32_t sK = smem_u32(sKp), sV = sK + L::kTile;
    // staged V rows past the unit's end, up to the next 16-row group: zero
    for (int t = tid; t < (((kn + 15) & ~15) - kn) * (D / 8); t += 128)
      sts_u4(tile_chunk(sV, kn + t / (D / 8), t % (D / 8)), make_uint4(0u, 0u, 0u, 0u));
    // ---- the new tokens (rows Lb .. Lb + S - 1) in this chunk: rotated keys
    // and values into the cache and into the staged copy
    const int r_lo = max(Lb, k_lo + k0), r_hi = min(Lb + S, k_lo + k0 + kn);
    for (int r = r_lo; r < r_hi; ++r) {  // uniform across the block
      const int t = r - Lb, rr = r - (k_lo + k0);
      if (kSpan) {  // (S = 1: scs already holds the angles of p + Lb)
        if (tid < HALF) scs[tid] = rope_cs_turns_fast(f.turns[tid], a.p + r);
        __syncthreads();
      }
      const long long crow = ((static_cast<long long>(b) * a.rows + r) * a.Hkv + g) * D;
      const long long nrow = ((static_cast<long long>(b) * S + t) * a.Hkv + g) * D;
      for (int j = tid; j < HALF; j += 128) {
        float y0, y1;
        rope_pair(__bfloat162float(a.k_new[nrow + j]), __bfloat162float(a.k_new[nrow + j + HALF]),
                  scs[j], y0, y1);
        const __nv_bfloat16 h0 = __float2bfloat16_rn(y0), h1 = __float2bfloat16_rn(y1);
        a.k_cache[crow + j] = h0;
        a.k_cache[crow + j + HALF] = h1;
        const int j1 = j + HALF;
        *reinterpret_cast<__nv_bfloat16*>(sKp + tile_chunk(0, rr, j >> 3) + (j & 7) * 2) = h0;
        *reinterpret_cast<__nv_bfloat16*>(sKp + tile_chunk(0, rr, j1 >> 3) + (j1 & 7) * 2) = h1;
      }
      for (int j = tid; j < D; j += 128) {
        const __nv_bfloat16 v = a.v_new[nrow + j];
        a.v_cache[crow + j] = v;
        *reinterpret_cast<__nv_bfloat16*>(sKp + L::kTile + tile_chunk(0, rr, j >> 3) + (j & 7) * 2) =
            v;
      }
      __syncthreads();  // scs and the patched rows
    }

    // ---- S^T = K Q^T for this warp's 16 keys, every query tile
    float sacc[QN][4];
    {
      // lane -> row address: matrices (rows 0-7,k lo), (rows 8-15,k lo),
      // (rows 0-7,k hi), (rows 8-15,k hi)
      const int row = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int j = 0; j < QN; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[j][e] = 0.f;
      if constexpr (QN == 1) {
        // one query tile: two independent accumulation chains over the d steps
        float s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < D / 16; k += 2) {
          uint32_t af[4], ag[4];
          ldsm_x4(tile_chunk(sK, row, 2 * k + (lane >> 4)), af);
          ldsm_x4(tile_chunk(sK, row, 2 * k + 2 + (lane >> 4)), ag);
          mma_bf16_16816(sacc[0], af, bq[0][k][0], bq[0][k][1]);
          mma_bf16_16816(s2, ag, bq[0][k + 1][0], bq[0][k + 1][1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[0][e] += s2[e];
      } else {
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          uint32_t af[4];
          ldsm_x4(tile_chunk(sK, row, 2 * k + (lane >> 4)), af);
#pragma unroll
          for (int j = 0; j < QN; ++j) mma_bf16_16816(sacc[j], af, bq[j][k][0], bq[j][k][1]);
        }
      }
    }
    // thread holds keys warp*16 + g8 (+8) and columns j*8 + 2tig + qq; a key
    // is visible to a column when it is a row of the unit at or before the
    // column's own position
#pragma unroll
    for (int j = 0; j < QN; ++j)
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        float mx = -INFINITY;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int key = warp * 16 + g8 + 8 * hf;
          float sv = sacc[j][2 * hf + qq] * scale_log2;
          // (the window: row >= the column's position - window + 1)
          const int r = k_lo + k0 + key;
          const bool vis = key < kn && (!kSpan || r <= qlast[j][qq]) &&
                           (W <= 0 || r >= (kSpan ? qlast[j][qq] - W + 1 : lo0));
          sv = vis ? sv : -INFINITY;
          sacc[j][2 * hf + qq] = sv;
          mx = fmaxf(mx, sv);
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        if (g8 == 0) sred[warp * 8 * QN + j * 8 + 2 * tig + qq] = mx;
      }
    __syncthreads();
    float alpha[QN][2];
#pragma unroll
    for (int j = 0; j < QN; ++j)
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        const int q = j * 8 + 2 * tig + qq;
        const float cm = fmaxf(fmaxf(sred[q], sred[8 * QN + q]),
                               fmaxf(sred[16 * QN + q], sred[24 * QN + q]));
        const float mnew = fmaxf(mrun[j][qq], cm);
        // a span column may see no key yet (its position precedes the
        // chunk); with S = 1 every chunk holds a visible key
        const bool none = kSpan && mnew == -INFINITY;
        alpha[j][qq] = none ? 1.f : exp2_approx(mrun[j][qq] - mnew);  // 0 on the first keys
        mrun[j][qq] = mnew;
        float sum = 0.f;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int key = warp * 16 + g8 + 8 * hf;
          const float pv = none ? 0.f : exp2_approx(sacc[j][2 * hf + qq] - mnew);  // 0 if masked
          sum += pv;
          sP[q * L::kPStride + key] = __float2bfloat16_rn(pv);
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        sum += __shfl_xor_sync(0xffffffffu, sum, 8);
        sum += __shfl_xor_sync(0xffffffffu, sum, 16);
        if (g8 == 0) sred[32 * QN + warp * 8 * QN + q] = sum;  // this warp's partial sum
      }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < QN; ++j)
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        const int q = j * 8 + 2 * tig + qq;
        const float cs = (sred[32 * QN + q] + sred[40 * QN + q]) +
                         (sred[48 * QN + q] + sred[56 * QN + q]);
        lrun[j][qq] = lrun[j][qq] * alpha[j][qq] + cs;
      }

    // ---- O^T = alpha O^T + V^T P^T
    const int kgroups = (kn + 15) / 16;
#pragma unroll
    for (int i = 0; i < kTilesPerWarp; ++i) {
      const int dt = warp * kTilesPerWarp + i;
#pragma unroll
      for (int j = 0; j < QN; ++j) {
        oacc[i][j][0] *= alpha[j][0];
        oacc[i][j][1] *= alpha[j][1];
        oacc[i][j][2] *= alpha[j][0];
        oacc[i][j][3] *= alpha[j][1];
      }
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
#pragma unroll
        for (int j = 0; j < QN; ++j) {
          const __nv_bfloat16* pr = sP + (j * 8 + g8) * L::kPStride + 16 * k;
          const uint32_t b0 = *reinterpret_cast<const uint32_t*>(pr + 2 * tig);
          const uint32_t b1 = *reinterpret_cast<const uint32_t*>(pr + 8 + 2 * tig);
          mma_bf16_16816(oacc[i][j], af, b0, b1);
        }
      }
    }
    fence_proxy_async_smem();  // generic writes to the slot before its next copy
    __syncthreads();  // the ring slot, P and the reduction slots are free again
    if (c + kPrivStages < nc) stage(c + kPrivStages);
  }

  // ---- the unit's normalised output and log-sum-exp (log2) per column; a
  // column that saw no row of this unit leaves O = 0 and lse = -inf
  const long long pidx = ((static_cast<long long>(b) * a.Hkv + g) * a.max_units + u) * QC;
#pragma unroll
  for (int j = 0; j < QN; ++j)
#pragma unroll
    for (int qq = 0; qq < 2; ++qq) {
      const int q = j * 8 + 2 * tig + qq;
      if (q >= QC) continue;
      const bool empty = lrun[j][qq] == 0.f;
      const float inv = empty ? 0.f : 1.f / lrun[j][qq];
      float* out = a.priv_part + (pidx + q) * D;
#pragma unroll
      for (int i = 0; i < kTilesPerWarp; ++i) {
        const int dt = warp * kTilesPerWarp + i;
        out[16 * dt + g8] = oacc[i][j][qq] * inv;
        out[16 * dt + g8 + 8] = oacc[i][j][2 + qq] * inv;
      }
      if (warp == 0 && g8 == 0)
        a.priv_lse[pidx + q] = empty ? -INFINITY : mrun[j][qq] + __log2f(lrun[j][qq]);
    }

  // The merge kernel may launch once every CTA of this grid is here.  One CTA
  // also waits for the cartridge grid this one depends on, so that this
  // grid's completion, which the merge kernel waits for, implies both.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (a.n_cart_splits > 0 && g == 0 && b == 0 && u == 0)
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int D, int QN, int kG>
cudaError_t launch_private_dq(const DecodeLaunch& a, const RopeFreqs& f, bool dependent,
                              cudaStream_t st) {
  using L = PrivSmem<D, QN>;
  cudaError_t e = set_smem_once<decode_private_kernel<D, QN, kG>>(L::kAlloc);
  if (e != cudaSuccess) return e;
  // private caches [B, rows, Hkv, d] as (d, Hkv, rows, B), (64, 1, CH, 1)
  // boxes, and (64, 1, 16, 1) boxes for the tails
  CUtensorMap mKs, mVs, mKt, mVt;
  const uint64_t e2 = 2;
  const uint64_t dims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.Hkv),
                            static_cast<uint64_t>(a.rows), static_cast<uint64_t>(a.B)};
  const uint64_t str[3] = {D * e2, static_cast<uint64_t>(a.Hkv) * D * e2,
                           static_cast<uint64_t>(a.rows) * a.Hkv * D * e2};
  const uint32_t box[4] = {64, 1, static_cast<uint32_t>(kPrivCH), 1};
  const uint32_t box16[4] = {64, 1, 16, 1};
  if (!make_bf16_map4(&mKs, a.k_cache, dims, str, box) ||
      !make_bf16_map4(&mVs, a.v_cache, dims, str, box) ||
      !make_bf16_map4(&mKt, a.k_cache, dims, str, box16) ||
      !make_bf16_map4(&mVt, a.v_cache, dims, str, box16))
    return cudaErrorInvalidValue;
  DecodeLaunch pa = a;
  pa.status = device_status_ptr();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.Hkv, a.B, a.max_units);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  const float scale_log2 = a.scale * 1.4426950408889634f;
  return cudaLaunchKernelEx(&cfg, decode_private_kernel<D, QN, kG>, mKs, mVs, mKt, mVt, pa, f,
                            scale_log2);
}

// --------------------------------------------------------------- merge ----
// grid: (Hkv, B*span); block: G warps; warp hh of block (g, b*span + t)
// merges query head g*G + hh of span position t of conversation b:
// cartridge splits s < S (cart_part / cart_lse) and private units
// u < ceil((len+span)/U) (priv_part / priv_lse), all normalised outputs
// with log2-domain log-sum-exps: o = sum_i 2^(lse_i - M) o_i / sum_i
// 2^(lse_i - M).  Lane owns d/32 dims; parts go in rounds of 32 (one log-sum-
// exp per lane), their rows 16 at a time, so a round costs three dependent
// L2 trips.  Runs as the programmatic dependent of the private pass.
template <int D>
__global__ void decode_merge_kernel(DecodeLaunch a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int G = a.Hq / a.Hkv;
  const int g = blockIdx.x, vb = blockIdx.y;
  const int b = vb / a.span, t = vb % a.span, QC = G * a.span;
  const int hh = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = a.B * QC, r = vb * G + hh;
  const int Lb = clamp_len(a.len, b, a.rows - a.span + 1);
  // parts in the sliding window: cartridge splits s_lo .. n_cart_splits - 1
  // (a split wholly before the row's window may not have been written: the
  // cartridge pass skips splits no row of its CTA sees), then private units
  // u_lo .. the last
  int s_lo = 0, u_lo = 0;
  if (a.window > 0) {
    const int lo_c = a.p + Lb + t - a.window + 1;  // first visible key position
    if (lo_c >= a.p)
      s_lo = a.n_cart_splits;
    else if (lo_c > 0 && a.cart_tiles_per_split > 0)
      s_lo = (lo_c / kTile) / a.cart_tiles_per_split;
    const int lo0 = Lb - a.window + 1;  // (t = 0: the parts every column shares)
    u_lo = lo0 > 0 ? lo0 / kDecodeUnit : 0;
  }
  const int S = a.n_cart_splits - s_lo;  // cartridge parts of this row
  const int np = S + (Lb + a.span - 1) / kDecodeUnit + 1 - u_lo;
  const long long pbase =
      (static_cast<long long>(b) * a.Hkv + g) * a.max_units * QC + t * G + hh;
  auto part_row = [&](int pt) -> const float* {
    return pt < S ? a.cart_part + ((static_cast<long long>(s_lo + pt) * a.Hkv + g) * R + r) * D
                  : a.priv_part + (pbase + static_cast<long long>(u_lo + pt - S) * QC) * D;
  };
  auto part_lse = [&](int pt) -> float {
    return pt < S ? __ldcg(a.cart_lse + (static_cast<long long>(s_lo + pt) * a.Hkv + g) * R + r)
                  : __ldcg(a.priv_lse + pbase + static_cast<long long>(u_lo + pt - S) * QC);
  };
  constexpr int PL = D / 32;  // dims per lane: 4 or 2
  float M = -INFINITY, lse0 = -INFINITY;
  for (int p0 = 0; p0 < np; p0 += 32)
    if (p0 + lane < np) {
      const float v = part_lse(p0 + lane);
      if (p0 == 0) lse0 = v;
      M = fmaxf(M, v);
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float num[4] = {0.f, 0.f, 0.f, 0.f}, den = 0.f;
  for (int p0 = 0; p0 < np; p0 += 32) {
    const bool have = p0 + lane < np;
    const float lse = p0 == 0 ? lse0 : (have ? part_lse(p0 + lane) : -INFINITY);
    const float w = have ? exp2_approx(lse - M) : 0.f;
    den += w;
    const int cnt = min(32, np - p0);
    for (int j0 = 0; j0 < cnt; j0 += 16) {
      float4 v[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        v[t] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j0 + t < cnt) {
          const float* src = part_row(p0 + j0 + t);
          if (PL == 4) {
            v[t] = __ldcg(reinterpret_cast<const float4*>(src) + lane);
          } else {
            const float2 t2 = __ldcg(reinterpret_cast<const float2*>(src) + lane);
            v[t] = make_float4(t2.x, t2.y, 0.f, 0.f);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const float wj = __shfl_sync(0xffffffffu, w, (j0 + t) & 31);
        if (j0 + t < cnt) {
          num[0] = fmaf(wj, v[t].x, num[0]);
          num[1] = fmaf(wj, v[t].y, num[1]);
          num[2] = fmaf(wj, v[t].z, num[2]);
          num[3] = fmaf(wj, v[t].w, num[3]);
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  const float inv = 1.f / den;
  __nv_bfloat16* out = a.o + (static_cast<long long>(vb) * a.Hq + g * G + hh) * D + lane * PL;
  if (PL == 4)
    *reinterpret_cast<uint2*>(out) = make_uint2(pack_bf16x2(num[0] * inv, num[1] * inv),
                                                pack_bf16x2(num[2] * inv, num[3] * inv));
  else
    *reinterpret_cast<uint32_t*>(out) = pack_bf16x2(num[0] * inv, num[1] * inv);
}

template <int D>
cudaError_t launch_merge_d(const DecodeLaunch& a, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.Hkv, a.B * a.span, 1);
  cfg.blockDim = dim3(32 * (a.Hq / a.Hkv), 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_merge_kernel<D>, a);
}

}  // namespace

cudaError_t launch_decode(const DecodeLaunch& a, const RopeFreqs& f, cudaStream_t st) {
  const int G = a.Hq / a.Hkv;
  if (a.max_units != (a.rows + kDecodeUnit - 1) / kDecodeUnit) return cudaErrorInvalidValue;
  if (a.span < 1 || G * a.span > kDecodeMaxColumns || a.span > a.rows) return cudaErrorInvalidValue;
  // one trace scope for the whole step: events between the chained kernels
  // would end their overlap
  TraceScope tr("decode", st);
  cudaError_t e = cudaSuccess;
  if (a.p > 0) {
    // raw queries [B, span, Hkv, G, d] as (d, G, Hkv, B*span): a
    // (64, G, 1, 128/G) box is 128 rows r = (b*span + t)*G + hh of one kv head
    CUtensorMap mQ, mKc, mVc;
    const uint64_t e2 = 2;
    const uint64_t qdims[4] = {static_cast<uint64_t>(a.d), static_cast<uint64_t>(G),
                               static_cast<uint64_t>(a.Hkv),
                               static_cast<uint64_t>(a.B) * a.span};
    const uint64_t qstr[3] = {a.d * e2, static_cast<uint64_t>(G) * a.d * e2,
                              static_cast<uint64_t>(a.Hkv) * G * a.d * e2};
    const uint32_t qbox[4] = {64, static_cast<uint32_t>(G), 1, static_cast<uint32_t>(kTile / G)};
    if (!make_bf16_map4(&mQ, a.q, qdims, qstr, qbox) ||
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
    l.n_rows = a.B * a.span * G;
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
    // f32 partials [S, Hkv, R, d] as (d, R, Hkv, S): 32 x 32 blocks by TMA
    CUtensorMap mOd;
    const int R = a.B * a.span * G;
    const uint64_t e4 = 4;
    const uint64_t odims[4] = {static_cast<uint64_t>(a.d), static_cast<uint64_t>(R),
                               static_cast<uint64_t>(a.Hkv),
                               static_cast<uint64_t>(a.n_cart_splits)};
    const uint64_t ostr[3] = {a.d * e4, static_cast<uint64_t>(R) * a.d * e4,
                              static_cast<uint64_t>(a.Hkv) * R * a.d * e4};
    const uint32_t obox[4] = {32, 32, 1, 1};
    if (!make_f32_map4(&mOd, a.cart_part, odims, ostr, obox)) return cudaErrorInvalidValue;
    l.mO32 = &mOd;
    l.lse = const_cast<float*>(a.cart_lse);
    l.decode = true;
    l.pdl = false;
    l.dec_len = a.len;
    l.dec_B = a.B * a.span;
    l.dec_G = G;
    l.dec_rows = a.rows;
    l.dec_s = a.span;
    l.window = a.window;
    l.freqs = &f;
    e = launch_fwd(l, st);
    if (e != cudaSuccess) return e;
  }
  const bool dep = a.p > 0;
  e = cudaErrorInvalidValue;
  const int qn = (G * a.span + 7) / 8;  // 8-column query tiles of the private pass
  if (a.span == 1) {  // the single-token step: G as a constant
    switch (G * (a.d == 128 ? 1 : -1)) {
      case 1: e = launch_private_dq<128, 1, 1>(a, f, dep, st); break;
      case 2: e = launch_private_dq<128, 1, 2>(a, f, dep, st); break;
      case 4: e = launch_private_dq<128, 1, 4>(a, f, dep, st); break;
      case 8: e = launch_private_dq<128, 1, 8>(a, f, dep, st); break;
      case -1: e = launch_private_dq<64, 1, 1>(a, f, dep, st); break;
      case -2: e = launch_private_dq<64, 1, 2>(a, f, dep, st); break;
      case -4: e = launch_private_dq<64, 1, 4>(a, f, dep, st); break;
      case -8: e = launch_private_dq<64, 1, 8>(a, f, dep, st); break;
    }
  } else if (a.d == 128) {
    switch (qn) {
      case 1: e = launch_private_dq<128, 1, 0>(a, f, dep, st); break;
      case 2: e = launch_private_dq<128, 2, 0>(a, f, dep, st); break;
      case 3: e = launch_private_dq<128, 3, 0>(a, f, dep, st); break;
      case 4: e = launch_private_dq<128, 4, 0>(a, f, dep, st); break;
    }
  } else if (a.d == 64) {
    switch (qn) {
      case 1: e = launch_private_dq<64, 1, 0>(a, f, dep, st); break;
      case 2: e = launch_private_dq<64, 2, 0>(a, f, dep, st); break;
      case 3: e = launch_private_dq<64, 3, 0>(a, f, dep, st); break;
      case 4: e = launch_private_dq<64, 4, 0>(a, f, dep, st); break;
    }
  }
  if (e != cudaSuccess) return e;
  return a.d == 128 ? launch_merge_d<128>(a, st) : launch_merge_d<64>(a, st);
}

}  // namespace cart
