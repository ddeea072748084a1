// misc.cu -- bandwidth-bound helper kernels of the cartridge-attention path:
//   * the cartridge cache write (f32 leaves -> cache dtype), which also makes
//     the bf16 shadow the tensor-core kernels read;
//   * the RoPE cos/sin table for a run of positions (fp64 angle reduction);
//   * rotation of real-token Q/K rows at positions p + i into bf16;
//   * the backward's per-row D = rowsum(dO * O) and log2-domain lse.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "internal.cuh"
#include "ptx.cuh"

namespace cart {
namespace {

constexpr int kThreads = 256;

int grid_for(long long work, int per_block = kThreads) {
  long long g = (work + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > 152 * 64) g = 152 * 64;  // grid-stride loops cover the rest
  return static_cast<int>(g);
}

// ---------------------------------------------------------- cache write ----
// One thread converts kCacheBatch runs of 8 consecutive values of a
// cartridge row, one grid stride apart, with all their loads issued before
// any store; the second tensor (src1 -> dst1, may be absent) continues the
// index range of the first, so K and V go in one launch.
constexpr int kCacheBatch = 4;

__global__ void write_to_cache_kernel(const float* __restrict__ src0, void* __restrict__ dst0,
                                      const float* __restrict__ src1, void* __restrict__ dst1,
                                      int p, int row_elems, long long row_stride, int dst_row0,
                                      int dst_bf16) {
  pdl_wait();
  pdl_release();
  const int vec_per_row = row_elems / 8;
  const long long per = static_cast<long long>(p) * vec_per_row;
  const long long total = src1 ? 2 * per : per;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long t0 = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t0 < total;
       t0 += stride * kCacheBatch) {
    float4 a[kCacheBatch], b[kCacheBatch];
#pragma unroll
    for (int u = 0; u < kCacheBatch; ++u) {
      const long long t1 = t0 + u * stride;
      if (t1 < total) {
        const bool second = t1 >= per;
        const long long t = second ? t1 - per : t1;
        const float4* s = reinterpret_cast<const float4*>((second ? src1 : src0) + t * 8);
        a[u] = __ldg(s);
        b[u] = __ldg(s + 1);
      }
    }
#pragma unroll
    for (int u = 0; u < kCacheBatch; ++u) {
      const long long t1 = t0 + u * stride;
      if (t1 >= total) break;
      const bool second = t1 >= per;
      const long long t = second ? t1 - per : t1;
      void* dst = second ? dst1 : dst0;
      const int r = static_cast<int>(t / vec_per_row);
      const int c = static_cast<int>(t % vec_per_row) * 8;
      const long long off = static_cast<long long>(dst_row0 + r) * row_stride + c;
      if (dst_bf16) {
        uint4 o;
        o.x = pack_bf16x2(a[u].x, a[u].y);
        o.y = pack_bf16x2(a[u].z, a[u].w);
        o.z = pack_bf16x2(b[u].x, b[u].y);
        o.w = pack_bf16x2(b[u].z, b[u].w);
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(dst) + off) = o;
      } else {
        float4* d = reinterpret_cast<float4*>(static_cast<float*>(dst) + off);
        d[0] = a[u];
        d[1] = b[u];
      }
    }
  }
}

// ----------------------------------------------------------- rope table ----
// table[i * (d/2) + j] = (cos, sin) of (pos0 + i) * inv_freq[j].  The angle
// is formed and reduced modulo 2*pi in fp64 (two-part 2*pi); the reduced
// angle is split into an f32 head and tail so that cos/sin of the head plus
// a first-order tail correction keep the table accurate to ~1e-7.
__device__ __forceinline__ float2 rope_table_entry(double pos, double inv_freq) {
  const double ang = pos * inv_freq;
  const double kTwoPiHi = 6.283185307179586232;   // nearest double to 2*pi
  const double kTwoPiLo = 2.4492935982947064e-16;  // 2*pi - kTwoPiHi
  const double k = rint(ang * 0.15915494309189535);
  double r = fma(-k, kTwoPiHi, ang);
  r = fma(-k, kTwoPiLo, r);
  const float rh = static_cast<float>(r);
  const float rl = static_cast<float>(r - static_cast<double>(rh));
  float s, c;
  sincosf(rh, &s, &c);
  return make_float2(c - s * rl, s + c * rl);
}

__global__ void rope_table_kernel(float2* __restrict__ table, int pos0, int npos, int half,
                                  const RopeFreqs f, int* sched) {
  if (sched && blockIdx.x == 0 && threadIdx.x == 0) *sched = 0;
  const long long total = static_cast<long long>(npos) * half;
  for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < total;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int i = static_cast<int>(t / half), j = static_cast<int>(t % half);
    table[t] = rope_table_entry(static_cast<double>(pos0 + i), f.inv_freq[j]);
  }
}

// ----------------------------------------------------------- rope rows ----
// x [B, n, H, d] -> out bf16 same layout.  One thread owns 8 consecutive
// pair indices j..j+7 of one row: elements j.. and j+d/2.. .
// Packed layout (cu given): the same (b, i < n) index space, tokens past a
// segment's end skipped, row (g0 + i) * H + h.
template <bool kF32>
__global__ void rope_rows_kernel(const void* __restrict__ xv, __nv_bfloat16* __restrict__ out,
                                 const float2* __restrict__ table, int B, int n, int H, int d,
                                 int rotate, const int* __restrict__ cu, int ntok) {
  const int half = d / 2;
  const int chunks = half / 8;
  const long long total = static_cast<long long>(B) * n * H * chunks;
  for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < total;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long bih = t / chunks;  // (b * n + i) * H + h
    const int j0 = static_cast<int>(t % chunks) * 8;
    const int i = static_cast<int>((bih / H) % n);
    const SeqRows sr = seq_rows(cu, ntok, n, static_cast<int>(bih / (static_cast<long long>(H) * n)));
    if (i >= sr.len) continue;
    const long long row = (static_cast<long long>(sr.g0) + i) * H + bih % H;
    float x0[8], x1[8];
    if (kF32) {
      const float* x = static_cast<const float*>(xv) + row * d;
      const float4* a = reinterpret_cast<const float4*>(x + j0);
      const float4* b = reinterpret_cast<const float4*>(x + j0 + half);
      float4 a0 = __ldg(a), a1 = __ldg(a + 1), b0 = __ldg(b), b1 = __ldg(b + 1);
      x0[0] = a0.x; x0[1] = a0.y; x0[2] = a0.z; x0[3] = a0.w;
      x0[4] = a1.x; x0[5] = a1.y; x0[6] = a1.z; x0[7] = a1.w;
      x1[0] = b0.x; x1[1] = b0.y; x1[2] = b0.z; x1[3] = b0.w;
      x1[4] = b1.x; x1[5] = b1.y; x1[6] = b1.z; x1[7] = b1.w;
    } else {
      const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(xv) + row * d;
      uint4 a = __ldg(reinterpret_cast<const uint4*>(x + j0));
      uint4 b = __ldg(reinterpret_cast<const uint4*>(x + j0 + half));
      const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float2 fa = __bfloat1622float2(pa[e]);
        float2 fb = __bfloat1622float2(pb[e]);
        x0[2 * e] = fa.x; x0[2 * e + 1] = fa.y;
        x1[2 * e] = fb.x; x1[2 * e + 1] = fb.y;
      }
    }
    float y0[8], y1[8];
    if (rotate) {
      const float2* tb = table + static_cast<long long>(i) * half + j0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        rope_pair(x0[e], x1[e], __ldg(tb + e), y0[e], y1[e]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) { y0[e] = x0[e]; y1[e] = x1[e]; }
    }
    uint4 o0, o1;
    o0.x = pack_bf16x2(y0[0], y0[1]); o0.y = pack_bf16x2(y0[2], y0[3]);
    o0.z = pack_bf16x2(y0[4], y0[5]); o0.w = pack_bf16x2(y0[6], y0[7]);
    o1.x = pack_bf16x2(y1[0], y1[1]); o1.y = pack_bf16x2(y1[2], y1[3]);
    o1.z = pack_bf16x2(y1[4], y1[5]); o1.w = pack_bf16x2(y1[6], y1[7]);
    __nv_bfloat16* orow = out + row * d;
    *reinterpret_cast<uint4*>(orow + j0) = o0;
    *reinterpret_cast<uint4*>(orow + j0 + half) = o1;
  }
}

// ------------------------------------------------------- training prep ----
// Everything the training kernels need before they start, for bf16 inputs,
// in one launch over blocks of ppc (1..kPrepPos) real-token positions i:
//   * the RoPE table rows of positions p + i (all-f32 angle reduction, see
//     rope_cs_turns; positions must stay below 2^24);
//   * K rotated at p + i for every (sequence, kv head), and Q for every
//     (sequence, head) when qr is given (the forward rotates Q itself);
//   * the bf16 copies of f32 cartridge leaves when cast.kc is given;
//   * with o given (backward): the negated row vectors -D = -rowsum(dO * O)
//     and -lse * log2(e) in [B, Hq, npad] (stored negated so that the
//     backward kernels add them with packed two-lane arithmetic), padding
//     rows npad > i >= n set to -D = 0 and -lse2 = -inf.
// Packed layout (cu given, see SeqRows): sequence b is segment b, its token
// i at flat row cu[b] + i; positions past a segment's end are padding of
// the row vectors; block 0 also checks the segment table.
constexpr int kPrepPos = 4;

__device__ __forceinline__ void rotate_chunk8(const __nv_bfloat16* x, __nv_bfloat16* y,
                                              const float2* cs, int half) {
  // elements j0..j0+7 and their rotate-half partners j0+half.. ; cs = the
  // 8 (cos, sin) of these pairs
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(x));
  const uint4 b = __ldg(reinterpret_cast<const uint4*>(x + half));
  const uint32_t pa[4] = {a.x, a.y, a.z, a.w};
  const uint32_t pb[4] = {b.x, b.y, b.z, b.w};
  uint32_t ya[4], yb[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 fa = bf16x2_to_float2(pa[e]), fb = bf16x2_to_float2(pb[e]);
    float y0a, y1a, y0b, y1b;
    rope_pair(fa.x, fb.x, cs[2 * e], y0a, y1a);
    rope_pair(fa.y, fb.y, cs[2 * e + 1], y0b, y1b);
    ya[e] = pack_bf16x2(y0a, y0b);
    yb[e] = pack_bf16x2(y1a, y1b);
  }
  *reinterpret_cast<uint4*>(y) = make_uint4(ya[0], ya[1], ya[2], ya[3]);
  *reinterpret_cast<uint4*>(y + half) = make_uint4(yb[0], yb[1], yb[2], yb[3]);
}

template <bool kPacked>
__global__ void __launch_bounds__(kThreads) train_prep_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
    __nv_bfloat16* __restrict__ qr, __nv_bfloat16* __restrict__ kr, float2* __restrict__ table,
    const RopeFreqs f, int p, int B, int n, int Hq, int Hkv, int d,
    const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
    const float* __restrict__ lse, float* __restrict__ nDvec, float* __restrict__ nlse2, int npad,
    int ppc, const int* __restrict__ cu_arg, int ntok, int* sched, uint32_t* status,
    const CartCast cast) {
  const int* const cu = kPacked ? cu_arg : nullptr;
  pdl_wait();
  pdl_release();
  if (sched && blockIdx.x == 0 && threadIdx.x == 0) *sched = 0;
  __shared__ float2 cs[kPrepPos][kMaxHeadDim / 2];
  const int half = d / 2, chunks = half / 8;
  if (cu && blockIdx.x == 0) {
    // the packed table: rising from 0 to ntok, no segment longer than n
    bool bad = threadIdx.x == 0 && (__ldg(cu) != 0 || __ldg(cu + B) != ntok);
    for (int s = threadIdx.x; s < B; s += blockDim.x) {
      const int len = __ldg(cu + s + 1) - __ldg(cu + s);
      bad |= len < 0 || len > n;
    }
    if (bad && status) atomicOr(status, kDevErrSegments);
  }
  const int i0 = blockIdx.x * ppc;
  const int np = max(0, min(ppc, n - i0));  // real positions in this block
  if (table || kr || qr) {  // (the backward vectors alone need no angles)
    for (int t = threadIdx.x; t < np * half; t += blockDim.x) {
      const int pl = t / half, j = t % half;
      const float2 v = rope_cs_turns(f.turns[j], p + i0 + pl);
      cs[pl][j] = v;
      if (table) table[static_cast<long long>(i0 + pl) * half + j] = v;
    }
    __syncthreads();
  }
  // rotations: task = ((pos, b), head, chunk)
  auto rotate_all = [&](const __nv_bfloat16* x, __nv_bfloat16* y, int H) {
    const int tasks = np * B * H * chunks;
#pragma unroll 4
    for (int t = threadIdx.x; t < tasks; t += blockDim.x) {
      const int jc = t % chunks;
      const int h = (t / chunks) % H;
      const int pb = t / (chunks * H);
      const int b = pb % B, pl = pb / B;
      const SeqRows sr = seq_rows(cu, ntok, n, b);
      if (kPacked && i0 + pl >= sr.len) continue;  // past a segment's end
      const long long row = (static_cast<long long>(sr.g0) + i0 + pl) * H + h;
      rotate_chunk8(x + row * d + jc * 8, y + row * d + jc * 8, &cs[pl][jc * 8], half);
    }
  };
  if (kr) rotate_all(k, kr, Hkv);
  if (qr) rotate_all(q, qr, Hq);
  if (cast.kc) {
    // the cartridge leaves' bf16 copies: eight values per thread and step
    // over the whole grid, K's then V's
    const long long per = cast.elems / 8, all = 2 * per;
    for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < all;
         t += static_cast<long long>(gridDim.x) * blockDim.x) {
      const bool second = t >= per;
      const long long u = second ? t - per : t;
      const float4* src = reinterpret_cast<const float4*>((second ? cast.vc : cast.kc) + u * 8);
      const float4 a = __ldg(src), b = __ldg(src + 1);
      *reinterpret_cast<uint4*>((second ? cast.vcb : cast.kcb) + u * 8) =
          make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                     pack_bf16x2(b.z, b.w));
    }
  }
  if (!o) return;
  // -D and -lse2: 8 lanes per (b, i, h) row, 4 rows per warp (uniform trip count)
  const int lane8 = threadIdx.x & 7;
  const int rows = np * B * Hq;
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int rows_pad = ((rows + 3) / 4) * 4;
#pragma unroll 2
  for (int base = warp * 4; base < rows_pad; base += nwarps * 4) {
    const int rr = base + ((threadIdx.x & 31) >> 3);
    float acc = 0.f;
    int h = 0, b = 0, pl = 0;
    SeqRows sr{};
    bool live = false;  // a token of its sequence (not past a packed segment's end)
    if (rr < rows) {
      h = rr % Hq;
      b = (rr / Hq) % B;
      pl = rr / (Hq * B);
      sr = seq_rows(cu, ntok, n, b);
      live = !kPacked || i0 + pl < sr.len;
    }
    float lv = 0.f;
    if (live) {
      // every load of the row in flight at once (d is 64 or 128: one or two
      // 16-byte pieces of o and of dO per lane), the lse with them
      const long long row = (static_cast<long long>(sr.g0) + i0 + pl) * Hq + h;
      const uint4* po = reinterpret_cast<const uint4*>(o + row * d + lane8 * 8);
      const uint4* pg = reinterpret_cast<const uint4*>(dout + row * d + lane8 * 8);
      if (lane8 == 0) lv = __ldg(lse + lse_index(cu, ntok, n, Hq, b, h, sr, i0 + pl));
      uint4 ov[2], gv[2];
      ov[0] = __ldg(po);
      gv[0] = __ldg(pg);
      ov[1] = d > 64 ? __ldg(po + 8) : make_uint4(0u, 0u, 0u, 0u);
      gv[1] = d > 64 ? __ldg(pg + 8) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const uint32_t a4[4] = {ov[k].x, ov[k].y, ov[k].z, ov[k].w};
        const uint32_t g4[4] = {gv[k].x, gv[k].y, gv[k].z, gv[k].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 fo = bf16x2_to_float2(a4[e]), fg = bf16x2_to_float2(g4[e]);
          acc += fo.x * fg.x + fo.y * fg.y;
        }
      }
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    if (lane8 == 0 && rr < rows) {
      const long long bh = static_cast<long long>(b) * Hq + h;
      nDvec[bh * npad + i0 + pl] = live ? -acc : 0.f;
      nlse2[bh * npad + i0 + pl] = live ? lv * -1.4426950408889634f : -INFINITY;
    }
  }
  // padding rows of this block's positions
  const int pad_lo = max(i0, n), pad_hi = min(i0 + ppc, npad);
  for (int t = threadIdx.x; t < B * Hq * max(0, pad_hi - pad_lo); t += blockDim.x) {
    const int i = pad_lo + t % (pad_hi - pad_lo);
    const long long bh = t / (pad_hi - pad_lo);
    nDvec[bh * npad + i] = 0.f;
    nlse2[bh * npad + i] = -INFINITY;
  }
}

// ------------------------------------------------------------- bwd vec ----
// Per query row of the backward, in [B, Hq, npad] layout (npad >= n, rows
// n..npad-1 are padding that reads as "no probability mass"):
//   nDvec[b, h, i] = -sum_c dO[b,i,h,c] * O[b,i,h,c]  (0 for padding)
//   nlse2[b, h, i] = -lse[b, h, i] * log2(e)          (-inf for padding)
// 8 lanes per row, 4 rows per warp; the loop trip count is uniform across
// the warp.
// Packed layout (cu given): the same (b, i < n, h) index space; tokens past
// a segment's end are padding.
template <bool kF32>
__global__ void bwd_vec_kernel(const void* __restrict__ ov, const void* __restrict__ dov,
                               const float* __restrict__ lse, float* __restrict__ nDvec,
                               float* __restrict__ nlse2, int B, int n, int npad, int Hq, int d,
                               const int* __restrict__ cu, int ntok) {
  const long long rows = static_cast<long long>(B) * n * Hq;
  const int lane8 = threadIdx.x & 7;
  const int group = (threadIdx.x & 31) >> 3;
  const long long tid = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long warp_id = tid >> 5;
  const long long warps = nthreads >> 5;
  for (long long base = warp_id * 4; base < rows; base += warps * 4) {
    const long long bih = base + group;  // (b * n + i) * Hq + h
    float acc = 0.f;
    int h = 0, i = 0, b = 0;
    SeqRows sr{};
    bool live = false;
    long long row = 0;
    if (bih < rows) {
      h = static_cast<int>(bih % Hq);
      i = static_cast<int>((bih / Hq) % n);
      b = static_cast<int>(bih / (static_cast<long long>(Hq) * n));
      sr = seq_rows(cu, ntok, n, b);
      live = i < sr.len;
      row = (static_cast<long long>(sr.g0) + i) * Hq + h;
    }
    if (live) {
      for (int c = lane8 * 8; c < d; c += 64) {
        if (kF32) {
          const float4* o =
              reinterpret_cast<const float4*>(static_cast<const float*>(ov) + row * d + c);
          const float4* g =
              reinterpret_cast<const float4*>(static_cast<const float*>(dov) + row * d + c);
          float4 o0 = __ldg(o), o1 = __ldg(o + 1), g0 = __ldg(g), g1 = __ldg(g + 1);
          acc += o0.x * g0.x + o0.y * g0.y + o0.z * g0.z + o0.w * g0.w;
          acc += o1.x * g1.x + o1.y * g1.y + o1.z * g1.z + o1.w * g1.w;
        } else {
          uint4 o = __ldg(reinterpret_cast<const uint4*>(
              static_cast<const __nv_bfloat16*>(ov) + row * d + c));
          uint4 g = __ldg(reinterpret_cast<const uint4*>(
              static_cast<const __nv_bfloat16*>(dov) + row * d + c));
          const __nv_bfloat162* po = reinterpret_cast<const __nv_bfloat162*>(&o);
          const __nv_bfloat162* pg = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float2 fo = __bfloat1622float2(po[e]);
            float2 fg = __bfloat1622float2(pg[e]);
            acc += fo.x * fg.x + fo.y * fg.y;
          }
        }
      }
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    if (lane8 == 0 && bih < rows) {
      const long long bh = static_cast<long long>(b) * Hq + h;
      nDvec[bh * npad + i] = live ? -acc : 0.f;
      nlse2[bh * npad + i] =
          live ? __ldg(lse + lse_index(cu, ntok, n, Hq, b, h, sr, i)) * -1.4426950408889634f
               : -INFINITY;
    }
  }
  const long long pad_rows = static_cast<long long>(B) * Hq * (npad - n);
  for (long long t = tid; t < pad_rows; t += nthreads) {
    const long long bh = t / (npad - n);
    const int i = n + static_cast<int>(t % (npad - n));
    nDvec[bh * npad + i] = 0.f;
    nlse2[bh * npad + i] = -INFINITY;
  }
}

}  // namespace

RopeFreqs make_rope_freqs(int d, double theta) {
  RopeFreqs f{};
  for (int j = 0; j < d / 2 && j < kMaxHeadDim / 2; ++j) {
    f.inv_freq[j] = std::pow(theta, -2.0 * static_cast<double>(j) / static_cast<double>(d));
    const double t = f.inv_freq[j] / 6.283185307179586476925;
    const float hi = static_cast<float>(t);
    f.turns[j] = make_float2(hi, static_cast<float>(t - static_cast<double>(hi)));
  }
  return f;
}

cudaError_t launch_write_to_cache(const float* src0, void* dst0, const float* src1, void* dst1,
                                  int p, int row_elems, long long row_stride, int dst_row0,
                                  bool dst_bf16, cudaStream_t st) {
  if (p <= 0) return cudaSuccess;
  if (!src0) {  // only the second tensor
    src0 = src1;
    dst0 = dst1;
    src1 = nullptr;
  }
  if (!src0) return cudaSuccess;
  const long long work = static_cast<long long>(p) * (row_elems / 8) * (src1 ? 2 : 1);
  TraceScope tr("write_to_cache", st);
  return launch_dependent(write_to_cache_kernel,
                          dim3(grid_for((work + kCacheBatch - 1) / kCacheBatch)), dim3(kThreads), 0,
                          st, src0, dst0, src1, src1 ? dst1 : nullptr, p, row_elems, row_stride,
                          dst_row0, dst_bf16 ? 1 : 0);
}

cudaError_t launch_train_prep(const __nv_bfloat16* q, const __nv_bfloat16* k, __nv_bfloat16* qr,
                              __nv_bfloat16* kr, float2* table, const RopeFreqs& f, int p, int B,
                              int n, int Hq, int Hkv, int d, const __nv_bfloat16* o,
                              const __nv_bfloat16* dout, const float* lse, float* nDvec,
                              float* nlse2, int npad, const int* cu, int total, int* sched,
                              cudaStream_t st, const CartCast& cast) {
  const int span = o ? max(n, npad) : n;
  // positions per CTA: enough CTAs for about eight per SM, at most kPrepPos
  const int ppc = max(1, min(kPrepPos, (span + 152 * 8 - 1) / (152 * 8)));
  const int grid = (span + ppc - 1) / ppc;
  if (grid <= 0) return cudaSuccess;
  TraceScope tr(o ? "bwd_prep" : "fwd_prep", st);
  auto* kern = cu ? train_prep_kernel<true> : train_prep_kernel<false>;
  return launch_dependent(kern, dim3(grid), dim3(kThreads), 0, st, q, k, qr, kr, table, f, p, B, n,
                          Hq, Hkv, d, o, dout, lse, nDvec, nlse2, npad, ppc, cu, total, sched,
                          device_status_ptr(), cast);
}

cudaError_t launch_rope_table(float2* table, int pos0, int npos, int d, const RopeFreqs& f,
                              int* sched, cudaStream_t st) {
  if (npos <= 0 && !sched) return cudaSuccess;
  const long long work = static_cast<long long>(npos > 0 ? npos : 0) * (d / 2);
  TraceScope tr("rope_table", st);
  rope_table_kernel<<<grid_for(work), kThreads, 0, st>>>(table, pos0, npos, d / 2, f, sched);
  return cudaGetLastError();
}

cudaError_t launch_rope_rows(const void* x, bool x_f32, __nv_bfloat16* out, const float2* table,
                             int B, int n, int H, int d, bool rotate, const int* cu, int total,
                             cudaStream_t st) {
  const long long work = static_cast<long long>(B) * n * H * (d / 16);
  if (work <= 0) return cudaSuccess;
  TraceScope tr(rotate ? "rope_rows" : "to_bf16", st);
  if (x_f32)
    rope_rows_kernel<true><<<grid_for(work), kThreads, 0, st>>>(x, out, table, B, n, H, d,
                                                                rotate ? 1 : 0, cu, total);
  else
    rope_rows_kernel<false><<<grid_for(work), kThreads, 0, st>>>(x, out, table, B, n, H, d,
                                                                 rotate ? 1 : 0, cu, total);
  return cudaGetLastError();
}

cudaError_t launch_bwd_vec(const void* o, const void* dout, bool f32, const float* lse,
                           float* nDvec, float* nlse2, int B, int n, int npad, int Hq, int d,
                           const int* cu, int total, cudaStream_t st) {
  const long long rows = static_cast<long long>(B) * n * Hq;
  if (rows <= 0 || npad < n) return cudaSuccess;
  const int grid = grid_for(rows * 8);  // 8 threads per row
  TraceScope tr("bwd_vec", st);
  if (f32)
    bwd_vec_kernel<true><<<grid, kThreads, 0, st>>>(o, dout, lse, nDvec, nlse2, B, n, npad, Hq, d,
                                                    cu, total);
  else
    bwd_vec_kernel<false><<<grid, kThreads, 0, st>>>(o, dout, lse, nDvec, nlse2, B, n, npad, Hq, d,
                                                     cu, total);
  return cudaGetLastError();
}

}  // namespace cart
