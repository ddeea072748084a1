// decode.cu -- q_seq = 1 decode of B conversations behind one shared cartridge.
// (Cartridges guide, "Semantics", serving bullet: decoding continues at
// position p with the training-time layout.)
//
// Work split:
//   prep      per conversation: rotate the new query and key at position
//             p + len[b] (fp64 angle reduction once per conversation, shared
//             by all heads), append the rotated key / value at private row
//             len[b], and lay the rotated queries out per kv head as
//             [B*G rows, Hkv, d] so that the cartridge part runs as ONE
//             tensor-core problem per kv head (rows of all conversations
//             batched into M) -- see fwd.cu.
//   private   split-KV over each conversation's own rows 0..len[b]:
//             bandwidth-bound, CUDA cores, 16-byte loads, warp shuffles.
//   combine   merges the cartridge splits and the private chunks of every
//             (conversation, head) with their log-sum-exps.
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
// grid: B blocks; block: 128 threads.
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
  // rows: Hq query heads, then Hkv new keys, then Hkv new values (copy only)
  const int chunks = half / 8;  // 8 pair indices per task
  const int tasks = (a.Hq + a.Hkv) * chunks + a.Hkv * (d / 8);
  for (int t = threadIdx.x; t < tasks; t += blockDim.x) {
    if (t < (a.Hq + a.Hkv) * chunks) {
      const int hrow = t / chunks, j0 = (t % chunks) * 8;
      const __nv_bfloat16* src;
      __nv_bfloat16* dst;
      if (hrow < a.Hq) {
        const int h = hrow, g = h / G, hh = h % G;
        src = a.q + (static_cast<long long>(b) * a.Hq + h) * d;
        dst = a.q_rot + (static_cast<long long>(b * G + hh) * a.Hkv + g) * d;
      } else {
        const int g = hrow - a.Hq;
        src = a.k_new + (static_cast<long long>(b) * a.Hkv + g) * d;
        dst = a.k_cache + ((static_cast<long long>(b) * a.rows + L) * a.Hkv + g) * d;
      }
      float x0[8], x1[8];
      bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(src + j0)), x0);
      bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(src + j0 + half)), x1);
      uint4 o0, o1;
      float y0[8], y1[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float2 c = cs[j0 + e];
        y0[e] = x0[e] * c.x - x1[e] * c.y;
        y1[e] = x1[e] * c.x + x0[e] * c.y;
      }
      o0 = make_uint4(pack_bf16x2(y0[0], y0[1]), pack_bf16x2(y0[2], y0[3]),
                      pack_bf16x2(y0[4], y0[5]), pack_bf16x2(y0[6], y0[7]));
      o1 = make_uint4(pack_bf16x2(y1[0], y1[1]), pack_bf16x2(y1[2], y1[3]),
                      pack_bf16x2(y1[4], y1[5]), pack_bf16x2(y1[6], y1[7]));
      *reinterpret_cast<uint4*>(dst + j0) = o0;
      *reinterpret_cast<uint4*>(dst + j0 + half) = o1;
    } else {
      const int u = t - (a.Hq + a.Hkv) * chunks;
      const int g = u / (d / 8), c0 = (u % (d / 8)) * 8;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(
          a.v_new + (static_cast<long long>(b) * a.Hkv + g) * d + c0));
      *reinterpret_cast<uint4*>(a.v_cache + ((static_cast<long long>(b) * a.rows + L) * a.Hkv + g) * d +
                                c0) = v;
    }
  }
}

// ------------------------------------------------------------- private ----
// grid: (chunks, Hkv, B); block: 128 threads (4 warps).  Keys of the chunk:
// private rows [c*CH, min((c+1)*CH, len+1)).  Output per query head of the
// group: unnormalised acc[d] against the chunk's own max m (log2 domain) and
// sum l.
template <int D, int G, int CH>
__global__ void __launch_bounds__(128) decode_private_kernel(DecodeLaunch a, float scale_log2) {
  constexpr int DL = D / 8;    // dims per lane in the score phase (8 lanes per key)
  constexpr int DV = D / 32;   // dims per lane in the PV phase
  __shared__ float s_q[G][D];
  __shared__ float s_p[CH][G];
  __shared__ float s_red[4][G][D];
  const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int L = clamp_len(a.len, b, a.rows);
  const int k0 = c * CH;
  if (k0 > L) return;  // whole chunk beyond this conversation's rows
  const int kn = min(CH, L + 1 - k0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row_stride = static_cast<long long>(a.Hkv) * D;
  const __nv_bfloat16* kbase = a.k_cache + (static_cast<long long>(b) * a.rows + k0) * row_stride + g * D;
  const __nv_bfloat16* vbase = a.v_cache + (static_cast<long long>(b) * a.rows + k0) * row_stride + g * D;

  for (int t = threadIdx.x; t < G * D; t += 128) {
    const int hh = t / D, e = t % D;
    s_q[hh][e] = __bfloat162float(a.q_rot[(static_cast<long long>(b * G + hh) * a.Hkv + g) * D + e]);
  }
  __syncthreads();

  // ---- scores: 8 lanes per key, 4 keys per warp step, 16 keys per CTA step
  {
    const int sub = lane & 7, kq = lane >> 3;
    float qr[G][DL];
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
#pragma unroll
      for (int e = 0; e < DL; ++e) qr[hh][e] = s_q[hh][sub * DL + e];
    for (int kk0 = warp * 4; kk0 < kn; kk0 += 16) {
      const int kk = kk0 + kq;
      float dot[G];
#pragma unroll
      for (int hh = 0; hh < G; ++hh) dot[hh] = 0.f;
      if (kk < kn) {
        const __nv_bfloat16* kr = kbase + static_cast<long long>(kk) * row_stride + sub * DL;
#pragma unroll
        for (int v8 = 0; v8 < DL / 8; ++v8) {
          float kf[8];
          bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(kr + v8 * 8)), kf);
#pragma unroll
          for (int hh = 0; hh < G; ++hh)
#pragma unroll
            for (int e = 0; e < 8; ++e) dot[hh] = fmaf(qr[hh][v8 * 8 + e], kf[e], dot[hh]);
        }
      }
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        float v = dot[hh];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        dot[hh] = v;
      }
      if (sub == 0 && kk < kn) {
#pragma unroll
        for (int hh = 0; hh < G; ++hh) s_p[kk][hh] = dot[hh] * scale_log2;
      }
    }
  }
  __syncthreads();

  // ---- chunk softmax statistics: warp w handles heads w, w+4, ...
  float* ml = a.priv_ml;
  const int n_chunks = (a.rows + CH - 1) / CH;
  const long long part_idx = ((static_cast<long long>(b) * a.Hkv + g) * n_chunks + c) * G;
  for (int hh = warp; hh < G; hh += 4) {
    float m = -INFINITY;
    for (int kk = lane; kk < kn; kk += 32) m = fmaxf(m, s_p[kk][hh]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.f;
    for (int kk = lane; kk < kn; kk += 32) {
      const float pv = exp2_approx(s_p[kk][hh] - m);
      s_p[kk][hh] = pv;
      l += pv;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) {
      ml[(part_idx + hh) * 2 + 0] = m;
      ml[(part_idx + hh) * 2 + 1] = l;
    }
  }
  __syncthreads();

  // ---- P V: warp w takes keys w, w+4, ...; lane owns DV dims
  float acc[G][DV];
#pragma unroll
  for (int hh = 0; hh < G; ++hh)
#pragma unroll
    for (int e = 0; e < DV; ++e) acc[hh][e] = 0.f;
#pragma unroll 4
  for (int kk = warp; kk < kn; kk += 4) {
    const __nv_bfloat16* vr = vbase + static_cast<long long>(kk) * row_stride + lane * DV;
    float vf[DV];
    if constexpr (DV == 4) {
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(vr));
      const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&u);
      float2 t0 = __bfloat1622float2(p2[0]), t1 = __bfloat1622float2(p2[1]);
      vf[0] = t0.x; vf[1] = t0.y; vf[2] = t1.x; vf[3] = t1.y;
    } else {
      const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(vr));
      float2 t0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
      vf[0] = t0.x; vf[1] = t0.y;
    }
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      const float pv = s_p[kk][hh];
#pragma unroll
      for (int e = 0; e < DV; ++e) acc[hh][e] = fmaf(pv, vf[e], acc[hh][e]);
    }
  }
#pragma unroll
  for (int hh = 0; hh < G; ++hh)
#pragma unroll
    for (int e = 0; e < DV; ++e) s_red[warp][hh][lane * DV + e] = acc[hh][e];
  __syncthreads();
  float* out = a.priv_part + part_idx * D;
  for (int t = threadIdx.x; t < G * D; t += 128) {
    const int hh = t / D, e = t % D;
    out[static_cast<long long>(hh) * D + e] =
        s_red[0][hh][e] + s_red[1][hh][e] + s_red[2][hh][e] + s_red[3][hh][e];
  }
}

// ------------------------------------------------------------- combine ----
// grid: B * Hq blocks of d threads.  All log-sum-exps are in the log2 domain.
template <int CH>
__global__ void decode_combine_kernel(DecodeLaunch a) {
  const int bh = blockIdx.x;
  const int b = bh / a.Hq, h = bh % a.Hq;
  const int G = a.Hq / a.Hkv, g = h / G, hh = h % G;
  const int d = a.d, e = threadIdx.x;
  const int R = a.B * G, r = b * G + hh;
  const int L = clamp_len(a.len, b, a.rows);
  const int n_chunks = (a.rows + CH - 1) / CH;
  const int used = L / CH + 1;
  float M = -INFINITY;
  for (int s = 0; s < a.n_cart_splits; ++s)
    M = fmaxf(M, a.cart_lse[(static_cast<long long>(s) * a.Hkv + g) * R + r]);
  const long long pbase = ((static_cast<long long>(b) * a.Hkv + g) * n_chunks) * G + hh;
  for (int c = 0; c < used; ++c) {
    const float m = a.priv_ml[(pbase + static_cast<long long>(c) * G) * 2];
    const float l = a.priv_ml[(pbase + static_cast<long long>(c) * G) * 2 + 1];
    M = fmaxf(M, m + __log2f(l));
  }
  float num = 0.f, den = 0.f;
  for (int s = 0; s < a.n_cart_splits; ++s) {
    const long long ri = (static_cast<long long>(s) * a.Hkv + g) * R + r;
    const float w = exp2_approx(a.cart_lse[ri] - M);
    den += w;
    num += w * a.cart_part[ri * d + e];
  }
  for (int c = 0; c < used; ++c) {
    const long long pi = pbase + static_cast<long long>(c) * G;
    const float m = a.priv_ml[pi * 2], l = a.priv_ml[pi * 2 + 1];
    // acc is relative to exp2(m): weight of the chunk's normalised output is
    // l * exp2(m - M); multiply its acc / l by that.
    const float w = exp2_approx(m - M);
    den += l * w;
    num += w * a.priv_part[pi * d + e];
  }
  a.o[(static_cast<long long>(b) * a.Hq + h) * d + e] = __float2bfloat16_rn(num / den);
}

template <int D, int G>
cudaError_t launch_private_dg(const DecodeLaunch& a, cudaStream_t st) {
  constexpr int CH = 128;
  const dim3 grid((a.rows + CH - 1) / CH, a.Hkv, a.B);
  const float scale_log2 = a.scale * 1.4426950408889634f;
  TraceScope tr("decode_private", st);
  decode_private_kernel<D, G, CH><<<grid, 128, 0, st>>>(a, scale_log2);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_prep(const DecodeLaunch& a, const RopeFreqs& f, cudaStream_t st) {
  TraceScope tr("decode_prep", st);
  decode_prep_kernel<<<a.B, 128, 0, st>>>(a, f);
  return cudaGetLastError();
}

cudaError_t launch_decode_private(const DecodeLaunch& a, cudaStream_t st) {
  const int G = a.Hq / a.Hkv;
  if (a.chunk != 128) return cudaErrorInvalidValue;
  if (a.d == 128) {
    switch (G) {
      case 1: return launch_private_dg<128, 1>(a, st);
      case 2: return launch_private_dg<128, 2>(a, st);
      case 4: return launch_private_dg<128, 4>(a, st);
      case 8: return launch_private_dg<128, 8>(a, st);
    }
  } else if (a.d == 64) {
    switch (G) {
      case 1: return launch_private_dg<64, 1>(a, st);
      case 2: return launch_private_dg<64, 2>(a, st);
      case 4: return launch_private_dg<64, 4>(a, st);
      case 8: return launch_private_dg<64, 8>(a, st);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_combine(const DecodeLaunch& a, cudaStream_t st) {
  TraceScope tr("decode_combine", st);
  decode_combine_kernel<128><<<a.B * a.Hq, a.d, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace cart
