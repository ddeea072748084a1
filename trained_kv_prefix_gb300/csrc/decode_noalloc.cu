// decode_noalloc.cu -- cart_attn_decode_noalloc: the decode step of
// cart_attn_decode with its scratch in a static device array, for callers
// that cannot allocate device memory themselves.
//
// Who needs it: a serving loop that runs under a fixed device-memory budget
// planned once at start-up, where a cudaMalloc on the decode path would
// synchronize the device and stall the other streams; and a plain C host
// that links only this library and has no device allocator (no PyTorch, no
// caching allocator) to carve a workspace from.  Such a caller passes only
// its inputs and outputs.
//
// The scratch is one file-scope array of CART_DECODE_NOALLOC_SCRATCH_BYTES
// bytes.  Every GPU that loads the library holds it until the process exits.
// Host code cannot use the array's name as a device address, so the first
// call on each device looks the address up with cudaGetSymbolAddress (with
// that device current) and caches it; that first call should come before any
// stream capture.  All calls share the one array: calls whose work overlaps
// on the GPU (different streams, or different host threads without ordering)
// race on it.  No scratch word needs to start at zero: every word a call
// reads is written earlier in the same call.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "internal.cuh"

static __device__ __align__(256) unsigned char g_decode_noalloc_scratch[CART_DECODE_NOALLOC_SCRATCH_BYTES];

namespace cart {
namespace {

struct NoallocLayout {
  size_t cart_part = 0, cart_lse = 0, priv_part = 0, priv_lse = 0, total = 0;
  int splits = 0, tiles_per_split = 0, max_units = 0;
};

size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

NoallocLayout layout(int B, int Hq, int Hkv, int d, int p, int rows) {
  NoallocLayout w;
  const int n_ct = (p + 127) / 128;
  const int R = B * (Hq / Hkv);
  const int qpairs = ((R + 127) / 128 + 1) / 2;  // the cartridge pass takes two row tiles per CTA
  if (n_ct > 0) {
    const long long units = static_cast<long long>(n_ct) * Hkv * qpairs;
    int per = static_cast<int>((units + kDecodeCartCtas - 1) / kDecodeCartCtas);
    if (per < 1) per = 1;
    w.tiles_per_split = per;
    w.splits = (n_ct + per - 1) / per;
  }
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += up256(bytes);
    return o;
  };
  w.max_units = (rows + kDecodeUnit - 1) / kDecodeUnit;
  w.cart_part = take(static_cast<size_t>(w.splits) * Hkv * R * d * 4);
  w.cart_lse = take(static_cast<size_t>(w.splits) * Hkv * R * 4);
  w.priv_part = take(static_cast<size_t>(B) * Hq * w.max_units * d * 4);
  w.priv_lse = take(static_cast<size_t>(B) * Hq * w.max_units * 4);
  w.total = off;
  return w;
}

// Device address of the scratch array for the current device, looked up once
// per device with that device current.
std::mutex g_mu;
void* g_addr[64] = {};

int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CART_ERR_CUDA;
  if (dev < 0 || dev >= 64) return CART_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_noalloc_scratch) != cudaSuccess || !ptr)
      return CART_ERR_CUDA;
    g_addr[dev] = ptr;
  }
  *out = g_addr[dev];
  return CART_OK;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace cart

using namespace cart;

extern "C" CART_API int cart_attn_decode_noalloc(int B, int Hq, int Hkv, int d, int p, float scale,
                                                 double rope_theta, const void* q,
                                                 const void* k_new, const void* v_new,
                                                 const void* kc, const void* vc, void* k_cache,
                                                 void* v_cache, int cache_rows,
                                                 const int* priv_len, void* o, void* stream) {
  // ---- the same argument rules as cart_attn_decode
  if (B < 1 || B > 65535 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || p < 0 || cache_rows < 1)
    return CART_ERR_GEOMETRY;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return CART_ERR_GEOMETRY;
  if (d != 64 && d != 128) return CART_ERR_GEOMETRY;
  if (!std::isfinite(scale) || !(scale > 0.f) || !(rope_theta > 0.0) || !std::isfinite(rope_theta))
    return CART_ERR_GEOMETRY;
  if ((static_cast<long long>(B) * G + 127) / 128 > 65535) return CART_ERR_GEOMETRY;
  if (cache_rows > 32768) return CART_ERR_GEOMETRY;
  if (static_cast<long long>(p) + cache_rows >= (1ll << 24)) return CART_ERR_GEOMETRY;
  const void* ptrs[] = {q, k_new, v_new, k_cache, v_cache, o};
  for (const void* ptr : ptrs)
    if (!ptr || !al16(ptr)) return CART_ERR_POINTER;
  if (!priv_len || (reinterpret_cast<uintptr_t>(priv_len) & 3u)) return CART_ERR_POINTER;
  if (p > 0 && (!kc || !vc || !al16(kc) || !al16(vc))) return CART_ERR_POINTER;
  // ---- the problem must fit the static scratch
  const NoallocLayout w = layout(B, Hq, Hkv, d, p, cache_rows);
  if (w.total > static_cast<size_t>(CART_DECODE_NOALLOC_SCRATCH_BYTES)) return CART_ERR_WORKSPACE;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return CART_ERR_CUDA;
  if (major != 10 || minor != 3) return CART_ERR_DEVICE;
  void* base = nullptr;
  int rc = scratch_address(&base);
  if (rc) return rc;
  uint8_t* ws = static_cast<uint8_t*>(base);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  DecodeLaunch a{};
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.p = p;
  a.rows = cache_rows;
  a.scale = scale;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k_new = static_cast<const __nv_bfloat16*>(k_new);
  a.v_new = static_cast<const __nv_bfloat16*>(v_new);
  a.kc = static_cast<const __nv_bfloat16*>(kc);
  a.vc = static_cast<const __nv_bfloat16*>(vc);
  a.k_cache = static_cast<__nv_bfloat16*>(k_cache);
  a.v_cache = static_cast<__nv_bfloat16*>(v_cache);
  a.len = priv_len;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.n_cart_splits = w.splits;
  a.cart_tiles_per_split = w.tiles_per_split;
  a.cart_part = reinterpret_cast<float*>(ws + w.cart_part);
  a.cart_lse = reinterpret_cast<float*>(ws + w.cart_lse);
  a.priv_part = reinterpret_cast<float*>(ws + w.priv_part);
  a.priv_lse = reinterpret_cast<float*>(ws + w.priv_lse);
  a.max_units = w.max_units;
  if (launch_decode(a, make_rope_freqs(d, rope_theta), st) != cudaSuccess) return CART_ERR_CUDA;
  return CART_OK;
}
