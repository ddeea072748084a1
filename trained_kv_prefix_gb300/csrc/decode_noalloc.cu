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

#include <cstdint>
#include <mutex>

#include "internal.cuh"

static __device__ __align__(256) unsigned char g_decode_noalloc_scratch[CART_DECODE_NOALLOC_SCRATCH_BYTES];

namespace cart {
namespace {

// Device address of the scratch array for the current device, looked up once
// per device with that device current.  The address belongs to the library's
// module in the device's current context: after cudaDeviceReset (a new
// context) it is stale, so a process that resets a device must not call this
// entry point on that device again.
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
  // ---- the problem must fit the static scratch: checked first, so that a
  // problem too large for it is refused before anything else is looked at
  int rc = check_decode(B, Hq, Hkv, d, p, scale, rope_theta, cache_rows);
  if (rc) return rc;
  const DecodeWs w = decode_ws(B, Hq, Hkv, d, p, cache_rows);
  if (w.total > static_cast<size_t>(CART_DECODE_NOALLOC_SCRATCH_BYTES)) return CART_ERR_WORKSPACE;
  // ---- the same pointer rules as cart_attn_decode
  const void* ptrs[] = {q, k_new, v_new, k_cache, v_cache, o};
  for (const void* ptr : ptrs)
    if (!ptr || !al16(ptr)) return CART_ERR_POINTER;
  if (!priv_len || (reinterpret_cast<uintptr_t>(priv_len) & 3u)) return CART_ERR_POINTER;
  if (p > 0 && (!kc || !vc || !al16(kc) || !al16(vc))) return CART_ERR_POINTER;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return CART_ERR_CUDA;
  if (major != 10 || minor != 3) return CART_ERR_DEVICE;
  void* base = nullptr;
  rc = scratch_address(&base);
  if (rc) return rc;
  // the same decode step as cart_attn_decode, its workspace being the array
  return run_decode(B, 1, 0, Hq, Hkv, d, p, scale, rope_theta, q, k_new, v_new, kc, vc, k_cache,
                    v_cache, cache_rows, priv_len, o, base, w, static_cast<cudaStream_t>(stream));
}
