// trace.cu -- optional launch tracing.  While enabled, every kernel launch the
// library makes is bracketed by two CUDA events recorded on the launching
// stream, so a caller can read back per-kernel device times and the number
// of launches.  Off by default; when off a launch pays one relaxed load.
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.cuh"

namespace cart {
namespace {

struct Rec {
  char name[32];
  cudaEvent_t a = nullptr, b = nullptr;
  bool valid = false;
};

std::atomic<bool> g_on{false};
std::mutex g_mu;
std::vector<Rec> g_recs;   // event pool; grows, never shrinks until release
size_t g_used = 0;
constexpr size_t kMaxRecs = 1 << 16;

}  // namespace

int trace_begin(const char* name, cudaStream_t st) {
  if (!name || !g_on.load(std::memory_order_relaxed)) return -1;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_used >= kMaxRecs) return -1;
  if (g_used == g_recs.size()) {
    Rec r;
    if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) return -1;
    g_recs.push_back(r);
  }
  Rec& r = g_recs[g_used];
  std::strncpy(r.name, name, sizeof r.name - 1);
  r.name[sizeof r.name - 1] = 0;
  r.valid = cudaEventRecord(r.a, st) == cudaSuccess;
  return static_cast<int>(g_used++);
}

void trace_end(int slot, cudaStream_t st) {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (static_cast<size_t>(slot) >= g_recs.size()) return;
  Rec& r = g_recs[slot];
  r.valid = r.valid && cudaEventRecord(r.b, st) == cudaSuccess;
}

}  // namespace cart

using namespace cart;

extern "C" {

CART_API int cart_trace_enable(int on) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (on) g_used = 0;  // starting clears; stopping keeps the records
  g_on.store(on != 0);
  return CART_OK;
}

CART_API int cart_trace_count(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  return static_cast<int>(g_used);
}

CART_API int cart_trace_get(int i, char* name, int name_len, float* ms) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (i < 0 || static_cast<size_t>(i) >= g_used) return CART_ERR_GEOMETRY;
  Rec& r = g_recs[i];
  if (name && name_len > 0) {
    std::strncpy(name, r.name, static_cast<size_t>(name_len) - 1);
    name[name_len - 1] = 0;
  }
  if (ms) {
    *ms = -1.f;
    if (!r.valid) return CART_ERR_CUDA;
    if (cudaEventSynchronize(r.b) != cudaSuccess) return CART_ERR_CUDA;
    if (cudaEventElapsedTime(ms, r.a, r.b) != cudaSuccess) return CART_ERR_CUDA;
  }
  return CART_OK;
}

}  // extern "C"
