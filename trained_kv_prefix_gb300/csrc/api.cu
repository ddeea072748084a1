// api.cu -- the C ABI (include/cartattn.h): host-side validation, workspace
// carving, TMA descriptor construction and kernel launches.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <algorithm>
#include <cstring>
#include <mutex>
#include <queue>

#include "internal.cuh"

namespace cart {

__device__ uint32_t g_device_status;

uint32_t* device_status_ptr() {
  // One address per device, looked up once with that device current.  The
  // address belongs to the library's module in the device's current context:
  // after cudaDeviceReset (a new context) the cached address is stale, so a
  // process that resets a device must not call the library on it again.
  static std::mutex mu;
  static uint32_t* cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<uint32_t*>(p);
  }
  return cache[dev];
}

int sm_count() {
  static std::mutex mu;
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (!cache[dev] &&
      cudaDeviceGetAttribute(&cache[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    cache[dev] = 0;
  return cache[dev];
}

void build_work_plan(const std::vector<double>& cost, int grid, std::vector<uint16_t>* items,
                     std::vector<uint16_t>* off) {
  const int n = static_cast<int>(cost.size());
  std::vector<std::vector<int>> per(grid);
  std::vector<double> load(grid, 0.0);
  std::vector<int> order(n);
  for (int w = 0; w < n; ++w) order[w] = w;
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return cost[x] > cost[y]; });
  using Slot = std::pair<double, int>;
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> q;
  for (int c = 0; c < grid; ++c) q.push({0.0, c});
  for (int w : order) {
    const Slot sl = q.top();
    q.pop();
    per[sl.second].push_back(w);
    load[sl.second] += cost[w];
    q.push({load[sl.second], sl.second});
  }
  for (int iter = 0; iter < 100000; ++iter) {
    const int cm = static_cast<int>(std::max_element(load.begin(), load.end()) - load.begin());
    double best = load[cm];
    int bj = -1, ba = -1, bb = -1;  // move per[cm][ba] to CTA bj (bb < 0) or swap with per[bj][bb]
    for (int j = 0; j < grid; ++j) {
      if (j == cm) continue;
      for (int ia = 0; ia < static_cast<int>(per[cm].size()); ++ia) {
        const double ca = cost[per[cm][ia]];
        const double mv = std::max(load[cm] - ca, load[j] + ca);
        if (mv < best - 1e-9) {
          best = mv;
          bj = j;
          ba = ia;
          bb = -1;
        }
        for (int ib = 0; ib < static_cast<int>(per[j].size()); ++ib) {
          const double d = ca - cost[per[j][ib]];
          if (d <= 1e-9) continue;
          const double sw = std::max(load[cm] - d, load[j] + d);
          if (sw < best - 1e-9) {
            best = sw;
            bj = j;
            ba = ia;
            bb = ib;
          }
        }
      }
    }
    if (bj < 0) break;
    const int wa = per[cm][ba];
    per[cm].erase(per[cm].begin() + ba);
    per[bj].push_back(wa);
    load[cm] -= cost[wa];
    load[bj] += cost[wa];
    if (bb >= 0) {
      const int wb = per[bj][bb];
      per[bj].erase(per[bj].begin() + bb);
      per[cm].push_back(wb);
      load[bj] -= cost[wb];
      load[cm] += cost[wb];
    }
  }
  items->clear();
  off->assign(1, 0);
  for (int c = 0; c < grid; ++c) {
    std::sort(per[c].begin(), per[c].end(), [&](int x, int y) { return cost[x] > cost[y]; });
    for (int w : per[c]) items->push_back(static_cast<uint16_t>(w));
    off->push_back(static_cast<uint16_t>(items->size()));
  }
}

namespace {

// ------------------------------------------------------------ utilities ----
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tensor-map encoding through a small per-process cache.  A map depends only
// on its arguments (type, base address, sizes, strides, box), so an entry
// can be reused by any later call with the same arguments; caching takes the
// driver's encode (microseconds each, several per decode step) off the
// host's launch path.  Entries are replaced round robin.
struct MapKey {
  int dtype, rank;
  const void* base;
  uint64_t dims[5], strides[4];
  uint32_t box[5];
  bool operator==(const MapKey& o) const {
    return dtype == o.dtype && rank == o.rank && base == o.base &&
           std::memcmp(dims, o.dims, sizeof dims) == 0 &&
           std::memcmp(strides, o.strides, sizeof strides) == 0 &&
           std::memcmp(box, o.box, sizeof box) == 0;
  }
};
constexpr int kMapCacheSize = 64;
struct MapCache {
  std::mutex mu;
  MapKey key[kMapCacheSize];
  CUtensorMap map[kMapCacheSize];
  bool used[kMapCacheSize] = {};
  int next = 0;
};
MapCache& map_cache() {
  static MapCache c;
  return c;
}

bool encode_cached(CUtensorMap* m, CUtensorMapDataType dtype, int rank, const void* base,
                   const uint64_t* dims, const uint64_t* strides, const uint32_t* box) {
  MapKey k{};
  k.dtype = static_cast<int>(dtype);
  k.rank = rank;
  k.base = base;
  for (int i = 0; i < rank; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) k.strides[i] = strides[i];
  MapCache& c = map_cache();
  {
    std::lock_guard<std::mutex> lk(c.mu);
    for (int i = 0; i < kMapCacheSize; ++i)
      if (c.used[i] && c.key[i] == k) {
        *m = c.map[i];
        return true;
      }
  }
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dd[5], ss[4];
  cuuint32_t bb[5], es[5];
  for (int i = 0; i < rank; ++i) {
    dd[i] = dims[i];
    bb[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) ss[i] = strides[i];
  if (fn(m, dtype, rank, const_cast<void*>(base), dd, ss, bb, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lk(c.mu);
  c.key[c.next] = k;
  c.map[c.next] = *m;
  c.used[c.next] = true;
  c.next = (c.next + 1) % kMapCacheSize;
  return true;
}

// 4D bf16 map with a 64 x 1 x rows x 1 box, 128-byte swizzle.  dims innermost
// first; strides in bytes for dims 1..3.
bool make_map(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
              uint64_t d3, uint64_t s1, uint64_t s2, uint64_t s3, uint32_t box_rows) {
  const uint64_t dims[4] = {d0, d1, d2, d3};
  const uint64_t strides[3] = {s1, s2, s3};
  const uint32_t box[4] = {64, 1, box_rows, 1};
  return encode_cached(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box);
}

// [blocks, rows, H, d] bf16 tensor as (d, H, rows, blocks).
bool make_rows_map(CUtensorMap* m, const void* base, int blocks, int rows, int H, int d,
                   uint32_t box_rows) {
  const uint64_t e = 2;
  return make_map(m, base, d, H, rows, blocks, d * e, static_cast<uint64_t>(H) * d * e,
                  static_cast<uint64_t>(rows) * H * d * e, box_rows);
}

}  // namespace

bool make_bf16_rows_map(CUtensorMap* m, const void* base, int blocks, int rows, int H, int d,
                        unsigned box_rows) {
  return make_rows_map(m, base, blocks, rows, H, d, box_rows);
}

bool make_bf16_map4(CUtensorMap* m, const void* base, const uint64_t (&dims)[4],
                    const uint64_t (&strides)[3], const uint32_t (&box)[4]) {
  return encode_cached(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box);
}

bool make_f32_map4(CUtensorMap* m, const void* base, const uint64_t (&dims)[4],
                   const uint64_t (&strides)[3], const uint32_t (&box)[4]) {
  return encode_cached(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, dims, strides, box);
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A second stream per device on which the backward's dQ kernel runs
// concurrently with the dK/dV kernel (they read the same inputs and write
// disjoint outputs).  Forked from and joined back into the caller's stream
// with two events, so the caller sees one ordered call.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

SideStream g_side[64];  // per device, created on first use
std::mutex g_side_mu;

// Destroys what a SideStream holds (callers hold g_side_mu).
void destroy_side(SideStream& x) {
  if (x.fork) cudaEventDestroy(x.fork);
  if (x.join) cudaEventDestroy(x.join);
  if (x.s) cudaStreamDestroy(x.s);
  x = SideStream{};
}

SideStream* side_stream() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_side_mu);
  SideStream& x = g_side[dev];
  if (!x.s) {
    if (cudaStreamCreateWithFlags(&x.s, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&x.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&x.join, cudaEventDisableTiming) != cudaSuccess) {
      destroy_side(x);
      return nullptr;
    }
  }
  return &x;
}

int check_device() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CART_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return CART_ERR_CUDA;
  if (major != 10 || minor != 3) return CART_ERR_DEVICE;
  return CART_OK;
}

int check_geom(const cart_geom* g) {
  if (!g) return CART_ERR_POINTER;
  if (g->B < 1 || g->n < 1 || g->Hq < 1 || g->Hkv < 1 || g->Hq % g->Hkv != 0) return CART_ERR_GEOMETRY;
  if (g->d != 64 && g->d != 128) return CART_ERR_GEOMETRY;
  if (g->p < 0 || g->frozen_prefix < 0 || g->frozen_prefix > g->p) return CART_ERR_GEOMETRY;
  if (g->window < 0) return CART_ERR_GEOMETRY;
  if (!(std::isfinite(g->scale)) || !(g->scale > 0.f) || !(g->rope_theta > 0.0) ||
      !std::isfinite(g->rope_theta))
    return CART_ERR_GEOMETRY;
  if (g->B > 65535 || g->Hq > 65535 || (g->n + 127) / 128 > 65535) return CART_ERR_GEOMETRY;
  // RoPE positions p + i are reduced in f32 and must be exact there
  if (static_cast<long long>(g->p) + g->n >= (1ll << 24)) return CART_ERR_GEOMETRY;
  return CART_OK;
}

bool dtype_ok(cart_dtype t) { return t == CART_BF16 || t == CART_F32; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Workspace carving shared by the size query and the call.
struct TrainWs {
  size_t table = 0, qr = 0, kr = 0, vb = 0, kcb = 0, vcb = 0, dob = 0, dvec = 0, nlse2 = 0,
         sched = SIZE_MAX, total = 0;
  int npad = 0;
};

// Packed layout (see SeqRows): cu == nullptr for the fixed [B, n, ...] one.
struct Packing {
  const int* cu = nullptr;
  int total = 0;
};

// Tokens on the training tensors' token axis.
long long token_rows(const cart_geom* g, const Packing& pk) {
  return pk.cu ? pk.total : static_cast<long long>(g->B) * g->n;
}

// reuse (backward only): the forward's workspace supplies the table, the
// rotated Q / K and the bf16 copies, so this workspace holds only the
// backward's own parts.
TrainWs train_ws(const cart_geom* g, cart_dtype in, cart_dtype cd, bool bwd,
                 const Packing& pk = Packing(), bool reuse = false) {
  TrainWs w;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += align256(bytes);
    return o;
  };
  const size_t e16 = 2;
  const size_t rows_q = static_cast<size_t>(token_rows(g, pk)) * g->Hq * g->d;
  const size_t rows_k = static_cast<size_t>(token_rows(g, pk)) * g->Hkv * g->d;
  const size_t cart = static_cast<size_t>(g->p) * g->Hkv * g->d;
  if (!reuse) {
    w.table = take(static_cast<size_t>(g->n) * (g->d / 2) * sizeof(float2));
    w.qr = take(rows_q * e16);
    w.kr = take(rows_k * e16);
    w.vb = (in == CART_F32) ? take(rows_k * e16) : SIZE_MAX;
    w.kcb = (cd == CART_F32 && g->p > 0) ? take(cart * e16) : SIZE_MAX;
    w.vcb = (cd == CART_F32 && g->p > 0) ? take(cart * e16) : SIZE_MAX;
  }
  w.sched = take(sizeof(int));  // the forward's / the dQ kernel's work-item counter
  if (bwd) {
    w.dob = (in == CART_F32) ? take(rows_q * e16) : SIZE_MAX;
    w.npad = (g->n + 127) / 128 * 128;
    w.dvec = take(static_cast<size_t>(g->B) * g->Hq * w.npad * sizeof(float));
    w.nlse2 = take(static_cast<size_t>(g->B) * g->Hq * w.npad * sizeof(float));
  }
  w.total = off;
  return w;
}

// TMA map over a training tensor [B, n, H, d] (fixed) or [total, H, d]
// (packed) as (d, H, n, B) or (d, H, total, 1).
bool make_tokens_map(CUtensorMap* m, const void* base, const cart_geom* g, const Packing& pk,
                     int H, uint32_t box_rows) {
  return pk.cu ? make_rows_map(m, base, 1, pk.total, H, g->d, box_rows)
               : make_rows_map(m, base, g->B, g->n, H, g->d, box_rows);
}

#define CART_CUDA(x)                                  \
  do {                                                \
    if ((x) != cudaSuccess) return CART_ERR_CUDA;     \
  } while (0)

// Shared front half of fwd and bwd: rope table, rotated Q/K, bf16 V and
// cartridge, and the TMA maps over them.
struct TrainPrep {
  const float2* table;
  RopeFreqs freqs;
  const void* qr;  // rotated bf16 queries
  const void* kr;
  const void* vb;
  const void* kcb;
  const void* vcb;
  CUtensorMap mQ, mK, mV, mKc, mVc;
};

// The backward's per-row vectors, produced by the same prep launch for bf16
// inputs (o == nullptr: none).
struct PrepVec {
  const void* o = nullptr;
  const void* dout = nullptr;
  const float* lse = nullptr;
  float* nDvec = nullptr;
  float* nlse2 = nullptr;
  int npad = 0;
};

// The TMA maps over the prepared tensors.
int prep_maps(const cart_geom* g, const Packing& pk, TrainPrep* out) {
  bool ok = make_tokens_map(&out->mQ, out->qr, g, pk, g->Hq, 128) &&
            make_tokens_map(&out->mK, out->kr, g, pk, g->Hkv, 128) &&
            make_tokens_map(&out->mV, out->vb, g, pk, g->Hkv, 128);
  if (g->p > 0)
    ok = ok && make_rows_map(&out->mKc, out->kcb, 1, g->p, g->Hkv, g->d, 128) &&
         make_rows_map(&out->mVc, out->vcb, 1, g->p, g->Hkv, g->d, 128);
  else  // never loaded when there are no cartridge tiles
    ok = ok && make_rows_map(&out->mKc, out->kr, 1, 1, g->Hkv, g->d, 128) &&
         make_rows_map(&out->mVc, out->kr, 1, 1, g->Hkv, g->d, 128);
  return ok ? CART_OK : CART_ERR_CUDA;
}

// bf16 inputs take one fused launch (table, rotated K and Q, backward
// vectors); f32 inputs take the generic kernels and the caller computes the
// vectors.  The workspace's work-item counter (of the persistent forward or
// dQ kernel that follows) is zeroed here, by the first launch of the call.
// With fwd_ws (the backward reusing a forward's workspace) nothing is
// recomputed: the table, the rotated Q / K and the bf16 copies are read from
// the forward's workspace (its layout: train_ws(..., bwd = false)), and only
// the backward's vectors are computed (bf16 inputs; f32 callers compute them).
int train_prep(const cart_geom* g, cart_dtype in, cart_dtype cd, const void* q, const void* k,
               const void* v, const void* kc, const void* vc, uint8_t* ws, const TrainWs& w,
               cudaStream_t st, TrainPrep* out, const PrepVec& vec, const Packing& pk,
               const uint8_t* fwd_ws = nullptr) {
  const bool f32 = in == CART_F32;
  const RopeFreqs freqs = make_rope_freqs(g->d, g->rope_theta);
  // the work-item counter of the kernel that follows (zeroed by the first
  // launch of this prep)
  int* sched = w.sched == SIZE_MAX ? nullptr : reinterpret_cast<int*>(ws + w.sched);
  if (fwd_ws) {
    const TrainWs wf = train_ws(g, in, cd, false, pk);
    if (!f32 && vec.o)
      CART_CUDA(launch_train_prep(
          static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), nullptr,
          nullptr, nullptr, freqs, g->p, g->B, g->n, g->Hq, g->Hkv, g->d,
          static_cast<const __nv_bfloat16*>(vec.o), static_cast<const __nv_bfloat16*>(vec.dout),
          vec.lse, vec.nDvec, vec.nlse2, vec.npad, pk.cu, pk.total, sched, st));
    else if (sched)
      CART_CUDA(cudaMemsetAsync(sched, 0, sizeof(int), st));
    const bool cart_f32 = cd == CART_F32 && g->p > 0;
    out->table = reinterpret_cast<const float2*>(fwd_ws + wf.table);
    out->freqs = freqs;
    out->qr = fwd_ws + wf.qr;
    out->kr = fwd_ws + wf.kr;
    out->vb = f32 ? static_cast<const void*>(fwd_ws + wf.vb) : v;
    out->kcb = cart_f32 ? static_cast<const void*>(fwd_ws + wf.kcb) : kc;
    out->vcb = cart_f32 ? static_cast<const void*>(fwd_ws + wf.vcb) : vc;
    return prep_maps(g, pk, out);
  }
  float2* table = reinterpret_cast<float2*>(ws + w.table);
  __nv_bfloat16* qr = reinterpret_cast<__nv_bfloat16*>(ws + w.qr);
  __nv_bfloat16* kr = reinterpret_cast<__nv_bfloat16*>(ws + w.kr);
  const bool cart_f32 = cd == CART_F32 && g->p > 0;
  if (!f32) {
    // f32 cartridge leaves: their bf16 copies come from the same launch
    CartCast cast;
    if (cart_f32) {
      cast.kc = static_cast<const float*>(kc);
      cast.vc = static_cast<const float*>(vc);
      cast.kcb = reinterpret_cast<__nv_bfloat16*>(ws + w.kcb);
      cast.vcb = reinterpret_cast<__nv_bfloat16*>(ws + w.vcb);
      cast.elems = static_cast<long long>(g->p) * g->Hkv * g->d;
    }
    CART_CUDA(launch_train_prep(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
        qr, kr, table, freqs, g->p, g->B, g->n, g->Hq, g->Hkv, g->d,
        static_cast<const __nv_bfloat16*>(vec.o), static_cast<const __nv_bfloat16*>(vec.dout),
        vec.lse, vec.nDvec, vec.nlse2, vec.npad, pk.cu, pk.total, sched, st, cast));
  } else {
    CART_CUDA(launch_rope_table(table, g->p, g->n, g->d, freqs, sched, st));
    CART_CUDA(launch_rope_rows(q, f32, qr, table, g->B, g->n, g->Hq, g->d, true, pk.cu, pk.total,
                               st));
    CART_CUDA(launch_rope_rows(k, f32, kr, table, g->B, g->n, g->Hkv, g->d, true, pk.cu, pk.total,
                               st));
  }
  const void* vb = v;
  if (f32) {
    __nv_bfloat16* t = reinterpret_cast<__nv_bfloat16*>(ws + w.vb);
    CART_CUDA(launch_rope_rows(v, true, t, table, g->B, g->n, g->Hkv, g->d, false, pk.cu, pk.total,
                               st));
    vb = t;
  }
  const void* kcb = kc;
  const void* vcb = vc;
  if (cart_f32) {
    __nv_bfloat16* tk = reinterpret_cast<__nv_bfloat16*>(ws + w.kcb);
    __nv_bfloat16* tv = reinterpret_cast<__nv_bfloat16*>(ws + w.vcb);
    if (f32) {  // (bf16 inputs: made by the prep launch above)
      const int row = g->Hkv * g->d;
      CART_CUDA(launch_write_to_cache(static_cast<const float*>(kc), tk,
                                      static_cast<const float*>(vc), tv, g->p, row, row, 0, true,
                                      st));
    }
    kcb = tk;
    vcb = tv;
  }
  out->table = table;
  out->freqs = freqs;
  out->qr = qr;
  out->kr = kr;
  out->vb = vb;
  out->kcb = kcb;
  out->vcb = vcb;
  return prep_maps(g, pk, out);
}

// Packed layout: at least one token, no more than B segments of n tokens
// hold, a 4-byte aligned table (its contents are checked on the device).
int check_packing(const cart_geom* g, const Packing& pk) {
  if (!pk.cu) return CART_OK;
  if (pk.total < 1 || static_cast<long long>(pk.total) > static_cast<long long>(g->B) * g->n)
    return CART_ERR_GEOMETRY;
  if (reinterpret_cast<uintptr_t>(pk.cu) & 3u) return CART_ERR_POINTER;
  return CART_OK;
}

int train_common_checks(const cart_geom* g, cart_dtype in, cart_dtype cd, const void* q,
                        const void* k, const void* v, const void* kc, const void* vc,
                        const Packing& pk) {
  int rc = check_geom(g);
  if (rc) return rc;
  rc = check_packing(g, pk);
  if (rc) return rc;
  if (!dtype_ok(in) || !dtype_ok(cd)) return CART_ERR_DTYPE;
  if (!q || !k || !v || !aligned16(q) || !aligned16(k) || !aligned16(v)) return CART_ERR_POINTER;
  if (g->p > 0 && (!kc || !vc || !aligned16(kc) || !aligned16(vc))) return CART_ERR_POINTER;
  return CART_OK;
}

}  // namespace
}  // namespace cart

using namespace cart;

extern "C" {

const char* cart_status_string(int s) {
  switch (s) {
    case CART_OK: return "ok";
    case CART_ERR_GEOMETRY: return "bad geometry";
    case CART_ERR_POINTER: return "null or misaligned pointer";
    case CART_ERR_DTYPE: return "unsupported dtype";
    case CART_ERR_WORKSPACE: return "workspace too small";
    case CART_ERR_CUDA: return "CUDA error";
    case CART_ERR_DEVICE: return "device is not sm_103";
    case CART_ERR_TIMEOUT: return "a kernel gave up waiting";
    default: return "unknown status";
  }
}

int cart_release(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return CART_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_side_mu);
  SideStream& x = g_side[dev];
  if (x.s && cudaStreamSynchronize(x.s) != cudaSuccess) return CART_ERR_CUDA;
  destroy_side(x);
  return CART_OK;
}

int cart_device_status(unsigned* bits_out, int clear) {
  uint32_t* p = device_status_ptr();
  if (!p) return CART_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return CART_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return CART_ERR_CUDA;
  if (clear && cudaMemset(p, 0, sizeof v) != cudaSuccess) return CART_ERR_CUDA;
  if (bits_out) *bits_out = v;
  return v ? CART_ERR_TIMEOUT : CART_OK;
}

int cart_write_to_cache(const float* kc, const float* vc, int p, int Hkv, int d, void* k_dst,
                        void* v_dst, long long row_stride_elems, int dst_row0,
                        cart_dtype dst_dtype, void* stream) {
  if (p < 0 || Hkv < 1 || d < 8 || d % 8 != 0 || dst_row0 < 0) return CART_ERR_GEOMETRY;
  const long long row = static_cast<long long>(Hkv) * d;
  if (row_stride_elems < row || row_stride_elems % 8 != 0) return CART_ERR_GEOMETRY;
  if (!dtype_ok(dst_dtype)) return CART_ERR_DTYPE;
  if ((!kc || !k_dst) && (!vc || !v_dst)) return CART_ERR_POINTER;
  if ((kc && !aligned16(kc)) || (vc && !aligned16(vc)) || (k_dst && !aligned16(k_dst)) ||
      (v_dst && !aligned16(v_dst)))
    return CART_ERR_POINTER;
  int rc = check_device();
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool bf16 = dst_dtype == CART_BF16;
  CART_CUDA(launch_write_to_cache(kc && k_dst ? kc : nullptr, kc && k_dst ? k_dst : nullptr,
                                  vc && v_dst ? vc : nullptr, vc && v_dst ? v_dst : nullptr, p,
                                  static_cast<int>(row), row_stride_elems, dst_row0, bf16, st));
  return CART_OK;
}

static int fwd_impl(const cart_geom* g, const Packing& pk, cart_dtype in, cart_dtype cd,
                    const void* q, const void* k, const void* v, const void* kc, const void* vc,
                    void* o, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = train_common_checks(g, in, cd, q, k, v, kc, vc, pk);
  if (rc) return rc;
  if (!o || !lse || !aligned16(o) || !aligned16(lse)) return CART_ERR_POINTER;
  const TrainWs w = train_ws(g, in, cd, false, pk);
  if (!workspace || workspace_bytes < w.total || !aligned16(workspace)) return CART_ERR_WORKSPACE;
  rc = check_device();
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  TrainPrep tp;
  rc = train_prep(g, in, cd, q, k, v, kc, vc, static_cast<uint8_t*>(workspace), w, st, &tp,
                  PrepVec(), pk);
  if (rc) return rc;
  FwdLaunch l{};
  l.mQ = &tp.mQ;
  l.mKc = &tp.mKc;
  l.mVc = &tp.mVc;
  l.mK = &tp.mK;
  l.mV = &tp.mV;
  l.d = g->d;
  l.n_rows = g->n;
  l.n_qblocks = g->B;
  l.Hq_map = g->Hq;
  l.G = g->Hq / g->Hkv;
  l.p = g->p;
  l.n_real = g->n;
  l.cart_tiles_per_split = 0;
  l.n_splits = 1;
  l.scale_log2 = g->scale * 1.4426950408889634f;
  l.out = o;
  l.out_f32 = in == CART_F32;
  l.lse = lse;
  l.decode = false;
  l.pdl = true;  // the kernel waits for the prep launch before it reads anything
  l.sched = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + w.sched);
  l.cu = pk.cu;
  l.total = pk.total;
  l.window = g->window;
  CUtensorMap mO32;
  if (in == CART_BF16) {
    if (!make_tokens_map(&mO32, o, g, pk, g->Hq, 32)) return CART_ERR_CUDA;
    l.mO32 = &mO32;
  }
  CART_CUDA(launch_fwd(l, st));
  return CART_OK;
}

size_t cart_attn_fwd_workspace_size(const cart_geom* g, cart_dtype in, cart_dtype cd) {
  if (check_geom(g) || !dtype_ok(in) || !dtype_ok(cd)) return 0;
  return train_ws(g, in, cd, false).total;
}

int cart_attn_fwd(const cart_geom* g, cart_dtype in, cart_dtype cd, const void* q, const void* k,
                  const void* v, const void* kc, const void* vc, void* o, float* lse,
                  void* workspace, size_t workspace_bytes, void* stream) {
  return fwd_impl(g, Packing(), in, cd, q, k, v, kc, vc, o, lse, workspace, workspace_bytes,
                  stream);
}

size_t cart_attn_fwd_packed_workspace_size(const cart_geom* g, int total, cart_dtype in,
                                           cart_dtype cd) {
  Packing pk;
  pk.cu = reinterpret_cast<const int*>(16);  // any non-null table: sizes only
  pk.total = total;
  if (check_geom(g) || check_packing(g, pk) || !dtype_ok(in) || !dtype_ok(cd)) return 0;
  return train_ws(g, in, cd, false, pk).total;
}

int cart_attn_fwd_packed(const cart_geom* g, int total, const int* cu_seqlens, cart_dtype in,
                         cart_dtype cd, const void* q, const void* k, const void* v,
                         const void* kc, const void* vc, void* o, float* lse, void* workspace,
                         size_t workspace_bytes, void* stream) {
  Packing pk;
  pk.cu = cu_seqlens;
  pk.total = total;
  if (!cu_seqlens) return CART_ERR_POINTER;
  return fwd_impl(g, pk, in, cd, q, k, v, kc, vc, o, lse, workspace, workspace_bytes, stream);
}

size_t cart_attn_bwd_workspace_size(const cart_geom* g, cart_dtype in, cart_dtype cd) {
  if (check_geom(g) || !dtype_ok(in) || !dtype_ok(cd)) return 0;
  return train_ws(g, in, cd, true).total;
}

static int bwd_impl(const cart_geom* g, const Packing& pk, cart_dtype in, cart_dtype cd,
                    const void* q, const void* k, const void* v, const void* kc, const void* vc,
                    const void* o, const float* lse, const void* dout, void* dq, void* dk,
                    void* dv, float* dkc, float* dvc, const int* frozen_rows, int n_frozen,
                    int accumulate, void* workspace, size_t workspace_bytes, void* stream,
                    const void* fwd_ws = nullptr, size_t fwd_ws_bytes = 0) {
  int rc = train_common_checks(g, in, cd, q, k, v, kc, vc, pk);
  if (rc) return rc;
  if (n_frozen < 0 || n_frozen > CART_MAX_FROZEN_ROWS || (n_frozen > 0 && !frozen_rows))
    return CART_ERR_GEOMETRY;
  for (int i = 0; i < n_frozen; ++i)
    if (frozen_rows[i] < 0 || frozen_rows[i] >= g->p) return CART_ERR_GEOMETRY;
  if (!o || !lse || !dout || !dq || !dk || !dv || !aligned16(o) || !aligned16(lse) ||
      !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return CART_ERR_POINTER;
  if (g->p > 0 && (!dkc || !dvc || !aligned16(dkc) || !aligned16(dvc))) return CART_ERR_POINTER;
  if (accumulate != 0 && accumulate != 1) return CART_ERR_GEOMETRY;
  const TrainWs w = train_ws(g, in, cd, true, pk, fwd_ws != nullptr);
  if (!workspace || workspace_bytes < w.total || !aligned16(workspace)) return CART_ERR_WORKSPACE;
  if (fwd_ws && (fwd_ws_bytes < train_ws(g, in, cd, false, pk).total || !aligned16(fwd_ws)))
    return CART_ERR_WORKSPACE;
  rc = check_device();
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  TrainPrep tp;
  const bool f32 = in == CART_F32;
  float* nDvec = reinterpret_cast<float*>(ws + w.dvec);
  float* nlse2 = reinterpret_cast<float*>(ws + w.nlse2);
  PrepVec vec;  // bf16: the per-row vectors come out of the same prep launch
  if (!f32) {
    vec.o = o;
    vec.dout = dout;
    vec.lse = lse;
    vec.nDvec = nDvec;
    vec.nlse2 = nlse2;
    vec.npad = w.npad;
  }
  rc = train_prep(g, in, cd, q, k, v, kc, vc, ws, w, st, &tp, vec, pk,
                  static_cast<const uint8_t*>(fwd_ws));
  if (rc) return rc;
  const void* dob = dout;
  if (f32) {
    __nv_bfloat16* t = reinterpret_cast<__nv_bfloat16*>(ws + w.dob);
    CART_CUDA(launch_rope_rows(dout, true, t, tp.table, g->B, g->n, g->Hq, g->d, false, pk.cu,
                               pk.total, st));
    dob = t;
    CART_CUDA(launch_bwd_vec(o, dout, f32, lse, nDvec, nlse2, g->B, g->n, w.npad, g->Hq, g->d,
                             pk.cu, pk.total, st));
  }
  CUtensorMap mdO;
  if (!make_tokens_map(&mdO, dob, g, pk, g->Hq, 128)) return CART_ERR_CUDA;
  BwdLaunch l{};
  l.mQ = &tp.mQ;
  l.mdO = &mdO;
  l.mKc = &tp.mKc;
  l.mVc = &tp.mVc;
  l.mK = &tp.mK;
  l.mV = &tp.mV;
  l.B = g->B;
  l.n = g->n;
  l.Hq = g->Hq;
  l.Hkv = g->Hkv;
  l.d = g->d;
  l.p = g->p;
  l.frozen_prefix = g->frozen_prefix;
  l.n_frozen = n_frozen;
  for (int i = 0; i < n_frozen; ++i) l.frozen_rows[i] = frozen_rows[i];
  l.scale = g->scale;
  l.nlse2 = nlse2;
  l.nDvec = nDvec;
  l.npad = w.npad;
  l.dq = dq;
  l.dk = dk;
  l.dv = dv;
  l.out_f32 = f32;
  l.dkc = dkc;
  l.dvc = dvc;
  l.accumulate = accumulate;
  l.table = tp.table;
  l.freqs = &tp.freqs;
  l.cu = pk.cu;
  l.total = pk.total;
  l.window = g->window;
  l.sched = reinterpret_cast<int*>(ws + w.sched);
  SideStream* side = side_stream();
  if (!side) {
    CART_CUDA(launch_bwd(l, st, st));
    return CART_OK;
  }
  CART_CUDA(cudaEventRecord(side->fork, st));
  CART_CUDA(cudaStreamWaitEvent(side->s, side->fork, 0));
  const cudaError_t e = launch_bwd(l, st, side->s);
  // join even when a launch failed, so the side stream never runs ahead
  CART_CUDA(cudaEventRecord(side->join, side->s));
  CART_CUDA(cudaStreamWaitEvent(st, side->join, 0));
  CART_CUDA(e);
  return CART_OK;
}


int cart_attn_bwd(const cart_geom* g, cart_dtype in, cart_dtype cd, const void* q, const void* k,
                  const void* v, const void* kc, const void* vc, const void* o, const float* lse,
                  const void* dout, void* dq, void* dk, void* dv, float* dkc, float* dvc,
                  int accumulate, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(g, Packing(), in, cd, q, k, v, kc, vc, o, lse, dout, dq, dk, dv, dkc, dvc,
                  nullptr, 0, accumulate, workspace, workspace_bytes, stream);
}

size_t cart_attn_bwd_reuse_workspace_size(const cart_geom* g, cart_dtype in, cart_dtype cd) {
  if (check_geom(g) || !dtype_ok(in) || !dtype_ok(cd)) return 0;
  return train_ws(g, in, cd, true, Packing(), true).total;
}

int cart_attn_bwd_reuse(const cart_geom* g, cart_dtype in, cart_dtype cd, const void* q,
                        const void* k, const void* v, const void* kc, const void* vc,
                        const void* o, const float* lse, const void* dout, void* dq, void* dk,
                        void* dv, float* dkc, float* dvc, int accumulate,
                        const void* fwd_workspace, size_t fwd_workspace_bytes, void* workspace,
                        size_t workspace_bytes, void* stream) {
  if (!fwd_workspace) return CART_ERR_WORKSPACE;
  return bwd_impl(g, Packing(), in, cd, q, k, v, kc, vc, o, lse, dout, dq, dk, dv, dkc, dvc,
                  nullptr, 0, accumulate, workspace, workspace_bytes, stream, fwd_workspace,
                  fwd_workspace_bytes);
}

int cart_attn_bwd_parts(const cart_geom* g, cart_dtype in, cart_dtype cd, const void* q,
                        const void* k, const void* v, const void* kc, const void* vc,
                        const void* o, const float* lse, const void* dout, void* dq, void* dk,
                        void* dv, float* dkc, float* dvc, const int* frozen_rows, int n_frozen,
                        int accumulate, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(g, Packing(), in, cd, q, k, v, kc, vc, o, lse, dout, dq, dk, dv, dkc, dvc,
                  frozen_rows, n_frozen, accumulate, workspace, workspace_bytes, stream);
}

size_t cart_attn_bwd_packed_workspace_size(const cart_geom* g, int total, cart_dtype in,
                                           cart_dtype cd) {
  Packing pk;
  pk.cu = reinterpret_cast<const int*>(16);  // any non-null table: sizes only
  pk.total = total;
  if (check_geom(g) || check_packing(g, pk) || !dtype_ok(in) || !dtype_ok(cd)) return 0;
  return train_ws(g, in, cd, true, pk).total;
}

int cart_attn_bwd_packed(const cart_geom* g, int total, const int* cu_seqlens, cart_dtype in,
                         cart_dtype cd, const void* q, const void* k, const void* v,
                         const void* kc, const void* vc, const void* o, const float* lse,
                         const void* dout, void* dq, void* dk, void* dv, float* dkc, float* dvc,
                         const int* frozen_rows, int n_frozen, int accumulate, void* workspace,
                         size_t workspace_bytes, void* stream) {
  Packing pk;
  pk.cu = cu_seqlens;
  pk.total = total;
  if (!cu_seqlens) return CART_ERR_POINTER;
  return bwd_impl(g, pk, in, cd, q, k, v, kc, vc, o, lse, dout, dq, dk, dv, dkc, dvc,
                  frozen_rows, n_frozen, accumulate, workspace, workspace_bytes, stream);
}

// ------------------------------------------------------------------ decode --
}  // extern "C"

namespace cart {

DecodeWs decode_ws(int B, int Hq, int Hkv, int d, int p, int rows, int span) {
  DecodeWs w;
  const int n_ct = (p + 127) / 128;
  const int R = B * span * (Hq / Hkv);
  const int qpairs = ((R + 127) / 128 + 1) / 2;  // the cartridge pass takes two row tiles per CTA
  if (n_ct > 0) {
    // about kDecodeCartCtas CTAs for the cartridge part
    const long long units = static_cast<long long>(n_ct) * Hkv * qpairs;
    int per = static_cast<int>((units + kDecodeCartCtas - 1) / kDecodeCartCtas);
    if (per < 1) per = 1;
    w.tiles_per_split = per;
    w.splits = (n_ct + per - 1) / per;
  }
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += align256(bytes);
    return o;
  };
  w.max_units = (rows + kDecodeUnit - 1) / kDecodeUnit;
  w.cart_part = take(static_cast<size_t>(w.splits) * Hkv * R * d * 4);
  w.cart_lse = take(static_cast<size_t>(w.splits) * Hkv * R * 4);
  w.priv_part = take(static_cast<size_t>(B) * span * Hq * w.max_units * d * 4);
  w.priv_lse = take(static_cast<size_t>(B) * span * Hq * w.max_units * 4);
  w.total = off;
  return w;
}

int check_decode(int B, int Hq, int Hkv, int d, int p, float scale, double theta, int rows,
                 int span) {
  if (B < 1 || B > 65535 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || p < 0 || rows < 1)
    return CART_ERR_GEOMETRY;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return CART_ERR_GEOMETRY;
  if (span < 1 || span > rows || G * span > kDecodeMaxColumns) return CART_ERR_GEOMETRY;
  if (static_cast<long long>(B) * span > 65535) return CART_ERR_GEOMETRY;
  if (d != 64 && d != 128) return CART_ERR_GEOMETRY;
  if (!std::isfinite(scale) || !(scale > 0.f) || !(theta > 0.0) || !std::isfinite(theta))
    return CART_ERR_GEOMETRY;
  if ((static_cast<long long>(B) * span * G + 127) / 128 > 65535) return CART_ERR_GEOMETRY;
  if (rows > 32768) return CART_ERR_GEOMETRY;
  // positions p + len must be exact in f32 (the query rotation of the
  // cartridge pass reduces its angles in f32)
  if (static_cast<long long>(p) + rows >= (1ll << 24)) return CART_ERR_GEOMETRY;
  return CART_OK;
}

int run_decode(int B, int span, int window, int Hq, int Hkv, int d, int p, float scale,
               double rope_theta, const void* q, const void* k_new, const void* v_new,
               const void* kc, const void* vc, void* k_cache, void* v_cache, int cache_rows,
               const int* priv_len, void* o, void* workspace, const DecodeWs& w,
               cudaStream_t stream) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeLaunch a{};
  a.span = span;
  a.window = window;
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
  a.max_units = w.max_units;
  a.priv_part = reinterpret_cast<float*>(ws + w.priv_part);
  a.priv_lse = reinterpret_cast<float*>(ws + w.priv_lse);
  return launch_decode(a, make_rope_freqs(d, rope_theta), stream) == cudaSuccess ? CART_OK
                                                                                   : CART_ERR_CUDA;
}

}  // namespace cart

extern "C" {

size_t cart_attn_decode_workspace_size(int B, int Hq, int Hkv, int d, int p, int cache_rows) {
  return cart_attn_decode_span_workspace_size(B, 1, Hq, Hkv, d, p, cache_rows);
}

size_t cart_attn_decode_span_workspace_size(int B, int span, int Hq, int Hkv, int d, int p,
                                            int cache_rows) {
  if (check_decode(B, Hq, Hkv, d, p, 1.f, 1.0, cache_rows, span)) return 0;
  return decode_ws(B, Hq, Hkv, d, p, cache_rows, span).total;
}

int cart_attn_decode(int B, int Hq, int Hkv, int d, int p, float scale, double rope_theta,
                     const void* q, const void* k_new, const void* v_new, const void* kc,
                     const void* vc, void* k_cache, void* v_cache, int cache_rows,
                     const int* priv_len, void* o, void* workspace, size_t workspace_bytes,
                     void* stream) {
  return cart_attn_decode_span(B, 1, 0, Hq, Hkv, d, p, scale, rope_theta, q, k_new, v_new, kc,
                               vc, k_cache, v_cache, cache_rows, priv_len, o, workspace,
                               workspace_bytes, stream);
}

int cart_attn_decode_span(int B, int span, int window, int Hq, int Hkv, int d, int p, float scale,
                          double rope_theta, const void* q, const void* k_new, const void* v_new,
                          const void* kc, const void* vc, void* k_cache, void* v_cache,
                          int cache_rows, const int* priv_len, void* o, void* workspace,
                          size_t workspace_bytes, void* stream) {
  if (window < 0) return CART_ERR_GEOMETRY;
  int rc = check_decode(B, Hq, Hkv, d, p, scale, rope_theta, cache_rows, span);
  if (rc) return rc;
  const void* ptrs[] = {q, k_new, v_new, k_cache, v_cache, o};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return CART_ERR_POINTER;
  if (!priv_len || (reinterpret_cast<uintptr_t>(priv_len) & 3u)) return CART_ERR_POINTER;
  if (p > 0 && (!kc || !vc || !aligned16(kc) || !aligned16(vc))) return CART_ERR_POINTER;
  const DecodeWs w = decode_ws(B, Hq, Hkv, d, p, cache_rows, span);
  if (!workspace || workspace_bytes < w.total || !aligned16(workspace)) return CART_ERR_WORKSPACE;
  rc = check_device();
  if (rc) return rc;
  return run_decode(B, span, window, Hq, Hkv, d, p, scale, rope_theta, q, k_new, v_new, kc, vc,
                    k_cache, v_cache, cache_rows, priv_len, o, workspace, w,
                    static_cast<cudaStream_t>(stream));
}

}  // extern "C"
