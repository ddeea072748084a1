// internal.cuh -- declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <vector>

#include "../../include/cartattn.h"

namespace cart {

constexpr int kTile = 128;          // query rows / key rows per tcgen05 tile
constexpr int kMaxHeadDim = 128;

// Raises a kernel's dynamic shared-memory limit once per device (the call is
// comparatively slow and the setting persists for the process).
template <auto Kernel>
cudaError_t set_smem_once(int bytes) {
  static std::atomic<unsigned long long> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_relaxed) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.fetch_or(bit);
  return e;
}

// Launches kern<<<grid, block, smem, st>>>(args...) as the programmatic
// dependent of the previous kernel on st: it may start while that kernel
// still runs, and calls pdl_wait() (ptx.cuh) in every thread before it
// touches global memory, so the stream order of memory effects is kept.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Device status word (bits from ptx.cuh); one per device.
uint32_t* device_status_ptr();

// Launch tracing (trace.cu): brackets a launch with events on its stream
// while tracing is enabled (a null name records nothing: kernels chained by
// programmatic dependent launch are traced as one scope, since an event
// between them would end the overlap).
int trace_begin(const char* name, cudaStream_t st);
void trace_end(int slot, cudaStream_t st);
struct TraceScope {
  int slot;
  cudaStream_t st;
  TraceScope(const char* name, cudaStream_t s) : slot(trace_begin(name, s)), st(s) {}
  ~TraceScope() { trace_end(slot, st); }
  TraceScope(const TraceScope&) = delete;
  TraceScope& operator=(const TraceScope&) = delete;
};

// 4D bf16 TMA map over a [blocks, rows, H, d] tensor as (d, H, rows, blocks)
// with a 64 x 1 x box_rows x 1 box and 128-byte swizzle (api.cu).
bool make_bf16_rows_map(CUtensorMap* m, const void* base, int blocks, int rows, int H, int d,
                        unsigned box_rows);

// fp64 inverse frequencies theta^(-2j/d), j < d/2, passed by value, and the
// same frequencies in turns per position, inv_freq / (2 pi), as an f32
// (hi, lo) pair for the all-f32 angle reduction below.
struct RopeFreqs {
  double inv_freq[kMaxHeadDim / 2];
  float2 turns[kMaxHeadDim / 2];
};
RopeFreqs make_rope_freqs(int d, double theta);

// (cos, sin) of pos * inv_freq with an all-f32 argument reduction, for
// kernels that need many angles (fp64 is slow on this part).  The angle in
// turns is pos * (hi + lo): pos * hi is split exactly into its rounded value
// and the fma remainder (pos < 2^24 is exact in f32), the whole turns are
// dropped from the rounded value (exact for |x| < 2^23), and the remaining
// fraction r in [-1/2, 1/2] is what is left to evaluate.
__device__ __forceinline__ float rope_turn_fraction(float2 turns, int pos) {
  const float pf = static_cast<float>(pos);
  const float th = pf * turns.x;
  const float te = fmaf(pf, turns.x, -th);
  return (th - rintf(th)) + (te + pf * turns.y);
}
// ... with sincospif (error about 2e-7 in all): the training table.
__device__ __forceinline__ float2 rope_cs_turns(float2 turns, int pos) {
  float s, c;
  sincospif(2.f * rope_turn_fraction(turns, pos), &s, &c);
  return make_float2(c, s);
}
// ... with the hardware sine / cosine (error about 5e-7): the many per-row
// angles of the decode cartridge pass.
__device__ __forceinline__ float2 rope_cs_turns_fast(float2 turns, int pos) {
  float s, c;
  __sincosf(6.28318530717958648f * rope_turn_fraction(turns, pos), &s, &c);
  return make_float2(c, s);
}

// Token axis of the training tensors.
//   fixed layout (cu == nullptr): B sequences of n tokens, tensors
//     [B, n, H, d], TMA maps (d, H, n, B);
//   packed layout: B segments back to back on one axis of `total` tokens,
//     segment b = tokens cu[b] .. cu[b+1] - 1 (at most n of them), tensors
//     [total, H, d], TMA maps (d, H, total, 1).
// In both, token i of sequence b sits at RoPE position p + i.
struct SeqRows {
  int row0;  // map row coordinate of the sequence's token 0
  int blk;   // map block coordinate
  int g0;    // flat token index of token 0 (plain addressing: (g0 + i) * H + h)
  int len;   // tokens of the sequence
};
// A packed table is clamped so that every access stays inside the tensors
// (a table that needed clamping is reported by the prep kernels).
__device__ __forceinline__ SeqRows seq_rows(const int* cu, int total, int n, int b) {
  SeqRows r;
  if (!cu) {
    r.row0 = 0;
    r.blk = b;
    r.g0 = b * n;
    r.len = n;
    return r;
  }
  int s0 = __ldg(cu + b), s1 = __ldg(cu + b + 1);
  s0 = min(max(s0, 0), total);
  s1 = min(max(s1, s0), min(total, s0 + n));
  r.row0 = s0;
  r.blk = 0;
  r.g0 = s0;
  r.len = s1 - s0;
  return r;
}
// Index of (sequence b, head h, token i) in a forward log-sum-exp:
// [B, Hq, n] for the fixed layout, [Hq, total] for the packed one.
__device__ __forceinline__ long long lse_index(const int* cu, int total, int n, int Hq, int b,
                                               int h, const SeqRows& r, int i) {
  return cu ? static_cast<long long>(h) * total + r.g0 + i
            : (static_cast<long long>(b) * Hq + h) * n + i;
}

// 4D bf16 TMA map with an arbitrary box and 128-byte swizzle; dims innermost
// first, strides in bytes for dims 1..3 (api.cu).
bool make_bf16_map4(CUtensorMap* m, const void* base, const uint64_t (&dims)[4],
                    const uint64_t (&strides)[3], const uint32_t (&box)[4]);
// The same for f32 data (api.cu).
bool make_f32_map4(CUtensorMap* m, const void* base, const uint64_t (&dims)[4],
                   const uint64_t (&strides)[3], const uint32_t (&box)[4]);

// ----------------------------------------------------------------- misc ----
// f32 -> bf16 / f32 row copy into a strided destination, for one or two
// tensors (K and V) in one launch; an absent pair is (nullptr, nullptr).
cudaError_t launch_write_to_cache(const float* src0, void* dst0, const float* src1, void* dst1,
                                  int p, int row_elems, long long row_stride, int dst_row0,
                                  bool dst_bf16, cudaStream_t st);

// bf16 training inputs, one launch: RoPE table rows for positions p..p+n-1
// (if table), K rotated into kr (if kr), Q into qr (if qr), and with o given
// the backward's
// [B, Hq, npad] vectors -D = -rowsum(dO * O) and -lse * log2(e), stored
// negated (padding rows 0 and -inf).
// cu / total: the packed layout (see SeqRows; cu == nullptr: fixed); the
// packed table is checked here (status bit kDevErrSegments).
// sched (may be null): the forward's work-item counter, set to 0.
// bf16 copies of f32 cartridge leaves, made by the same prep launch:
// kcb/vcb[e] = bf16(kc/vc[e]) for e < elems (a multiple of 8); kc null: none.
struct CartCast {
  const float* kc = nullptr;
  const float* vc = nullptr;
  __nv_bfloat16* kcb = nullptr;
  __nv_bfloat16* vcb = nullptr;
  long long elems = 0;
};
cudaError_t launch_train_prep(const __nv_bfloat16* q, const __nv_bfloat16* k, __nv_bfloat16* qr,
                              __nv_bfloat16* kr, float2* table, const RopeFreqs& f, int p, int B,
                              int n, int Hq, int Hkv, int d, const __nv_bfloat16* o,
                              const __nv_bfloat16* dout, const float* lse, float* nDvec,
                              float* nlse2, int npad, const int* cu, int total, int* sched,
                              cudaStream_t st, const CartCast& cast = CartCast());

// cos/sin table for positions [pos0, pos0 + npos): float2 [npos, d/2]; sets
// *sched to 0 when sched is given (as launch_train_prep).
cudaError_t launch_rope_table(float2* table, int pos0, int npos, int d, const RopeFreqs& f,
                              int* sched, cudaStream_t st);

// Multiprocessors of the current device (cached per device; 0 on error).
int sm_count();

// A static schedule of work items over persistent CTAs, passed as a kernel
// parameter: CTA c takes items[off[c] .. off[c+1]) in that order (n == 0: no
// plan; the CTAs take items from a counter instead).
constexpr int kPlanCtas = 160;
constexpr int kPlanItems = 4096;
template <int N>
struct WorkPlan {
  int n;
  uint16_t off[kPlanCtas + 1];
  uint16_t items[N];
};
// Host: items 0..cost.size()-1 onto `grid` CTAs -- longest processing time
// first onto the least loaded CTA, then moves and swaps that lower the most
// loaded CTA's total while any does (a tighter fit than taking items in
// order from a counter when every CTA gets only a few).  Each CTA's items
// come heaviest first.  cost.size() <= kPlanItems, grid <= kPlanCtas.
void build_work_plan(const std::vector<double>& cost, int grid, std::vector<uint16_t>* items,
                     std::vector<uint16_t>* off);

// Rotate rows of x [B, n, H, d] (bf16 or f32) at positions pos0 + i using the
// table (row i of the table = position pos0 + i) and write bf16 to out (same
// layout).  With rotate == false this is a plain convert/copy.
cudaError_t launch_rope_rows(const void* x, bool x_f32, __nv_bfloat16* out, const float2* table,
                             int B, int n, int H, int d, bool rotate, const int* cu, int total,
                             cudaStream_t st);

// Per-row vectors of the backward in [B, Hq, npad] layout (npad >= n):
// nDvec = -sum_c dO[b,i,h,c] * O[b,i,h,c], nlse2 = -lse * log2(e); padding
// rows get 0 and -inf (zero probability).
cudaError_t launch_bwd_vec(const void* o, const void* dout, bool f32, const float* lse,
                           float* nDvec, float* nlse2, int B, int n, int npad, int Hq, int d,
                           const int* cu, int total, cudaStream_t st);

// ------------------------------------------------------------- forward ----
struct FwdLaunch {
  const CUtensorMap* mQ;   // 4D (d, Hq_map, rows, blocks) bf16, 64x1x128x1 box, SW128
  const CUtensorMap* mKc;  // 4D (d, Hkv, p, 1)
  const CUtensorMap* mVc;
  const CUtensorMap* mK;   // 4D (d, Hkv, n, B) rotated real keys
  const CUtensorMap* mV;   // 4D (d, Hkv, n, B)
  const CUtensorMap* mO32; // training, bf16 output: 4D (d, Hq, n, B) over o, 64x1x32x1 box
                           // (each warp stores its 32 rows by TMA); decode: f32
                           // (d, R, Hkv, S) over the partials, 32x32x1x1 box; or null
  int d;
  int n_rows;              // query rows per query block (n, or B*G for decode)
  int n_qblocks;           // query blocks: B for training, 1 for decode
  int Hq_map;              // heads in the query map
  int G;                   // query heads per kv head (1 for decode: rows carry the group)
  int p;                   // cartridge rows
  int n_real;              // real key rows (0 for decode)
  int cart_tiles_per_split;// decode: cartridge tiles per split (0 = all)
  int n_splits;            // decode: number of splits
  float scale_log2;        // scale * log2(e)
  void* out;               // training: o [B, n, Hq, d]; decode: f32 partial [S, Hkv, R, d]
  bool out_f32;
  float* lse;              // training: [B, Hq, n]; decode: [S, Hkv, R]
  bool decode;
  int* sched;              // training: the work-item counter, zero at launch
  // decode mode: mQ maps the raw queries [B, Hkv, G, d] as (d, G, Hkv, B)
  // with a (64, G, 1, 128/G) box, so that a 128-row tile is rows b*G + hh;
  // the kernel rotates row (b, hh) at position p + len[b] in shared memory.
  const int* dec_len;
  int dec_B, dec_G, dec_rows;  // dec_B counts (conversation, span position) pairs
  int dec_s = 1;               // span length
  const RopeFreqs* freqs;  // host copy, read at launch
  bool pdl;                // launch as the programmatic dependent of the
                           // previous kernel on the stream
  // training, packed layout (SeqRows): n_qblocks segments, n_rows = n_real
  // = the longest; maps over (d, H, total, 1)
  const int* cu = nullptr;
  int total = 0;
  int window = 0;          // sliding window in keys (0: none)
};
// Two 128-row query tiles per work item (training: one query tile of two
// heads of a kv group, or consecutive row tiles of one (sequence, head);
// decode: rows 0-127 / 128-255 of a kv head's stacked rows).
cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t st);

// ------------------------------------------------------------ backward ----
struct BwdLaunch {
  const CUtensorMap* mQ;    // 4D (d, Hq, n, B) rotated queries (bf16), 128-row box
  const CUtensorMap* mdO;   // 4D (d, Hq, n, B) dO (bf16), 128-row box
  const CUtensorMap* mKc;   // 4D (d, Hkv, p, 1)
  const CUtensorMap* mVc;
  const CUtensorMap* mK;    // 4D (d, Hkv, n, B) rotated real keys
  const CUtensorMap* mV;
  int B, n, Hq, Hkv, d, p, frozen_prefix;
  int n_frozen;                            // cartridge rows also frozen (parts' sinks)
  int frozen_rows[CART_MAX_FROZEN_ROWS];
  float scale;
  const float* nlse2;       // [B, Hq, npad] -lse * log2(e), -inf past n
  const float* nDvec;       // [B, Hq, npad] -D, 0 past n
  int npad;                 // n rounded up to a multiple of 128
  void* dq;                 // [B, n, Hq, d] output dtype
  void* dk;                 // [B, n, Hkv, d]
  void* dv;
  bool out_f32;
  float* dkc;               // [p, Hkv, d]
  float* dvc;
  int accumulate;
  const float2* table;      // rope table for positions p .. p+n-1
  const RopeFreqs* freqs;   // rope angles (the epilogues' inverse rotation)
  // packed layout (SeqRows): B segments of at most n tokens, maps over
  // (d, H, total, 1); the row vectors stay [B, Hq, npad]
  const int* cu = nullptr;
  int total = 0;
  int window = 0;           // sliding window in keys (0: none)
  int* sched = nullptr;     // the dQ kernel's work-item counter, zero at launch
};
// dK/dV kernel on st_dkdv, dQ kernel on st_dq (the two are independent).
cudaError_t launch_bwd(const BwdLaunch& a, cudaStream_t st_dkdv, cudaStream_t st_dq);

// -------------------------------------------------------------- decode ----
struct DecodeLaunch {
  int B, Hq, Hkv, d, p, rows;
  float scale;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  const __nv_bfloat16* kc;
  const __nv_bfloat16* vc;
  __nv_bfloat16* k_cache;
  __nv_bfloat16* v_cache;
  const int* len;
  __nv_bfloat16* o;
  int n_cart_splits;
  const float* cart_part;   // [S, Hkv, R, d], R = B*span*G rows (b*span + t)*G + hh
  const float* cart_lse;    // [S, Hkv, R]
  int cart_tiles_per_split; // cartridge tiles per split CTA
  float* priv_part;         // [B, Hkv, units, span*G, d] normalised private partials
  float* priv_lse;          // [B, Hkv, units, span*G] their log2-domain lse
  int max_units;            // ceil(rows / kDecodeUnit)
  uint32_t* status;         // device status word (set by the launcher)
  int span = 1;             // queries per conversation (q, k_new, v_new, o are [B, span, ...])
  int window = 0;           // sliding window in keys (0: none)
};
// The whole decode step on one stream, three kernels chained by
// programmatic dependent launch: the cartridge split pass (fwd kernel in
// decode mode, which rotates the queries itself) starts first on a few SMs;
// the private pass (fixed units of kDecodeUnit private rows per CTA) fills
// the rest of the GPU next to it; the merge kernel combines every
// (conversation, head)'s parts once both are done.
constexpr int kDecodeChunk = 64;    // private rows per pipeline stage
constexpr int kDecodeUnit = 256;    // private rows per CTA
constexpr int kDecodeMaxColumns = 32;  // G * span: query columns of the private pass
// The cartridge pass gets about this many CTAs (one SM each), so that the
// private pass runs next to it on the remaining SMs.
constexpr int kDecodeCartCtas = 48;
cudaError_t launch_decode(const DecodeLaunch& a, const RopeFreqs& f, cudaStream_t st);

// Decode workspace layout (api.cu): byte offsets of each part inside the
// caller's workspace (or the static scratch of the allocation-free entry).
struct DecodeWs {
  size_t cart_part = 0, cart_lse = 0, priv_part = 0, priv_lse = 0, total = 0;
  int splits = 0, tiles_per_split = 0, max_units = 0;
};
DecodeWs decode_ws(int B, int Hq, int Hkv, int d, int p, int rows, int span = 1);
// Host-side argument rules shared by every decode entry point (a cart_status).
int check_decode(int B, int Hq, int Hkv, int d, int p, float scale, double theta, int rows,
                 int span = 1);
// Carves the workspace and enqueues the decode step (arguments already
// checked); returns a cart_status.
int run_decode(int B, int span, int window, int Hq, int Hkv, int d, int p, float scale,
               double rope_theta, const void* q, const void* k_new, const void* v_new,
               const void* kc, const void* vc, void* k_cache, void* v_cache, int cache_rows,
               const int* priv_len, void* o, void* workspace, const DecodeWs& w,
               cudaStream_t stream);

}  // namespace cart
