/*
 * cartattn.h -- C ABI of the GB300 (sm_103a) cartridge-attention library.
 *
 * A cartridge is a trained KV prefix: per layer a [p, kv_head, d] pair of
 * key/value rows living in KV-cache row space.  Cartridge keys are already
 * rotated (RoPE) at positions 0..p-1 and are never rotated again; the real
 * tokens that follow sit at RoPE positions p, p+1, ...  The first
 * `frozen_prefix` rows (1 by default: the attention sink) are frozen
 * constants; the remaining rows are trainable leaves.
 * (Cartridges guide, section "Semantics", parameterization bullet.)
 *
 * Attention runs over concat(sink, trainable rows, real-token K/V) along the
 * sequence with the end-aligned causal mask, source_offset = kv_seq - q_seq:
 * every query sees every cartridge row and is causal over the real tokens.
 * Query head h reads kv head h / (Hq / Hkv).
 * (Cartridges guide, "Semantics", attention bullet.)
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers, row-major, innermost last,
 *     16-byte aligned, owned by the caller.  The library never frees them.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     validate their arguments synchronously on the host, then enqueue work
 *     asynchronously on `stream`; nothing is written when validation fails.
 *   - RoPE is the rotate-half form: element j pairs with j + d/2 at angle
 *     position * theta^(-2j/d).  Angles are reduced in f32: the frequency
 *     in turns is held as an f32 (hi, lo) pair, position * hi is split
 *     exactly into its rounded value and the fma remainder, and whole turns
 *     are dropped; positions must stay below 2^24.  Training with bf16
 *     inputs evaluates the remaining fraction with sincospif (absolute
 *     error about 2e-7), decode with the hardware sine/cosine (about 5e-7).
 *     Training with f32 inputs forms each angle in fp64 and reduces it
 *     modulo 2*pi in fp64 before an f32 sine/cosine.
 *   - Return value: CART_OK (0) or a negative cart_status.
 *   - The library holds no per-call state.  It caches, per process, the
 *     CUDA driver entry point used to build TMA descriptors and, per device,
 *     one helper stream with two events on which cart_attn_bwd runs its dQ
 *     kernel concurrently with its dK/dV kernel (forked from and joined back
 *     into the caller's stream).  Calls on one device from several host
 *     threads at once must therefore be serialised by the caller.
 */
#ifndef CARTATTN_H_
#define CARTATTN_H_

#include <stddef.h>

#if defined(__GNUC__)
#define CART_API __attribute__((visibility("default")))
#else
#define CART_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum cart_status {
  CART_OK = 0,
  CART_ERR_GEOMETRY = -1,   /* bad sizes: Hq % Hkv, d not 64/128, p < frozen_prefix, n < 1 ... */
  CART_ERR_POINTER = -2,    /* NULL or not 16-byte aligned */
  CART_ERR_DTYPE = -3,      /* dtype not supported for this argument */
  CART_ERR_WORKSPACE = -4,  /* workspace NULL or smaller than the *_workspace_size() answer */
  CART_ERR_CUDA = -5,       /* a CUDA runtime / driver call failed (launch, attribute, TMA map) */
  CART_ERR_DEVICE = -6,     /* current device is not a compute capability 10.3 GPU */
  CART_ERR_TIMEOUT = -7     /* a kernel gave up waiting (see cart_device_status) */
} cart_status;

typedef enum cart_dtype { CART_BF16 = 0, CART_F32 = 1 } cart_dtype;

/* Geometry of one training-shape call.
 *   B      independent sequences sharing ONE cartridge (the packed group)
 *   n      real tokens per sequence (q_seq); kv_seq = p + n < 2^24
 *   Hq     query heads;  Hkv  kv heads;  Hq % Hkv == 0
 *   d      head dimension, 64 or 128
 *   p      cartridge rows INCLUDING the frozen sink rows (p >= 0)
 *   frozen_prefix  leading cartridge rows whose gradient is exactly 0
 *   scale  softmax scale (normally 1/sqrt(d)); finite and > 0
 *   rope_theta     RoPE base (1e6 for the Qwen3 family)
 *   window sliding window in keys, 0 = none: the query at position P sees
 *          the keys at positions P - window + 1 .. P (cartridge row j sits
 *          at position j, so the window may cut through the cartridge and
 *          its sink).  (Cartridges guide, "gemma4 (measured)": on a local-SWA
 *          layer a cartridge is visible exactly as a real prefix, within
 *          the window.)                                                  */
typedef struct cart_geom {
  int B, n, Hq, Hkv, d, p, frozen_prefix;
  float scale;
  double rope_theta;
  int window;
} cart_geom;

/* ------------------------------------------------------------------------
 * cart_write_to_cache -- write the whole cartridge into a cache, converting
 * f32 leaf rows to the cache dtype (round to nearest even for bf16).
 * (Cartridges guide, "Semantics", serving bullet: the prefix is written into
 * an empty KV cache, converted to the cache dtype, and the cache advances to
 * p.  The same conversion produces the bf16 shadow the attention kernels
 * read once per optimizer step.)
 *   kc, vc        [p, Hkv, d] f32 (device)
 *   k_dst, v_dst  destination rows; row r of the cartridge goes to row
 *                 dst_row0 + r, rows are row_stride_elems elements apart
 *                 (row_stride_elems >= Hkv*d, a multiple of 8)
 *   dst_dtype     CART_BF16 or CART_F32
 * Either pair member may be NULL to skip it (not both).                   */
CART_API int cart_write_to_cache(const float* kc, const float* vc, int p, int Hkv, int d, void* k_dst,
                        void* v_dst, long long row_stride_elems, int dst_row0,
                        cart_dtype dst_dtype, void* stream);

/* ------------------------------------------------------------------------
 * cart_attn_fwd -- training forward.
 *   q   [B, n, Hq, d]  in_dtype, NOT rotated (rotated in the library at p+i)
 *   k,v [B, n, Hkv, d] in_dtype, k NOT rotated
 *   kc, vc [p, Hkv, d] cart_dtype (bf16 shadow or f32 leaves), already in
 *          attended space (never rotated)
 *   o   [B, n, Hq, d]  in_dtype (output)
 *   lse [B, Hq, n]     f32 (output): natural-log log-sum-exp of the scaled
 *                      logits of each query row; the backward consumes it.
 * Arithmetic: bf16 tensor-core products with f32 accumulation; f32 inputs
 * are rounded to bf16 on load.  Workspace: cart_attn_fwd_workspace_size().  */
CART_API size_t cart_attn_fwd_workspace_size(const cart_geom* g, cart_dtype in_dtype,
                                    cart_dtype cart_dtype);
CART_API int cart_attn_fwd(const cart_geom* g, cart_dtype in_dtype, cart_dtype cart_dtype,
                  const void* q, const void* k, const void* v, const void* kc, const void* vc,
                  void* o, float* lse, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * cart_attn_bwd -- training backward through the concat into the cartridge.
 * (Cartridges guide, "Semantics": the backward routes gradients through the
 * concat into the trainable rows; row 0 is the frozen attention sink.)
 *   q,k,v,kc,vc,o,lse  as given to / returned by cart_attn_fwd
 *   dout [B, n, Hq, d] in_dtype: gradient of the loss w.r.t. o
 *   dq [B, n, Hq, d], dk, dv [B, n, Hkv, d]  in_dtype outputs, gradients
 *        w.r.t. the UN-rotated inputs q and k (the transpose rotation at
 *        position p+i is applied) and v
 *   dkc, dvc [p, Hkv, d] f32 outputs: gradient w.r.t. the cartridge rows,
 *        summed over the batch and over the query heads of each group.
 *        accumulate == 0 overwrites, 1 adds to the existing contents.  Rows
 *        < frozen_prefix are set to exactly 0.0 in both modes.
 * Workspace: cart_attn_bwd_workspace_size().                              */
CART_API size_t cart_attn_bwd_workspace_size(const cart_geom* g, cart_dtype in_dtype,
                                    cart_dtype cart_dtype);
CART_API int cart_attn_bwd(const cart_geom* g, cart_dtype in_dtype, cart_dtype cart_dtype,
                  const void* q, const void* k, const void* v, const void* kc, const void* vc,
                  const void* o, const float* lse, const void* dout, void* dq, void* dk,
                  void* dv, float* dkc, float* dvc, int accumulate, void* workspace,
                  size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * cart_attn_bwd_reuse -- cart_attn_bwd that takes the rotated queries and
 * keys, the RoPE table and the bf16 copies from the workspace of the
 * forward call that produced o and lse, instead of recomputing them.
 * (Cartridges guide, "Semantics": the backward of the same attention.)
 *   fwd_workspace [fwd_workspace_bytes]: the workspace passed to that
 *        cart_attn_fwd (same geometry, dtypes and inputs), read only; it
 *        must not have been reused since.  At least
 *        cart_attn_fwd_workspace_size() bytes, 16-byte aligned.
 *   workspace: cart_attn_bwd_reuse_workspace_size() bytes (the backward's
 *        own per-row vectors only).
 *   Everything else, outputs included, is as in cart_attn_bwd; the results
 *   are bit-identical to cart_attn_bwd on the same inputs.  The contents of
 *   fwd_workspace are not checked: a stale one gives wrong gradients.
 *   Returns CART_ERR_WORKSPACE for a missing or short workspace.         */
CART_API size_t cart_attn_bwd_reuse_workspace_size(const cart_geom* g, cart_dtype in_dtype,
                                                   cart_dtype cart_dtype);
CART_API int cart_attn_bwd_reuse(const cart_geom* g, cart_dtype in_dtype, cart_dtype cart_dtype,
                                 const void* q, const void* k, const void* v, const void* kc,
                                 const void* vc, const void* o, const float* lse,
                                 const void* dout, void* dq, void* dk, void* dv, float* dkc,
                                 float* dvc, int accumulate, const void* fwd_workspace,
                                 size_t fwd_workspace_bytes, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * cart_attn_bwd_parts -- cart_attn_bwd for a cartridge composed of several
 * independently trained parts concatenated along the rows, each with its
 * own frozen sink row.  (Cartridges guide, composition: parts are simply
 * concatenated, and every part keeps its sink.)
 *   frozen_rows [n_frozen] host int32: cartridge rows whose gradient is set
 *        to exactly 0.0 in both accumulate modes, in addition to the rows
 *        < frozen_prefix (e.g. each part's first row); any order, repeats
 *        allowed; 0 <= row < p; 0 <= n_frozen <= CART_MAX_FROZEN_ROWS.
 *        The list is copied into the launch: the caller may reuse it after
 *        the call returns.  frozen_rows may be NULL when n_frozen == 0.
 *   Everything else is as in cart_attn_bwd, which equals this call with
 *   n_frozen == 0.  Returns CART_ERR_GEOMETRY for a bad list.            */
#define CART_MAX_FROZEN_ROWS 64
CART_API int cart_attn_bwd_parts(const cart_geom* g, cart_dtype in_dtype, cart_dtype cart_dtype,
                                 const void* q, const void* k, const void* v, const void* kc,
                                 const void* vc, const void* o, const float* lse,
                                 const void* dout, void* dq, void* dk, void* dv, float* dkc,
                                 float* dvc, const int* frozen_rows, int n_frozen,
                                 int accumulate, void* workspace, size_t workspace_bytes,
                                 void* stream);

/* ------------------------------------------------------------------------
 * cart_attn_fwd_packed / cart_attn_bwd_packed -- training on packed
 * segments: the group's sequences lie back to back along ONE token axis
 * instead of in a [B, n] batch.  RoPE restarts in every segment (its token i
 * sits at position p + i) and attention runs per segment behind the one
 * shared cartridge, so each segment is exactly one sequence of
 * cart_attn_fwd / cart_attn_bwd.  (Cartridges guide, "Deliberate
 * divergences from the reference", packing bullet; "Batched self-study
 * (measured)", packed training step.)
 *   g->B   number of segments S;  g->n  the longest segment (an upper bound:
 *          it sizes the launch grids and the RoPE table)
 *   total  packed tokens T, 1 <= T <= S * n
 *   cu_seqlens [S + 1] DEVICE int32, 4-byte aligned: 0 = cu[0] <= cu[1] <=
 *          ... <= cu[S] = T, every segment cu[s+1] - cu[s] <= n (empty
 *          segments allowed).  A table that breaks these rules sets device
 *          status bit 6; the kernels clamp it so that every access stays
 *          inside the tensors (the results are then undefined).
 *   q, o, dout, dq [T, Hq, d]; k, v, dk, dv [T, Hkv, d] (dtypes as in the
 *          unpacked calls); lse [Hq, T] f32 (natural log), written by the
 *          forward and read by the backward.
 *   dkc, dvc [p, Hkv, d] f32: summed over every segment; frozen rows as in
 *          cart_attn_bwd_parts (frozen_rows may be NULL when n_frozen == 0).
 * Workspace: the *_packed_workspace_size() answers (0 for bad sizes).     */
CART_API size_t cart_attn_fwd_packed_workspace_size(const cart_geom* g, int total,
                                                    cart_dtype in_dtype, cart_dtype cart_dtype);
CART_API int cart_attn_fwd_packed(const cart_geom* g, int total, const int* cu_seqlens,
                                  cart_dtype in_dtype, cart_dtype cart_dtype, const void* q,
                                  const void* k, const void* v, const void* kc, const void* vc,
                                  void* o, float* lse, void* workspace, size_t workspace_bytes,
                                  void* stream);
CART_API size_t cart_attn_bwd_packed_workspace_size(const cart_geom* g, int total,
                                                    cart_dtype in_dtype, cart_dtype cart_dtype);
CART_API int cart_attn_bwd_packed(const cart_geom* g, int total, const int* cu_seqlens,
                                  cart_dtype in_dtype, cart_dtype cart_dtype, const void* q,
                                  const void* k, const void* v, const void* kc, const void* vc,
                                  const void* o, const float* lse, const void* dout, void* dq,
                                  void* dk, void* dv, float* dkc, float* dvc,
                                  const int* frozen_rows, int n_frozen, int accumulate,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * cart_attn_decode -- one q_seq = 1 decode step for B conversations behind
 * ONE shared cartridge.  (Cartridges guide, "Semantics", serving bullet: a
 * normal decode continues at position p with the training-time layout.)
 *   q      [B, Hq, d]  bf16, new token's query, NOT rotated
 *   k_new, v_new [B, Hkv, d] bf16, new token's key (NOT rotated) and value
 *   kc, vc [p, Hkv, d] bf16 shared cartridge (e.g. from cart_write_to_cache)
 *   k_cache, v_cache [B, cache_rows, Hkv, d] bf16 private caches; rows
 *          0..len[b]-1 hold already-rotated keys at positions p..p+len[b]-1
 *   priv_len [B] int32 (device): len[b], 0 <= len[b] < cache_rows (entries
 *          outside that range are clamped into it); cache_rows <= 32768 and
 *          p + cache_rows < 2^24
 *   o      [B, Hq, d] bf16 (output)
 * The new token sits at position p + len[b]: its rotated key and its value
 * are written to private row len[b], then it attends to the p cartridge rows
 * and private rows 0..len[b].  The caller advances len afterwards.
 * Workspace: cart_attn_decode_workspace_size().                           */
CART_API size_t cart_attn_decode_workspace_size(int B, int Hq, int Hkv, int d, int p, int cache_rows);
CART_API int cart_attn_decode(int B, int Hq, int Hkv, int d, int p, float scale, double rope_theta,
                     const void* q, const void* k_new, const void* v_new, const void* kc,
                     const void* vc, void* k_cache, void* v_cache, int cache_rows,
                     const int* priv_len, void* o, void* workspace, size_t workspace_bytes,
                     void* stream);

/* ------------------------------------------------------------------------
 * cart_attn_decode_span -- span verify: `span` consecutive new tokens per
 * conversation in one step (q_seq = span), behind the shared cartridge.
 * (Cartridges guide, "Batched self-study (measured)", the --spec-b bullet:
 * each stream's span of carried and drafted tokens attends to its own cache
 * behind the prefix in one pass; the mask is the end-aligned causal one.)
 *   q      [B, span, Hq, d] bf16, the span's queries, NOT rotated
 *   k_new, v_new [B, span, Hkv, d] bf16, the span's keys (NOT rotated) and
 *          values
 *   o      [B, span, Hq, d] bf16 (output)
 *   priv_len [B]: len[b], clamped into 0 <= len[b] <= cache_rows - span
 *   Token t of conversation b sits at position p + len[b] + t: the span's
 *   rotated keys and values are written to private rows len[b] .. len[b] +
 *   span - 1, and query t attends to the p cartridge rows and private rows
 *   0 .. len[b] + t.  Requires 1 <= span <= cache_rows and
 *   (Hq / Hkv) * span <= 32.  Everything else is as in cart_attn_decode,
 *   which equals this call with span == 1.
 *   window  sliding window in keys (0: none), as in cart_geom: token t
 *   sees the keys at positions p + len[b] + t - window + 1 .. p + len[b] + t.
 * Workspace: cart_attn_decode_span_workspace_size().                      */
CART_API size_t cart_attn_decode_span_workspace_size(int B, int span, int Hq, int Hkv, int d,
                                                     int p, int cache_rows);
CART_API int cart_attn_decode_span(int B, int span, int window, int Hq, int Hkv, int d, int p,
                                   float scale,
                                   double rope_theta, const void* q, const void* k_new,
                                   const void* v_new, const void* kc, const void* vc,
                                   void* k_cache, void* v_cache, int cache_rows,
                                   const int* priv_len, void* o, void* workspace,
                                   size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * cart_attn_decode_noalloc -- the decode step of cart_attn_decode for
 * callers that cannot allocate device memory: a serving loop running under a
 * fixed device-memory budget planned at start-up (a cudaMalloc on the decode
 * path would synchronize the device and stall the other streams), or a plain
 * C host that links only this library and has no device allocator to carve a
 * workspace from.  The paper has no counterpart; this is a library service.
 *   Arguments, layouts and results are those of cart_attn_decode, without
 *   the workspace: the scratch is a static device array of
 *   CART_DECODE_NOALLOC_SCRATCH_BYTES bytes that every GPU loading the
 *   library holds until the process exits.  (The 64-conversation, p = 4096,
 *   1025-row serving shape needs about 10 MiB.)
 *   Returns CART_ERR_WORKSPACE, without touching the device, when the
 *   problem needs more scratch than that; otherwise as cart_attn_decode.
 *   Calls no cudaMalloc / cudaFree or allocating library routine.
 *   The first call on each device looks up the array's device address (with
 *   that device current) and caches it; make that first call before any
 *   stream capture.  All calls share the one array: calls whose work can
 *   overlap on the GPU (other streams, or other host threads without
 *   ordering) race on it and must be serialised by the caller.  No scratch
 *   word needs to start at zero: each call writes what it reads.          */
#define CART_DECODE_NOALLOC_SCRATCH_BYTES (32u << 20)
CART_API int cart_attn_decode_noalloc(int B, int Hq, int Hkv, int d, int p, float scale,
                                      double rope_theta, const void* q, const void* k_new,
                                      const void* v_new, const void* kc, const void* vc,
                                      void* k_cache, void* v_cache, int cache_rows,
                                      const int* priv_len, void* o, void* stream);

/* Human-readable name of a cart_status value (static string). */
CART_API const char* cart_status_string(int status);

/* Reads (and with clear != 0 resets) the device status word that kernels set
 * when a bounded wait gives up (bit 0: a TMA copy, 1: an MMA, 2: the softmax
 * warps, 3: the epilogue), when a work schedule is inconsistent (bit 4), or
 * when the dynamic shared memory does not start 1024-byte aligned (bit 5;
 * the kernel then does nothing), or when a packed segment table breaks its
 * rules (bit 6).  Synchronizes the current device.  Writes
 * the bits to *bits_out (may be NULL); returns CART_OK, CART_ERR_TIMEOUT when
 * any bit is set, or CART_ERR_CUDA. */
CART_API int cart_device_status(unsigned* bits_out, int clear);

/* cart_release -- destroys the current device's helper stream and events
 * (created by the first cart_attn_bwd on that device; see the conventions
 * above) after waiting for the work queued on that stream.  The next
 * backward call creates them again.  Call it with no library call in
 * flight on the device from another host thread.  The library holds no
 * other per-device state besides the static scratch array of
 * cart_attn_decode_noalloc, which lives as long as the loaded library.
 * Returns CART_OK or CART_ERR_CUDA (no usable current device).            */
CART_API int cart_release(void);

/* ------------------------------------------------------------------------
 * Launch tracing (off by default).  cart_trace_enable(1) clears the trace
 * and starts recording: every later kernel launch of the library is
 * bracketed by two CUDA events recorded on the launching stream.
 * cart_trace_enable(0) stops recording and keeps what was recorded.
 * cart_trace_count() returns the number of recorded launches (at most
 * 65536).  cart_trace_get(i, ...) copies the kernel's name (NUL-terminated,
 * truncated to name_len) and, if ms != NULL, waits for launch i to finish
 * and writes its device time in milliseconds.  Not meant for use while a
 * stream is being captured into a CUDA graph. */
CART_API int cart_trace_enable(int on);
CART_API int cart_trace_count(void);
CART_API int cart_trace_get(int i, char* name, int name_len, float* ms);

#ifdef __cplusplus
}
#endif

#endif /* CARTATTN_H_ */
