/*
 * cart_oracle.c -- plain fp64 CPU oracle for cartridge attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this code.  It shares nothing with the
 * CUDA path (no headers, helpers or tables) and is written as the plain
 * definition, loop by loop, so that it can be checked against the pages by eye.
 *
 * What it computes (Cartridges guide, section "Semantics"):
 *   - "Parameterization": a cartridge is a per-layer [p, kv_head, d] key/value
 *     pair in KV-cache row space; keys are already rotated at positions
 *     0..p-1 and are never rotated again; real tokens sit at RoPE positions
 *     p, p+1, ...; the first `frozen_prefix` rows (default 1, the attention
 *     sink) are frozen constants, the rest are trainable leaves.
 *   - "Attention": keys/values are concat(sink, trainable, tokens) along the
 *     sequence, attended by grouped attention with the end-aligned causal mask
 *     (source_offset = kv_seq - q_seq): every query sees the whole cartridge and
 *     is causal over real tokens.  The backward routes gradients through the
 *     concat into the trainable rows.
 *   - "Serving": the prefix is written into an empty cache and decoding
 *     continues at position p.
 *
 * Readings where the pages are silent:
 *   - RoPE is the rotate-half (NeoX / HF) form: element j pairs with j + d/2,
 *     angle = position * theta^(-2j/d).  Angles are computed in fp64.
 *   - GQA: query head h reads kv head h / (Hq / Hkv) (contiguous groups).
 *   - p counts the sink row.  Cartridge gradients are summed over the batch and
 *     over the query heads of each group; rows < frozen_prefix are exactly 0.
 *   - Real-token gradients dQ, dK, dV are returned in the pre-RoPE space of
 *     the inputs (the transpose rotation is applied to dQ and dK).
 *   - Decode: the private cache holds L_b already-rotated rows at positions
 *     p..p+L_b-1; the new token sits at position p+L_b, its key is rotated and
 *     appended at private row L_b, and it attends to p + L_b + 1 keys.
 *   - Sliding window (Cartridges guide, "gemma4 (measured)": on a local-SWA
 *     layer a served cartridge is visible exactly as a real prefix, within
 *     the window, so the window may cut through the cartridge): with
 *     window W > 0 a query at position P sees the keys at positions
 *     P - W + 1 .. P (W keys counting itself); cartridge row j sits at
 *     position j, so the sink gets no exemption.  W = 0: no window.
 *
 * Layouts (row-major, innermost last):
 *   q, o, dout, dq   [B, n, Hq, d]
 *   k, v, dk, dv     [B, n, Hkv, d]
 *   kc, vc, dkc, dvc [p, Hkv, d]
 *   lse              [B, Hq, n]   (natural log of sum_j exp(s_j))
 *
 * Parity: pinned by the "not gpu" tests (library attention with an explicit
 * mask matrix and a complex-number RoPE, central finite differences, the
 * p = 0 reduction to causal attention, the prefill-equivalence gate and
 * invariants).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int B, n, Hq, Hkv, d, p, frozen_prefix;
    double scale, theta;
    int window; /* sliding window in keys (0: none) */
} cart_ogeom;

/* First visible key (= key position) of the query at position pos. */
static int first_key(int pos, int window) {
    int lo = window > 0 ? pos - window + 1 : 0;
    return lo > 0 ? lo : 0;
}

/* ---- RoPE (rotate-half) --------------------------------------------------- */

/* y = R(pos) x ; with inverse != 0, y = R(pos)^T x (rotation by -angle). */
static void rope_vec(const double* x, double* y, int d, double pos, double theta,
                     int inverse) {
    int h = d / 2;
    for (int j = 0; j < h; ++j) {
        double inv_freq = pow(theta, -2.0 * (double)j / (double)d);
        double ang = pos * inv_freq;
        double c = cos(ang), s = sin(ang);
        if (inverse) s = -s;
        double x0 = x[j], x1 = x[j + h];
        y[j] = x0 * c - x1 * s;
        y[j + h] = x1 * c + x0 * s;
    }
}

/* out[r, hh, :] = R(pos0 + r) x[r, hh, :] for r < rows, hh < H. */
void cart_oracle_rope(const double* x, double* out, int rows, int H, int d,
                      double pos0, double theta, int inverse) {
    for (int r = 0; r < rows; ++r)
        for (int hh = 0; hh < H; ++hh)
            rope_vec(x + ((size_t)r * H + hh) * d, out + ((size_t)r * H + hh) * d, d,
                     pos0 + r, theta, inverse);
}

static int geom_ok(const cart_ogeom* g) {
    if (g->B < 1 || g->n < 0 || g->Hq < 1 || g->Hkv < 1 || g->d < 2 || (g->d & 1)) return 0;
    if (g->Hq % g->Hkv) return 0;
    if (g->p < 0 || g->frozen_prefix < 0 || g->frozen_prefix > g->p) return 0;
    if (g->p + g->n < 1) return 0;
    if (g->window < 0) return 0;
    return 1;
}

/* Keys and values of one (batch b, kv head kh) as the attention sees them:
 * rows 0..p-1 are the cartridge rows as stored, rows p..p+n-1 are the real
 * tokens, keys rotated at their position p + r. */
static void build_kv(const cart_ogeom* g, const double* k, const double* v,
                     const double* kc, const double* vc, int b, int kh,
                     double* kt, double* vt) {
    int d = g->d, p = g->p, n = g->n, Hkv = g->Hkv;
    for (int j = 0; j < p; ++j) {
        memcpy(kt + (size_t)j * d, kc + ((size_t)j * Hkv + kh) * d, sizeof(double) * d);
        memcpy(vt + (size_t)j * d, vc + ((size_t)j * Hkv + kh) * d, sizeof(double) * d);
    }
    for (int r = 0; r < n; ++r) {
        const double* kr = k + (((size_t)b * n + r) * Hkv + kh) * d;
        const double* vr = v + (((size_t)b * n + r) * Hkv + kh) * d;
        rope_vec(kr, kt + (size_t)(p + r) * d, d, (double)(p + r), g->theta, 0);
        memcpy(vt + (size_t)(p + r) * d, vr, sizeof(double) * d);
    }
}

/* ---- forward ------------------------------------------------------------- */

/* Computes o and lse for query heads [h_lo, h_hi) and query rows [i_lo, i_hi)
 * of every batch; other entries are left untouched.  Returns 0, or -1 on a bad
 * geometry or range. */
int cart_oracle_fwd(const cart_ogeom* g, const double* q, const double* k,
                    const double* v, const double* kc, const double* vc,
                    double* o, double* lse, int h_lo, int h_hi, int i_lo, int i_hi) {
    if (!geom_ok(g)) return -1;
    if (h_lo < 0 || h_hi > g->Hq || h_lo > h_hi || i_lo < 0 || i_hi > g->n || i_lo > i_hi)
        return -1;
    const int B = g->B, n = g->n, Hq = g->Hq, Hkv = g->Hkv, d = g->d, p = g->p;
    const int G = Hq / Hkv, kv = p + n;
    const int nh = h_hi - h_lo;
    int failed = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : failed)
    for (int t = 0; t < B * nh; ++t) {
        int b = t / nh, h = h_lo + t % nh, kh = h / G;
        double* kt = (double*)malloc(sizeof(double) * (size_t)kv * d);
        double* vt = (double*)malloc(sizeof(double) * (size_t)kv * d);
        double* qt = (double*)malloc(sizeof(double) * d);
        double* s = (double*)malloc(sizeof(double) * (size_t)(kv > 0 ? kv : 1));
        if (!kt || !vt || !qt || !s) { failed = 1; free(kt); free(vt); free(qt); free(s); continue; }
        build_kv(g, k, v, kc, vc, b, kh, kt, vt);
        for (int i = i_lo; i < i_hi; ++i) {
            const double* qi = q + (((size_t)b * n + i) * Hq + h) * d;
            rope_vec(qi, qt, d, (double)(p + i), g->theta, 0);
            /* end-aligned causal mask: key j is visible iff j <= i + (kv - n)
             * (key j sits at position j, query i at p + i = i + (kv - n)),
             * and within the window: j >= p + i - W + 1 */
            int nvis = i + (kv - n) + 1;
            int j0 = first_key(p + i, g->window);
            double m = -INFINITY;
            for (int j = j0; j < nvis; ++j) {
                double acc = 0.0;
                for (int c = 0; c < d; ++c) acc += qt[c] * kt[(size_t)j * d + c];
                s[j] = g->scale * acc;
                if (s[j] > m) m = s[j];
            }
            double l = 0.0;
            for (int j = j0; j < nvis; ++j) { s[j] = exp(s[j] - m); l += s[j]; }
            /* o_i = sum_j softmax_j * v_j */
            double* oi = o + (((size_t)b * n + i) * Hq + h) * d;
            for (int c = 0; c < d; ++c) oi[c] = 0.0;
            for (int j = j0; j < nvis; ++j) {
                double w = s[j] / l;
                for (int c = 0; c < d; ++c) oi[c] += w * vt[(size_t)j * d + c];
            }
            lse[((size_t)b * Hq + h) * n + i] = m + log(l);
        }
        free(kt); free(vt); free(qt); free(s);
    }
    return failed ? -2 : 0;
}

/* ---- backward ------------------------------------------------------------ */

/* Gradients of sum(dout * o) for kv heads [kh_lo, kh_hi) and the query heads
 * that read them, counting only the query rows [i_lo, i_hi) of the loss (the
 * full gradient when the range is [0, n)).  dq of rows outside the range and
 * entries of other heads are untouched; dk/dv/dkc/dvc of the selected kv
 * heads are overwritten (cartridge rows summed over the batch). */
int cart_oracle_bwd(const cart_ogeom* g, const double* q, const double* k,
                    const double* v, const double* kc, const double* vc,
                    const double* dout, double* dq, double* dk, double* dv,
                    double* dkc, double* dvc, int kh_lo, int kh_hi, int i_lo, int i_hi) {
    if (!geom_ok(g)) return -1;
    if (kh_lo < 0 || kh_hi > g->Hkv || kh_lo > kh_hi) return -1;
    if (i_lo < 0 || i_hi > g->n || i_lo > i_hi) return -1;
    const int B = g->B, n = g->n, Hq = g->Hq, Hkv = g->Hkv, d = g->d, p = g->p;
    const int G = Hq / Hkv, kv = p + n;
    const int nk = kh_hi - kh_lo;
    /* per (b, kv head) gradient w.r.t. the attended (rotated) keys and values */
    double* dkt_all = (double*)calloc((size_t)B * nk * kv * d, sizeof(double));
    double* dvt_all = (double*)calloc((size_t)B * nk * kv * d, sizeof(double));
    if (!dkt_all || !dvt_all) { free(dkt_all); free(dvt_all); return -2; }
    int failed = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : failed)
    for (int t = 0; t < B * nk; ++t) {
        int b = t / nk, kh = kh_lo + t % nk;
        double* dkt = dkt_all + (size_t)t * kv * d;
        double* dvt = dvt_all + (size_t)t * kv * d;
        double* kt = (double*)malloc(sizeof(double) * (size_t)kv * d);
        double* vt = (double*)malloc(sizeof(double) * (size_t)kv * d);
        double* qt = (double*)malloc(sizeof(double) * d);
        double* dqt = (double*)malloc(sizeof(double) * d);
        double* a = (double*)malloc(sizeof(double) * (size_t)kv);
        double* dp = (double*)malloc(sizeof(double) * (size_t)kv);
        if (!kt || !vt || !qt || !dqt || !a || !dp) {
            failed = 1; free(kt); free(vt); free(qt); free(dqt); free(a); free(dp); continue;
        }
        build_kv(g, k, v, kc, vc, b, kh, kt, vt);
        for (int h = kh * G; h < (kh + 1) * G; ++h) {
            for (int i = i_lo; i < i_hi; ++i) {
                const double* qi = q + (((size_t)b * n + i) * Hq + h) * d;
                const double* gi = dout + (((size_t)b * n + i) * Hq + h) * d;
                rope_vec(qi, qt, d, (double)(p + i), g->theta, 0);
                int nvis = i + (kv - n) + 1;
                int j0 = first_key(p + i, g->window);
                /* attention weights a_j = softmax_j(scale * qt . kt_j) */
                double m = -INFINITY;
                for (int j = j0; j < nvis; ++j) {
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c) acc += qt[c] * kt[(size_t)j * d + c];
                    a[j] = g->scale * acc;
                    if (a[j] > m) m = a[j];
                }
                double l = 0.0;
                for (int j = j0; j < nvis; ++j) { a[j] = exp(a[j] - m); l += a[j]; }
                for (int j = j0; j < nvis; ++j) a[j] /= l;
                /* d(loss)/d(a_j) = dout . vt_j ; softmax Jacobian:
                 * d(loss)/d(s_j) = a_j (dp_j - sum_k a_k dp_k) */
                double Dsum = 0.0;
                for (int j = j0; j < nvis; ++j) {
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c) acc += gi[c] * vt[(size_t)j * d + c];
                    dp[j] = acc;
                    Dsum += a[j] * acc;
                }
                for (int c = 0; c < d; ++c) dqt[c] = 0.0;
                for (int j = j0; j < nvis; ++j) {
                    double ds = a[j] * (dp[j] - Dsum);
                    for (int c = 0; c < d; ++c) {
                        dqt[c] += g->scale * ds * kt[(size_t)j * d + c];
                        dkt[(size_t)j * d + c] += g->scale * ds * qt[c];
                        dvt[(size_t)j * d + c] += a[j] * gi[c];
                    }
                }
                /* back through the rotation of q at position p + i */
                rope_vec(dqt, dq + (((size_t)b * n + i) * Hq + h) * d, d, (double)(p + i),
                         g->theta, 1);
            }
        }
        /* real-token rows: back through the key rotation at position p + r */
        for (int r = 0; r < n; ++r) {
            rope_vec(dkt + (size_t)(p + r) * d, dk + (((size_t)b * n + r) * Hkv + kh) * d, d,
                     (double)(p + r), g->theta, 1);
            memcpy(dv + (((size_t)b * n + r) * Hkv + kh) * d, dvt + (size_t)(p + r) * d,
                   sizeof(double) * d);
        }
        free(kt); free(vt); free(qt); free(dqt); free(a); free(dp);
    }
    if (!failed) {
        /* cartridge rows: the rows are leaves as stored (no rotation to undo);
         * sum over the batch; frozen rows get exactly zero */
        for (int kh = kh_lo; kh < kh_hi; ++kh) {
            for (int j = 0; j < p; ++j) {
                double* gk = dkc + ((size_t)j * Hkv + kh) * d;
                double* gv = dvc + ((size_t)j * Hkv + kh) * d;
                for (int c = 0; c < d; ++c) { gk[c] = 0.0; gv[c] = 0.0; }
                if (j < g->frozen_prefix) continue;
                for (int b = 0; b < B; ++b) {
                    size_t t = (size_t)b * nk + (kh - kh_lo);
                    const double* sk = dkt_all + (t * kv + j) * d;
                    const double* sv = dvt_all + (t * kv + j) * d;
                    for (int c = 0; c < d; ++c) { gk[c] += sk[c]; gv[c] += sv[c]; }
                }
            }
        }
    }
    free(dkt_all); free(dvt_all);
    return failed ? -2 : 0;
}

/* ---- decode behind a shared cartridge ------------------------------------ */

/* q [B, Hq, d], k_new/v_new [B, Hkv, d] (un-rotated new token), shared
 * kc/vc [p, Hkv, d], private caches [B, rows, Hkv, d] holding already-rotated
 * rows 0..len[b]-1.  Writes the new token's rotated key and its value at
 * private row len[b] (so rows must exceed len[b]) and o [B, Hq, d]. */
int cart_oracle_decode(int B, int Hq, int Hkv, int d, int p, double scale, double theta,
                       const double* q, const double* k_new, const double* v_new,
                       const double* kc, const double* vc, double* k_cache,
                       double* v_cache, int rows, const int* len, double* o, int window) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || d < 2 || (d & 1) || p < 0 || rows < 1 ||
        window < 0)
        return -1;
    for (int b = 0; b < B; ++b)
        if (len[b] < 0 || len[b] >= rows) return -1;
    const int G = Hq / Hkv;
    for (int b = 0; b < B; ++b)
        for (int kh = 0; kh < Hkv; ++kh) {
            double pos = (double)(p + len[b]);
            double* krow = k_cache + (((size_t)b * rows + len[b]) * Hkv + kh) * d;
            double* vrow = v_cache + (((size_t)b * rows + len[b]) * Hkv + kh) * d;
            rope_vec(k_new + ((size_t)b * Hkv + kh) * d, krow, d, pos, theta, 0);
            memcpy(vrow, v_new + ((size_t)b * Hkv + kh) * d, sizeof(double) * d);
        }
    int failed = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : failed)
    for (int t = 0; t < B * Hq; ++t) {
        int b = t / Hq, h = t % Hq, kh = h / G;
        int nkey = p + len[b] + 1;
        int j0 = first_key(p + len[b], window); /* keys j0 .. p + len[b] */
        double* qt = (double*)malloc(sizeof(double) * d);
        double* s = (double*)malloc(sizeof(double) * (size_t)nkey);
        if (!qt || !s) { failed = 1; free(qt); free(s); continue; }
        rope_vec(q + ((size_t)b * Hq + h) * d, qt, d, (double)(p + len[b]), theta, 0);
        double m = -INFINITY;
        for (int j = j0; j < nkey; ++j) {
            const double* kj = j < p ? kc + ((size_t)j * Hkv + kh) * d
                                     : k_cache + (((size_t)b * rows + (j - p)) * Hkv + kh) * d;
            double acc = 0.0;
            for (int c = 0; c < d; ++c) acc += qt[c] * kj[c];
            s[j] = scale * acc;
            if (s[j] > m) m = s[j];
        }
        double l = 0.0;
        for (int j = j0; j < nkey; ++j) l += exp(s[j] - m);
        double* ob = o + ((size_t)b * Hq + h) * d;
        for (int c = 0; c < d; ++c) ob[c] = 0.0;
        for (int j = j0; j < nkey; ++j) {
            const double* vj = j < p ? vc + ((size_t)j * Hkv + kh) * d
                                     : v_cache + (((size_t)b * rows + (j - p)) * Hkv + kh) * d;
            double w = exp(s[j] - m) / l;
            for (int c = 0; c < d; ++c) ob[c] += w * vj[c];
        }
        free(qt); free(s);
    }
    return failed ? -2 : 0;
}

/* ---- cache write: f32 -> bf16, round to nearest, ties to even ------------ */

/* bf16 keeps the top 16 bits of an IEEE binary32.  Rounding to nearest with
 * ties to even adds 0x7FFF plus the lowest kept bit before truncating; NaNs
 * are kept quiet.  Destination rows dst_row0 .. dst_row0 + p - 1 of a buffer
 * whose rows are row_stride elements apart receive the p * Hkv * d values. */
static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

void cart_oracle_write_to_cache(const float* src, int p, int Hkv, int d, uint16_t* dst,
                                long long row_stride, int dst_row0) {
    for (int j = 0; j < p; ++j)
        for (int e = 0; e < Hkv * d; ++e)
            dst[(size_t)(dst_row0 + j) * row_stride + e] = f32_to_bf16_rne(src[(size_t)j * Hkv * d + e]);
}

int cart_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
