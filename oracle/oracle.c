/*
 * oracle.c - plain float64 CPU oracle for blockwise exact attention.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg load this library; the CUDA library never does,
 * and the two share no source, header, table or helper.  It is slow on
 * purpose: every formula is written the way the pages define it, in double
 * precision, with no blocking, fusion or reordering beyond what the pages'
 * own definition states.  Compile with -ffp-contract=off (no FMA contraction)
 * and without -ffast-math.
 *
 * Sources (page title, section / function):
 *   [bpt]  "bpt.py" (Ring Attention / Blockwise Parallel Transformer):
 *          the commented einsum versions inside _ring_attention_fwd and
 *          _ring_attention_bwd (materialised softmax and its gradients),
 *          _blockwise_attention_fwd / scan_kv_block (the running
 *          max / numerator / denominator carry), _ring_attention_fwd
 *          (ring order: step idx uses KV block (my_idx - idx) mod n).
 *   [te]   "JAX: Single-GPU Attention with TransformerEngine", section 1
 *          (_repeat_kv_for_gqa, _make_causal_swa_mask,
 *          FlaxNativeGQAAttention): GQA head map, inclusive causal/window
 *          mask, scale d^-0.5 applied to fp32/f64 scores.
 *   [ann]  "AnnAttention", faiss_block_attention.py: select_block (block
 *          means, strictly earlier blocks, sorted indices) and
 *          faiss_block_attention (local window + selected blocks).
 *
 * Readings where the pages are silent or garbled (each is listed in the
 * design notes):
 *   - masked entries are excluded exactly (not added as finfo.min); a row with
 *     no allowed key gives O = 0, m = -inf, l = 0 and zero gradients;
 *   - the scale multiplies the f64 dot product; the bias is added after it;
 *   - the bias is indexed at global (q, k) positions; a bias dim of 1
 *     broadcasts (stride 0);
 *   - window bounds are inclusive, -1 means unbounded on either side, causal
 *     and window intersect, positions share one origin (top-left);
 *   - q head h reads kv head h / (Hq / Hkv);
 *   - block selection: block-mean Q against block-mean K by exact dot
 *     product over strictly earlier blocks; the sums (not means) rank the
 *     same; ties go to the lower block; fewer than top_n candidates pad
 *     with -1; the local window (keys q-W+1..q) and the selected blocks
 *     combine as a set union;
 *   - variable lengths ([te] section 1, SequenceDescriptor.from_seqlens):
 *     batch b holds Lq = seqlens_q[b] queries and Lk = seqlens_kv[b] keys
 *     (NULL: S; seqlens_kv NULL: the query lengths); later positions are
 *     padding, take part in nothing and get O = 0, m = -inf, l = 0 and zero
 *     gradients; the causal / window rule compares k with q + off, off = 0
 *     (top-left) or Lk - Lq (bottom-right: the queries are the last Lq
 *     positions of the key sequence);
 *   - sink attention ([te] "Other attention knobs", softmax_type off_by_one
 *     or learnable; the page names it without a formula): every valid row's
 *     softmax denominator gains exp(sink[h]), an extra logit with no value
 *     vector (off_by_one: sink = 0):  P = exp(z) / (exp(sink) + sum exp(z));
 *     m and l include it (m = max(max z, sink)), so a row with no allowed key
 *     has O = 0, m = sink, l = 1; the sink's gradient is
 *     dsink[h] = -sum over rows of P_sink * <dO, O>;
 *   - attention dropout ([bpt] _blockwise_attention_fwd / _bwd and the
 *     blockwise attention helper: a Bernoulli(p) mask over (batch, head, q, k)
 *     whose dropped entries get the dtype minimum added to the score, i.e.
 *     they leave the softmax, which renormalises over the kept keys; no
 *     1/(1-p) factor): the JAX generator is not available, so the mask comes
 *     from the counter-based generator Philox4x32-10 (Salmon, Moraes, Dror,
 *     Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011) with the
 *     64-bit seed as key and the position as counter, {k / 4, q, h, b}; word
 *     k % 4 of the output is the entry's 32-bit draw, and the entry is
 *     dropped when the draw is below the threshold p * 2^32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORA_F64 = 0, ORA_F32 = 1, ORA_BF16 = 2 };

typedef struct {
    int32_t B, S, Hq, Hkv, d, dv;
    double scale;
    int32_t causal, window_left, window_right;
    int32_t in_dtype;               /* dtype of q, k, v, dout */
    const double* bias;             /* NULL or f64, indexed with bias_strides */
    int64_t bias_strides[4];        /* b, h, q, k in elements; 0 broadcasts */
    const int32_t* block_idx;       /* NULL or [B][Hq][S/sel_block][top_n] */
    int32_t sel_block, top_n, local_window;
    const int32_t* seqlens_q;       /* NULL or [B]: valid queries per batch entry */
    const int32_t* seqlens_kv;      /* NULL or [B]: valid keys (NULL: seqlens_q) */
    int32_t bottom_right;           /* 1: causal / window diagonal at k = q + Lk - Lq */
    const double* sink;             /* NULL or [Hq]: extra softmax logit per q head */
    double* dsink;                  /* NULL or [Hq]: gradient of sink (written by ora_bwd) */
    uint32_t drop_threshold;        /* 0: no dropout; else drop entries whose draw < this */
    uint32_t drop_seed_lo, drop_seed_hi;
} ora_desc;

/* ---- element access: inputs are widened exactly to double ------------- */

static double widen(const void* p, int dt, int64_t i) {
    if (dt == ORA_F64) return ((const double*)p)[i];
    if (dt == ORA_F32) return (double)((const float*)p)[i];
    uint32_t u = ((uint32_t)((const uint16_t*)p)[i]) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* row r of head h at batch b of a contiguous [B][S][H][w] tensor */
static void load_row(double* dst, const void* src, int dt, int B_, int S, int H,
                     int w, int b, int s, int h) {
    (void)B_;
    int64_t base = (((int64_t)b * S + s) * H + h) * (int64_t)w;
    for (int c = 0; c < w; ++c) dst[c] = widen(src, dt, base + c);
}

/* K or V widened once, head-major: out[((b*Hkv + g)*S + k)*w + c] */
static double* widen_kv(const ora_desc* D, const void* src, int w) {
    int64_t n = (int64_t)D->B * D->Hkv * D->S * w;
    double* out = (double*)malloc((size_t)n * sizeof(double));
    if (!out) return NULL;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < D->B; ++b)
        for (int k = 0; k < D->S; ++k)
            for (int g = 0; g < D->Hkv; ++g) {
                int64_t s = (((int64_t)b * D->S + k) * D->Hkv + g) * (int64_t)w;
                int64_t t = (((int64_t)b * D->Hkv + g) * D->S + k) * (int64_t)w;
                for (int c = 0; c < w; ++c) out[t + c] = widen(src, D->in_dtype, s + c);
            }
    return out;
}

/* ---- Philox4x32-10 (the SC 2011 paper's definition) --------------------
 * One round maps the counter (c0, c1, c2, c3) with key (k0, k1) to
 *   (hi(B c2) ^ c1 ^ k0, lo(B c2), hi(A c0) ^ c3 ^ k1, lo(A c0))
 * with A = 0xD2511F53, B = 0xCD9E8D57 (hi / lo: the halves of the 64-bit
 * product); between rounds the key grows by the Weyl increments
 * (0x9E3779B9, 0xBB67AE85).  Ten rounds. */
static void philox4x32_10(const uint32_t ctr[4], uint32_t k0, uint32_t k1, uint32_t out[4]) {
    uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint64_t pa = (uint64_t)0xD2511F53u * c[0];
        const uint64_t pb = (uint64_t)0xCD9E8D57u * c[2];
        const uint32_t n0 = (uint32_t)(pb >> 32) ^ c[1] ^ k0;
        const uint32_t n1 = (uint32_t)pb;
        const uint32_t n2 = (uint32_t)(pa >> 32) ^ c[3] ^ k1;
        const uint32_t n3 = (uint32_t)pa;
        c[0] = n0;
        c[1] = n1;
        c[2] = n2;
        c[3] = n3;
    }
    for (int i = 0; i < 4; ++i) out[i] = c[i];
}

/* The 32-bit draw of score entry (b, h, q, k): counter {k / 4, q, h, b}, word k % 4. */
static uint32_t drop_draw(const ora_desc* D, int b, int h, int q, int k) {
    const uint32_t ctr[4] = {(uint32_t)k >> 2, (uint32_t)q, (uint32_t)h, (uint32_t)b};
    uint32_t out[4];
    philox4x32_10(ctr, D->drop_seed_lo, D->drop_seed_hi, out);
    return out[k & 3];
}

/* ---- the mask ([te] _make_causal_swa_mask; [bpt] causal; [ann]) -------- */

/* Valid query / key counts of batch entry b and the offset of the causal /
 * window diagonal. */
static void lengths(const ora_desc* D, int b, int* lq, int* lk, int* off) {
    int nq = D->seqlens_q ? D->seqlens_q[b] : D->S;
    int nk = D->seqlens_kv ? D->seqlens_kv[b] : nq;
    *lq = nq;
    *lk = nk;
    *off = D->bottom_right ? nk - nq : 0;
}

/* Keys that can be allowed for query q lie in [lo, hi]; used only to skip
 * keys that the length / causal / window rule excludes anyway. */
static void key_range(const ora_desc* D, int b, int q, int* lo, int* hi) {
    int lq, lk, off;
    lengths(D, b, &lq, &lk, &off);
    int a = 0, z = lk - 1, c = q + off;
    if (q >= lq) z = -1;
    if (D->causal && c < z) z = c;
    if (D->window_right >= 0 && c + D->window_right < z) z = c + D->window_right;
    if (D->window_left >= 0 && c - D->window_left > a) a = c - D->window_left;
    *lo = a;
    *hi = z;
}

static int allowed(const ora_desc* D, int b, int h, int q, int k) {
    int lq, lk, off;
    lengths(D, b, &lq, &lk, &off);
    if (q >= lq || k >= lk) return 0;
    if (D->causal && k > q + off) return 0;
    if (D->window_left >= 0 && k < q + off - D->window_left) return 0;
    if (D->window_right >= 0 && k > q + off + D->window_right) return 0;
    if (D->drop_threshold && drop_draw(D, b, h, q, k) < D->drop_threshold) return 0;   /* dropped */
    if (D->block_idx) {
        int in_local = (k <= q) && (k >= q - (D->local_window - 1));
        int in_sel = 0;
        int nblk = D->S / D->sel_block;
        const int32_t* sel =
            D->block_idx + (((int64_t)b * D->Hq + h) * nblk + q / D->sel_block) * D->top_n;
        for (int t = 0; t < D->top_n; ++t)
            if (sel[t] >= 0 && k / D->sel_block == sel[t]) in_sel = 1;
        if (!(in_local || in_sel)) return 0;
    }
    return 1;
}

static double bias_at(const ora_desc* D, int b, int h, int q, int k) {
    if (!D->bias) return 0.0;
    const int64_t* st = D->bias_strides;
    return D->bias[b * st[0] + h * st[1] + q * st[2] + k * st[3]];
}

/* Selection order: a larger score first.  A NaN score (only non-finite inputs give one;
 * the pages do not say how to rank it) ranks below every number. */
static int ranks_above(double a, double b) {
    if (isnan(b)) return !isnan(a);
    return a > b;
}

static double dot(const double* a, const double* b, int n) {
    double acc = 0.0;
    for (int c = 0; c < n; ++c) acc = acc + a[c] * b[c];
    return acc;
}

/* z = s * <q, k> + bias   ([bpt] scan_kv_block: scores / sqrt(d) + bias) */
static double score(const ora_desc* D, const double* qrow, const double* Kh, int b,
                    int h, int q, int k) {
    return D->scale * dot(qrow, Kh + (int64_t)k * D->d, D->d) + bias_at(D, b, h, q, k);
}

/* ---- one query row of the plain softmax definition ----------------------
 * m = max over allowed z, l = sum exp(z - m), O = sum (exp(z - m) / l) V.
 * z[] (length S) is scratch; entries for keys that are not allowed are
 * set to -inf.  Returns 0 when the row has no allowed key. */
static int row_forward(const ora_desc* D, const double* qrow, const double* Kh,
                       const double* Vh, int b, int h, int q, double* z, double* o,
                       double* m_out, double* l_out) {
    int lo, hi;
    key_range(D, b, q, &lo, &hi);
    double m = -INFINITY;
    int any = 0;
    for (int k = lo; k <= hi; ++k) {
        if (allowed(D, b, h, q, k)) {
            z[k] = score(D, qrow, Kh, b, h, q, k);
            if (z[k] > m) m = z[k];
            any = 1;
        } else {
            z[k] = -INFINITY;
        }
    }
    int lq, lk, off;
    lengths(D, b, &lq, &lk, &off);
    const int with_sink = D->sink != NULL && q < lq;   /* padding rows take part in nothing */
    const double sk = with_sink ? D->sink[h] : -INFINITY;
    if (sk > m) m = sk;
    for (int c = 0; c < D->dv; ++c) o[c] = 0.0;
    if (m == -INFINITY) {
        *m_out = -INFINITY;
        *l_out = 0.0;
        return 0;
    }
    double l = with_sink ? exp(sk - m) : 0.0;
    for (int k = lo; k <= hi; ++k)
        if (z[k] != -INFINITY) l = l + exp(z[k] - m);
    for (int k = lo; k <= hi; ++k) {
        if (z[k] == -INFINITY) continue;
        double p = exp(z[k] - m) / l;
        const double* vk = Vh + (int64_t)k * D->dv;
        for (int c = 0; c < D->dv; ++c) o[c] = o[c] + p * vk[c];
    }
    *m_out = m;
    *l_out = l;
    return any;
}

static const double* head(const double* X, const ora_desc* D, int b, int g, int w) {
    return X + ((int64_t)b * D->Hkv + g) * D->S * (int64_t)w;
}

/* ---- exported: one-shot forward ----------------------------------------- */

int ora_fwd(const ora_desc* D, const void* q, const void* k, const void* v, double* o,
            double* m, double* l) {
    double* Kw = widen_kv(D, k, D->d);
    double* Vw = widen_kv(D, v, D->dv);
    if (!Kw || !Vw) { free(Kw); free(Vw); return 1; }
    int G = D->Hq / D->Hkv;
    int64_t nrows = (int64_t)D->B * D->Hq * D->S;
    int fail = 0;
#pragma omp parallel
    {
        double* z = (double*)malloc((size_t)D->S * sizeof(double));
        double* qrow = (double*)malloc((size_t)D->d * sizeof(double));
        if (!z || !qrow) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t r = 0; r < nrows; ++r) {
                int b = (int)(r / ((int64_t)D->Hq * D->S));
                int h = (int)((r / D->S) % D->Hq);
                int s = (int)(r % D->S);
                int g = h / G;
                load_row(qrow, q, D->in_dtype, D->B, D->S, D->Hq, D->d, b, s, h);
                double* orow = o + (((int64_t)b * D->S + s) * D->Hq + h) * D->dv;
                int64_t ml = ((int64_t)b * D->Hq + h) * D->S + s;
                row_forward(D, qrow, head(Kw, D, b, g, D->d), head(Vw, D, b, g, D->dv), b, h,
                            s, z, orow, &m[ml], &l[ml]);
            }
        }
        free(z);
        free(qrow);
    }
    free(Kw);
    free(Vw);
    return fail;
}

/* ---- exported: backward from the plain definition -----------------------
 * ([bpt] commented einsum version in _ring_attention_bwd and
 *  _blockwise_attention_bwd):
 *   D  = <dO, O>            (O is this oracle's own forward output)
 *   P  = exp(z - m) / l,  dP = <dO, V_k>,  dS = P (dP - D)
 *   dQ = s sum_k dS K_k,  dK_k += s dS Q,  dV_k += P dO
 * summed over every q head of the kv head's group. */
int ora_bwd(const ora_desc* D, const void* q, const void* k, const void* v,
            const void* dout, double* dq, double* dk, double* dv, double* o_out,
            double* m_out, double* l_out) {
    double* Kw = widen_kv(D, k, D->d);
    double* Vw = widen_kv(D, v, D->dv);
    if (!Kw || !Vw) { free(Kw); free(Vw); return 1; }
    int G = D->Hq / D->Hkv;
    int units = D->B * D->Hkv;
    int fail = 0;
    memset(dq, 0, sizeof(double) * (size_t)D->B * D->S * D->Hq * D->d);
    memset(dk, 0, sizeof(double) * (size_t)D->B * D->S * D->Hkv * D->d);
    memset(dv, 0, sizeof(double) * (size_t)D->B * D->S * D->Hkv * D->dv);
    /* per (b, h) partial sums of the sink gradient, added in a fixed order at the end */
    double* ds_part = D->dsink ? (double*)calloc((size_t)D->B * D->Hq, sizeof(double)) : NULL;
    if (D->dsink && !ds_part) { free(Kw); free(Vw); return 1; }
#pragma omp parallel
    {
        double* z = (double*)malloc((size_t)D->S * sizeof(double));
        double* qrow = (double*)malloc((size_t)D->d * sizeof(double));
        double* dorow = (double*)malloc((size_t)D->dv * sizeof(double));
        double* orow = (double*)malloc((size_t)D->dv * sizeof(double));
        if (!z || !qrow || !dorow || !orow) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int u = 0; u < units; ++u) {
                int b = u / D->Hkv, g = u % D->Hkv;
                const double* Kh = head(Kw, D, b, g, D->d);
                const double* Vh = head(Vw, D, b, g, D->dv);
                for (int h = g * G; h < (g + 1) * G; ++h) {
                    for (int s = 0; s < D->S; ++s) {
                        double m, l;
                        load_row(qrow, q, D->in_dtype, D->B, D->S, D->Hq, D->d, b, s, h);
                        load_row(dorow, dout, D->in_dtype, D->B, D->S, D->Hq, D->dv, b, s, h);
                        int any = row_forward(D, qrow, Kh, Vh, b, h, s, z, orow, &m, &l);
                        int64_t ml = ((int64_t)b * D->Hq + h) * D->S + s;
                        if (o_out) {
                            double* od = o_out + (((int64_t)b * D->S + s) * D->Hq + h) * D->dv;
                            for (int c = 0; c < D->dv; ++c) od[c] = orow[c];
                        }
                        if (m_out) m_out[ml] = m;
                        if (l_out) l_out[ml] = l;
                        if (!any) continue;
                        double Dq = dot(dorow, orow, D->dv);
                        if (ds_part) ds_part[b * D->Hq + h] -= exp(D->sink[h] - m) / l * Dq;
                        double* dqrow = dq + (((int64_t)b * D->S + s) * D->Hq + h) * D->d;
                        int lo, hi;
                        key_range(D, b, s, &lo, &hi);
                        for (int kk = lo; kk <= hi; ++kk) {
                            if (z[kk] == -INFINITY) continue;
                            double P = exp(z[kk] - m) / l;
                            const double* kr = Kh + (int64_t)kk * D->d;
                            const double* vr = Vh + (int64_t)kk * D->dv;
                            double dP = dot(dorow, vr, D->dv);
                            double dS = P * (dP - Dq);
                            double* dkr = dk + (((int64_t)b * D->S + kk) * D->Hkv + g) * D->d;
                            double* dvr = dv + (((int64_t)b * D->S + kk) * D->Hkv + g) * D->dv;
                            for (int c = 0; c < D->d; ++c) {
                                dqrow[c] = dqrow[c] + D->scale * dS * kr[c];
                                dkr[c] = dkr[c] + D->scale * dS * qrow[c];
                            }
                            for (int c = 0; c < D->dv; ++c) dvr[c] = dvr[c] + P * dorow[c];
                        }
                    }
                }
            }
        }
        free(z);
        free(qrow);
        free(dorow);
        free(orow);
    }
    if (ds_part) {
        for (int h = 0; h < D->Hq; ++h) {
            double acc = 0.0;
            for (int b = 0; b < D->B; ++b) acc = acc + ds_part[b * D->Hq + h];
            D->dsink[h] = acc;
        }
        free(ds_part);
    }
    free(Kw);
    free(Vw);
    return fail;
}

/* ---- exported: the blockwise carry, literally ---------------------------
 * [bpt] _blockwise_attention_fwd / scan_kv_block and _ring_attention_fwd:
 * the queries are split into ring_size blocks (one per device of the ring);
 * query block i visits KV block (i - idx) mod n at step idx; inside a step
 * each query chunk folds the key chunks of that KV block in ascending order
 * into a running (max, numerator, denominator) carry:
 *   m' = max(m, rowmax z);  c = exp(m - m');  p = exp(z - m')
 *   num = num * c + p V;    den = den * c + rowsum p
 * A key chunk is skipped when no (query, key) pair of the chunk pair is
 * allowed (position-based skip).  A row whose running max is still -inf
 * keeps its carry.  At the end O = num / den. */
int ora_blockwise_fwd(const ora_desc* D, const void* q, const void* k, const void* v,
                      int32_t query_chunk, int32_t key_chunk, int32_t ring_size, double* o,
                      double* m_out, double* l_out) {
    int n = ring_size, S = D->S;
    if (n < 1 || S % n) return 2;
    int blk = S / n;
    if (query_chunk < 1 || key_chunk < 1 || blk % query_chunk || blk % key_chunk) return 2;
    double* Kw = widen_kv(D, k, D->d);
    double* Vw = widen_kv(D, v, D->dv);
    if (!Kw || !Vw) { free(Kw); free(Vw); return 1; }
    int G = D->Hq / D->Hkv;
    int nqc = S / query_chunk;
    int64_t units = (int64_t)D->B * D->Hq * nqc;
    int fail = 0;
#pragma omp parallel
    {
        int qc = query_chunk, kc = key_chunk;
        double* num = (double*)malloc((size_t)qc * D->dv * sizeof(double));
        double* den = (double*)malloc((size_t)qc * sizeof(double));
        double* mx = (double*)malloc((size_t)qc * sizeof(double));
        double* qrows = (double*)malloc((size_t)qc * D->d * sizeof(double));
        double* z = (double*)malloc((size_t)kc * sizeof(double));
        if (!num || !den || !mx || !qrows || !z) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t u = 0; u < units; ++u) {
                int b = (int)(u / ((int64_t)D->Hq * nqc));
                int h = (int)((u / nqc) % D->Hq);
                int c0 = (int)(u % nqc) * qc; /* first query of this chunk */
                int g = h / G;
                int i = c0 / blk; /* the ring device that holds this chunk */
                const double* Kh = head(Kw, D, b, g, D->d);
                const double* Vh = head(Vw, D, b, g, D->dv);
                for (int r = 0; r < qc; ++r) {
                    load_row(qrows + (int64_t)r * D->d, q, D->in_dtype, D->B, S, D->Hq, D->d, b,
                             c0 + r, h);
                    den[r] = 0.0;
                    mx[r] = -INFINITY;
                    for (int c = 0; c < D->dv; ++c) num[(int64_t)r * D->dv + c] = 0.0;
                }
                for (int idx = 0; idx < n; ++idx) {
                    int j = ((i - idx) % n + n) % n;
                    for (int k0 = j * blk; k0 < (j + 1) * blk; k0 += kc) {
                        int any = 0;
                        for (int r = 0; r < qc && !any; ++r)
                            for (int kk = 0; kk < kc && !any; ++kk)
                                if (allowed(D, b, h, c0 + r, k0 + kk)) any = 1;
                        if (!any) continue; /* skip by position */
                        for (int r = 0; r < qc; ++r) {
                            int qpos = c0 + r;
                            double cm = -INFINITY;
                            for (int kk = 0; kk < kc; ++kk) {
                                if (allowed(D, b, h, qpos, k0 + kk)) {
                                    z[kk] = score(D, qrows + (int64_t)r * D->d, Kh, b, h, qpos,
                                                  k0 + kk);
                                    if (z[kk] > cm) cm = z[kk];
                                } else {
                                    z[kk] = -INFINITY;
                                }
                            }
                            double mnew = mx[r] > cm ? mx[r] : cm;
                            if (mnew == -INFINITY) continue;
                            double corr = exp(mx[r] - mnew);
                            double* nr = num + (int64_t)r * D->dv;
                            for (int c = 0; c < D->dv; ++c) nr[c] = nr[c] * corr;
                            double rs = 0.0;
                            for (int kk = 0; kk < kc; ++kk) {
                                if (z[kk] == -INFINITY) continue;
                                double p = exp(z[kk] - mnew);
                                rs = rs + p;
                                const double* vk = Vh + (int64_t)(k0 + kk) * D->dv;
                                for (int c = 0; c < D->dv; ++c) nr[c] = nr[c] + p * vk[c];
                            }
                            den[r] = den[r] * corr + rs;
                            mx[r] = mnew;
                        }
                    }
                }
                for (int r = 0; r < qc; ++r) {
                    int s = c0 + r;
                    double* orow = o + (((int64_t)b * S + s) * D->Hq + h) * D->dv;
                    int64_t ml = ((int64_t)b * D->Hq + h) * S + s;
                    for (int c = 0; c < D->dv; ++c)
                        orow[c] = den[r] > 0.0 ? num[(int64_t)r * D->dv + c] / den[r] : 0.0;
                    m_out[ml] = mx[r];
                    l_out[ml] = den[r];
                }
            }
        }
        free(num);
        free(den);
        free(mx);
        free(qrows);
        free(z);
    }
    free(Kw);
    free(Vw);
    return fail;
}

/* ---- exported: sampled rows (for workloads too large for a full run) ----
 * rows[] holds (b, h, q) triples.  O, m, l and dQ of exactly those rows,
 * from the same definitions as ora_fwd / ora_bwd. */
int ora_rows(const ora_desc* D, const void* q, const void* k, const void* v,
             const void* dout, int32_t nrows, const int32_t* rows, double* o, double* m,
             double* l, double* dq) {
    double* Kw = widen_kv(D, k, D->d);
    double* Vw = widen_kv(D, v, D->dv);
    if (!Kw || !Vw) { free(Kw); free(Vw); return 1; }
    int G = D->Hq / D->Hkv;
    int fail = 0;
#pragma omp parallel
    {
        double* z = (double*)malloc((size_t)D->S * sizeof(double));
        double* qrow = (double*)malloc((size_t)D->d * sizeof(double));
        double* dorow = (double*)malloc((size_t)D->dv * sizeof(double));
        if (!z || !qrow || !dorow) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int r = 0; r < nrows; ++r) {
                int b = rows[3 * r], h = rows[3 * r + 1], s = rows[3 * r + 2];
                int g = h / G;
                const double* Kh = head(Kw, D, b, g, D->d);
                const double* Vh = head(Vw, D, b, g, D->dv);
                double* orow = o + (int64_t)r * D->dv;
                double* dqrow = dq ? dq + (int64_t)r * D->d : NULL;
                load_row(qrow, q, D->in_dtype, D->B, D->S, D->Hq, D->d, b, s, h);
                int any = row_forward(D, qrow, Kh, Vh, b, h, s, z, orow, &m[r], &l[r]);
                if (!dqrow) continue;
                for (int c = 0; c < D->d; ++c) dqrow[c] = 0.0;
                if (!any) continue;
                load_row(dorow, dout, D->in_dtype, D->B, D->S, D->Hq, D->dv, b, s, h);
                double Dq = dot(dorow, orow, D->dv);
                int lo, hi;
                key_range(D, b, s, &lo, &hi);
                for (int kk = lo; kk <= hi; ++kk) {
                    if (z[kk] == -INFINITY) continue;
                    double P = exp(z[kk] - m[r]) / l[r];
                    double dS = P * (dot(dorow, Vh + (int64_t)kk * D->dv, D->dv) - Dq);
                    const double* kr = Kh + (int64_t)kk * D->d;
                    for (int c = 0; c < D->d; ++c) dqrow[c] = dqrow[c] + D->scale * dS * kr[c];
                }
            }
        }
        free(z);
        free(qrow);
        free(dorow);
    }
    free(Kw);
    free(Vw);
    return fail;
}

/* dK and dV of the sampled keys keys[0..nkeys) of kv head g at batch b.
 * Every query row of the group that may attend to one of them is evaluated
 * in full (m, l, O, D), then each key sums its terms over those rows. */
int ora_keys(const ora_desc* D, const void* q, const void* k, const void* v,
             const void* dout, int32_t b, int32_t g, int32_t nkeys, const int32_t* keys,
             double* dk, double* dv) {
    double* Kw = widen_kv(D, k, D->d);
    double* Vw = widen_kv(D, v, D->dv);
    if (!Kw || !Vw) { free(Kw); free(Vw); return 1; }
    int G = D->Hq / D->Hkv, S = D->S;
    const double* Kh = head(Kw, D, b, g, D->d);
    const double* Vh = head(Vw, D, b, g, D->dv);
    int kmin = S;
    for (int t = 0; t < nkeys; ++t)
        if (keys[t] < kmin) kmin = keys[t];
    /* rows that may see a sampled key: all rows when there is no causal
     * rule or the diagonal is shifted, rows q >= kmin otherwise */
    int q0 = (D->causal && !D->bottom_right) ? kmin : 0;
    int nq = S - q0;
    int64_t nr = (int64_t)G * nq;
    double* M = (double*)malloc((size_t)nr * sizeof(double));
    double* L = (double*)malloc((size_t)nr * sizeof(double));
    double* Dv = (double*)malloc((size_t)nr * sizeof(double));
    int fail = (!M || !L || !Dv);
    if (!fail) {
#pragma omp parallel
        {
            double* z = (double*)malloc((size_t)S * sizeof(double));
            double* qrow = (double*)malloc((size_t)D->d * sizeof(double));
            double* dorow = (double*)malloc((size_t)D->dv * sizeof(double));
            double* orow = (double*)malloc((size_t)D->dv * sizeof(double));
            if (!z || !qrow || !dorow || !orow) {
#pragma omp atomic write
                fail = 1;
            } else {
#pragma omp for schedule(dynamic, 4)
                for (int64_t r = 0; r < nr; ++r) {
                    int h = g * G + (int)(r / nq), s = q0 + (int)(r % nq);
                    load_row(qrow, q, D->in_dtype, D->B, S, D->Hq, D->d, b, s, h);
                    load_row(dorow, dout, D->in_dtype, D->B, S, D->Hq, D->dv, b, s, h);
                    row_forward(D, qrow, Kh, Vh, b, h, s, z, orow, &M[r], &L[r]);
                    Dv[r] = dot(dorow, orow, D->dv);
                }
            }
            free(z);
            free(qrow);
            free(dorow);
            free(orow);
        }
    }
    if (!fail) {
#pragma omp parallel
        {
            double* qrow = (double*)malloc((size_t)D->d * sizeof(double));
            double* dorow = (double*)malloc((size_t)D->dv * sizeof(double));
            if (!qrow || !dorow) {
#pragma omp atomic write
                fail = 1;
            } else {
#pragma omp for schedule(dynamic, 1)
                for (int t = 0; t < nkeys; ++t) {
                    int kk = keys[t];
                    double* dkr = dk + (int64_t)t * D->d;
                    double* dvr = dv + (int64_t)t * D->dv;
                    for (int c = 0; c < D->d; ++c) dkr[c] = 0.0;
                    for (int c = 0; c < D->dv; ++c) dvr[c] = 0.0;
                    for (int64_t r = 0; r < nr; ++r) {
                        int h = g * G + (int)(r / nq), s = q0 + (int)(r % nq);
                        if (M[r] == -INFINITY || !allowed(D, b, h, s, kk)) continue;
                        load_row(qrow, q, D->in_dtype, D->B, S, D->Hq, D->d, b, s, h);
                        load_row(dorow, dout, D->in_dtype, D->B, S, D->Hq, D->dv, b, s, h);
                        double zz = score(D, qrow, Kh, b, h, s, kk);
                        double P = exp(zz - M[r]) / L[r];
                        double dP = dot(dorow, Vh + (int64_t)kk * D->dv, D->dv);
                        double dS = P * (dP - Dv[r]);
                        for (int c = 0; c < D->d; ++c) dkr[c] = dkr[c] + D->scale * dS * qrow[c];
                        for (int c = 0; c < D->dv; ++c) dvr[c] = dvr[c] + P * dorow[c];
                    }
                }
            }
            free(qrow);
            free(dorow);
        }
    }
    free(M);
    free(L);
    free(Dv);
    free(Kw);
    free(Vw);
    return fail;
}

/* ---- exported: exact top-n block selection ([ann] select_block) ---------
 * Per (b, h): Qs[i] = sum of the block_size rows of query block i, Ks[j]
 * likewise for keys (sums accumulate in row order; they rank exactly like
 * the means).  For j < i: score(i, j) = sum_c Qs[i][c] * Ks[j][c], summed in
 * channel order without fused multiply-add.  Block i keeps the min(top_n, i)
 * best scores (a larger score wins; equal scores keep the lower j), written
 * in ascending j, padded with -1.  Output [B][H][S/block_size][top_n]. */
int ora_select(const void* q, const void* k, int32_t in_dtype, int32_t B, int32_t S,
               int32_t H, int32_t d, int32_t block_size, int32_t top_n, int32_t* out) {
    if (block_size < 1 || S % block_size || top_n < 1) return 2;
    int nblk = S / block_size;
    int fail = 0;
#pragma omp parallel
    {
        double* Qs = (double*)malloc((size_t)nblk * d * sizeof(double));
        double* Ks = (double*)malloc((size_t)nblk * d * sizeof(double));
        double* sc = (double*)malloc((size_t)(nblk > 0 ? nblk : 1) * sizeof(double));
        int* pick = (int*)malloc((size_t)(nblk > 0 ? nblk : 1) * sizeof(int));
        if (!Qs || !Ks || !sc || !pick) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int u = 0; u < B * H; ++u) {
                int b = u / H, h = u % H;
                for (int i = 0; i < nblk; ++i)
                    for (int c = 0; c < d; ++c) {
                        double sq = 0.0, sk = 0.0;
                        for (int r = 0; r < block_size; ++r) {
                            int64_t e = (((int64_t)b * S + (int64_t)i * block_size + r) * H + h) * d + c;
                            sq = sq + widen(q, in_dtype, e);
                            sk = sk + widen(k, in_dtype, e);
                        }
                        Qs[(int64_t)i * d + c] = sq;
                        Ks[(int64_t)i * d + c] = sk;
                    }
                for (int i = 0; i < nblk; ++i) {
                    int32_t* dst = out + (((int64_t)b * H + h) * nblk + i) * top_n;
                    for (int j = 0; j < i; ++j) sc[j] = dot(Qs + (int64_t)i * d, Ks + (int64_t)j * d, d);
                    int take = i < top_n ? i : top_n;
                    /* repeated arg-max: the best remaining score, lowest j on ties */
                    for (int j = 0; j < i; ++j) pick[j] = 0;
                    for (int t = 0; t < take; ++t) {
                        int best = -1;
                        for (int j = 0; j < i; ++j) {
                            if (pick[j]) continue;
                            if (best < 0 || ranks_above(sc[j], sc[best])) best = j;
                        }
                        pick[best] = 1;
                    }
                    int w = 0;
                    for (int j = 0; j < i; ++j)
                        if (pick[j]) dst[w++] = j;
                    for (; w < top_n; ++w) dst[w] = -1;
                }
            }
        }
        free(Qs);
        free(Ks);
        free(sc);
        free(pick);
    }
    return fail;
}

/* The dropout decisions of one (b, h) block: keep[q * S + k] = 1 unless the
 * entry's draw falls below the threshold (positions only; other masks are not
 * applied).  For the pins. */
int ora_dropout_keep(const ora_desc* D, int32_t b, int32_t h, uint8_t* keep) {
    for (int q = 0; q < D->S; ++q)
        for (int k = 0; k < D->S; ++k)
            keep[(int64_t)q * D->S + k] = !(D->drop_threshold && drop_draw(D, b, h, q, k) < D->drop_threshold);
    return 0;
}

/* Philox4x32-10 itself, for the pins. */
int ora_philox4x32_10(const uint32_t* ctr, uint32_t k0, uint32_t k1, uint32_t* out) {
    philox4x32_10(ctr, k0, k1, out);
    return 0;
}

int ora_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
