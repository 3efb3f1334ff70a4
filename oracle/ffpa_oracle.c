/*
 * Float64 CPU oracle for exact scaled-dot-product attention: the forward
 * and, at the end of the file, its gradients.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the tests, the package smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table
 * or helper with the CUDA library.
 *
 * What it computes (FFPA API reference, "ffpa_attn.ffpa_attn_func",
 * description of `query`/`key`/`value`, `attn_mask`, `is_causal`, `scale`,
 * `enable_gqa` and "Returns"):
 *
 *   O = softmax(scale * Q K^T + mask) V            per (batch, query head)
 *
 *   - query head hq reads key/value head hq / (Hq / Hkv)  (grouped heads,
 *     the query head count is a whole multiple of the key/value head count);
 *   - a boolean mask keeps an element where it is true (a true entry takes
 *     part in the softmax); a floating mask is an additive bias;
 *   - is_causal: query row r sees key k only when k <= r + (Nkv - Nq)
 *     (the query rows line up with the end of the key sequence);
 *   - scale defaults to 1/sqrt(D) (chosen by the caller of this file).
 *
 * The log-sum-exp returned beside O is the natural logarithm of
 * sum_k exp(scale * q.k + mask) (FFPA API reference,
 * "ffpa_attn.ffpa_attn_varlen_func", `return_lse`: fp32, "CUDA convention").
 * A row whose every key is masked has no softmax; it is given O = 0 and
 * LSE = -inf (the FlashAttention convention; the pages say nothing).
 *
 * Packed variable-length input (FFPA API reference,
 * "ffpa_attn.ffpa_attn_varlen_func"): q is [T_q, H_q, D], k/v are
 * [T_k, H_kv, D]; sequence s owns rows cu_q[s]..cu_q[s+1]-1 of q and
 * cu_k[s]..cu_k[s+1]-1 of k/v, and is attended exactly like a dense
 * problem of those lengths (causal alignment is per sequence, lower right).
 * LSE is stored as [H_q, T_q].
 *
 * Inputs are read as the raw 16-bit patterns of bf16 or fp16 and widened
 * exactly to double; every sum, exponential and logarithm is in double.
 * No blocking, fusion or reordering beyond the definition above.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_BF16 = 0, ORACLE_FP16 = 1 };
enum { ORACLE_MASK_NONE = 0, ORACLE_MASK_BOOL = 1, ORACLE_MASK_F32 = 2, ORACLE_MASK_QTYPE = 3 };

/* bf16 is the top half of an IEEE binary32: widen by shifting. */
static double widen_bf16(uint16_t h) {
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* IEEE binary16: sign, 5-bit exponent (bias 15), 10-bit fraction. */
static double widen_fp16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -24);                 /* subnormal: frac * 2^-24 */
    else if (expo == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(frac | 0x400), expo - 25); /* (1024+frac) * 2^(e-15-10) */
    return sign ? -mag : mag;
}

static double widen(const uint16_t* p, int dtype) {
    return dtype == ORACLE_FP16 ? widen_fp16(*p) : widen_bf16(*p);
}

/* One attention row: query vector qrow (stride 1 over D, element stride
 * given), keys/values for n_keys rows.  mask_* describe this row's mask
 * entries over keys (stride mk_str, elements).  causal_limit is the
 * largest visible key index (or n_keys-1 when not causal).  Writes D
 * doubles to out and returns the LSE. */
static double attend_row(const uint16_t* qrow, const uint16_t* kbase, const uint16_t* vbase,
                         int64_t k_row_stride, int64_t v_row_stride, int n_keys, int D, int dtype, double scale,
                         int mask_kind, const void* mask_row, int64_t mk_str, int64_t causal_limit,
                         double* s /* scratch, n_keys */, double* out) {
    double m = -INFINITY;
    for (int kk = 0; kk < n_keys; ++kk) {
        const uint16_t* krow = kbase + (int64_t)kk * k_row_stride;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += widen(qrow + d, dtype) * widen(krow + d, dtype);
        double x = scale * dot;
        if (mask_kind == ORACLE_MASK_BOOL) {
            if (((const uint8_t*)mask_row)[kk * mk_str] == 0) x = -INFINITY;
        } else if (mask_kind == ORACLE_MASK_F32) {
            x += (double)((const float*)mask_row)[kk * mk_str];
        } else if (mask_kind == ORACLE_MASK_QTYPE) {
            x += widen((const uint16_t*)mask_row + kk * mk_str, dtype);
        }
        if ((int64_t)kk > causal_limit) x = -INFINITY;
        s[kk] = x;
        if (x > m) m = x;
    }
    if (m == -INFINITY) {               /* every key masked: no softmax */
        for (int d = 0; d < D; ++d) out[d] = 0.0;
        return -INFINITY;
    }
    double l = 0.0;
    for (int kk = 0; kk < n_keys; ++kk) {
        s[kk] = exp(s[kk] - m);         /* unnormalised weight */
        l += s[kk];
    }
    for (int d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int kk = 0; kk < n_keys; ++kk)
            acc += s[kk] * widen(vbase + (int64_t)kk * v_row_stride + d, dtype);
        out[d] = acc / l;
    }
    return m + log(l);
}

/*
 * Dense layout.  q: [B, Hq, Nq, D] with element strides q_str[4]; k, v:
 * [B, Hkv, Nkv, D] with k_str / v_str (the D stride must be 1 for all).
 * mask: broadcastable to [B, Hq, Nq, Nkv], element strides m_str[4]
 * (0 on a broadcast dimension), kind ORACLE_MASK_*.
 *
 * rows == NULL: every row; o is [B, Hq, Nq, D] and lse [B, Hq, Nq],
 * both contiguous.  Otherwise rows[r] is the flat index
 * (b*Hq + hq)*Nq + i of the r-th requested row; o is [nrows, D] and lse
 * [nrows].  Returns 0, or -1 on a bad argument.
 */
int oracle_attn_dense(const uint16_t* q, const uint16_t* k, const uint16_t* v, int dtype,
                      int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                      const int64_t* q_str, const int64_t* k_str, const int64_t* v_str,
                      const void* mask, int mask_kind, const int64_t* m_str,
                      double scale, int causal,
                      const int64_t* rows, int64_t nrows,
                      double* o, double* lse, int nthreads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || Nq < 0 || Nkv < 0 || D <= 0) return -1;
    const int group = Hq / Hkv;
    const int64_t total = rows ? nrows : (int64_t)B * Hq * Nq;
    int err = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(Nkv > 0 ? Nkv : 1));
        if (!s) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < total; ++r) {
            if (!s) continue;
            int64_t flat = rows ? rows[r] : r;
            int64_t i = flat % Nq;
            int64_t bh = flat / Nq;
            int hq = (int)(bh % Hq);
            int b = (int)(bh / Hq);
            int hk = hq / group;
            const uint16_t* qrow = q + b * q_str[0] + hq * q_str[1] + i * q_str[2];
            const uint16_t* kb = k + b * k_str[0] + hk * k_str[1];
            const uint16_t* vb = v + b * v_str[0] + hk * v_str[1];
            const void* mrow = NULL;
            int64_t mk = 0;
            if (mask_kind != ORACLE_MASK_NONE) {
                int64_t off = b * m_str[0] + hq * m_str[1] + i * m_str[2];
                size_t esz = mask_kind == ORACLE_MASK_BOOL ? 1 : mask_kind == ORACLE_MASK_F32 ? 4 : 2;
                mrow = (const char*)mask + off * (int64_t)esz;
                mk = m_str[3];
            }
            int64_t limit = causal ? i + (int64_t)Nkv - Nq : (int64_t)Nkv - 1;
            double* out = o + r * D;
            lse[r] = attend_row(qrow, kb, vb, k_str[2], v_str[2], Nkv, D, dtype, scale, mask_kind, mrow,
                                mk, limit, s, out);
        }
        free(s);
    }
    return err ? -1 : 0;
}

/*
 * Packed variable-length layout.  q: [Tq, Hq, D] (element strides
 * q_str[3] over T, H, D); k, v: [Tk, Hkv, D].  cu_q, cu_k: nseq+1 row
 * offsets (cu_k may equal cu_q).  o: [Tq, Hq, D] contiguous;
 * lse: [Hq, Tq] contiguous.  Returns 0, or -1 on a bad argument.
 */
int oracle_attn_varlen(const uint16_t* q, const uint16_t* k, const uint16_t* v, int dtype,
                       int Hq, int Hkv, int D,
                       const int64_t* q_str, const int64_t* k_str, const int64_t* v_str,
                       const int32_t* cu_q, const int32_t* cu_k, int nseq,
                       double scale, int causal, double* o, double* lse, int nthreads) {
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || nseq < 1) return -1;
    const int group = Hq / Hkv;
    const int64_t Tq = cu_q[nseq];
    int64_t maxk = 1;
    for (int sq = 0; sq < nseq; ++sq) {
        int64_t lk = cu_k[sq + 1] - cu_k[sq];
        if (cu_q[sq + 1] < cu_q[sq] || lk < 0) return -1;
        if (lk > maxk) maxk = lk;
    }
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)maxk);
        if (!s) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < Tq * Hq; ++r) {
            if (!s) continue;
            int64_t t = r / Hq;         /* packed query row */
            int hq = (int)(r % Hq);
            int sq = 0;                 /* owning sequence */
            while (!(t >= cu_q[sq] && t < cu_q[sq + 1])) ++sq;
            int64_t i = t - cu_q[sq];   /* row within the sequence */
            int64_t nq = cu_q[sq + 1] - cu_q[sq];
            int nk = cu_k[sq + 1] - cu_k[sq];
            int hk = hq / group;
            const uint16_t* qrow = q + t * q_str[0] + hq * q_str[1];
            const uint16_t* kb = k + (int64_t)cu_k[sq] * k_str[0] + hk * k_str[1];
            const uint16_t* vb = v + (int64_t)cu_k[sq] * v_str[0] + hk * v_str[1];
            int64_t limit = causal ? i + (int64_t)nk - nq : (int64_t)nk - 1;
            lse[(int64_t)hq * Tq + t] =
                attend_row(qrow, kb, vb, k_str[0], v_str[0], nk, D, dtype, scale, ORACLE_MASK_NONE, NULL,
                           0, limit, s, o + (t * Hq + hq) * D);
        }
        free(s);
    }
    return err ? -1 : 0;
}

/* ------------------------------------------------------------------ backward
 *
 * Gradients of the dense forward above (FFPA API reference,
 * "ffpa_attn.ffpa_attn_func": "Backward pass is supported via
 * FFPAAttnFunc"): for an upstream gradient dO of O, the derivatives of the
 * scalar L = sum(O * dO) with respect to Q, K and V.  The pages give no
 * formulas; these are the chain rule through the definition, per (batch,
 * query head, row i) with P_i = softmax(s_i) the weights of row i:
 *
 *   O_i    = sum_j P_ij V_j                =>  dV_j += P_ij dO_i
 *   dP_ij  = dO_i . V_j
 *   dS_ij  = P_ij (dP_ij - sum_k P_ik dP_ik)    (Jacobian of the softmax)
 *   s_ij   = scale q_i . k_j (+ mask)      =>  dQ_i  = scale sum_j dS_ij K_j
 *                                              dK_j += scale dS_ij Q_i
 *
 * Query heads of one group read the same key/value head, so their dK and dV
 * contributions add up there.  A masked score has P = 0 and contributes
 * nothing; a fully masked row (no softmax) contributes nothing either.
 */

/* Row statistics of query row i: scores s[] (masked entries -inf), the
 * weights P[] and dP[] over all keys, and returns sum_k P_k dP_k.  *dead is
 * set when every key is masked (then P = 0). */
static double grad_row(const uint16_t* qrow, const uint16_t* dorow, const uint16_t* kbase,
                       const uint16_t* vbase, int64_t k_row_stride, int64_t v_row_stride, int n_keys,
                       int D, int dtype, double scale, int mask_kind, const void* mask_row,
                       int64_t mk_str, int64_t causal_limit, double* P, double* dP, int* dead) {
    double m = -INFINITY;
    for (int kk = 0; kk < n_keys; ++kk) {
        const uint16_t* krow = kbase + (int64_t)kk * k_row_stride;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += widen(qrow + d, dtype) * widen(krow + d, dtype);
        double x = scale * dot;
        if (mask_kind == ORACLE_MASK_BOOL) {
            if (((const uint8_t*)mask_row)[kk * mk_str] == 0) x = -INFINITY;
        } else if (mask_kind == ORACLE_MASK_F32) {
            x += (double)((const float*)mask_row)[kk * mk_str];
        } else if (mask_kind == ORACLE_MASK_QTYPE) {
            x += widen((const uint16_t*)mask_row + kk * mk_str, dtype);
        }
        if ((int64_t)kk > causal_limit) x = -INFINITY;
        P[kk] = x;
        if (x > m) m = x;
    }
    *dead = m == -INFINITY;
    double l = 0.0;
    for (int kk = 0; kk < n_keys; ++kk) {
        P[kk] = *dead ? 0.0 : exp(P[kk] - m);
        l += P[kk];
    }
    double delta = 0.0;
    for (int kk = 0; kk < n_keys; ++kk) {
        if (!*dead) P[kk] /= l;
        const uint16_t* vrow = vbase + (int64_t)kk * v_row_stride;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += widen(dorow + d, dtype) * widen(vrow + d, dtype);
        dP[kk] = dot;
        delta += P[kk] * dot;
    }
    return delta;
}

/* Pointers of one dense row (b, hq, i): its query, upstream gradient, the
 * key/value bases of its head and its mask row. */
typedef struct {
    const uint16_t *qrow, *dorow, *kb, *vb;
    const void* mrow;
    int64_t mk, limit;
} dense_row;

static dense_row dense_row_at(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                              const uint16_t* dout, int Hq, int Hkv, int Nq, int Nkv,
                              const int64_t* q_str, const int64_t* k_str, const int64_t* v_str,
                              const int64_t* do_str, const void* mask, int mask_kind,
                              const int64_t* m_str, int causal, int b, int hq, int64_t i) {
    dense_row r;
    int hk = hq / (Hq / Hkv);
    r.qrow = q + b * q_str[0] + hq * q_str[1] + i * q_str[2];
    r.dorow = dout + b * do_str[0] + hq * do_str[1] + i * do_str[2];
    r.kb = k + b * k_str[0] + hk * k_str[1];
    r.vb = v + b * v_str[0] + hk * v_str[1];
    r.mrow = NULL;
    r.mk = 0;
    if (mask_kind != ORACLE_MASK_NONE) {
        int64_t off = b * m_str[0] + hq * m_str[1] + i * m_str[2];
        size_t esz = mask_kind == ORACLE_MASK_BOOL ? 1 : mask_kind == ORACLE_MASK_F32 ? 4 : 2;
        r.mrow = (const char*)mask + off * (int64_t)esz;
        r.mk = m_str[3];
    }
    r.limit = causal ? i + (int64_t)Nkv - Nq : (int64_t)Nkv - 1;
    return r;
}

/*
 * Full backward, dense layout.  dout has the layout of q (strides
 * do_str[4]).  dq: [B, Hq, Nq, D]; dk, dv: [B, Hkv, Nkv, D]; all three
 * contiguous float64.  One (batch, key/value head) per task, so the group's
 * additions into dK and dV never race.  Returns 0, or -1 on a bad argument.
 */
int oracle_attn_bwd_dense(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          const uint16_t* dout, int dtype, int B, int Hq, int Hkv, int Nq, int Nkv,
                          int D, const int64_t* q_str, const int64_t* k_str, const int64_t* v_str,
                          const int64_t* do_str, const void* mask, int mask_kind,
                          const int64_t* m_str, double scale, int causal, double* dq, double* dk,
                          double* dv, int nthreads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || Nq < 0 || Nkv < 0 || D <= 0) return -1;
    const int group = Hq / Hkv;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = 0;
#pragma omp parallel
    {
        size_t n = (size_t)(Nkv > 0 ? Nkv : 1);
        double* P = (double*)malloc(sizeof(double) * n);
        double* dP = (double*)malloc(sizeof(double) * n);
        if (!P || !dP) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < (int64_t)B * Hkv; ++u) {
            if (!P || !dP) continue;
            int b = (int)(u / Hkv), hk = (int)(u % Hkv);
            double* dkh = dk + u * Nkv * (int64_t)D;
            double* dvh = dv + u * Nkv * (int64_t)D;
            for (int64_t e = 0; e < (int64_t)Nkv * D; ++e) dkh[e] = dvh[e] = 0.0;
            for (int hq = hk * group; hq < (hk + 1) * group; ++hq) {
                for (int64_t i = 0; i < Nq; ++i) {
                    dense_row r = dense_row_at(q, k, v, dout, Hq, Hkv, Nq, Nkv, q_str, k_str, v_str,
                                               do_str, mask, mask_kind, m_str, causal, b, hq, i);
                    int dead;
                    double delta = grad_row(r.qrow, r.dorow, r.kb, r.vb, k_str[2], v_str[2], Nkv, D,
                                            dtype, scale, mask_kind, r.mrow, r.mk, r.limit, P, dP, &dead);
                    double* dqi = dq + (((int64_t)b * Hq + hq) * Nq + i) * D;
                    for (int d = 0; d < D; ++d) dqi[d] = 0.0;
                    if (dead) continue;
                    for (int kk = 0; kk < Nkv; ++kk) {
                        double ds = P[kk] * (dP[kk] - delta);
                        const uint16_t* krow = r.kb + (int64_t)kk * k_str[2];
                        for (int d = 0; d < D; ++d) {
                            dqi[d] += scale * ds * widen(krow + d, dtype);
                            dkh[(int64_t)kk * D + d] += scale * ds * widen(r.qrow + d, dtype);
                            dvh[(int64_t)kk * D + d] += P[kk] * widen(r.dorow + d, dtype);
                        }
                    }
                }
            }
        }
        free(P);
        free(dP);
    }
    return err ? -1 : 0;
}

/*
 * Sampled backward, dense layout, for problems too large for the full
 * routine.  q_rows[r] = (b*Hq + hq)*Nq + i selects dQ rows (dq: [nq_rows, D]);
 * k_rows[r] = (b*Hkv + hk)*Nkv + j selects dK/dV rows (dk, dv: [nk_rows, D]).
 * A dK/dV row needs, for every query row of its group, the row's softmax
 * and sum_k P dP; these are recomputed per query row from the definition.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_attn_bwd_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         const uint16_t* dout, int dtype, int B, int Hq, int Hkv, int Nq, int Nkv,
                         int D, const int64_t* q_str, const int64_t* k_str, const int64_t* v_str,
                         const int64_t* do_str, double scale, int causal,
                         const int64_t* q_rows, int64_t nq_rows, const int64_t* k_rows,
                         int64_t nk_rows, double* dq, double* dk, double* dv, int nthreads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || Nq < 0 || Nkv < 0 || D <= 0) return -1;
    const int group = Hq / Hkv;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = 0;
    for (int64_t e = 0; e < nk_rows * D; ++e) dk[e] = dv[e] = 0.0;
#pragma omp parallel
    {
        size_t n = (size_t)(Nkv > 0 ? Nkv : 1);
        double* P = (double*)malloc(sizeof(double) * n);
        double* dP = (double*)malloc(sizeof(double) * n);
        double* acc = (double*)calloc((size_t)(nk_rows > 0 ? nk_rows : 1) * 2 * (size_t)D,
                                      sizeof(double));
        if (!P || !dP || !acc) {
#pragma omp atomic write
            err = 1;
        }
        /* dQ rows: one row's softmax at a time. */
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < nq_rows; ++r) {
            if (!P || !dP || !acc) continue;
            int64_t flat = q_rows[r];
            int64_t i = flat % Nq, bh = flat / Nq;
            int hq = (int)(bh % Hq), b = (int)(bh / Hq);
            dense_row w = dense_row_at(q, k, v, dout, Hq, Hkv, Nq, Nkv, q_str, k_str, v_str, do_str,
                                       NULL, ORACLE_MASK_NONE, NULL, causal, b, hq, i);
            int dead;
            double delta = grad_row(w.qrow, w.dorow, w.kb, w.vb, k_str[2], v_str[2], Nkv, D, dtype,
                                    scale, ORACLE_MASK_NONE, NULL, 0, w.limit, P, dP, &dead);
            double* dqi = dq + r * D;
            for (int d = 0; d < D; ++d) dqi[d] = 0.0;
            if (dead) continue;
            for (int kk = 0; kk < Nkv; ++kk) {
                double ds = P[kk] * (dP[kk] - delta);
                const uint16_t* krow = w.kb + (int64_t)kk * k_str[2];
                for (int d = 0; d < D; ++d) dqi[d] += scale * ds * widen(krow + d, dtype);
            }
        }
        /* dK/dV rows: every query row of every (batch, query head) that
         * reads one of the selected key/value heads; each thread adds its
         * query rows' contributions into a private accumulator. */
#pragma omp for schedule(dynamic, 8)
        for (int64_t t = 0; t < (int64_t)B * Hq * Nq; ++t) {
            if (!P || !dP || !acc) continue;
            int64_t i = t % Nq, bh = t / Nq;
            int hq = (int)(bh % Hq), b = (int)(bh / Hq);
            int64_t head_kv = (int64_t)b * Hkv + hq / group;
            int wanted = 0;
            for (int64_t r = 0; r < nk_rows && !wanted; ++r) wanted = k_rows[r] / Nkv == head_kv;
            if (!wanted) continue;
            dense_row w = dense_row_at(q, k, v, dout, Hq, Hkv, Nq, Nkv, q_str, k_str, v_str, do_str,
                                       NULL, ORACLE_MASK_NONE, NULL, causal, b, hq, i);
            int dead;
            double delta = grad_row(w.qrow, w.dorow, w.kb, w.vb, k_str[2], v_str[2], Nkv, D, dtype,
                                    scale, ORACLE_MASK_NONE, NULL, 0, w.limit, P, dP, &dead);
            if (dead) continue;
            for (int64_t r = 0; r < nk_rows; ++r) {
                if (k_rows[r] / Nkv != head_kv) continue;
                int64_t j = k_rows[r] % Nkv;
                double ds = P[j] * (dP[j] - delta);
                double* ak = acc + r * 2 * D;
                double* av = ak + D;
                for (int d = 0; d < D; ++d) {
                    ak[d] += scale * ds * widen(w.qrow + d, dtype);
                    av[d] += P[j] * widen(w.dorow + d, dtype);
                }
            }
        }
#pragma omp critical
        {
            if (acc)
                for (int64_t r = 0; r < nk_rows; ++r)
                    for (int d = 0; d < D; ++d) {
                        dk[r * D + d] += acc[r * 2 * D + d];
                        dv[r * D + d] += acc[r * 2 * D + D + d];
                    }
        }
        free(P);
        free(dP);
        free(acc);
    }
    return err ? -1 : 0;
}

/*
 * Backward of the packed variable-length forward: q, dout [Tq, Hq, D]
 * (strides q_str[3], do_str[3] over T, H, D); k, v [Tk, Hkv, D]; cu_q,
 * cu_k as for oracle_attn_varlen.  Sequence s is differentiated exactly like
 * a dense problem of its own lengths (causal alignment lower right within
 * the sequence).  dq: [Tq, Hq, D]; dk, dv: [Tk, Hkv, D]; contiguous float64.
 * One (sequence, key/value head) per task.  Returns 0, or -1 on a bad
 * argument.
 */
int oracle_attn_bwd_varlen(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           const uint16_t* dout, int dtype, int Hq, int Hkv, int D,
                           const int64_t* q_str, const int64_t* k_str, const int64_t* v_str,
                           const int64_t* do_str, const int32_t* cu_q, const int32_t* cu_k, int nseq,
                           double scale, int causal, double* dq, double* dk, double* dv, int nthreads) {
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || nseq < 1) return -1;
    const int group = Hq / Hkv;
    int64_t maxk = 1;
    for (int sq = 0; sq < nseq; ++sq) {
        int64_t lk = cu_k[sq + 1] - cu_k[sq];
        if (cu_q[sq + 1] < cu_q[sq] || lk < 0) return -1;
        if (lk > maxk) maxk = lk;
    }
    const int64_t Tq = cu_q[nseq], Tk = cu_k[nseq];
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    for (int64_t e = 0; e < Tk * Hkv * D; ++e) dk[e] = dv[e] = 0.0;
    for (int64_t e = 0; e < Tq * Hq * D; ++e) dq[e] = 0.0;
    int err = 0;
#pragma omp parallel
    {
        double* P = (double*)malloc(sizeof(double) * (size_t)maxk);
        double* dP = (double*)malloc(sizeof(double) * (size_t)maxk);
        if (!P || !dP) {
#pragma omp atomic write
            err = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < (int64_t)nseq * Hkv; ++u) {
            if (!P || !dP) continue;
            int sq = (int)(u / Hkv), hk = (int)(u % Hkv);
            int64_t q0 = cu_q[sq], nq = cu_q[sq + 1] - cu_q[sq];
            int64_t k0 = cu_k[sq];
            int nk = cu_k[sq + 1] - cu_k[sq];
            const uint16_t* kb = k + k0 * k_str[0] + hk * k_str[1];
            const uint16_t* vb = v + k0 * v_str[0] + hk * v_str[1];
            for (int hq = hk * group; hq < (hk + 1) * group; ++hq) {
                for (int64_t i = 0; i < nq; ++i) {
                    const uint16_t* qrow = q + (q0 + i) * q_str[0] + hq * q_str[1];
                    const uint16_t* dorow = dout + (q0 + i) * do_str[0] + hq * do_str[1];
                    int64_t limit = causal ? i + (int64_t)nk - nq : (int64_t)nk - 1;
                    int dead;
                    double delta = grad_row(qrow, dorow, kb, vb, k_str[0], v_str[0], nk, D, dtype, scale,
                                            ORACLE_MASK_NONE, NULL, 0, limit, P, dP, &dead);
                    if (dead) continue;
                    double* dqi = dq + ((q0 + i) * Hq + hq) * D;
                    for (int kk = 0; kk < nk; ++kk) {
                        double ds = P[kk] * (dP[kk] - delta);
                        const uint16_t* krow = kb + (int64_t)kk * k_str[0];
                        double* dkr = dk + ((k0 + kk) * Hkv + hk) * D;
                        double* dvr = dv + ((k0 + kk) * Hkv + hk) * D;
                        for (int d = 0; d < D; ++d) {
                            dqi[d] += scale * ds * widen(krow + d, dtype);
                            dkr[d] += scale * ds * widen(qrow + d, dtype);
                            dvr[d] += P[kk] * widen(dorow + d, dtype);
                        }
                    }
                }
            }
        }
        free(P);
        free(dP);
    }
    return err ? -1 : 0;
}

/* ====================================================================
 * FP8 forward (FFPA README, "Backends" and "Latest News": FP8 attention
 * kernels for head dims 64..1024 that take bf16/fp16 tensors and return the
 * input type; the pages name scale folding but print no quantisation
 * formula, so the scheme below is this build's reading).
 *
 * Each of Q, K and V is quantised per (batch, head, block of 128 rows):
 *   amax = max |x| over the block's rows (those below N) and all D columns;
 *   if amax > 0 and 448 / amax is finite in float:
 *       inv = fl(448 / amax), s = fl(amax / 448)
 *   else inv = 0, s = 1;
 *   code(x) = e4m3(clamp(fl(x * inv), -448, 448)), rounded to nearest,
 *             ties to even (fl = one float operation, rounded to nearest);
 *   dequantised x = value(code) * s.
 * The FP8 attention is then the exact definition (in double) on the
 * dequantised Q, K and V, with the mask, scale, causal rule and GQA map of
 * the 16-bit path; its P is not rounded here (the kernel's e4m3 P is
 * covered by the tolerance the tests derive).
 * ==================================================================== */

enum { ORACLE_FP8_BLOCK = 128 };

/* e4m3 (1 sign, 4 exponent bits with bias 7, 3 fraction bits; no
 * infinities; largest finite 448 = 1.75 * 2^8; smallest subnormal 2^-9) of a
 * finite y with |y| <= 448, rounded to nearest, ties to even. */
static uint8_t e4m3_encode(float y) {
    const uint8_t sign = signbit(y) ? 0x80 : 0x00;
    const double a = fabs((double)y);
    if (a == 0.0) return sign;
    int e2;
    frexp(a, &e2);            /* a = f * 2^e2, f in [0.5, 1): a in [2^(e2-1), 2^e2) */
    const int E = e2 - 1;     /* a = 1.m * 2^E */
    if (E < -6) {             /* subnormal range: multiples of 2^-9 */
        const double q = nearbyint(ldexp(a, 9));   /* ties to even (default rounding mode) */
        return (uint8_t)(sign | (uint8_t)q);       /* q == 8 is the smallest normal, code 0x08 */
    }
    double q = nearbyint(ldexp(a, 3 - E));          /* eighths of 2^E: 8 .. 16 */
    int ex = E;
    if (q == 16.0) {
        q = 8.0;
        ++ex;
    }
    return (uint8_t)(sign | (uint8_t)((ex + 7) << 3) | (uint8_t)((int)q - 8));
}

static double e4m3_value(uint8_t c) {
    const int ex = (c >> 3) & 0x0f, fr = c & 0x07;
    const double mag = ex == 0 ? ldexp((double)fr, -9) : ldexp(8.0 + fr, ex - 10);
    return (c & 0x80) ? -mag : mag;
}

/* e4m3 codes of n floats (each clamped to [-448, 448] first). */
int oracle_e4m3_encode(const float* x, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) {
        float y = x[i];
        if (!(y == y)) return -1;
        if (y > 448.0f) y = 448.0f;
        if (y < -448.0f) y = -448.0f;
        out[i] = e4m3_encode(y);
    }
    return 0;
}

/* Quantises x [B, H, N, D] (element strides x_str, D stride 1) block by
 * block: codes [B, H, Npad, D] contiguous with Npad = N rounded up to 128
 * (rows >= N are zero), scales s [B, H, Npad/128] contiguous. */
int oracle_fp8_quantize(const uint16_t* x, int dtype, int B, int H, int N, int D,
                        const int64_t* x_str, uint8_t* codes, float* scales) {
    if (B < 0 || H <= 0 || N < 0 || D <= 0) return -1;
    const int nblk = (N + ORACLE_FP8_BLOCK - 1) / ORACLE_FP8_BLOCK;
    const int64_t npad = (int64_t)nblk * ORACLE_FP8_BLOCK;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int blk = 0; blk < nblk; ++blk) {
                const int r0 = blk * ORACLE_FP8_BLOCK;
                const int r1 = r0 + ORACLE_FP8_BLOCK < N ? r0 + ORACLE_FP8_BLOCK : N;
                const uint16_t* base = x + b * x_str[0] + h * x_str[1];
                float amax = 0.0f;
                for (int r = r0; r < r1; ++r)
                    for (int d = 0; d < D; ++d) {
                        const float a = (float)fabs(widen(base + (int64_t)r * x_str[2] + d, dtype));
                        if (a > amax) amax = a;
                    }
                float inv = 0.0f, s = 1.0f;
                if (amax > 0.0f && isfinite(448.0f / amax)) {
                    inv = 448.0f / amax;
                    s = amax / 448.0f;
                }
                scales[((int64_t)b * H + h) * nblk + blk] = s;
                uint8_t* out = codes + (((int64_t)b * H + h) * npad + r0) * D;
                for (int r = r0; r < r0 + ORACLE_FP8_BLOCK; ++r)
                    for (int d = 0; d < D; ++d) {
                        uint8_t c = 0;
                        if (r < r1) {
                            float y = (float)widen(base + (int64_t)r * x_str[2] + d, dtype) * inv;
                            if (y > 448.0f) y = 448.0f;
                            if (y < -448.0f) y = -448.0f;
                            c = e4m3_encode(y);
                        }
                        out[(int64_t)(r - r0) * D + d] = c;
                    }
            }
    return 0;
}

/* Dequantised [B, H, Npad, D] doubles of a quantised tensor. */
static double* fp8_dequantize(const uint8_t* codes, const float* scales, int B, int H, int N, int D) {
    const int nblk = (N + ORACLE_FP8_BLOCK - 1) / ORACLE_FP8_BLOCK;
    const int64_t npad = (int64_t)nblk * ORACLE_FP8_BLOCK;
    double* out = (double*)malloc(sizeof(double) * (size_t)((int64_t)B * H * npad * D + 1));
    if (!out) return NULL;
    for (int64_t bh = 0; bh < (int64_t)B * H; ++bh)
        for (int64_t r = 0; r < npad; ++r) {
            const double s = scales[bh * nblk + r / ORACLE_FP8_BLOCK];
            for (int d = 0; d < D; ++d)
                out[(bh * npad + r) * D + d] = e4m3_value(codes[(bh * npad + r) * D + d]) * s;
        }
    return out;
}

/* One attention row on double inputs (the definition, as attend_row). */
static double attend_row_f64(const double* qrow, const double* kbase, const double* vbase, int n_keys,
                             int D, double scale, int mask_kind, int dtype, const void* mask_row,
                             int64_t mk_str, int64_t causal_limit, double* s, double* out) {
    double m = -INFINITY;
    for (int kk = 0; kk < n_keys; ++kk) {
        const double* krow = kbase + (int64_t)kk * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qrow[d] * krow[d];
        double x = scale * dot;
        if (mask_kind == ORACLE_MASK_BOOL) {
            if (((const uint8_t*)mask_row)[kk * mk_str] == 0) x = -INFINITY;
        } else if (mask_kind == ORACLE_MASK_F32) {
            x += (double)((const float*)mask_row)[kk * mk_str];
        } else if (mask_kind == ORACLE_MASK_QTYPE) {
            x += widen((const uint16_t*)mask_row + kk * mk_str, dtype);
        }
        if ((int64_t)kk > causal_limit) x = -INFINITY;
        s[kk] = x;
        if (x > m) m = x;
    }
    if (m == -INFINITY) {
        for (int d = 0; d < D; ++d) out[d] = 0.0;
        return -INFINITY;
    }
    double l = 0.0;
    for (int kk = 0; kk < n_keys; ++kk) {
        s[kk] = exp(s[kk] - m);
        l += s[kk];
    }
    for (int d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int kk = 0; kk < n_keys; ++kk) acc += s[kk] * vbase[(int64_t)kk * D + d];
        out[d] = acc / l;
    }
    return m + log(l);
}

/* The FP8 forward's reference: quantise Q, K, V as above, then exact
 * attention on the dequantised values.  Arguments and outputs as for
 * oracle_attn_dense.  Returns 0, or -1 on a bad argument. */
int oracle_attn_fp8(const uint16_t* q, const uint16_t* k, const uint16_t* v, int dtype,
                    int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                    const int64_t* q_str, const int64_t* k_str, const int64_t* v_str,
                    const void* mask, int mask_kind, const int64_t* m_str,
                    double scale, int causal, const int64_t* rows, int64_t nrows,
                    double* o, double* lse, int nthreads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || Nq < 0 || Nkv < 0 || D <= 0) return -1;
    const int group = Hq / Hkv;
    const int64_t nqp = (int64_t)((Nq + ORACLE_FP8_BLOCK - 1) / ORACLE_FP8_BLOCK) * ORACLE_FP8_BLOCK;
    const int64_t nkp = (int64_t)((Nkv + ORACLE_FP8_BLOCK - 1) / ORACLE_FP8_BLOCK) * ORACLE_FP8_BLOCK;
    uint8_t* cq = (uint8_t*)malloc((size_t)((int64_t)B * Hq * nqp * D + 1));
    uint8_t* ck = (uint8_t*)malloc((size_t)((int64_t)B * Hkv * nkp * D + 1));
    uint8_t* cv = (uint8_t*)malloc((size_t)((int64_t)B * Hkv * nkp * D + 1));
    float* sq = (float*)malloc(sizeof(float) * (size_t)((int64_t)B * Hq * (nqp / ORACLE_FP8_BLOCK) + 1));
    float* sk = (float*)malloc(sizeof(float) * (size_t)((int64_t)B * Hkv * (nkp / ORACLE_FP8_BLOCK) + 1));
    float* sv = (float*)malloc(sizeof(float) * (size_t)((int64_t)B * Hkv * (nkp / ORACLE_FP8_BLOCK) + 1));
    double *dq = NULL, *dk = NULL, *dv = NULL;
    int err = !cq || !ck || !cv || !sq || !sk || !sv;
    if (!err)
        err = oracle_fp8_quantize(q, dtype, B, Hq, Nq, D, q_str, cq, sq) ||
              oracle_fp8_quantize(k, dtype, B, Hkv, Nkv, D, k_str, ck, sk) ||
              oracle_fp8_quantize(v, dtype, B, Hkv, Nkv, D, v_str, cv, sv);
    if (!err) {
        dq = fp8_dequantize(cq, sq, B, Hq, Nq, D);
        dk = fp8_dequantize(ck, sk, B, Hkv, Nkv, D);
        dv = fp8_dequantize(cv, sv, B, Hkv, Nkv, D);
        err = !dq || !dk || !dv;
    }
    const int64_t total = rows ? nrows : (int64_t)B * Hq * Nq;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    if (!err) {
#pragma omp parallel
        {
            double* s = (double*)malloc(sizeof(double) * (size_t)(Nkv > 0 ? Nkv : 1));
            if (!s) {
#pragma omp atomic write
                err = 1;
            }
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < total; ++r) {
                if (!s) continue;
                const int64_t flat = rows ? rows[r] : r;
                const int64_t i = flat % Nq;
                const int64_t bh = flat / Nq;
                const int hq = (int)(bh % Hq);
                const int b = (int)(bh / Hq);
                const int hk = hq / group;
                const double* qrow = dq + (((int64_t)b * Hq + hq) * nqp + i) * D;
                const double* kb = dk + ((int64_t)b * Hkv + hk) * nkp * D;
                const double* vb = dv + ((int64_t)b * Hkv + hk) * nkp * D;
                const void* mrow = NULL;
                int64_t mk = 0;
                if (mask_kind != ORACLE_MASK_NONE) {
                    const int64_t off = b * m_str[0] + hq * m_str[1] + i * m_str[2];
                    const size_t esz = mask_kind == ORACLE_MASK_BOOL ? 1 : mask_kind == ORACLE_MASK_F32 ? 4 : 2;
                    mrow = (const char*)mask + off * (int64_t)esz;
                    mk = m_str[3];
                }
                const int64_t limit = causal ? i + (int64_t)Nkv - Nq : (int64_t)Nkv - 1;
                lse[r] = attend_row_f64(qrow, kb, vb, Nkv, D, scale, mask_kind, dtype, mrow, mk, limit, s,
                                        o + r * D);
            }
            free(s);
        }
    }
    free(cq); free(ck); free(cv); free(sq); free(sk); free(sv);
    free(dq); free(dk); free(dv);
    return err ? -1 : 0;
}
