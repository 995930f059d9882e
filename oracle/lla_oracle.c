/*
 * Plain CPU oracle for the causal log-linear Mamba-2 attention operator and
 * for its Gated DeltaNet counterpart (end of the file).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it. It shares no code with the CUDA library.
 *
 * Everything is fp64, single-threaded, and written as the definition reads,
 * without blocking, fusion or reordering.
 *
 * Sources ("Log-Linear Attention", gist.science summaries of arXiv 2506.04761,
 * pages in Portuguese (pt) and French (fr)):
 *   - pt §2 "Particionamento Hierarquico (Arvore Fenwick)" and fr §2
 *     "Partitionnement par Arbre de Fenwick": the prefix of each query is cut
 *     into Fenwick-tree buckets of sizes 1, 2, 4, 8, ...; O(log T) of them are
 *     active at any time t.
 *   - pt §2 "Mascara Hierarquica (M_H)" and fr §2 "Matrice de Masque
 *     Hierarchique": O = (Q K^T (.) M_H) V, with one data-dependent weight
 *     lambda_t^(l) per level l of query t.
 *   - pt §2 "Generalizacao" and fr §3 "Cadre General": the hierarchical mask
 *     is applied on top of a linear-attention variant's own mask; for Mamba-2
 *     that is the semiseparable scalar-decay mask M^S.
 *   - pt §2 "Forma Recorrente e Paralela" and fr §2 "Algorithmes Efficaces"
 *     (Inference): the decode keeps O(log T) states S_t^(l); each new token
 *     updates the finest level and the levels are merged along the Fenwick
 *     structure.
 *
 * Readings taken where the pages are silent:
 *   - positions are 0-indexed; the query token itself is its own level 0;
 *   - M^S[t,s] = prod_{r=s+1..t} a_r (exclusive of s, so the diagonal is 1);
 *   - lambda is indexed by the query: lambda[b,h,t,l];
 *   - no 1/sqrt(d) scale, no normalisation, no gating beyond M^S.
 *
 * Layouts are row-major: q,k [B,H,T,dk]; v,out [B,H,T,dv]; log_a [B,H,T];
 * lambda [B,H,T,L]. Decode: q,k [B,H,dk]; v,out [B,H,dv]; log_a [B,H];
 * lambda [B,H,Lmax]; states [B,H,Lmax,dk,dv]; t [B].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Fenwick bucket of key s for query t (s <= t), found by walking the Fenwick
 * decomposition of t's prefix: the query token alone is level 0; then, from
 * b = t, the bucket [b - lowbit(b), b) holds 2^(l-1) keys and has level
 * l = log2(lowbit(b)) + 1, and b steps down to b - lowbit(b). Returns -1 when
 * s > t (the key is in the future). */
int lla_oracle_level(int64_t t, int64_t s)
{
    if (s > t || s < 0) return -1;
    if (s == t) return 0;
    int64_t b = t;
    while (b > 0) {
        int64_t low = b & (-b);
        int level = 1;
        for (int64_t w = low; w > 1; w >>= 1) level++;
        if (s >= b - low && s < b) return level;
        b -= low;
    }
    return -1; /* unreachable for 0 <= s < t */
}

/* Number of Fenwick levels for a sequence of length T: the largest level any
 * (t, s) pair reaches, plus one, found by enumeration. */
int lla_oracle_num_levels(int64_t T)
{
    int best = 0;
    for (int64_t t = 0; t < T; t++)
        for (int64_t s = 0; s <= t; s++) {
            int l = lla_oracle_level(t, s);
            if (l > best) best = l;
        }
    return T > 0 ? best + 1 : 0;
}

/* Explicit O(T^2) form: for every query t,
 *   o_t = sum_{s<=t} lambda_t^(l(t,s)) * exp(sum_{r=s+1..t} log_a_r) * (q_t . k_s) * v_s,
 * i.e. row t of (Q K^T (.) M^S (.) M^H) V. The decay exponent is accumulated
 * while s walks down from t, so it is the plain sum over r in (s, t]. */
void lla_oracle_explicit(const double* q, const double* k, const double* v,
                         const double* log_a, const double* lambda, double* out,
                         int B, int H, int T, int dk, int dv, int L)
{
    for (int bh = 0; bh < B * H; bh++) {
        const double* qh = q + (size_t)bh * T * dk;
        const double* kh = k + (size_t)bh * T * dk;
        const double* vh = v + (size_t)bh * T * dv;
        const double* ah = log_a + (size_t)bh * T;
        const double* lh = lambda + (size_t)bh * T * L;
        double* oh = out + (size_t)bh * T * dv;
        for (int t = 0; t < T; t++) {
            double* o = oh + (size_t)t * dv;
            for (int j = 0; j < dv; j++) o[j] = 0.0;
            double decay_exp = 0.0; /* sum of log_a over (s, t] */
            for (int s = t; s >= 0; s--) {
                int l = lla_oracle_level(t, s);
                double qk = 0.0;
                for (int i = 0; i < dk; i++) qk += qh[(size_t)t * dk + i] * kh[(size_t)s * dk + i];
                double w = lh[(size_t)t * L + l] * exp(decay_exp) * qk;
                for (int j = 0; j < dv; j++) o[j] += w * vh[(size_t)s * dv + j];
                decay_exp += ah[s];
            }
        }
    }
}

/* The explicit form restricted to chosen query rows of one head (bh), for
 * spot checks of long sequences: o_t for each t in rows[0..nrows), written to
 * out[r * dv ...]. Same definition and summation order as lla_oracle_explicit. */
void lla_oracle_explicit_rows(const double* q, const double* k, const double* v,
                              const double* log_a, const double* lambda, double* out,
                              int bh, int T, int dk, int dv, int L,
                              const int64_t* rows, int nrows)
{
    const double* qh = q + (size_t)bh * T * dk;
    const double* kh = k + (size_t)bh * T * dk;
    const double* vh = v + (size_t)bh * T * dv;
    const double* ah = log_a + (size_t)bh * T;
    const double* lh = lambda + (size_t)bh * T * L;
    for (int r = 0; r < nrows; r++) {
        int64_t t = rows[r];
        double* o = out + (size_t)r * dv;
        for (int j = 0; j < dv; j++) o[j] = 0.0;
        double decay_exp = 0.0;
        for (int64_t s = t; s >= 0; s--) {
            int l = lla_oracle_level(t, s);
            double qk = 0.0;
            for (int i = 0; i < dk; i++) qk += qh[(size_t)t * dk + i] * kh[(size_t)s * dk + i];
            double w = lh[(size_t)t * L + l] * exp(decay_exp) * qk;
            for (int j = 0; j < dv; j++) o[j] += w * vh[(size_t)s * dv + j];
            decay_exp += ah[s];
        }
    }
}

/* Gradients of the explicit form for an upstream gradient dout = dL/dO, with
 * the loss L = sum_t dout_t . o_t. For every pair s <= t write
 *   D_ts = exp(sum_{r=s+1..t} log_a_r), l = l(t,s), lam = lambda_t^(l),
 *   qk = q_t . k_s,  gv = dout_t . v_s;
 * the pair adds lam * D_ts * qk * (dout_t . v_s) to L, so
 *   dq_t += lam D gv k_s,   dk_s += lam D gv q_t,   dv_s += lam D qk dout_t,
 *   dlambda_t^(l) += D qk gv,
 * and every log_a_r with s < r <= t (the factors of D_ts) gets lam D qk gv.
 * That last sum over pairs is accumulated as +E at r = s+1 and -E at r = t+1
 * followed by a running sum over r, which adds E exactly to r in (s, t].
 * Outputs are overwritten. */
void lla_oracle_backward(const double* q, const double* k, const double* v,
                         const double* log_a, const double* lambda, const double* dout,
                         double* dq, double* dk, double* dv, double* dlog_a, double* dlambda,
                         int B, int H, int T, int dkk, int dvv, int L)
{
    double* diff = (double*)malloc(sizeof(double) * (size_t)(T + 1));
    for (int bh = 0; bh < B * H; bh++) {
        const double* qh = q + (size_t)bh * T * dkk;
        const double* kh = k + (size_t)bh * T * dkk;
        const double* vh = v + (size_t)bh * T * dvv;
        const double* ah = log_a + (size_t)bh * T;
        const double* lh = lambda + (size_t)bh * T * L;
        const double* gh = dout + (size_t)bh * T * dvv;
        double* dqh = dq + (size_t)bh * T * dkk;
        double* dkh = dk + (size_t)bh * T * dkk;
        double* dvh = dv + (size_t)bh * T * dvv;
        double* dah = dlog_a + (size_t)bh * T;
        double* dlh = dlambda + (size_t)bh * T * L;
        memset(dqh, 0, sizeof(double) * (size_t)T * dkk);
        memset(dkh, 0, sizeof(double) * (size_t)T * dkk);
        memset(dvh, 0, sizeof(double) * (size_t)T * dvv);
        memset(dlh, 0, sizeof(double) * (size_t)T * L);
        for (int r = 0; r <= T; r++) diff[r] = 0.0;
        for (int t = 0; t < T; t++) {
            double decay_exp = 0.0; /* sum of log_a over (s, t] */
            for (int s = t; s >= 0; s--) {
                int l = lla_oracle_level(t, s);
                double qk = 0.0, gv = 0.0;
                for (int i = 0; i < dkk; i++) qk += qh[(size_t)t * dkk + i] * kh[(size_t)s * dkk + i];
                for (int j = 0; j < dvv; j++) gv += gh[(size_t)t * dvv + j] * vh[(size_t)s * dvv + j];
                double D = exp(decay_exp);
                double lam = lh[(size_t)t * L + l];
                for (int i = 0; i < dkk; i++) {
                    dqh[(size_t)t * dkk + i] += lam * D * gv * kh[(size_t)s * dkk + i];
                    dkh[(size_t)s * dkk + i] += lam * D * gv * qh[(size_t)t * dkk + i];
                }
                for (int j = 0; j < dvv; j++) dvh[(size_t)s * dvv + j] += lam * D * qk * gh[(size_t)t * dvv + j];
                dlh[(size_t)t * L + l] += D * qk * gv;
                double E = lam * D * qk * gv;
                diff[s + 1] += E;
                diff[t + 1] -= E;
                decay_exp += ah[s];
            }
        }
        double run = 0.0;
        for (int r = 0; r < T; r++) {
            run += diff[r];
            dah[r] = run;
        }
    }
    free(diff);
}

/* The backward restricted to chosen positions x of one head (bh), for spot
 * checks of long sequences. For each x in rows[0..nrows):
 *   dq_x, dlambda_x  from the pairs (x, s), s <= x   (x as the query),
 *   dk_x, dv_x       from the pairs (t, x), t >= x   (x as the key),
 *   dcum_x = sum_s E_xs - sum_t E_tx, the derivative with respect to
 *            cum_x = sum_{r<=x} log_a_r, so that dlog_a_x - dlog_a_{x+1} = dcum_x,
 * with the same per-pair terms as lla_oracle_backward. Outputs are overwritten:
 * dq [nrows][dk], dk [nrows][dk], dv [nrows][dv], dlambda [nrows][L], dcum [nrows]. */
void lla_oracle_backward_rows(const double* q, const double* k, const double* v,
                              const double* log_a, const double* lambda, const double* dout,
                              int bh, int T, int dkk, int dvv, int L, const int64_t* rows, int nrows,
                              double* dq, double* dk, double* dv, double* dlambda, double* dcum)
{
    const double* qh = q + (size_t)bh * T * dkk;
    const double* kh = k + (size_t)bh * T * dkk;
    const double* vh = v + (size_t)bh * T * dvv;
    const double* ah = log_a + (size_t)bh * T;
    const double* lh = lambda + (size_t)bh * T * L;
    const double* gh = dout + (size_t)bh * T * dvv;
    for (int r = 0; r < nrows; r++) {
        int64_t x = rows[r];
        double* dqr = dq + (size_t)r * dkk;
        double* dkr = dk + (size_t)r * dkk;
        double* dvr = dv + (size_t)r * dvv;
        double* dlr = dlambda + (size_t)r * L;
        memset(dqr, 0, sizeof(double) * dkk);
        memset(dkr, 0, sizeof(double) * dkk);
        memset(dvr, 0, sizeof(double) * dvv);
        memset(dlr, 0, sizeof(double) * L);
        double dc = 0.0;
        /* x as the query: pairs (x, s) */
        double decay_exp = 0.0;
        for (int64_t s = x; s >= 0; s--) {
            int l = lla_oracle_level(x, s);
            double qk = 0.0, gv = 0.0;
            for (int i = 0; i < dkk; i++) qk += qh[(size_t)x * dkk + i] * kh[(size_t)s * dkk + i];
            for (int j = 0; j < dvv; j++) gv += gh[(size_t)x * dvv + j] * vh[(size_t)s * dvv + j];
            double D = exp(decay_exp);
            double lam = lh[(size_t)x * L + l];
            for (int i = 0; i < dkk; i++) dqr[i] += lam * D * gv * kh[(size_t)s * dkk + i];
            dlr[l] += D * qk * gv;
            dc += lam * D * qk * gv;
            decay_exp += ah[s];
        }
        /* x as the key: pairs (t, x) */
        decay_exp = 0.0; /* sum of log_a over (x, t] */
        for (int64_t t = x; t < T; t++) {
            if (t > x) decay_exp += ah[t];
            int l = lla_oracle_level(t, x);
            double qk = 0.0, gv = 0.0;
            for (int i = 0; i < dkk; i++) qk += qh[(size_t)t * dkk + i] * kh[(size_t)x * dkk + i];
            for (int j = 0; j < dvv; j++) gv += gh[(size_t)t * dvv + j] * vh[(size_t)x * dvv + j];
            double D = exp(decay_exp);
            double lam = lh[(size_t)t * L + l];
            for (int i = 0; i < dkk; i++) dkr[i] += lam * D * gv * qh[(size_t)t * dkk + i];
            for (int j = 0; j < dvv; j++) dvr[j] += lam * D * qk * gh[(size_t)t * dvv + j];
            dc -= lam * D * qk * gv;
        }
        dcum[r] = dc;
    }
}

/* Lowest set bit position of t > 0. */
static int trailing_zeros(int64_t t)
{
    int c = 0;
    while (((t >> c) & 1) == 0) c++;
    return c;
}

/* Is level l of the state set held after token u nonempty? Level 0 is the
 * token u itself; level l >= 1 is nonempty exactly when bit l-1 of u is set
 * (the Fenwick bucket of that size exists in u's prefix). */
static int level_nonempty(int64_t u, int l)
{
    if (l == 0) return 1;
    return (int)((u >> (l - 1)) & 1);
}

/* One recurrent step on one head's state set, in place.
 * On entry `S` (Lmax matrices dk x dv) holds, for query t-1, each Fenwick
 * bucket's keys summed as exp(decay to t-1) k_s v_s^T; levels empty for t-1
 * are not read. On exit it holds the same for query t, and o = sum_l
 * lambda^(l) S^(l)^T q. For t > 0 with c = ctz(t): every held bucket is
 * decayed by a_t; buckets 0..c (together the 2^c keys t-2^c .. t-1) merge
 * into level c+1 and levels 1..c become empty (set to zero here); the new
 * token's k v^T becomes level 0. */
static void recurrent_step(double* S, const double* qt, const double* kt, const double* vt,
                           double log_a_t, const double* lam, int64_t t,
                           int dk, int dv, int Lmax, double* o)
{
    size_t msz = (size_t)dk * dv;
    if (t > 0) {
        int c = trailing_zeros(t);
        double a = exp(log_a_t);
        /* decay every bucket held for query t-1 */
        for (int l = 0; l < Lmax; l++) {
            if (!level_nonempty(t - 1, l)) continue;
            for (size_t e = 0; e < msz; e++) S[l * msz + e] *= a;
        }
        /* merge levels 0..c into level c+1 (level c+1 is empty for t-1) */
        double* dst = S + (size_t)(c + 1) * msz;
        for (size_t e = 0; e < msz; e++) dst[e] = 0.0;
        for (int l = 0; l <= c; l++) {
            for (size_t e = 0; e < msz; e++) dst[e] += S[l * msz + e];
            if (l > 0)
                for (size_t e = 0; e < msz; e++) S[l * msz + e] = 0.0;
        }
    }
    /* the new token is level 0 */
    for (int i = 0; i < dk; i++)
        for (int j = 0; j < dv; j++) S[(size_t)i * dv + j] = kt[i] * vt[j];
    /* read every nonempty level with its lambda */
    for (int j = 0; j < dv; j++) o[j] = 0.0;
    for (int l = 0; l < Lmax; l++) {
        if (!level_nonempty(t, l)) continue;
        const double* Sl = S + (size_t)l * msz;
        for (int j = 0; j < dv; j++) {
            double acc = 0.0;
            for (int i = 0; i < dk; i++) acc += qt[i] * Sl[(size_t)i * dv + j];
            o[j] += lam[l] * acc;
        }
    }
}

/* Recurrent form over whole sequences: one state set per head, stepped token
 * by token with the lowbit-carry merge of recurrent_step. Independent of the
 * explicit form: it never evaluates l(t,s) or a pairwise decay. */
int lla_oracle_recurrent(const double* q, const double* k, const double* v,
                         const double* log_a, const double* lambda, double* out,
                         int B, int H, int T, int dk, int dv, int L)
{
    int Lmax = L; /* for t < T every merge target and every read level is < L */
    size_t msz = (size_t)dk * dv;
    double* S = (double*)calloc((size_t)Lmax * msz, sizeof(double));
    if (!S) return -1;
    for (int bh = 0; bh < B * H; bh++) {
        memset(S, 0, (size_t)Lmax * msz * sizeof(double));
        for (int t = 0; t < T; t++) {
            size_t r = (size_t)bh * T + t;
            recurrent_step(S, q + r * dk, k + r * dk, v + r * dv, log_a[r],
                           lambda + r * L, t, dk, dv, Lmax, out + r * dv);
        }
    }
    free(S);
    return 0;
}

/* One decode step for a batch: the same recurrent step applied to each
 * (b, h) state set at its sequence position t[b]. Returns -1 if a position
 * needs more levels than Lmax holds. */
int lla_oracle_decode_step(const double* q, const double* k, const double* v,
                           const double* log_a, const double* lambda, double* states,
                           const int64_t* t, double* out,
                           int B, int H, int dk, int dv, int Lmax)
{
    size_t msz = (size_t)dk * dv;
    for (int b = 0; b < B; b++) {
        int64_t tb = t[b];
        if (tb < 0) return -1;
        int need = 1;
        for (int64_t x = tb; x > 0; x >>= 1) need++;
        if (need > Lmax) return -1;
        for (int h = 0; h < H; h++) {
            size_t bh = (size_t)b * H + h;
            recurrent_step(states + bh * Lmax * msz, q + bh * dk, k + bh * dk, v + bh * dv,
                           log_a[bh], lambda + bh * Lmax, tb, dk, dv, Lmax, out + bh * dv);
        }
    }
    return 0;
}

/* ======================================================================
 * Log-Linear Gated DeltaNet.
 *
 * Sources: pt §2 "Generalizacao" and pt §4, fr §3 "Cadre General" and
 * "Etudes de Cas" ("Log-Linear Attention"): the log-linear framework is
 * applied on top of an existing linear-attention model by replacing its
 * temporal mask with the hierarchical one, P = A (.) M_H (pt §2 "Mascara
 * Hierarquica"); Gated DeltaNet is the second model it is applied to. The
 * recurrent form keeps the same O(log T) Fenwick bucket states: the new token
 * updates the finest level and levels merge along the tree (pt §2 "Forma
 * Recorrente e Paralela", fr §2 "Algorithmes Efficaces").
 *
 * Readings (the pages do not define Gated DeltaNet itself; its published
 * recurrence is taken as the base model):
 *   - base recurrence, states dk x dv: S_t = A_t S_{t-1} + beta_t k_t v_t^T with
 *     the gated delta-rule transition A_t = alpha_t (I - beta_t k_t k_t^T),
 *     alpha_t = exp(log_a_t), beta_t in [0,1] a per-token input; o_t = S_t^T q_t;
 *   - its attention matrix (the coefficient of v_s in o_t) is
 *     A[t,s] = beta_s k_s^T A_{s+1} A_{s+2} ... A_t q_t (s <= t);
 *   - log-linear: o_t = sum_{s<=t} lambda_t^(l(t,s)) A[t,s] v_s, with the Fenwick
 *     level l(t,s) and query-indexed lambda of the Mamba-2 variant above;
 *   - recurrently: every held bucket state evolves under A_t, buckets merge on
 *     the lowbit carry, and the new token's beta_t k_t v_t^T is level 0.
 * Layouts as above, plus beta [B,H,T] (decode: [B,H]).
 * ====================================================================== */

/* x <- A_t x = alpha (x - beta k (k . x)) for one dk-vector x. */
static void gdn_transition_vec(double* x, const double* kt, double alpha, double beta, int dk)
{
    double kx = 0.0;
    for (int i = 0; i < dk; i++) kx += kt[i] * x[i];
    for (int i = 0; i < dk; i++) x[i] = alpha * (x[i] - beta * kt[i] * kx);
}

/* Explicit form: o_t = sum_{s<=t} lambda_t^(l(t,s)) A[t,s] v_s. For each query
 * the vector u = A_{s+1} ... A_t q_t is carried while s walks down from t:
 * u starts at q_t; key s contributes A[t,s] = beta_s (k_s . u); then u <- A_s u. */
void lla_oracle_gdn_explicit(const double* q, const double* k, const double* v,
                             const double* log_a, const double* beta, const double* lambda,
                             double* out, int B, int H, int T, int dk, int dv, int L)
{
    double* u = (double*)malloc((size_t)(dk > 0 ? dk : 1) * sizeof(double));
    if (!u) return;
    for (int bh = 0; bh < B * H; bh++) {
        const double* qh = q + (size_t)bh * T * dk;
        const double* kh = k + (size_t)bh * T * dk;
        const double* vh = v + (size_t)bh * T * dv;
        const double* ah = log_a + (size_t)bh * T;
        const double* bth = beta + (size_t)bh * T;
        const double* lh = lambda + (size_t)bh * T * L;
        double* oh = out + (size_t)bh * T * dv;
        for (int t = 0; t < T; t++) {
            double* o = oh + (size_t)t * dv;
            for (int j = 0; j < dv; j++) o[j] = 0.0;
            for (int i = 0; i < dk; i++) u[i] = qh[(size_t)t * dk + i];
            for (int s = t; s >= 0; s--) {
                const double* ks = kh + (size_t)s * dk;
                double ku = 0.0;
                for (int i = 0; i < dk; i++) ku += ks[i] * u[i];
                double w = lh[(size_t)t * L + lla_oracle_level(t, s)] * bth[s] * ku;
                for (int j = 0; j < dv; j++) o[j] += w * vh[(size_t)s * dv + j];
                gdn_transition_vec(u, ks, exp(ah[s]), bth[s], dk);
            }
        }
    }
    free(u);
}

/* One recurrent step of the log-linear Gated DeltaNet on one head's state set,
 * in place: as recurrent_step, with the scalar decay of every held bucket
 * replaced by the transition A_t (S <- alpha (S - beta k (k^T S)), column by
 * column) and the new level 0 = beta_t k_t v_t^T. */
static void gdn_step(double* S, const double* qt, const double* kt, const double* vt,
                     double log_a_t, double beta_t, const double* lam, int64_t t,
                     int dk, int dv, int Lmax, double* o)
{
    size_t msz = (size_t)dk * dv;
    if (t > 0) {
        int c = trailing_zeros(t);
        double alpha = exp(log_a_t);
        for (int l = 0; l < Lmax; l++) {
            if (!level_nonempty(t - 1, l)) continue;
            double* Sl = S + (size_t)l * msz;
            for (int j = 0; j < dv; j++) {
                double kS = 0.0;
                for (int i = 0; i < dk; i++) kS += kt[i] * Sl[(size_t)i * dv + j];
                for (int i = 0; i < dk; i++)
                    Sl[(size_t)i * dv + j] = alpha * (Sl[(size_t)i * dv + j] - beta_t * kt[i] * kS);
            }
        }
        double* dst = S + (size_t)(c + 1) * msz;
        for (size_t e = 0; e < msz; e++) dst[e] = 0.0;
        for (int l = 0; l <= c; l++) {
            for (size_t e = 0; e < msz; e++) dst[e] += S[l * msz + e];
            if (l > 0)
                for (size_t e = 0; e < msz; e++) S[l * msz + e] = 0.0;
        }
    }
    for (int i = 0; i < dk; i++)
        for (int j = 0; j < dv; j++) S[(size_t)i * dv + j] = beta_t * kt[i] * vt[j];
    for (int j = 0; j < dv; j++) o[j] = 0.0;
    for (int l = 0; l < Lmax; l++) {
        if (!level_nonempty(t, l)) continue;
        const double* Sl = S + (size_t)l * msz;
        for (int j = 0; j < dv; j++) {
            double acc = 0.0;
            for (int i = 0; i < dk; i++) acc += qt[i] * Sl[(size_t)i * dv + j];
            o[j] += lam[l] * acc;
        }
    }
}

/* Recurrent form of the log-linear Gated DeltaNet over whole sequences. It never
 * evaluates l(t,s) or a pairwise attention coefficient. */
int lla_oracle_gdn_recurrent(const double* q, const double* k, const double* v,
                             const double* log_a, const double* beta, const double* lambda,
                             double* out, int B, int H, int T, int dk, int dv, int L)
{
    size_t msz = (size_t)dk * dv;
    double* S = (double*)calloc((size_t)L * msz, sizeof(double));
    if (!S) return -1;
    for (int bh = 0; bh < B * H; bh++) {
        memset(S, 0, (size_t)L * msz * sizeof(double));
        for (int t = 0; t < T; t++) {
            size_t r = (size_t)bh * T + t;
            gdn_step(S, q + r * dk, k + r * dk, v + r * dv, log_a[r], beta[r], lambda + r * L, t, dk, dv, L,
                     out + r * dv);
        }
    }
    free(S);
    return 0;
}

/* One decode step of the log-linear Gated DeltaNet for a batch (states as in
 * lla_oracle_decode_step). */
int lla_oracle_gdn_decode_step(const double* q, const double* k, const double* v,
                               const double* log_a, const double* beta, const double* lambda,
                               double* states, const int64_t* t, double* out,
                               int B, int H, int dk, int dv, int Lmax)
{
    size_t msz = (size_t)dk * dv;
    for (int b = 0; b < B; b++) {
        int64_t tb = t[b];
        if (tb < 0) return -1;
        int need = 1;
        for (int64_t x = tb; x > 0; x >>= 1) need++;
        if (need > Lmax) return -1;
        for (int h = 0; h < H; h++) {
            size_t bh = (size_t)b * H + h;
            gdn_step(states + bh * Lmax * msz, q + bh * dk, k + bh * dk, v + bh * dv, log_a[bh], beta[bh],
                     lambda + bh * Lmax, tb, dk, dv, Lmax, out + bh * dv);
        }
    }
    return 0;
}

/* lla_oracle_gdn_explicit restricted to chosen query rows of one head (bh), for spot
 * checks of long sequences: o_t for each t in rows[0..nrows), written to out[r * dv ...].
 * Same definition and summation order. */
void lla_oracle_gdn_explicit_rows(const double* q, const double* k, const double* v,
                                  const double* log_a, const double* beta, const double* lambda,
                                  double* out, int bh, int T, int dk, int dv, int L,
                                  const int64_t* rows, int nrows)
{
    double* u = (double*)malloc((size_t)(dk > 0 ? dk : 1) * sizeof(double));
    if (!u) return;
    const double* qh = q + (size_t)bh * T * dk;
    const double* kh = k + (size_t)bh * T * dk;
    const double* vh = v + (size_t)bh * T * dv;
    const double* ah = log_a + (size_t)bh * T;
    const double* bth = beta + (size_t)bh * T;
    const double* lh = lambda + (size_t)bh * T * L;
    for (int rr = 0; rr < nrows; rr++) {
        int64_t t = rows[rr];
        double* o = out + (size_t)rr * dv;
        for (int j = 0; j < dv; j++) o[j] = 0.0;
        for (int i = 0; i < dk; i++) u[i] = qh[(size_t)t * dk + i];
        for (int64_t s = t; s >= 0; s--) {
            const double* ks = kh + (size_t)s * dk;
            double ku = 0.0;
            for (int i = 0; i < dk; i++) ku += ks[i] * u[i];
            double w = lh[(size_t)t * L + lla_oracle_level(t, s)] * bth[s] * ku;
            for (int j = 0; j < dv; j++) o[j] += w * vh[(size_t)s * dv + j];
            gdn_transition_vec(u, ks, exp(ah[s]), bth[s], dk);
        }
    }
    free(u);
}
