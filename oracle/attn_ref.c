/*
 * Oracle for ring attention (context parallelism): plain, slow, fp64, CPU.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline / reference legs may load this library.  It shares
 * no code, header or table with the CUDA path, and the CUDA path never calls it.
 *
 * What it computes (sources are the three pages on context parallelism):
 *
 *  - Full softmax attention, the definition the ring method must reproduce
 *    exactly: the ring's answer is full attention over the whole sequence
 *    (ultralytics glossary, "How Context Parallelism Works"); the
 *    43,200 x 43,200 score matrix of the "day 83" blog intro.
 *      s_ij  = (q_i . k_j) / sqrt(d)
 *      LSE_i = ln sum_{j in K(i)} exp(s_ij)
 *      O_i   = sum_{j in K(i)} exp(s_ij - LSE_i) v_j
 *    K(i) = all keys, or {j <= i} (causal, top-left aligned, by global token
 *    position), as SDPA's is_causal flag in the glossary's example.
 *
 *  - Ring attention as the pages describe it, step by step: every rank keeps
 *    its query chunk; at step s rank r holds KV block (r - s) mod P (k8ai
 *    "How context parallel works", ring diagram: after the first exchange
 *    rank 0 holds block 3 and rank 1 holds block 0); each block's partial result is folded into a running
 *    (max, sum, output) with the online-softmax rule (day 83 blog, "Context
 *    parallelism: splitting the sequence").  Used only to pin ring == full.
 *
 *  - The log-sum-exp merge of partial (O_i, LSE_i) pairs, the same online
 *    softmax rule applied to normalised partials.
 *
 *  - The sequence shard maps: contiguous (day 83 blog, "Context parallelism:
 *    splitting the sequence": S tokens over P GPUs, S/P each) and the balanced
 *    causal pattern (k8ai "How context parallel works", last paragraph), read
 *    as zigzag: 2P chunks, rank r holds chunk r then chunk 2P-1-r.
 *
 *  - Factored video attention (day 83 blog, "The spatial-temporal twist"):
 *    spatial = attention within each frame, temporal = attention across frames
 *    at one spatial position; token index t*N + n.
 *
 * Inputs are raw bf16 bit patterns, widened exactly to double.  All arithmetic
 * is double precision, straightforward loops, OpenMP over query rows only.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double widen_bf16(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_threads(void) { return omp_get_max_threads(); }

/* ------------------------------------------------------------------ maps -- */

/* Sharded position j (rank-major: rank r owns rows [r*L, (r+1)*L)) <-> global
 * token position g.  layout 0 = contiguous, 1 = zigzag.  Returns 0, or -1 on
 * bad arguments. */
int oracle_shard_index(int64_t S, int64_t P, int layout, int64_t *s2g, int64_t *g2s)
{
    if (S < 0 || P <= 0 || S % P != 0) return -1;
    if (layout == 1 && S % (2 * P) != 0) return -1;
    int64_t L = S / P;
    for (int64_t r = 0; r < P; ++r) {
        for (int64_t i = 0; i < L; ++i) {
            int64_t j = r * L + i, g;
            if (layout == 0) {
                g = r * L + i;
            } else {
                int64_t C = S / (2 * P);
                int64_t chunk = (i < C) ? r : (2 * P - 1 - r);
                g = chunk * C + (i < C ? i : i - C);
            }
            s2g[j] = g;
            g2s[g] = j;
        }
    }
    return 0;
}

/* ------------------------------------------------------------ definition -- */

/* One query row against the keys {start + t*stride : 0 <= t < count}. */
static void attend(const uint16_t *qrow, const uint16_t *K, const uint16_t *V, int64_t d,
                   int64_t start, int64_t count, int64_t stride, double scale,
                   double *out, double *lse, double *s)
{
    for (int64_t c = 0; c < d; ++c) out[c] = 0.0;
    if (count <= 0) {
        *lse = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (int64_t t = 0; t < count; ++t) {
        const uint16_t *krow = K + (start + t * stride) * d;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c) dot += widen_bf16(qrow[c]) * widen_bf16(krow[c]);
        s[t] = dot * scale;
        if (s[t] > m) m = s[t];
    }
    double z = 0.0;
    for (int64_t t = 0; t < count; ++t) z += exp(s[t] - m);
    double L = m + log(z);
    for (int64_t t = 0; t < count; ++t) {
        const uint16_t *vrow = V + (start + t * stride) * d;
        double p = exp(s[t] - L);
        for (int64_t c = 0; c < d; ++c) out[c] += p * widen_bf16(vrow[c]);
    }
    *lse = L;
}

/* Full attention.  q: [BH, Sq, d], k/v: [BH, Skv, d], all global order.  Query
 * i of a head sits at global position q_offset + i.  rows: flat indices
 * bh*Sq + i to compute (NULL = all).  o: [n_rows, d], lse: [n_rows]. */
int oracle_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     int64_t BH, int64_t Sq, int64_t Skv, int64_t d, int causal,
                     int64_t q_offset, const int64_t *rows, int64_t n_rows,
                     double *o, double *lse)
{
    if (rows == NULL) n_rows = BH * Sq;
    double scale = 1.0 / sqrt((double)d);
    int bad = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Skv > 0 ? Skv : 1));
        if (!s) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t n = 0; n < n_rows; ++n) {
            if (!s) continue;
            int64_t flat = rows ? rows[n] : n;
            int64_t bh = flat / Sq, i = flat % Sq;
            int64_t count = Skv;
            if (causal) {
                count = q_offset + i + 1;
                if (count > Skv) count = Skv;
            }
            attend(q + flat * d, k + bh * Skv * d, v + bh * Skv * d, d, 0, count, 1, scale,
                   o + n * d, lse + n, s);
        }
        free(s);
    }
    return bad ? -1 : 0;
}

/* Factored video attention.  q/k/v: [BH, T*N, d], token index t*N + n.
 * which = 0: spatial (keys = the query's frame); 1: temporal (keys = the
 * query's spatial position in every frame). */
int oracle_factored(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    int64_t BH, int64_t T, int64_t N, int64_t d, int which,
                    const int64_t *rows, int64_t n_rows, double *o, double *lse)
{
    int64_t S = T * N;
    if (rows == NULL) n_rows = BH * S;
    double scale = 1.0 / sqrt((double)d);
    int64_t buf = (which == 0) ? N : T;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(buf > 0 ? buf : 1));
#pragma omp for schedule(dynamic, 16)
        for (int64_t n = 0; n < n_rows; ++n) {
            int64_t flat = rows ? rows[n] : n;
            int64_t bh = flat / S, tok = flat % S;
            int64_t t = tok / N, pos = tok % N;
            const uint16_t *Kh = k + bh * S * d, *Vh = v + bh * S * d;
            if (which == 0)
                attend(q + flat * d, Kh, Vh, d, t * N, N, 1, scale, o + n * d, lse + n, s);
            else
                attend(q + flat * d, Kh, Vh, d, pos, T, N, scale, o + n * d, lse + n, s);
        }
        free(s);
    }
    return 0;
}

/* ------------------------------------------------------------ ring form -- */

/* Block held by rank r at ring step s: at step 0 its own, then the block of
 * the rank before it (k8ai ring diagram: after one exchange rank 0 holds block 3, rank 1
 * block 0). */
int64_t oracle_ring_source(int64_t P, int64_t r, int64_t s)
{
    return ((r - s) % P + P) % P;
}

/* Ring attention in the pages' step order, for the rows of a global-order
 * problem.  q/k/v: [BH, S, d] global order.  causal selects the zigzag
 * layout (and the causal mask); otherwise contiguous.  order: NULL for the
 * ring schedule (block (r - s) mod P at step s), or a [P][P] table giving the
 * block rank r visits at step s (used to test order invariance). */
int oracle_ring_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          int64_t BH, int64_t S, int64_t d, int64_t P, int causal,
                          const int64_t *order, const int64_t *rows, int64_t n_rows,
                          double *o, double *lse)
{
    if (P <= 0 || S % P != 0 || (causal && S % (2 * P) != 0)) return -1;
    int64_t L = S / P;
    int64_t *s2g = (int64_t *)malloc(sizeof(int64_t) * (size_t)(S ? S : 1));
    int64_t *g2s = (int64_t *)malloc(sizeof(int64_t) * (size_t)(S ? S : 1));
    if (!s2g || !g2s) return -1;
    oracle_shard_index(S, P, causal ? 1 : 0, s2g, g2s);
    if (rows == NULL) n_rows = BH * S;
    double scale = 1.0 / sqrt((double)d);
#pragma omp parallel
    {
        double *sb = (double *)malloc(sizeof(double) * (size_t)(L ? L : 1));
        double *acc = (double *)malloc(sizeof(double) * (size_t)d);
        double *accb = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int64_t n = 0; n < n_rows; ++n) {
            int64_t flat = rows ? rows[n] : n;
            int64_t bh = flat / S, g = flat % S;
            int64_t r = g2s[g] / L; /* the rank that owns this query */
            const uint16_t *qrow = q + flat * d;
            const uint16_t *Kh = k + bh * S * d, *Vh = v + bh * S * d;
            double m = -INFINITY, z = 0.0;
            for (int64_t c = 0; c < d; ++c) acc[c] = 0.0;
            for (int64_t step = 0; step < P; ++step) {
                int64_t src = order ? order[r * P + step] : oracle_ring_source(P, r, step);
                /* Block partial over the keys of block src (in sharded order). */
                double mb = -INFINITY;
                for (int64_t t = 0; t < L; ++t) {
                    int64_t gk = s2g[src * L + t];
                    if (causal && gk > g) { sb[t] = -INFINITY; continue; }
                    const uint16_t *krow = Kh + gk * d;
                    double dot = 0.0;
                    for (int64_t c = 0; c < d; ++c) dot += widen_bf16(qrow[c]) * widen_bf16(krow[c]);
                    sb[t] = dot * scale;
                    if (sb[t] > mb) mb = sb[t];
                }
                if (mb == -INFINITY) continue; /* every key of this block masked */
                double zb = 0.0;
                for (int64_t c = 0; c < d; ++c) accb[c] = 0.0;
                for (int64_t t = 0; t < L; ++t) {
                    if (sb[t] == -INFINITY) continue;
                    double p = exp(sb[t] - mb);
                    zb += p;
                    const uint16_t *vrow = Vh + s2g[src * L + t] * d;
                    for (int64_t c = 0; c < d; ++c) accb[c] += p * widen_bf16(vrow[c]);
                }
                /* Online-softmax fold of the block into the running state. */
                double mn = (mb > m) ? mb : m;
                double a = exp(m - mn), b = exp(mb - mn);
                z = z * a + zb * b;
                for (int64_t c = 0; c < d; ++c) acc[c] = acc[c] * a + accb[c] * b;
                m = mn;
            }
            if (z > 0.0) {
                for (int64_t c = 0; c < d; ++c) o[n * d + c] = acc[c] / z;
                lse[n] = m + log(z);
            } else {
                for (int64_t c = 0; c < d; ++c) o[n * d + c] = 0.0;
                lse[n] = -INFINITY;
            }
        }
        free(sb);
        free(acc);
        free(accb);
    }
    free(s2g);
    free(g2s);
    return 0;
}

/* ----------------------------------------------------------- backward -- */

/* Gradients of full attention (the definition, differentiated):
 *   s_ij = scale q_i.k_j,  P_ij = exp(s_ij - LSE_i),  O_i = sum_j P_ij v_j
 *   dV_j = sum_i P_ij dO_i
 *   dP_ij = dO_i . v_j,   D_i = sum_j P_ij dP_ij  (= dO_i . O_i)
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i
 * K(i) as in oracle_attention (causal: j <= i).  All of [BH, S, d] in global
 * order; dq/dk/dv: [BH, S, d] fp64 outputs.  Parallel over heads. */
int oracle_attention_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         const uint16_t *dout, int64_t BH, int64_t S, int64_t d, int causal,
                         double *dq, double *dk, double *dv)
{
    double scale = 1.0 / sqrt((double)d);
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < BH; ++bh) {
        const uint16_t *Q = q + bh * S * d, *K = k + bh * S * d, *V = v + bh * S * d;
        const uint16_t *dO = dout + bh * S * d;
        double *dQ = dq + bh * S * d, *dK = dk + bh * S * d, *dV = dv + bh * S * d;
        double *P = (double *)malloc(sizeof(double) * (size_t)(S ? S : 1));
        double *dP = (double *)malloc(sizeof(double) * (size_t)(S ? S : 1));
        if (!P || !dP) {
#pragma omp atomic write
            bad = 1;
            free(P);
            free(dP);
            continue;
        }
        for (int64_t x = 0; x < S * d; ++x) dQ[x] = dK[x] = dV[x] = 0.0;
        for (int64_t i = 0; i < S; ++i) {
            int64_t n = causal ? i + 1 : S;
            double m = -INFINITY;
            for (int64_t j = 0; j < n; ++j) {
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c) dot += widen_bf16(Q[i * d + c]) * widen_bf16(K[j * d + c]);
                P[j] = dot * scale;
                if (P[j] > m) m = P[j];
            }
            double z = 0.0;
            for (int64_t j = 0; j < n; ++j) z += exp(P[j] - m);
            double lse = m + log(z);
            double D = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                P[j] = exp(P[j] - lse);
                double t = 0.0;
                for (int64_t c = 0; c < d; ++c) t += widen_bf16(dO[i * d + c]) * widen_bf16(V[j * d + c]);
                dP[j] = t;
                D += P[j] * t;
            }
            for (int64_t j = 0; j < n; ++j) {
                double ds = P[j] * (dP[j] - D);
                for (int64_t c = 0; c < d; ++c) {
                    dV[j * d + c] += P[j] * widen_bf16(dO[i * d + c]);
                    dQ[i * d + c] += scale * ds * widen_bf16(K[j * d + c]);
                    dK[j * d + c] += scale * ds * widen_bf16(Q[i * d + c]);
                }
            }
        }
        free(P);
        free(dP);
    }
    return bad ? -1 : 0;
}

/* -------------------------------------------------------------- merge ---- */

/* Merge n normalised partials (O_i, LSE_i) of the same rows.
 *   M = max_i LSE_i;  w_i = exp(LSE_i - M);  LSE = M + ln sum w_i;
 *   O = sum_i w_i O_i / sum_i w_i.   All partials empty: O = 0, LSE = -inf.
 * o_parts: [n][rows][d], lse_parts: [n][rows]. */
int oracle_lse_merge(const double *o_parts, const double *lse_parts, int64_t n, int64_t rows,
                     int64_t d, double *o, double *lse)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int64_t i = 0; i < n; ++i)
            if (lse_parts[i * rows + r] > M) M = lse_parts[i * rows + r];
        for (int64_t c = 0; c < d; ++c) o[r * d + c] = 0.0;
        if (M == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double W = 0.0;
        for (int64_t i = 0; i < n; ++i) {
            double w = exp(lse_parts[i * rows + r] - M);
            W += w;
            for (int64_t c = 0; c < d; ++c) o[r * d + c] += w * o_parts[(i * rows + r) * d + c];
        }
        for (int64_t c = 0; c < d; ++c) o[r * d + c] /= W;
        lse[r] = M + log(W);
    }
    return 0;
}
