/*
 * dspark_oracle.c -- plain, slow CPU oracle for one DSpark draft round.
 *
 * TEST INFRASTRUCTURE ONLY (see dspark_oracle.h). All arithmetic is IEEE
 * double; every loop is the literal definition, with no blocking, fusion or
 * reordering beyond what the definition states.
 *
 * Method source: "DSpark: Confidence-Scheduled Speculative Decoding with
 * Semi-Autoregressive Generation", as described on
 *   - caijizhuo.github.io (section 4 "dspark_cycle" and "admit" sketches,
 *     section 3.2-3.3 survival / E / Theta table),
 *   - zhongzhuzhou.org reading notes (eq. 4, 5, 7, 8a-8c; Algorithm 1;
 *     Appendix A counterexample eq. 9-10; section 5.2 asynchronous capacity).
 *
 * Readings where the pages are silent (the same readings the CUDA path takes):
 *   - sampling rule: the pages say only "sample(softmax(U_k + B_k))". Draws use
 *     Gumbel-max with counter-based Philox noise, applied at two levels: a
 *     Gumbel-max over the log-masses of fixed vocabulary blocks of width
 *     noise_block picks a block, then a Gumbel-max over the log-weights inside
 *     that block picks the token. This samples exactly from the normalised
 *     weights (the block maximum of Gumbel-perturbed log-weights is a Gumbel
 *     centred on the block log-mass, independent of the arg-max inside the
 *     block). With V <= noise_block it is the flat Gumbel-max.
 *   - temperature T_r divides both the draft logits (U + B) and the target logits.
 *   - uniform u = (2*(x>>9)+1) * 2^-24 from a 32-bit Philox word x; Gumbel = -log(-log u).
 *   - ties: arg-max keeps the lowest index; the scheduler sorts by a descending,
 *     then request ascending, then position ascending.
 */
#include "dspark_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* random purposes (counter word 3 low bits) */
enum {
    PUR_DRAFT_ELEM = 0,   /* element-level Gumbel of a draft draw, per (req, pos, v) */
    PUR_ACCEPT = 1,       /* acceptance uniform, per (req, pos) */
    PUR_FINAL_ELEM = 2,   /* element-level Gumbel of the residual / bonus draw, per (req, v) */
    PUR_DRAFT_BLOCK = 3,  /* block-level Gumbel of a draft draw, per (req, pos, block) */
    PUR_FINAL_BLOCK = 4   /* block-level Gumbel of the residual / bonus draw, per (req, block) */
};

/* ------------------------------------------------------------------ Philox */

void dso_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    /* Salmon et al. SC'11, Philox-4x32 with 10 rounds:
     * round:  (c0,c1,c2,c3) -> (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0))
     * key schedule: k0 += 0x9E3779B9, k1 += 0xBB67AE85 between rounds. */
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint64_t p0 = (uint64_t)M0 * (uint64_t)c0;
        uint64_t p1 = (uint64_t)M1 * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0;
        c1 = n1;
        c2 = n2;
        c3 = n3;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

double dso_uniform(uint64_t seed, uint64_t round, uint32_t purpose, uint32_t req, uint32_t pos,
                   uint32_t elem)
{
    uint32_t ctr[4] = {elem >> 2, pos, req, (uint32_t)(round << 3) | purpose};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    dso_philox4x32_10(ctr, key, out);
    uint32_t x = out[elem & 3u];
    return ((double)(x >> 9) * 2.0 + 1.0) * ldexp(1.0, -24);
}

static double gumbel(double u) { return -log(-log(u)); }

/* ------------------------------------------------------------------ inputs */

static double load(const void* p, int dtype, size_t i)
{
    if (dtype == DSO_F64) return ((const double*)p)[i];
    if (dtype == DSO_F32) return (double)((const float*)p)[i];
    /* bf16: the upper 16 bits of an IEEE binary32 */
    uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double* to_double(const void* p, int dtype, size_t n)
{
    double* out = (double*)malloc(n * sizeof(double));
    if (!out) return NULL;
    for (size_t i = 0; i < n; ++i) out[i] = load(p, dtype, i);
    return out;
}

/* ------------------------------------------------------ two-level Gumbel-max */

static double logsumexp(const double* x, int n)
{
    double m = -INFINITY;
    for (int i = 0; i < n; ++i)
        if (x[i] > m) m = x[i];
    if (m == -INFINITY) return -INFINITY;
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += exp(x[i] - m);
    return m + log(s);
}

typedef struct {
    int token;    /* -1 when every weight is zero */
    int block;
    double gap1;  /* best minus second-best block-level value (+inf if one candidate) */
    double gap2;  /* best minus second-best element-level value */
    int second_block;
    int second_token;
} draw_t;

/* Draw an index with probability exp(logw[v]) / sum exp(logw). */
static draw_t two_level_draw(const double* logw, int V, int nb, uint64_t seed, uint64_t round,
                             uint32_t pur_block, uint32_t pur_elem, uint32_t req, uint32_t pos)
{
    draw_t d = {-1, -1, INFINITY, INFINITY, -1, -1};
    int nblk = (V + nb - 1) / nb;
    double best = -INFINITY, second = -INFINITY;
    for (int b = 0; b < nblk; ++b) {
        int v0 = b * nb, n = (V - v0 < nb) ? V - v0 : nb;
        double L = logsumexp(logw + v0, n);
        if (L == -INFINITY) continue;
        double z = L + gumbel(dso_uniform(seed, round, pur_block, req, pos, (uint32_t)b));
        if (z > best) {
            second = best;
            d.second_block = d.block;
            best = z;
            d.block = b;
        } else if (z > second) {
            second = z;
            d.second_block = b;
        }
    }
    if (d.block < 0) return d;
    d.gap1 = best - second;
    best = -INFINITY;
    second = -INFINITY;
    int v0 = d.block * nb, v1 = (v0 + nb < V) ? v0 + nb : V;
    for (int v = v0; v < v1; ++v) {
        if (logw[v] == -INFINITY) continue;
        double z = logw[v] + gumbel(dso_uniform(seed, round, pur_elem, req, pos, (uint32_t)v));
        if (z > best) {
            second = best;
            d.second_token = d.token;
            best = z;
            d.token = v;
        } else if (z > second) {
            second = z;
            d.second_token = v;
        }
    }
    d.gap2 = best - second;
    return d;
}

/* -------------------------------------------------------------- sampler */

/* logits l[v] = (U_k(v) + B_k(v)) / T with B_k = W_1[prev] W_2 (eq. 4-5), or 0 */
/* l = (U + B) / T with B = a^T W_2, a = arow if given, else W_1[prev] (Markov head) */
static void draft_logits(double* l, const void* U, int dtype, size_t u_off, int V, int r,
                         const double* Wd, const void* E, int use_bias, int prev, double T, const double* arow)
{
    for (int v = 0; v < V; ++v) l[v] = 0.0;
    if (use_bias) {
        for (int i = 0; i < r; ++i) {
            double e = arow ? arow[i] : load(E, dtype, (size_t)prev * r + i);
            const double* wrow = Wd + (size_t)i * V;
            for (int v = 0; v < V; ++v) l[v] += e * wrow[v];
        }
    }
    /* temperature 0 (greedy decoding) keeps the raw logits */
    const double div = T > 0.0 ? T : 1.0;
    for (int v = 0; v < V; ++v) l[v] = (load(U, dtype, u_off + v) + l[v]) / div;
}

/* Greedy decoding (temperature 0): the arg-max (lowest index on ties) and the gap between the
 * two largest values (both gaps of a draw report it). */
static draw_t argmax_draw(const double* l, int V)
{
    draw_t dr;
    memset(&dr, 0, sizeof dr);
    int best = 0;
    for (int v = 1; v < V; ++v)
        if (l[v] > l[best]) best = v;
    double second = -INFINITY;
    for (int v = 0; v < V; ++v)
        if (v != best && l[v] > second) second = l[v];
    dr.token = best;
    dr.second_token = -1;
    dr.block = dr.second_block = -1;
    dr.gap1 = dr.gap2 = l[best] - second;
    return dr;
}

int dso_sample_block(const dso_sample_args* a)
{
    if (!a || a->R < 0 || a->gamma_max < 1 || a->V < 1 || a->r < 1 || a->d < 1 || a->noise_block < 1)
        return 1;
    const int R = a->R, G = a->gamma_max, V = a->V, r = a->r, d = a->d;
    const int rnn = a->head == DSO_HEAD_RNN;
    if (rnn && !a->W_rnn) return 1;
    const int Z = 2 * r + d;
    double* Wd = to_double(a->W, a->dtype, (size_t)r * V);
    double* l = (double*)malloc((size_t)V * sizeof(double));
    double* st = (double*)malloc((size_t)r * sizeof(double));   /* RNN state s */
    double* z = (double*)malloc((size_t)Z * sizeof(double));
    double* o = (double*)malloc((size_t)r * sizeof(double));
    if (!Wd || !l || !st || !z || !o) {
        free(Wd);
        free(l);
        free(st);
        free(z);
        free(o);
        return 2;
    }
    for (int q = 0; q < R; ++q) {
        const uint32_t rid = (uint32_t)(a->req_ids ? a->req_ids[q] : q);
        const int g = a->gamma ? a->gamma[q] : G;
        const double T = (double)a->temperature[q];
        int prev = a->anchor[q];
        double s = 1.0;
        for (int i = 0; i < r; ++i) st[i] = 0.0;   /* s_0 = 0 */
        for (int k = 0; k < G; ++k) {
            const size_t idx = (size_t)q * G + k;
            if (k >= g) {
                a->tokens[idx] = -1;
                a->conf[idx] = a->surv[idx] = a->lse[idx] = a->logit[idx] = 0.0;
                a->gap1[idx] = a->gap2[idx] = INFINITY;
                if (a->a_rows)
                    for (int i = 0; i < r; ++i) a->a_rows[idx * r + i] = 0.0;
                if (a->logp)
                    for (int v = 0; v < V; ++v) a->logp[idx * V + v] = 0.0f;
                continue;
            }
            const int use_bias = (k > 0) || a->bias_first;
            if (rnn) {
                /* eq. (6): one packed projection of z_k = [s_{k-1}; W_1[x_{k-1}]; h_k], split into the
                 * gate, candidate and output parts */
                for (int i = 0; i < r; ++i) z[i] = st[i];
                for (int i = 0; i < r; ++i) z[r + i] = load(a->E, a->dtype, (size_t)prev * r + i);
                for (int j = 0; j < d; ++j) z[2 * r + j] = load(a->h, a->dtype, idx * d + j);
                for (int i = 0; i < r; ++i) {
                    double yg = 0.0, yc = 0.0, yo = 0.0;
                    for (int j = 0; j < Z; ++j) {
                        yg += load(a->W_rnn, a->dtype, (size_t)i * Z + j) * z[j];
                        yc += load(a->W_rnn, a->dtype, (size_t)(r + i) * Z + j) * z[j];
                        yo += load(a->W_rnn, a->dtype, (size_t)(2 * r + i) * Z + j) * z[j];
                    }
                    const double gate = 1.0 / (1.0 + exp(-yg));
                    st[i] = gate * st[i] + (1.0 - gate) * tanh(yc);   /* z keeps s_{k-1} for the other rows */
                    o[i] = tanh(yo);
                }
            } else {
                for (int i = 0; i < r; ++i) o[i] = load(a->E, a->dtype, (size_t)prev * r + i);
            }
            if (a->a_rows)
                for (int i = 0; i < r; ++i) a->a_rows[idx * r + i] = o[i];
            draft_logits(l, a->U, a->dtype, idx * V, V, r, Wd, a->E, use_bias, prev, T, o);
            draw_t dr = T == 0.0 ? argmax_draw(l, V) : two_level_draw(l, V, a->noise_block, a->seed, a->round, PUR_DRAFT_BLOCK,
                                       PUR_DRAFT_ELEM, rid, (uint32_t)k);
            const int commit = a->forced_tokens ? a->forced_tokens[idx] : dr.token;
            a->tokens[idx] = dr.token;
            a->gap1[idx] = dr.gap1;
            a->gap2[idx] = dr.gap2;
            /* temperature 0: the draft is a point mass, reported as lse = logit (log p_d = 0) */
            a->lse[idx] = T == 0.0 ? l[commit] : logsumexp(l, V);
            a->logit[idx] = l[commit];
            if (a->logp) {
                float* lp = a->logp + idx * V;
                for (int v = 0; v < V; ++v)
                    lp[v] = T == 0.0 ? (v == commit ? 0.0f : -INFINITY) : (float)(l[v] - a->lse[idx]);
            }
            /* eq. (7): c_k = sigmoid(w^T [h_k; W_1[x]]) + b */
            const int xc = a->conf_token ? commit : prev;
            double dot = (double)a->b;
            for (int j = 0; j < d; ++j) dot += (double)a->w_h[j] * load(a->h, a->dtype, idx * d + j);
            for (int i = 0; i < r; ++i) dot += (double)a->w_e[i] * load(a->E, a->dtype, (size_t)xc * r + i);
            /* sequential temperature scaling: the logit of position k over its temperature */
            if (a->sts_temp) dot /= a->sts_temp[k];
            const double c = 1.0 / (1.0 + exp(-dot));
            s *= c;
            a->conf[idx] = c;
            a->surv[idx] = s;
            prev = commit;
        }
    }
    free(Wd);
    free(l);
    free(st);
    free(z);
    free(o);
    return 0;
}

/* ------------------------------------------------------------ scheduler */

typedef struct {
    double a;
    int r, j;
} cand_t;

static int cand_cmp(const void* x, const void* y)
{
    const cand_t* p = (const cand_t*)x;
    const cand_t* q = (const cand_t*)y;
    if (p->a > q->a) return -1;
    if (p->a < q->a) return 1;
    if (p->r != q->r) return p->r < q->r ? -1 : 1;
    if (p->j != q->j) return p->j < q->j ? -1 : 1;
    return 0;
}

/* Algorithm 1, step 2: pool E = {(r,j) : a_{r,j} > 0}, sorted descending. */
static int build_pool(cand_t* pool, int R, int G, const int32_t* gamma, const double* surv)
{
    int n = 0;
    for (int q = 0; q < R; ++q) {
        const int g = gamma ? gamma[q] : G;
        for (int j = 1; j <= g; ++j) {
            const double a = surv[(size_t)q * G + (j - 1)];
            if (a > 0.0) {
                pool[n].a = a;
                pool[n].r = q;
                pool[n].j = j;
                ++n;
            }
        }
    }
    qsort(pool, (size_t)n, sizeof(cand_t), cand_cmp);
    return n;
}

static double sps_at(const double* sps, int B) { return sps[B - 1]; }

/* Algorithm 1 steps 3-6 over a sorted pool. early_stop = 1 breaks at the first
 * non-improvement (the causal rule); 0 scans every prefix and keeps the first
 * maximum. Returns the admitted count; keep[] receives the snapshot l*_r. */
static int greedy_scan(const cand_t* pool, int n, int R, const double* sps, int early_stop,
                       int32_t* keep, double* theta_best, double* margin)
{
    int* l = (int*)calloc((size_t)R, sizeof(int));
    int B = R;
    double tau = (double)R;
    double best = (double)R * sps_at(sps, R);
    int admitted = 0;
    double m = INFINITY;
    for (int q = 0; q < R; ++q) keep[q] = 0;
    for (int i = 0; i < n; ++i) {
        l[pool[i].r] = pool[i].j;
        B += 1;
        tau += pool[i].a;
        const double theta = tau * sps_at(sps, B);
        const double rel = fabs(theta - best) / best;
        if (rel < m) m = rel;
        if (theta > best) {
            best = theta;
            admitted = i + 1;
            for (int q = 0; q < R; ++q) keep[q] = l[q];
        } else if (early_stop) {
            break;
        }
    }
    free(l);
    *theta_best = best;
    if (!early_stop) {
        /* for the full scan the decisive margin is the gap between the maximum and
         * every other prefix value */
        double tau2 = (double)R;
        m = INFINITY;
        for (int i = 0; i <= n; ++i) {
            if (i > 0) tau2 += pool[i - 1].a;
            if (i == admitted) continue;
            const double theta = tau2 * sps_at(sps, R + i);
            const double rel = fabs(best - theta) / best;
            if (rel < m) m = rel;
        }
    }
    *margin = m;
    return admitted;
}

int dso_schedule(const dso_schedule_args* a)
{
    if (!a || a->P < 0 || a->R < 1 || a->gamma_max < 1) return 1;
    const int R = a->R, G = a->gamma_max;
    if (a->n_sps < R * (1 + G)) return 1;
    cand_t* pool = (cand_t*)malloc((size_t)R * G * sizeof(cand_t));
    cand_t* old = (cand_t*)malloc((size_t)R * G * sizeof(cand_t));
    if (!pool || !old) {
        free(pool);
        free(old);
        return 2;
    }
    for (int p = 0; p < a->P; ++p) {
        const int32_t* gamma = a->gamma ? a->gamma + (size_t)p * R : NULL;
        const double* surv = a->surv + (size_t)p * R * G;
        int32_t* keep = a->keep + (size_t)p * R;
        const int n = build_pool(pool, R, G, gamma, surv);
        double theta, margin;
        int admitted;
        a->capacity[p] = -1;
        if (a->mode == DSO_SCHED_THRESHOLD) {
            /* static confidence threshold: every candidate whose survival reaches the threshold,
             * l_r the largest such position; no throughput model decides anything */
            double tau = (double)R;
            admitted = 0;
            for (int q = 0; q < R; ++q) keep[q] = 0;
            for (int i = 0; i < n; ++i) {
                if (pool[i].a >= a->threshold) {
                    ++admitted;
                    tau += pool[i].a;
                    if (pool[i].j > keep[pool[i].r]) keep[pool[i].r] = pool[i].j;
                }
            }
            theta = tau * sps_at(a->sps, R + admitted);
            margin = INFINITY;
        } else if (a->mode == DSO_SCHED_SYNC) {
            admitted = greedy_scan(pool, n, R, a->sps, 1, keep, &theta, &margin);
        } else if (a->mode == DSO_SCHED_FULL_SCAN) {
            admitted = greedy_scan(pool, n, R, a->sps, 0, keep, &theta, &margin);
        } else {
            /* section 5.2: capacity K from the survivals two rounds old with an
             * unconstrained search; the current survivals choose which
             * candidates fill K */
            const double* cap = a->surv_capacity + (size_t)p * R * G;
            const int n_old = build_pool(old, R, G, gamma, cap);
            double theta_old;
            const int K = greedy_scan(old, n_old, R, a->sps, 0, keep, &theta_old, &margin);
            a->capacity[p] = K;
            admitted = K < n ? K : n;
            double tau = (double)R;
            for (int q = 0; q < R; ++q) keep[q] = 0;
            for (int i = 0; i < admitted; ++i) {
                tau += pool[i].a;
                if (pool[i].j > keep[pool[i].r]) keep[pool[i].r] = pool[i].j;
            }
            theta = tau * sps_at(a->sps, R + admitted);
        }
        if (a->theta_curve) {
            double* curve = a->theta_curve + (size_t)p * (R * G + 1);
            double tau = (double)R;
            for (int i = 0; i <= R * G; ++i) {
                if (i > n) {
                    curve[i] = NAN;
                    continue;
                }
                if (i > 0) tau += pool[i - 1].a;
                curve[i] = tau * sps_at(a->sps, R + i);
            }
        }
        a->theta_best[p] = theta;
        a->admitted[p] = admitted;
        a->pool[p] = n;
        a->min_margin[p] = margin;
    }
    free(pool);
    free(old);
    return 0;
}

/* ------------------------------------------------------------- verifier */

/* Margins of the residual draw ([P1] section 4 sample_residual) when every probability p_t(v),
 * p_d(v) is known only to a relative error e: a block's mass sum max(0, p_t - p_d) then lies
 * within e * sum (p_t + p_d) of its value, and so does each token's residual. m1 is the winning
 * block's lowest possible perturbed value log(mass) + G minus the highest possible value of any
 * other block; m2 the same for the tokens of the winning block. With e = 0 they are the draw's
 * top-two gaps. A negative margin means another candidate could win under such errors. */
static void residual_margins(const double* zt, double lse_t, const double* ld, double lse_d, int V, int nb,
                             double e, draw_t dr, uint64_t seed, uint64_t round, uint32_t req, double* m1,
                             double* m2)
{
    const int nblk = (V + nb - 1) / nb;
    double low_w = -INFINITY, up_o = -INFINITY;
    for (int b = 0; b < nblk; ++b) {
        const int v0 = b * nb, v1 = (v0 + nb < V) ? v0 + nb : V;
        double mass = 0.0, scale = 0.0;
        for (int v = v0; v < v1; ++v) {
            const double pt = exp(zt[v] - lse_t), pd = exp(ld[v] - lse_d);
            if (pt > pd) mass += pt - pd;
            scale += pt + pd;
        }
        const double g = gumbel(dso_uniform(seed, round, PUR_FINAL_BLOCK, req, 0, (uint32_t)b));
        if (b == dr.block) {
            const double lo = mass - e * scale;
            low_w = lo > 0.0 ? log(lo) + g : -INFINITY;
        } else {
            const double hi = mass + e * scale;
            if (hi > 0.0 && log(hi) + g > up_o) up_o = log(hi) + g;
        }
    }
    *m1 = up_o == -INFINITY ? INFINITY : low_w - up_o;
    low_w = -INFINITY;
    up_o = -INFINITY;
    const int v0 = dr.block * nb, v1 = (v0 + nb < V) ? v0 + nb : V;
    for (int v = v0; v < v1; ++v) {
        const double pt = exp(zt[v] - lse_t), pd = exp(ld[v] - lse_d);
        const double res = pt - pd, scale = pt + pd;
        const double g = gumbel(dso_uniform(seed, round, PUR_FINAL_ELEM, req, 0, (uint32_t)v));
        if (v == dr.token) {
            const double lo = res - e * scale;
            low_w = lo > 0.0 ? log(lo) + g : -INFINITY;
        } else {
            const double hi = res + e * scale;
            if (hi > 0.0 && log(hi) + g > up_o) up_o = log(hi) + g;
        }
    }
    *m2 = up_o == -INFINITY ? INFINITY : low_w - up_o;
}

int dso_verify(const dso_verify_args* a)
{
    if (!a || a->R < 0 || a->gamma_max < 1 || a->V < 1 || a->r < 1 || a->noise_block < 1) return 1;
    const int R = a->R, G = a->gamma_max, V = a->V, r = a->r, nb = a->noise_block;
    double* Wd = to_double(a->W, a->dtype, (size_t)r * V);
    double* zt = (double*)malloc((size_t)V * sizeof(double));
    double* ld = (double*)malloc((size_t)V * sizeof(double));
    double* lw = (double*)malloc((size_t)V * sizeof(double));
    if (!Wd || !zt || !ld || !lw) {
        free(Wd);
        free(zt);
        free(ld);
        free(lw);
        return 2;
    }
    for (int q = 0; q < R; ++q) {
        const uint32_t rid = (uint32_t)(a->req_ids ? a->req_ids[q] : q);
        const double T = (double)a->temperature[q];
        const int ell = a->keep[q];
        for (int k = 0; k < G; ++k) a->accept_margin[(size_t)q * G + k] = NAN;
        for (int i = 0; i <= G; ++i) a->lse_t[(size_t)q * (G + 1) + i] = NAN;
        if (T == 0.0) {
            /* greedy decoding: acceptance is an exact match with the target's arg-max; the first
             * mismatch is replaced by that arg-max, and if every admitted token matches, the
             * arg-max of row l_r is the bonus token */
            int n = ell, next = -1;
            double gap = INFINITY;
            for (int j = 0; j <= ell; ++j) {
                const size_t row = ((size_t)q * (G + 1) + j) * V;
                for (int v = 0; v < V; ++v) zt[v] = load(a->target, a->dtype, row + v);
                const draw_t t = argmax_draw(zt, V);
                if (j == ell || a->tokens[(size_t)q * G + j] != t.token) {
                    n = j;
                    next = t.token;
                    gap = t.gap1;
                    break;
                }
            }
            a->accepted[q] = n;
            a->next_token[q] = next;
            a->resampled[q] = n < ell ? 1 : 0;
            a->gap1[q] = a->gap2[q] = gap;
            a->rgap1[q] = a->rgap2[q] = gap;
            continue;
        }
        /* longest accepted prefix: accept x_j with probability min(1, p_t/p_d) */
        int n = ell;
        for (int j = 1; j <= ell; ++j) {
            const int k = j - 1;
            const size_t row = ((size_t)q * (G + 1) + k) * V;
            for (int v = 0; v < V; ++v) zt[v] = load(a->target, a->dtype, row + v) / T;
            const double lse_t = logsumexp(zt, V);
            a->lse_t[(size_t)q * (G + 1) + k] = lse_t;
            const int x = a->tokens[(size_t)q * G + k];
            const double log_pt = zt[x] - lse_t;
            const double log_pd = a->draft_logit[(size_t)q * G + k] - a->draft_lse[(size_t)q * G + k];
            const double u = dso_uniform(a->seed, a->round, PUR_ACCEPT, rid, (uint32_t)k, 0);
            const double diff = log(u) - (log_pt - log_pd);
            a->accept_margin[(size_t)q * G + k] = fabs(diff);
            if (!(diff < 0.0)) {
                n = k;
                break;
            }
        }
        a->accepted[q] = n;
        /* the target row that supplies the next token: row n in both cases */
        const size_t row = ((size_t)q * (G + 1) + n) * V;
        for (int v = 0; v < V; ++v) zt[v] = load(a->target, a->dtype, row + v) / T;
        const double lse_t = logsumexp(zt, V);
        a->lse_t[(size_t)q * (G + 1) + n] = lse_t;
        draw_t dr;
        if (n < ell) {
            /* rejected at draft position n: resample from norm(max(0, p_t - p_d)) */
            const int prev = n == 0 ? a->anchor[q] : a->tokens[(size_t)q * G + n - 1];
            const int use_bias = (n > 0) || a->bias_first;
            draft_logits(ld, a->U, a->dtype, ((size_t)q * G + n) * V, V, r, Wd, a->E, use_bias, prev, T,
                         a->a_rows ? a->a_rows + ((size_t)q * G + n) * r : NULL);
            const double lse_d = logsumexp(ld, V);
            int any = 0;
            for (int v = 0; v < V; ++v) {
                const double pt = exp(zt[v] - lse_t), pd = exp(ld[v] - lse_d);
                const double res = pt - pd;
                lw[v] = res > 0.0 ? log(res) : -INFINITY;
                if (res > 0.0) any = 1;
            }
            if (!any) {
                /* residual mass zero (possible only through rounding): fall back to p_t */
                for (int v = 0; v < V; ++v) lw[v] = zt[v];
            }
            dr = two_level_draw(lw, V, nb, a->seed, a->round, PUR_FINAL_BLOCK, PUR_FINAL_ELEM, rid, 0);
            if (any) {
                residual_margins(zt, lse_t, ld, lse_d, V, nb, a->res_rel_eps, dr, a->seed, a->round, rid,
                                 &a->rgap1[q], &a->rgap2[q]);
            } else {
                a->rgap1[q] = dr.gap1;
                a->rgap2[q] = dr.gap2;
            }
            a->resampled[q] = 1;
        } else {
            /* every admitted token accepted: bonus token from target row l_r */
            dr = two_level_draw(zt, V, nb, a->seed, a->round, PUR_FINAL_BLOCK, PUR_FINAL_ELEM, rid, 0);
            a->rgap1[q] = dr.gap1;
            a->rgap2[q] = dr.gap2;
            a->resampled[q] = 0;
        }
        a->next_token[q] = dr.token;
        a->gap1[q] = dr.gap1;
        a->gap2[q] = dr.gap2;
    }
    free(Wd);
    free(zt);
    free(ld);
    free(lw);
    return 0;
}

/* ------------------------------------------------------------- ragged verify batch */

int dso_assemble(const dso_assemble_args* a)
{
    if (!a || a->R < 0 || a->gamma_max < 1) return 1;
    const int R = a->R, G = a->gamma_max;
    const size_t cap = (size_t)R * (G + 1);
    for (size_t f = 0; f < cap; ++f) a->flat_tokens[f] = a->flat_request[f] = a->flat_position[f] = -1;
    int32_t off = 0;
    for (int q = 0; q < R; ++q) {
        const int ell = a->keep[q];
        if (ell < 0 || ell > G) return 1;
        a->offsets[q] = off;
        for (int j = 0; j <= ell; ++j) {
            a->flat_tokens[off + j] = j == 0 ? a->anchor[q] : a->tokens[(size_t)q * G + j - 1];
            a->flat_request[off + j] = q;
            a->flat_position[off + j] = j;
        }
        off += ell + 1;
    }
    a->offsets[R] = off;
    return 0;
}
