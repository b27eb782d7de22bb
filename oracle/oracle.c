/*
 * oracle.c -- plain, slow CPU oracle for the forward pass (and, for flat
 * gating, the backward pass) of the Sparsely-Gated Mixture-of-Experts layer
 * (Shazeer et al. 2017, "Outrageously Large Neural Networks").
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check of the package
 * entry file and the CPU-baseline leg of the benchmark may load or call this
 * library.  The CUDA path shares no code with it: no header, helper, table or
 * constant comes from here, and nothing here comes from there.
 *
 * Every value is taken in double precision (fp64) from the exact values of the
 * stored inputs (a bf16 or fp32 input converts to fp64 without loss).  No step
 * is blocked, fused or reordered beyond what the definition states; the only
 * library calls are libm's exp/log1p and libc's qsort.
 *
 * Sources (cited by page title and section):
 *   [MoE:稀疏门控混合专家] nengyongai.cn lesson "MoE:稀疏门控混合专家"
 *     section 二 "一层 MoE 长什么样": expert = 512 -> 1024 -> 512 feed-forward
 *       net with one hidden layer; y = G(x)_1 E_1(x) + ... + G(x)_n E_n(x);
 *       unselected experts have weight 0 and are not computed.
 *     section 三 "门控怎么挑": score = x . W_g (one column per expert);
 *       KeepTopK sets all but the k best scores to -inf; softmax turns the
 *       survivors into weights summing to 1 (worked example with 8 experts);
 *       hierarchical MoE-N-h: 4096 experts = 16 groups x 256, pick 2 groups,
 *       then 2 experts inside each chosen group.
 *     section 四 "为什么要加噪声": H(x)_i = (x.W_g)_i + eps * softplus((x.W_noise)_i),
 *       eps redrawn each time.
 *   [Outrageously Large Neural Networks - 中文验证版] ai-papers.xuzou.cn card,
 *     section "瓶颈": each expert receives about k*b/n rows;
 *     section "方法适配": importance loss and load loss keep samples spread.
 *   [Outrageously Large Neural Networks — MoE 怎样让模型“很大但不每次全算”]
 *     wudongming97 note, section "方法怎么做": importance loss constrains the
 *     total gate weight each expert receives, load loss the number of samples.
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * repository's design notes):
 *   - softplus(z) = log(1 + e^z), evaluated as max(z,0) + log1p(exp(-|z|)).
 *   - ties in KeepTopK go to the lower expert index; the k survivors are
 *     reported in descending H order (this fixes the slot index j).
 *   - bias b_g, when given, is added to the clean score x.W_g.
 *   - hierarchical weight of expert (g, e) = Gp[g] * Gi[e] (product of the two
 *     softmaxes); each level has its own eps columns.
 *   - importance[e] = sum over tokens of G(x)_e; CV^2 = population variance
 *     over the n experts / mean^2 (0 when the mean is 0).  PARITY UNPINNED for
 *     the hierarchical weight product and the CV^2 convention beyond the
 *     invariants the tests check: the pages print no value for either.
 *   - the expert has biases b1, b2; ReLU after the first layer only.
 *   - load estimate: the paper's smooth load (probability of staying in the
 *     top k under a redraw of the expert's own noise), summed over tokens;
 *     flat gating with noise only.  PARITY PINNED by a Monte Carlo redraw of
 *     one expert's noise, the k = n case and the vanishing-noise limit.
 *
 * Weight layouts (row-major):
 *   Wg, Wnoise : [d, C] where C = n (flat) or G + n (hierarchical: the first G
 *                columns score the groups, then G blocks of m = n/G columns,
 *                block g scoring the experts of group g)
 *   bg         : [C] or NULL;  eps : [T, C] or NULL (NULL = no noise)
 *   W1         : [n, h, d]  (expert e maps d -> h:  a = ReLU(W1[e] x + b1[e]))
 *   b1         : [n, h]
 *   W2         : [n, d, h]  (expert e maps h -> d:  E = W2[e] a + b2[e])
 *   b2         : [n, d]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* softplus(z) = log(1 + e^z) in its overflow-free form.
 * [MoE:稀疏门控混合专家] section 四: the noise scale is softplus((x.W_noise)_i). */
double oracle_softplus(double z) {
    return (z > 0.0 ? z : 0.0) + log1p(exp(-fabs(z)));
}

typedef struct {
    double h;
    int i;
} scored;

/* Order for KeepTopK: larger H first; equal H -> lower index first. */
static int by_desc_h_then_index(const void *pa, const void *pb) {
    const scored *a = (const scored *)pa, *b = (const scored *)pb;
    if (a->h > b->h) return -1;
    if (a->h < b->h) return 1;
    return (a->i > b->i) - (a->i < b->i);
}

/*
 * One noisy top-k gate over m consecutive score columns [col0, col0+m) of the
 * [d, ld] matrices Wg and Wn, for a single token x[0..d).
 *
 *   step 1  scores   c_i = sum_j x_j Wg[j, col0+i]  (+ bg[col0+i])
 *                    r_i = sum_j x_j Wn[j, col0+i]
 *   step 2  noise    H_i = c_i + eps_i * softplus(r_i)     ([MoE:稀疏门控混合专家] §四)
 *   step 3  KeepTopK H_i kept for the k best, -inf elsewhere  (§三, step ②)
 *   step 4  softmax  over all m entries; e^-inf = 0            (§三, step ③)
 *
 * Outputs: sel[0..k) local column indices in descending H order, w[0..k)
 * their softmax weights, H[0..m) the noisy scores (scratch owned by caller),
 * and *margin = H_(k) - H_(k+1) (+inf when k == m).
 */
static void noisy_top_k_gate(int d, const double *x, const double *Wg, const double *Wn,
                             int64_t ld, int col0, int m, const double *bg,
                             const double *eps_row, int k, int *sel, double *w,
                             double *H, scored *order, double *kept, double *margin) {
    for (int i = 0; i < m; ++i) {
        double c = 0.0, r = 0.0;
        for (int j = 0; j < d; ++j) c += x[j] * Wg[(int64_t)j * ld + col0 + i];
        if (bg) c += bg[col0 + i];
        /* Without eps the noise term is absent, and Wn may be absent too. */
        if (eps_row && Wn) {
            for (int j = 0; j < d; ++j) r += x[j] * Wn[(int64_t)j * ld + col0 + i];
            H[i] = c + eps_row[col0 + i] * oracle_softplus(r);
        } else {
            H[i] = c;
        }
    }
    /* KeepTopK: sort (H desc, index asc) and keep the first k. */
    for (int i = 0; i < m; ++i) {
        order[i].h = H[i];
        order[i].i = i;
    }
    qsort(order, (size_t)m, sizeof(scored), by_desc_h_then_index);
    for (int i = 0; i < m; ++i) kept[i] = -INFINITY;
    for (int q = 0; q < k; ++q) kept[order[q].i] = order[q].h;
    *margin = (k < m) ? order[k - 1].h - order[k].h : INFINITY;
    /* Softmax over the whole vector; exp(-inf - max) = 0 for the dropped ones. */
    double mx = -INFINITY;
    for (int i = 0; i < m; ++i)
        if (kept[i] > mx) mx = kept[i];
    double s = 0.0;
    for (int i = 0; i < m; ++i) {
        kept[i] = exp(kept[i] - mx);
        s += kept[i];
    }
    for (int q = 0; q < k; ++q) {
        sel[q] = order[q].i;
        w[q] = kept[order[q].i] / s;
    }
}

/*
 * Flat noisy top-k gating for T tokens.
 *   idx[T,k] (int32, descending H), G[T,k], H_out[T,n] (optional),
 *   margin[T] (optional): gap between the k-th and (k+1)-th noisy score.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_gate_flat(int64_t T, int d, int n, int k, const double *x, const double *Wg,
                     const double *Wn, const double *bg, const double *eps, int32_t *idx,
                     double *G, double *H_out, double *margin) {
    if (T < 0 || d <= 0 || n <= 0 || k <= 0 || k > n || (eps && !Wn)) return -1;
    int bad = 0;
#pragma omp parallel
    {
        double *H = (double *)malloc(sizeof(double) * (size_t)n);
        double *kept = (double *)malloc(sizeof(double) * (size_t)n);
        scored *order = (scored *)malloc(sizeof(scored) * (size_t)n);
        int *sel = (int *)malloc(sizeof(int) * (size_t)k);
        double *w = (double *)malloc(sizeof(double) * (size_t)k);
        if (!H || !kept || !order || !sel || !w) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 8)
            for (int64_t t = 0; t < T; ++t) {
                double mg;
                noisy_top_k_gate(d, x + t * d, Wg, Wn, n, 0, n, bg,
                                 eps ? eps + t * (int64_t)n : NULL, k, sel, w, H, order,
                                 kept, &mg);
                for (int q = 0; q < k; ++q) {
                    idx[t * k + q] = sel[q];
                    G[t * k + q] = w[q];
                }
                if (H_out) memcpy(H_out + t * (int64_t)n, H, sizeof(double) * (size_t)n);
                if (margin) margin[t] = mg;
            }
        }
        free(H);
        free(kept);
        free(order);
        free(sel);
        free(w);
    }
    return bad ? -1 : 0;
}

/*
 * Load estimate of the flat noisy gate.  [Outrageously Large Neural Networks
 * - 中文验证版] section 方法适配 and the wudongming97 note name a load loss
 * beside the importance loss: it balances how many samples each expert
 * receives.  A count is not smooth, so the load is estimated from the noise
 * (the pages are cut off before the formula; this follows the paper's
 * load-balancing appendix): for token t and expert i,
 *   P(t, i) = probability that expert i is among the k best when only its own
 *             noise is redrawn and the other experts' noisy scores stay fixed
 *           = Phi((c_i - kth_excluding(H, k, i)) / softplus(r_i)),
 * with c_i = (x.W_g)_i (+ bg_i), r_i = (x.W_noise)_i, H as in the gate, and
 * kth_excluding(H, k, i) the k-th largest H_j over j != i (-inf when fewer
 * than k others exist; ties ordered as in KeepTopK).  Phi(z) = erfc(-z/sqrt2)/2.
 *   load[i] = sum_t P(t, i);  cv2 = population variance of load / mean^2.
 * P[T,n] is written (caller-owned); the sums over t run in token order.
 */
int oracle_load(int64_t T, int d, int n, int k, const double *x, const double *Wg,
                const double *Wn, const double *bg, const double *eps, double *P, double *load,
                double *cv2) {
    if (T < 0 || d <= 0 || n <= 0 || k <= 0 || k > n || !Wn || !eps) return -1;
    int bad = 0;
#pragma omp parallel
    {
        double *c = (double *)malloc(sizeof(double) * (size_t)n);
        double *sp = (double *)malloc(sizeof(double) * (size_t)n);
        scored *order = (scored *)malloc(sizeof(scored) * (size_t)n);
        char *in_top = (char *)malloc((size_t)n);
        if (!c || !sp || !order || !in_top) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 8)
            for (int64_t t = 0; t < T; ++t) {
                const double *xt = x + t * d;
                for (int i = 0; i < n; ++i) {
                    double ci = 0.0, ri = 0.0;
                    for (int j = 0; j < d; ++j) {
                        ci += xt[j] * Wg[(int64_t)j * n + i];
                        ri += xt[j] * Wn[(int64_t)j * n + i];
                    }
                    if (bg) ci += bg[i];
                    c[i] = ci;
                    sp[i] = oracle_softplus(ri);
                    order[i].h = ci + eps[t * (int64_t)n + i] * sp[i];
                    order[i].i = i;
                }
                qsort(order, (size_t)n, sizeof(scored), by_desc_h_then_index);
                memset(in_top, 0, (size_t)n);
                for (int q = 0; q < k; ++q) in_top[order[q].i] = 1;
                /* k-th largest of the others: for a member the (k+1)-th overall,
                 * for a non-member the k-th overall */
                const double kth = order[k - 1].h;
                const double next = (k < n) ? order[k].h : -INFINITY;
                for (int i = 0; i < n; ++i) {
                    const double thr = in_top[i] ? next : kth;
                    P[t * (int64_t)n + i] =
                        (thr == -INFINITY) ? 1.0 : 0.5 * erfc(-(c[i] - thr) / (sp[i] * sqrt(2.0)));
                }
            }
        }
        free(c);
        free(sp);
        free(order);
        free(in_top);
    }
    if (bad) return -1;
    double sum = 0.0;
    for (int i = 0; i < n; ++i) {
        double acc = 0.0;
        for (int64_t t = 0; t < T; ++t) acc += P[t * (int64_t)n + i];
        load[i] = acc;
        sum += acc;
    }
    const double mean = sum / n;
    double var = 0.0;
    for (int i = 0; i < n; ++i) var += (load[i] - mean) * (load[i] - mean);
    var /= n;
    *cv2 = mean != 0.0 ? var / (mean * mean) : 0.0;
    return 0;
}

/*
 * Hierarchical (MoE-N-h) gating, [MoE:稀疏门控混合专家] section 三: the groups
 * are scored first and the k_g best kept (noisy top-k + softmax -> Gp); then,
 * inside each chosen group g (in descending primary order), the m = n/G
 * experts are scored with that group's own columns and the k_i = k/k_g best
 * kept (-> Gi).  Output slot j = (group rank) * k_i + (inner rank); expert
 * index g*m + e; weight Gp[g] * Gi[e].
 * margin[t] = smallest of the primary gap and every chosen group's inner gap.
 */
int oracle_gate_hier(int64_t T, int d, int groups, int m, int k_groups, int k_inner,
                     const double *x, const double *Wg, const double *Wn, const double *bg,
                     const double *eps, int32_t *idx, double *G, double *margin) {
    if (T < 0 || d <= 0 || groups <= 0 || m <= 0 || k_groups <= 0 || k_groups > groups ||
        k_inner <= 0 || k_inner > m || (eps && !Wn))
        return -1;
    const int64_t C = (int64_t)groups + (int64_t)groups * m; /* score columns */
    const int k = k_groups * k_inner;
    const int big = groups > m ? groups : m;
    int bad = 0;
#pragma omp parallel
    {
        double *H = (double *)malloc(sizeof(double) * (size_t)big);
        double *kept = (double *)malloc(sizeof(double) * (size_t)big);
        scored *order = (scored *)malloc(sizeof(scored) * (size_t)big);
        int *gsel = (int *)malloc(sizeof(int) * (size_t)k_groups);
        double *gw = (double *)malloc(sizeof(double) * (size_t)k_groups);
        int *esel = (int *)malloc(sizeof(int) * (size_t)k_inner);
        double *ew = (double *)malloc(sizeof(double) * (size_t)k_inner);
        if (!H || !kept || !order || !gsel || !gw || !esel || !ew) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 8)
            for (int64_t t = 0; t < T; ++t) {
                const double *xt = x + t * d;
                const double *et = eps ? eps + t * C : NULL;
                double mg, mg_in;
                noisy_top_k_gate(d, xt, Wg, Wn, C, 0, groups, bg, et, k_groups, gsel, gw, H,
                                 order, kept, &mg);
                for (int r = 0; r < k_groups; ++r) {
                    const int g = gsel[r];
                    noisy_top_k_gate(d, xt, Wg, Wn, C, groups + g * m, m, bg, et, k_inner, esel,
                                     ew, H, order, kept, &mg_in);
                    if (mg_in < mg) mg = mg_in;
                    for (int q = 0; q < k_inner; ++q) {
                        idx[t * k + r * k_inner + q] = g * m + esel[q];
                        G[t * k + r * k_inner + q] = gw[r] * ew[q];
                    }
                }
                if (margin) margin[t] = mg;
            }
        }
        free(H);
        free(kept);
        free(order);
        free(gsel);
        free(gw);
        free(esel);
        free(ew);
    }
    return bad ? -1 : 0;
}

typedef struct {
    int32_t e;
    int64_t s;
} slot_key;

static int by_expert_then_slot(const void *pa, const void *pb) {
    const slot_key *a = (const slot_key *)pa, *b = (const slot_key *)pb;
    if (a->e != b->e) return (a->e > b->e) - (a->e < b->e);
    return (a->s > b->s) - (a->s < b->s);
}

/*
 * Routing of the S = T*k slots (slot s = t*k + j) to expert-contiguous rows.
 * The pages' "conditional computation" (unselected experts are not computed)
 * needs each expert's rows gathered together; each expert sees about k*b/n
 * rows ([Outrageously Large Neural Networks - 中文验证版] section 瓶颈).
 *   counts[e]      number of slots routed to e (the discrete load)
 *   offsets[n+1]   exclusive prefix sum of counts
 *   perm[S]        row r -> slot, rows sorted by (expert, slot): stable
 *   inv_perm[S]    slot -> row
 *   importance[e]  sum of the gate weights of e's rows, summed in row order
 *                  ([MoE 怎样让模型“很大但不每次全算”] section 方法怎么做)
 *   *cv2           population variance of importance / mean^2 (0 if mean 0)
 * Returns 0, or -1 on a bad argument (an expert index outside [0, n)).
 */
int oracle_route(int64_t T, int n, int k, const int32_t *idx, const double *G, int32_t *counts,
                 int32_t *offsets, int32_t *perm, int32_t *inv_perm, double *importance,
                 double *cv2) {
    if (T < 0 || n <= 0 || k <= 0) return -1;
    const int64_t S = T * k;
    for (int e = 0; e < n; ++e) counts[e] = 0;
    for (int64_t s = 0; s < S; ++s) {
        if (idx[s] < 0 || idx[s] >= n) return -1;
        counts[idx[s]] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < n; ++e) offsets[e + 1] = offsets[e] + counts[e];
    slot_key *keys = (slot_key *)malloc(sizeof(slot_key) * (size_t)(S > 0 ? S : 1));
    if (!keys) return -1;
    for (int64_t s = 0; s < S; ++s) {
        keys[s].e = idx[s];
        keys[s].s = s;
    }
    qsort(keys, (size_t)S, sizeof(slot_key), by_expert_then_slot);
    for (int64_t r = 0; r < S; ++r) {
        perm[r] = (int32_t)keys[r].s;
        inv_perm[keys[r].s] = (int32_t)r;
    }
    free(keys);
    double total = 0.0;
    for (int e = 0; e < n; ++e) {
        double acc = 0.0;
        for (int64_t r = offsets[e]; r < offsets[e + 1]; ++r) acc += G[perm[r]];
        importance[e] = acc;
        total += acc;
    }
    const double mean = total / n;
    double var = 0.0;
    for (int e = 0; e < n; ++e) var += (importance[e] - mean) * (importance[e] - mean);
    var /= n;
    *cv2 = (mean != 0.0) ? var / (mean * mean) : 0.0;
    return 0;
}

/*
 * One expert on one token: E(x) = W2 . ReLU(W1 . x + b1) + b2, with no rounding
 * between the layers.  [MoE:稀疏门控混合专家] section 二: each expert is a
 * feed-forward network with one hidden layer of ReLU units (512 -> 1024 -> 512
 * in the pages' example).  W1e [h, d], b1e [h] or NULL, W2e [d, h], b2e [d] or
 * NULL; out [d].  a is caller scratch of length h.
 */
void oracle_expert(int d, int h, const double *x, const double *W1e, const double *b1e,
                   const double *W2e, const double *b2e, double *a, double *out) {
    for (int i = 0; i < h; ++i) {
        double z = b1e ? b1e[i] : 0.0;
        for (int j = 0; j < d; ++j) z += W1e[(int64_t)i * d + j] * x[j];
        a[i] = z > 0.0 ? z : 0.0;
    }
    for (int o = 0; o < d; ++o) {
        double z = b2e ? b2e[o] : 0.0;
        for (int i = 0; i < h; ++i) z += W2e[(int64_t)o * h + i] * a[i];
        out[o] = z;
    }
}

/*
 * Combine: y[t] = sum_j G[t,j] * E_{idx[t,j]}(x_t), j = 0..k-1 in slot order
 * ([MoE:稀疏门控混合专家] section 二, y = sum_i G(x)_i E_i(x), summed over the
 * selected experts only since the others have weight 0).
 * Experts are evaluated per (token, slot); no expert is evaluated for a token
 * that did not select it.
 */
int oracle_experts_combine(int64_t T, int d, int h, int n, int k, const double *x,
                           const int32_t *idx, const double *G, const double *W1,
                           const double *b1, const double *W2, const double *b2, double *y) {
    if (T < 0 || d <= 0 || h <= 0 || n <= 0 || k <= 0) return -1;
    int bad = 0;
#pragma omp parallel
    {
        double *a = (double *)malloc(sizeof(double) * (size_t)h);
        double *E = (double *)malloc(sizeof(double) * (size_t)d);
        if (!a || !E) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t t = 0; t < T; ++t) {
                double *yt = y + t * d;
                for (int o = 0; o < d; ++o) yt[o] = 0.0;
                for (int j = 0; j < k; ++j) {
                    const int e = idx[t * k + j];
                    if (e < 0 || e >= n) {
#pragma omp atomic write
                        bad = 1;
                        continue;
                    }
                    oracle_expert(d, h, x + t * d, W1 + (int64_t)e * h * d,
                                  b1 ? b1 + (int64_t)e * h : NULL, W2 + (int64_t)e * d * h,
                                  b2 ? b2 + (int64_t)e * d : NULL, a, E);
                    for (int o = 0; o < d; ++o) yt[o] += G[t * k + j] * E[o];
                }
            }
        }
        free(a);
        free(E);
    }
    return bad ? -1 : 0;
}

/*
 * The whole forward pass: gate (flat when groups == 0, else hierarchical with
 * k_groups groups kept and k/k_groups experts per kept group), then routing
 * (counts, perm, importance, CV^2), then the selected experts and the combine.
 * perm, inv_perm, offsets may be NULL if not wanted (they are computed anyway).
 */
int oracle_forward(int64_t T, int d, int h, int n, int k, int groups, int k_groups,
                   const double *x, const double *Wg, const double *Wn, const double *bg,
                   const double *eps, const double *W1, const double *b1, const double *W2,
                   const double *b2, double *y, double *G, int32_t *idx, double *importance,
                   double *cv2, int32_t *counts, int32_t *offsets, int32_t *perm,
                   int32_t *inv_perm) {
    int rc;
    if (groups == 0) {
        rc = oracle_gate_flat(T, d, n, k, x, Wg, Wn, bg, eps, idx, G, NULL, NULL);
    } else {
        if (k_groups <= 0 || k % k_groups != 0 || n % groups != 0) return -1;
        rc = oracle_gate_hier(T, d, groups, n / groups, k_groups, k / k_groups, x, Wg, Wn, bg,
                              eps, idx, G, NULL);
    }
    if (rc) return rc;
    const int64_t S = T * k;
    int32_t *off = offsets ? offsets : (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 1));
    int32_t *pm = perm ? perm : (int32_t *)malloc(sizeof(int32_t) * (size_t)(S > 0 ? S : 1));
    int32_t *ip = inv_perm ? inv_perm : (int32_t *)malloc(sizeof(int32_t) * (size_t)(S > 0 ? S : 1));
    if (!off || !pm || !ip) return -1;
    rc = oracle_route(T, n, k, idx, G, counts, off, pm, ip, importance, cv2);
    if (!offsets) free(off);
    if (!perm) free(pm);
    if (!inv_perm) free(ip);
    if (rc) return rc;
    return oracle_experts_combine(T, d, h, n, k, x, idx, G, W1, b1, W2, b2, y);
}

/*
 * Combine alone, from expert outputs already in expert-row order:
 * y[t] = sum_{j<k} G[t,j] * Y[inv_perm[t*k+j]]  (rows with inv_perm < 0 skipped).
 */
int oracle_combine_rows(int64_t T, int d, int k, int64_t S, const double *Y,
                        const int32_t *inv_perm, const double *G, double *y) {
    if (T < 0 || d <= 0 || k <= 0) return -1;
    for (int64_t t = 0; t < T; ++t) {
        for (int o = 0; o < d; ++o) y[t * d + o] = 0.0;
        for (int j = 0; j < k; ++j) {
            const int32_t r = inv_perm[t * k + j];
            if (r < 0) continue;
            if (r >= S) return -1;
            for (int o = 0; o < d; ++o) y[t * d + o] += G[t * k + j] * Y[(int64_t)r * d + o];
        }
    }
    return 0;
}

/*
 * Backward pass of the flat layer.  [MoE:稀疏门控混合专家] section 四 and the
 * wudongming97 note train the layer (noise during training, the importance
 * loss beside the task loss); the pages give no formula for the gradients, so
 * they are the chain rule of the forward definition above, taken with the
 * selection held fixed (KeepTopK is piecewise constant in its inputs), for
 *
 *   L = sum_t <dy_t, y_t>  +  w_imp * CV^2(importance)
 *
 * dy [T, d] is the upstream gradient of y, w_imp the weight of the importance
 * loss.  Written out, for token t and slot j with expert e = idx[t, j]:
 *   z = W1[e] x_t + b1[e],  a = max(z, 0),  E = W2[e] a + b2[e]
 *   dG_j   = <dy_t, E> + w_imp * dCV2/dimp_e
 *            dCV2/dimp_e = 2 (imp_e - mu) / (n mu^2) - 2 var / (n mu^3)
 *            (mu, var: mean and population variance of importance; 0 if mu = 0)
 *   dH_j   = G_j (dG_j - sum_l G_l dG_l)                   (softmax over the k kept)
 *   dc_j   = dH_j;  dr_j = dH_j * eps[t, e] * sigmoid(r_j),  r_j = x_t . Wn[:, e]
 *   dE     = G_j dy_t;  da = W2[e]^T dE;  dz = da * [z > 0]
 *   dx_t  += dc_j Wg[:, e] + dr_j Wn[:, e] + W1[e]^T dz
 *   dWg[:, e] += dc_j x_t;  dWn[:, e] += dr_j x_t;  dbg[e] += dc_j
 *   dW2[e] += dE a^T;  db2[e] += dE;  dW1[e] += dz x_t^T;  db1[e] += dz
 * The per-token part runs in parallel over tokens; the per-expert sums run in
 * parallel over experts, each over its slots in token order.  idx_out [T, k]
 * and G_out [T, k] (the gate of the forward) may be NULL.  eps NULL = no noise
 * (then dWn is all zeros).  Every output is overwritten.
 */
int oracle_backward_flat(int64_t T, int d, int h, int n, int k, const double *x,
                         const double *Wg, const double *Wn, const double *bg, const double *eps,
                         const double *W1, const double *b1, const double *W2, const double *b2,
                         const double *dy, double w_imp, double *dx, double *dWg, double *dWn,
                         double *dbg, double *dW1, double *db1, double *dW2, double *db2,
                         int32_t *idx_out, double *G_out) {
    if (T < 0 || d <= 0 || h <= 0 || n <= 0 || k <= 0 || k > n) return -1;
    const int64_t S = T * k;
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)(S > 0 ? S : 1));
    double *G = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
    double *dc = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
    double *dr = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
    double *imp = (double *)calloc((size_t)n, sizeof(double));
    double *gimp = (double *)calloc((size_t)n, sizeof(double));
    if (!idx || !G || !dc || !dr || !imp || !gimp) return -1;
    int rc = oracle_gate_flat(T, d, n, k, x, Wg, Wn, bg, eps, idx, G, NULL, NULL);
    if (rc) return rc;

    /* importance and the gradient of w_imp * CV^2 with respect to it */
    for (int64_t s = 0; s < S; ++s) imp[idx[s]] += G[s];
    double mu = 0.0, var = 0.0;
    for (int e = 0; e < n; ++e) mu += imp[e];
    mu /= n;
    for (int e = 0; e < n; ++e) var += (imp[e] - mu) * (imp[e] - mu);
    var /= n;
    if (mu != 0.0)
        for (int e = 0; e < n; ++e)
            gimp[e] = w_imp * (2.0 * (imp[e] - mu) / (n * mu * mu) - 2.0 * var / (n * mu * mu * mu));

    int bad = 0;
    /* per token: dG, dH, dc, dr and the whole of dx_t */
#pragma omp parallel
    {
        double *z = (double *)malloc(sizeof(double) * (size_t)h);
        double *a = (double *)malloc(sizeof(double) * (size_t)h);
        double *E = (double *)malloc(sizeof(double) * (size_t)d);
        double *dG = (double *)malloc(sizeof(double) * (size_t)k);
        if (!z || !a || !E || !dG) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t t = 0; t < T; ++t) {
                const double *xt = x + t * d;
                const double *dyt = dy + t * d;
                double *dxt = dx + t * d;
                for (int o = 0; o < d; ++o) dxt[o] = 0.0;
                for (int j = 0; j < k; ++j) {
                    const int e = idx[t * k + j];
                    const double *W1e = W1 + (int64_t)e * h * d, *W2e = W2 + (int64_t)e * d * h;
                    for (int i = 0; i < h; ++i) {
                        double v = b1 ? b1[(int64_t)e * h + i] : 0.0;
                        for (int q = 0; q < d; ++q) v += W1e[(int64_t)i * d + q] * xt[q];
                        z[i] = v;
                        a[i] = v > 0.0 ? v : 0.0;
                    }
                    double g = gimp[e];
                    for (int o = 0; o < d; ++o) {
                        double v = b2 ? b2[(int64_t)e * d + o] : 0.0;
                        for (int i = 0; i < h; ++i) v += W2e[(int64_t)o * h + i] * a[i];
                        E[o] = v;
                        g += dyt[o] * v;
                    }
                    dG[j] = g;
                }
                double sGdG = 0.0;
                for (int j = 0; j < k; ++j) sGdG += G[t * k + j] * dG[j];
                for (int j = 0; j < k; ++j) {
                    const int64_t s = t * k + j;
                    const int e = idx[s];
                    const double dH = G[s] * (dG[j] - sGdG);
                    double r = 0.0;
                    for (int q = 0; q < d; ++q) r += xt[q] * Wn[(int64_t)q * n + e];
                    const double dr_s = eps ? dH * eps[t * (int64_t)n + e] / (1.0 + exp(-r)) : 0.0;
                    dc[s] = dH;
                    dr[s] = dr_s;
                    for (int q = 0; q < d; ++q)
                        dxt[q] += dH * Wg[(int64_t)q * n + e] + dr_s * Wn[(int64_t)q * n + e];
                    /* expert part: dz = (W2[e]^T (G dy_t)) * [z > 0]; dx_t += W1[e]^T dz */
                    const double *W1e = W1 + (int64_t)e * h * d, *W2e = W2 + (int64_t)e * d * h;
                    for (int i = 0; i < h; ++i) {
                        double v = b1 ? b1[(int64_t)e * h + i] : 0.0;
                        for (int q = 0; q < d; ++q) v += W1e[(int64_t)i * d + q] * xt[q];
                        double da = 0.0;
                        for (int o = 0; o < d; ++o) da += W2e[(int64_t)o * h + i] * G[s] * dyt[o];
                        const double dz = v > 0.0 ? da : 0.0;
                        for (int q = 0; q < d; ++q) dxt[q] += W1e[(int64_t)i * d + q] * dz;
                    }
                }
            }
        }
        free(z);
        free(a);
        free(E);
        free(dG);
    }
    if (bad) return -1;

    /* per expert: weight and bias gradients, summed over its slots in token order */
#pragma omp parallel
    {
        double *a = (double *)malloc(sizeof(double) * (size_t)h);
        double *dz = (double *)malloc(sizeof(double) * (size_t)h);
        double *dE = (double *)malloc(sizeof(double) * (size_t)d);
        if (!a || !dz || !dE) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int e = 0; e < n; ++e) {
                const double *W1e = W1 + (int64_t)e * h * d, *W2e = W2 + (int64_t)e * d * h;
                double *dW1e = dW1 + (int64_t)e * h * d, *dW2e = dW2 + (int64_t)e * d * h;
                memset(dW1e, 0, sizeof(double) * (size_t)h * d);
                memset(dW2e, 0, sizeof(double) * (size_t)d * h);
                if (db1) memset(db1 + (int64_t)e * h, 0, sizeof(double) * (size_t)h);
                if (db2) memset(db2 + (int64_t)e * d, 0, sizeof(double) * (size_t)d);
                for (int q = 0; q < d; ++q) {
                    dWg[(int64_t)q * n + e] = 0.0;
                    if (dWn) dWn[(int64_t)q * n + e] = 0.0;
                }
                if (dbg) dbg[e] = 0.0;
                for (int64_t s = 0; s < S; ++s) {
                    if (idx[s] != e) continue;
                    const double *xt = x + (s / k) * d;
                    const double *dyt = dy + (s / k) * d;
                    for (int i = 0; i < h; ++i) {
                        double v = b1 ? b1[(int64_t)e * h + i] : 0.0;
                        for (int q = 0; q < d; ++q) v += W1e[(int64_t)i * d + q] * xt[q];
                        a[i] = v > 0.0 ? v : 0.0;
                        dz[i] = v;  /* pre-activation, masked below */
                    }
                    for (int o = 0; o < d; ++o) dE[o] = G[s] * dyt[o];
                    for (int i = 0; i < h; ++i) {
                        double da = 0.0;
                        for (int o = 0; o < d; ++o) da += W2e[(int64_t)o * h + i] * dE[o];
                        dz[i] = dz[i] > 0.0 ? da : 0.0;
                    }
                    for (int o = 0; o < d; ++o) {
                        for (int i = 0; i < h; ++i) dW2e[(int64_t)o * h + i] += dE[o] * a[i];
                        if (db2) db2[(int64_t)e * d + o] += dE[o];
                    }
                    for (int i = 0; i < h; ++i) {
                        for (int q = 0; q < d; ++q) dW1e[(int64_t)i * d + q] += dz[i] * xt[q];
                        if (db1) db1[(int64_t)e * h + i] += dz[i];
                    }
                    for (int q = 0; q < d; ++q) {
                        dWg[(int64_t)q * n + e] += dc[s] * xt[q];
                        if (dWn) dWn[(int64_t)q * n + e] += dr[s] * xt[q];
                    }
                    if (dbg) dbg[e] += dc[s];
                }
            }
        }
        free(a);
        free(dz);
        free(dE);
    }
    if (idx_out) memcpy(idx_out, idx, sizeof(int32_t) * (size_t)S);
    if (G_out) memcpy(G_out, G, sizeof(double) * (size_t)S);
    free(idx);
    free(G);
    free(dc);
    free(dr);
    free(imp);
    free(gimp);
    return bad ? -1 : 0;
}

/*
 * Balanced routing.  "Outrageously Large Neural Networks - 中文验证版", section
 * 方法适配: in some translation experiments a per-batch mask gives every
 * expert the same batch size during training, and per-expert thresholds
 * approximate that behaviour at inference.  The pages give no formula; the
 * plainest reading, written out here:
 *   H[t, e]   the noisy score of the flat gate (as in noisy_top_k_gate)
 *   batchwise (thr == NULL): m = floor(k*T/n); expert e keeps the m tokens
 *             with the largest H[:, e] (equal scores: the lower token index
 *             first)
 *   threshold (thr given):   expert e keeps token t iff H[t, e] > thr[e]
 *   weights   w[t, e] = softmax of H[t, .] over the experts that kept t
 *             (KeepTopK replaced by the mask); a token no expert kept has
 *             y_t = 0
 *   y[t]      = sum over the kept experts e, in increasing e, of w[t, e] E_e(x_t)
 * Outputs y [T, d], counts [n] (tokens kept per expert), W [T, n] (the
 * weights, 0 where not kept; may be NULL).  Returns 0, or -1 on bad arguments.
 */
typedef struct {
    double h;
    int64_t t;
} col_entry;

static int by_desc_h_then_token(const void *pa, const void *pb) {
    const col_entry *a = (const col_entry *)pa, *b = (const col_entry *)pb;
    if (a->h > b->h) return -1;
    if (a->h < b->h) return 1;
    return (a->t > b->t) - (a->t < b->t);
}

int oracle_forward_balanced(int64_t T, int d, int h, int n, int k, const double *x,
                            const double *Wg, const double *Wn, const double *bg,
                            const double *eps, const double *thr, const double *W1,
                            const double *b1, const double *W2, const double *b2, double *y,
                            int32_t *counts, double *W) {
    if (T < 0 || d <= 0 || h <= 0 || n <= 0 || k <= 0 || k > n) return -1;
    double *H = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * (size_t)n);
    unsigned char *keep = (unsigned char *)calloc((size_t)(T > 0 ? T : 1) * (size_t)n, 1);
    if (!H || !keep) return -1;
    /* noisy scores */
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int e = 0; e < n; ++e) {
            double c = bg ? bg[e] : 0.0, r = 0.0;
            for (int j = 0; j < d; ++j) {
                c += x[t * d + j] * Wg[(int64_t)j * n + e];
                r += x[t * d + j] * Wn[(int64_t)j * n + e];
            }
            H[t * n + e] = eps ? c + eps[t * (int64_t)n + e] * oracle_softplus(r) : c;
        }
    }
    /* the mask */
    if (thr) {
        for (int64_t t = 0; t < T; ++t)
            for (int e = 0; e < n; ++e) keep[t * n + e] = H[t * n + e] > thr[e];
    } else {
        const int64_t m = (int64_t)k * T / n;
        col_entry *col = (col_entry *)malloc(sizeof(col_entry) * (size_t)(T > 0 ? T : 1));
        if (!col) return -1;
        for (int e = 0; e < n; ++e) {
            for (int64_t t = 0; t < T; ++t) {
                col[t].h = H[t * n + e];
                col[t].t = t;
            }
            qsort(col, (size_t)T, sizeof(col_entry), by_desc_h_then_token);
            for (int64_t q = 0; q < m; ++q) keep[col[q].t * n + e] = 1;
        }
        free(col);
    }
    for (int e = 0; e < n; ++e) {
        int32_t c = 0;
        for (int64_t t = 0; t < T; ++t) c += keep[t * n + e];
        counts[e] = c;
    }
    /* weights and the experts */
    int bad = 0;
#pragma omp parallel
    {
        double *a = (double *)malloc(sizeof(double) * (size_t)h);
        double *E = (double *)malloc(sizeof(double) * (size_t)d);
        if (!a || !E) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t t = 0; t < T; ++t) {
                double *yt = y + t * d;
                for (int o = 0; o < d; ++o) yt[o] = 0.0;
                double mx = -INFINITY, sum = 0.0;
                for (int e = 0; e < n; ++e)
                    if (keep[t * n + e] && H[t * n + e] > mx) mx = H[t * n + e];
                for (int e = 0; e < n; ++e)
                    if (keep[t * n + e]) sum += exp(H[t * n + e] - mx);
                for (int e = 0; e < n; ++e) {
                    const double w = keep[t * n + e] ? exp(H[t * n + e] - mx) / sum : 0.0;
                    if (W) W[t * n + e] = w;
                    if (!keep[t * n + e]) continue;
                    oracle_expert(d, h, x + t * d, W1 + (int64_t)e * h * d,
                                  b1 ? b1 + (int64_t)e * h : NULL, W2 + (int64_t)e * d * h,
                                  b2 ? b2 + (int64_t)e * d : NULL, a, E);
                    for (int o = 0; o < d; ++o) yt[o] += w * E[o];
                }
            }
        }
        free(a);
        free(E);
    }
    free(H);
    free(keep);
    return bad ? -1 : 0;
}
