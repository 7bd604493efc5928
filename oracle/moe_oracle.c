/*
 * moe_oracle.c -- plain, slow, obviously correct CPU definition of the
 * routed-expert MoE layer. TEST INFRASTRUCTURE ONLY: the tests, the smoke
 * check and the benchmark's CPU-baseline leg call it; the CUDA library never
 * does, and the two share no code, header or table.
 *
 * Everything is accumulated in double precision with straight loops, in the
 * order the definitions are written. Where a floating-point value decides an
 * integer (which experts are the top k, whether a gate weight reaches the
 * substitution threshold) the decision is taken on the value rounded to fp32,
 * the precision of MLX's `softmax(..., precise=True)` in the lilting.ch router
 * article (section "hooking the router").
 *
 * Sources (page title, section):
 *  - lilting.ch "observing the Qwen MoE router": the three router steps
 *    gate -> softmax -> top-k; expert weights stacked as
 *    (num_experts, output_dims, input_dims) and gathered by expert index.
 *  - Qiita "custom Metal gather_qmm": section 4, routing indices are an input and
 *    only the routed experts are read; section 6, sym8 = symmetric linear int8
 *    with one scale per K-block of 32, and the gather equals the dequantised
 *    reference; section 7, gate/up share the token x while down is applied per
 *    slot to that expert's own gated activation, and int8 is sign-extended.
 *  - gist.science "Which expert misses are worth waiting for?": method section,
 *    the fetch-all / 0.15 / first-choice rules and the substituted gate mass m.
 *  - xyznot.com "The Other Half of the Memory Wall: Serving 35B MoEs from SSD
 *    with Trained Routing Prediction": method section, the prerouter head
 *    (input of d_model + 2E values, fc2(erf-gelu(fc1 f)) + a linear path) whose
 *    prediction is used as the routing, and the unmerged recovery LoRA
 *    y = W(x) + (alpha/r) B A x on the shared expert's projections.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define BLK 32

/* ---------------------------------------------------------------- helpers */

/* Signed value of code k in a row of codes: int8 directly, int4 from a packed
 * byte (element 2j in the low nibble of byte j, 2j+1 in the high nibble,
 * two's complement). */
static int code_at(const uint8_t* row, int qbits, int64_t k) {
    if (qbits == 8) return (int)(int8_t)row[k];
    uint8_t byte = row[k >> 1];
    int nib = (k & 1) ? (byte >> 4) : (byte & 0xF);
    return nib >= 8 ? nib - 16 : nib;
}

/* Dequantised weight w[n][k] = q[n][k] * s[n][k/32] of one [N][K] matrix. */
static double dq(const uint8_t* codes, const double* scales, int qbits, int64_t K,
                 int64_t n, int64_t k) {
    int64_t row_bytes = qbits == 8 ? K : K / 2;
    return (double)code_at(codes + n * row_bytes, qbits, k) * scales[n * (K / BLK) + k / BLK];
}

/* fp32 decision key with the lowest-index tie-break: a before b? */
static int ranks_before(float pa, int a, float pb, int b) {
    if (pa != pb) return pa > pb;
    return a < b;
}

/* ------------------------------------------------------------------ router */

/*
 * Router of one MoE block (lilting.ch, "hooking the router"):
 *   logits[t][e] = sum_d x[t][d] * Wr[e][d] + bias[e]
 *   probs[t]     = softmax(logits[t])              (max-subtracted)
 *   idx[t]       = the k experts of largest probs, largest first,
 *                  equal fp32 values ordered by lower expert index
 *   w[t][r]      = probs[t][idx[t][r]] / sum_r' probs[t][idx[t][r']]   (norm_topk=1)
 *                  probs[t][idx[t][r]]                                 (norm_topk=0)
 * bias may be NULL. Returns 0, or -1 on bad arguments.
 */
/* Softmax of one token's logits and its top k (the last two router steps):
 * probs = exp(l - max) / sum, the fp32-rounded probs ranked by a full insertion
 * sort with the lowest-index tie-break, and the k weights (renormalised if
 * norm_topk). `order` is scratch of E ints. */
static void softmax_topk(int E, int k, int norm_topk, const double* lt, double* pt, float* p32,
                         int* order, int32_t* idx_t, double* w_t) {
    double mx = lt[0];
    for (int e = 1; e < E; e++) if (lt[e] > mx) mx = lt[e];
    double sum = 0.0;
    for (int e = 0; e < E; e++) { pt[e] = exp(lt[e] - mx); sum += pt[e]; }
    for (int e = 0; e < E; e++) { pt[e] /= sum; p32[e] = (float)pt[e]; }
    /* full insertion sort of all experts by the fp32 key, then take k */
    for (int e = 0; e < E; e++) {
        int j = e;
        while (j > 0 && ranks_before(p32[e], e, p32[order[j - 1]], order[j - 1])) {
            order[j] = order[j - 1];
            j--;
        }
        order[j] = e;
    }
    double norm = 0.0;
    for (int r = 0; r < k; r++) norm += pt[order[r]];
    for (int r = 0; r < k; r++) {
        idx_t[r] = order[r];
        w_t[r] = norm_topk ? pt[order[r]] / norm : pt[order[r]];
    }
}

int oracle_router(int T, int E, int D, int k, int norm_topk, const double* x,
                  const double* Wr, const double* bias, double* logits, double* probs,
                  float* probs32, int32_t* idx, double* w) {
    if (T < 0 || E < 1 || D < 1 || k < 1 || k > E) return -1;
    int* order = (int*)malloc(sizeof(int) * E);
    if (!order) return -1;
    for (int t = 0; t < T; t++) {
        const double* xt = x + (int64_t)t * D;
        double* lt = logits + (int64_t)t * E;
        for (int e = 0; e < E; e++) {
            double acc = 0.0;
            for (int d = 0; d < D; d++) acc += xt[d] * Wr[(int64_t)e * D + d];
            lt[e] = acc + (bias ? bias[e] : 0.0);
        }
        softmax_topk(E, k, norm_topk, lt, probs + (int64_t)t * E, probs32 + (int64_t)t * E, order,
                     idx + (int64_t)t * k, w + (int64_t)t * k);
    }
    free(order);
    return 0;
}

/* ------------------------------------------------------------ substitution */

/*
 * Residency substitution (gist.science, method section). Slots are visited in
 * rank order r = 0..k-1. For slot r of token t with expert e = idx[t][r]:
 *   resident[e]                          -> kept, flag 0
 *   r == 0  or  w[t][r] >= threshold     -> kept and fetched, flag 1
 *   otherwise                            -> replaced by the resident expert of
 *        highest probability that is neither among the token's original k nor
 *        already chosen as a replacement (ties: lower index), flag 2; the
 *        replacement keeps the slot's weight; m[t] += w[t][r]
 *   no such resident expert              -> kept, flag 3
 * threshold = 0 is "fetch every miss"; threshold = +inf keeps only first-choice
 * misses. The threshold comparison is made on fp32 values.
 */
int oracle_substitute(int T, int E, int k, const float* probs32, const int32_t* idx,
                      const double* w, const uint8_t* resident, double threshold,
                      int32_t* idx_out, double* w_out, uint8_t* flag, double* mass) {
    if (T < 0 || E < 1 || k < 1 || k > E) return -1;
    uint8_t* taken = (uint8_t*)malloc(E);
    if (!taken) return -1;
    float thr32 = (float)threshold;
    for (int t = 0; t < T; t++) {
        const int32_t* it = idx + (int64_t)t * k;
        const float* pt = probs32 + (int64_t)t * E;
        memset(taken, 0, E);
        for (int r = 0; r < k; r++) taken[it[r]] = 1;
        double m = 0.0;
        for (int r = 0; r < k; r++) {
            int64_t o = (int64_t)t * k + r;
            int e = it[r];
            idx_out[o] = e;
            w_out[o] = w[o];
            if (resident[e]) { flag[o] = 0; continue; }
            if (r == 0 || (float)w[o] >= thr32) { flag[o] = 1; continue; }
            int best = -1;
            for (int c = 0; c < E; c++) {
                if (!resident[c] || taken[c]) continue;
                if (best < 0 || ranks_before(pt[c], c, pt[best], best)) best = c;
            }
            if (best < 0) { flag[o] = 3; continue; }
            taken[best] = 1;
            idx_out[o] = best;
            flag[o] = 2;
            m += w[o];
        }
        mass[t] = m;
    }
    free(taken);
    return 0;
}

/* ------------------------------------------------------------- expert MLP */

/*
 * One routed expert applied to one token (Qiita gather_qmm, sections 4 and 7):
 *   g[n] = sum_k Gate[e][n][k] * x[k]         (Gate dequantised, [F][D])
 *   u[n] = sum_k Up[e][n][k]   * x[k]         (Up dequantised,   [F][D])
 *   h[n] = g[n] * sigmoid(g[n]) * u[n]        (SwiGLU, silu(g) * u)
 *   o[d] = sum_n Down[e][d][n] * h[n]         (Down dequantised, [D][F])
 * Gate and up read the shared token x; down reads this expert's own h.
 */
static void expert_mlp(int D, int F, int qbits, const uint8_t* gq, const double* gs,
                       const uint8_t* uq, const double* us, const uint8_t* dq_codes,
                       const double* ds, const double* x, double* h, double* o) {
    for (int n = 0; n < F; n++) {
        double g = 0.0, u = 0.0;
        for (int kk = 0; kk < D; kk++) {
            g += dq(gq, gs, qbits, D, n, kk) * x[kk];
            u += dq(uq, us, qbits, D, n, kk) * x[kk];
        }
        h[n] = g / (1.0 + exp(-g)) * u;
    }
    for (int d = 0; d < D; d++) {
        double acc = 0.0;
        for (int n = 0; n < F; n++) acc += dq(dq_codes, ds, qbits, F, d, n) * h[n];
        o[d] = acc;
    }
}

/*
 * The MoE layer output for routed tokens:
 *   y[t][d] = sum_{r=0..k-1} w[t][r] * o_{t,r}[d],   o_{t,r} = expert_mlp(idx[t][r], x[t])
 * summed in slot order r = 0, 1, ..., k-1. Expert e's matrices start at
 * e * (rows * row_bytes) in the code arrays and e * rows * (K/32) in the scale
 * arrays. Scales arrive as double (exact conversions of fp16/fp32 values).
 * nthreads > 1 parallelises over (t, r) pairs; the combine order is fixed.
 * Out-of-range expert ids return -2 before any work.
 */
int oracle_moe(int T, int E, int k, int D, int F, int qbits, const uint8_t* gate_q,
               const double* gate_s, const uint8_t* up_q, const double* up_s,
               const uint8_t* down_q, const double* down_s, const double* x,
               const int32_t* idx, const double* w, double* y, int nthreads) {
    if (T < 0 || E < 1 || k < 1 || D % BLK || F % BLK || (qbits != 8 && qbits != 4)) return -1;
    for (int64_t i = 0; i < (int64_t)T * k; i++)
        if (idx[i] < 0 || idx[i] >= E) return -2;
    int64_t gu_row = qbits == 8 ? D : D / 2, dn_row = qbits == 8 ? F : F / 2;
    int64_t gu_codes = (int64_t)F * gu_row, dn_codes = (int64_t)D * dn_row;
    int64_t gu_sc = (int64_t)F * (D / BLK), dn_sc = (int64_t)D * (F / BLK);
    int64_t pairs = (int64_t)T * k;
    double* o = (double*)malloc(sizeof(double) * (pairs > 0 ? pairs : 1) * D);
    if (!o) return -1;
    int fail = 0;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t p = 0; p < pairs; p++) {
        double* h = (double*)malloc(sizeof(double) * F);
        if (!h) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            fail = 1;
            continue;
        }
        int64_t t = p / k;
        int64_t e = idx[p];
        expert_mlp(D, F, qbits, gate_q + e * gu_codes, gate_s + e * gu_sc,
                   up_q + e * gu_codes, up_s + e * gu_sc, down_q + e * dn_codes,
                   down_s + e * dn_sc, x + t * D, h, o + p * D);
        free(h);
    }
    if (!fail) {
        for (int64_t t = 0; t < T; t++)
            for (int d = 0; d < D; d++) {
                double acc = 0.0;
                for (int r = 0; r < k; r++) acc += w[t * k + r] * o[(t * k + r) * D + d];
                y[t * D + d] = acc;
            }
    }
    free(o);
    return fail ? -1 : 0;
}

/* ------------------------------------------- shared expert, unmerged LoRA */

/*
 * One projection served with an unmerged low-rank adapter (xyznot.com "The
 * Other Half of the Memory Wall", method section "unmerged adapter execution",
 * and its FAQ on why the adapter is not merged into the 4-bit weights): the
 * quantised base is kept as it is and the delta runs beside it,
 *   out[n] = sum_k dq(W)[n][k] * v[k]  +  scale * sum_j B[n][j] * (sum_k A[j][k] * v[k])
 * with W [N][K] codes/scales, A [r][K], B [N][r] and scale = alpha / r.
 * r = 0 is the base projection alone.
 */
static void lora_projection(int64_t N, int64_t K, int r, int qbits, const uint8_t* codes,
                            const double* scales, const double* A, const double* B, double scale,
                            const double* v, double* av, double* out) {
    for (int j = 0; j < r; j++) {
        double acc = 0.0;
        for (int64_t kk = 0; kk < K; kk++) acc += A[j * K + kk] * v[kk];
        av[j] = acc;
    }
    for (int64_t n = 0; n < N; n++) {
        double base = 0.0;
        for (int64_t kk = 0; kk < K; kk++) base += dq(codes, scales, qbits, K, n, kk) * v[kk];
        double delta = 0.0;
        for (int j = 0; j < r; j++) delta += B[n * r + j] * av[j];
        out[n] = base + scale * delta;
    }
}

/*
 * The shared expert of a MoE block with its recovery LoRA (same page: the
 * adapters sit on the attention, linear-attention and shared-expert
 * projections, never on the streamed experts), applied to each of T tokens:
 *   g = Gate(x), u = Up(x)       (gate/up codes [F][D], A [r][D], B [F][r])
 *   h = g * sigmoid(g) * u       (SwiGLU)
 *   y = Down(h)                  (down codes [D][F], A [r][F], B [D][r])
 * every projection as lora_projection above. Returns 0, or -1 on bad arguments.
 */
int oracle_shared_lora(int T, int D, int F, int r, int qbits, const uint8_t* gate_q,
                       const double* gate_s, const uint8_t* up_q, const double* up_s,
                       const uint8_t* down_q, const double* down_s, const double* gate_A,
                       const double* gate_B, const double* up_A, const double* up_B,
                       const double* down_A, const double* down_B, double scale, const double* x,
                       double* y) {
    if (T < 0 || D < BLK || F < BLK || D % BLK || F % BLK || r < 0 || (qbits != 8 && qbits != 4))
        return -1;
    double* g = (double*)malloc(sizeof(double) * F);
    double* u = (double*)malloc(sizeof(double) * F);
    double* h = (double*)malloc(sizeof(double) * F);
    double* av = (double*)malloc(sizeof(double) * (r > 0 ? r : 1));
    if (!g || !u || !h || !av) {
        free(g); free(u); free(h); free(av);
        return -1;
    }
    for (int64_t t = 0; t < T; t++) {
        const double* xt = x + t * D;
        lora_projection(F, D, r, qbits, gate_q, gate_s, gate_A, gate_B, scale, xt, av, g);
        lora_projection(F, D, r, qbits, up_q, up_s, up_A, up_B, scale, xt, av, u);
        for (int n = 0; n < F; n++) h[n] = g[n] / (1.0 + exp(-g[n])) * u[n];
        lora_projection(D, F, r, qbits, down_q, down_s, down_A, down_B, scale, h, av, y + t * D);
    }
    free(g); free(u); free(h); free(av);
    return 0;
}

/* ------------------------------------------------------- prerouter head */

/*
 * Prerouter head (xyznot.com "The Other Half of the Memory Wall", method
 * section "prerouter head architecture"; glossary "prerouter" and
 * "prediction-as-routing"). The head held by layer N runs at token t and
 * predicts the routing of layer N+1 at token t+1. Its input joins the hidden
 * state with two k-hot routing vectors, of the current and of the previous
 * token:
 *   f = [ x (D) ; hot(cur) (E) ; hot(prev) (E) ]      (D + 2E values)
 *   hot(S)[e] = 1 if e is among the ids S (negative ids: absent), else 0
 * and the head is
 *   z      = fc1 f + b1                               (fc1 [H][D+2E], b1 [H])
 *   a      = gelu(z) = z/2 * (1 + erf(z / sqrt(2)))   (the erf form)
 *   logits = fc2 a + L f + bias                       (fc2 [E][H], L [E][D+2E], bias [E])
 * L being the linear residual path warm-started from the next layer's router.
 * The prediction is consumed as the routing itself, so it goes through the
 * router's own last steps (softmax_topk above): probs, the k most probable
 * experts and their weights. b1 and bias may be NULL. Returns 0, -1 on bad
 * arguments, -2 for an id >= E.
 */
int oracle_prerouter(int T, int D, int E, int H, int k, int norm_topk, const double* x,
                     const int32_t* cur, const int32_t* prev, const double* fc1, const double* b1,
                     const double* fc2, const double* L, const double* bias, double* logits,
                     double* probs, float* probs32, int32_t* idx, double* w) {
    if (T < 0 || D < 1 || E < 1 || H < 1 || k < 1 || k > E) return -1;
    for (int64_t i = 0; i < (int64_t)T * k; i++)
        if (cur[i] >= E || prev[i] >= E) return -2;
    const int64_t nf = (int64_t)D + 2 * (int64_t)E;
    double* f = (double*)malloc(sizeof(double) * nf);
    double* a = (double*)malloc(sizeof(double) * H);
    int* order = (int*)malloc(sizeof(int) * E);
    if (!f || !a || !order) {
        free(f); free(a); free(order);
        return -1;
    }
    for (int64_t t = 0; t < T; t++) {
        for (int64_t i = 0; i < D; i++) f[i] = x[t * D + i];
        for (int64_t i = D; i < nf; i++) f[i] = 0.0;
        for (int r = 0; r < k; r++) {
            if (cur[t * k + r] >= 0) f[D + cur[t * k + r]] = 1.0;
            if (prev[t * k + r] >= 0) f[D + E + prev[t * k + r]] = 1.0;
        }
        for (int j = 0; j < H; j++) {
            double z = b1 ? b1[j] : 0.0;
            for (int64_t i = 0; i < nf; i++) z += fc1[j * nf + i] * f[i];
            a[j] = 0.5 * z * (1.0 + erf(z / sqrt(2.0)));
        }
        double* lt = logits + t * E;
        for (int e = 0; e < E; e++) {
            double head = 0.0;
            for (int j = 0; j < H; j++) head += fc2[(int64_t)e * H + j] * a[j];
            double lin = 0.0;
            for (int64_t i = 0; i < nf; i++) lin += L[e * nf + i] * f[i];
            lt[e] = head + lin + (bias ? bias[e] : 0.0);
        }
        softmax_topk(E, k, norm_topk, lt, probs + t * E, probs32 + t * E, order, idx + t * k,
                     w + t * k);
    }
    free(f); free(a); free(order);
    return 0;
}

/* ---------------------------------------------------- prefill permutation */

/*
 * Grouping of the T*k (token, slot) assignments by expert:
 *   cnt[e]  = number of assignments with idx == e
 *   off[e]  = sum_{e' < e} cnt[e'],  off[E] = T*k
 *   the assignments sorted by expert, keeping (t, r) order inside an expert:
 *   position p holds perm_tok[p] = t, perm_slot[p] = r, and inv[t][r] = p.
 * Written as a counting sort over assignments visited in (t, r) order.
 */
int oracle_permute(int T, int k, int E, const int32_t* idx, int32_t* cnt, int32_t* off,
                   int32_t* perm_tok, int32_t* perm_slot, int32_t* inv) {
    if (T < 0 || k < 1 || E < 1) return -1;
    for (int e = 0; e < E; e++) cnt[e] = 0;
    for (int64_t i = 0; i < (int64_t)T * k; i++) {
        if (idx[i] < 0 || idx[i] >= E) return -2;
        cnt[idx[i]]++;
    }
    off[0] = 0;
    for (int e = 0; e < E; e++) off[e + 1] = off[e] + cnt[e];
    int32_t* fill = (int32_t*)malloc(sizeof(int32_t) * E);
    if (!fill) return -1;
    for (int e = 0; e < E; e++) fill[e] = off[e];
    for (int t = 0; t < T; t++)
        for (int r = 0; r < k; r++) {
            int e = idx[(int64_t)t * k + r];
            int32_t p = fill[e]++;
            perm_tok[p] = t;
            perm_slot[p] = r;
            inv[(int64_t)t * k + r] = p;
        }
    free(fill);
    return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
