/*
 * oracle.c -- plain, slow CPU oracle for budgeted-KV decode attention with
 * heavy-hitter (H2O) eviction and the HashEvict LSH variant.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header, table or
 * constant with the CUDA library; the two meet only through the seeded
 * inputs that the tests hand to both.
 *
 * Arithmetic: IEEE fp64 throughout ("double"), compiled with
 * -ffp-contract=off so every product and sum is rounded exactly as written.
 * The one exception is the LSH sign projection, which the HashEvict variant
 * requires to be bit-exact across implementations: it is an fp32 fused
 * multiply-add chain (C99 fmaf) in index order, starting from 0.0f.
 *
 * Sources, by page title and section:
 *  [H2O]   "H2O: Heavy-Hitter Oracle for Efficient Generative Inference of
 *          Large Language Models" (review page), sections 提案手法 (method:
 *          heavy hitters are the tokens with concentrated accumulated
 *          attention; eviction is a greedy rule driven by per-decode-step
 *          local attention statistics) and 研究の動機と目的 (motivation:
 *          balance recency against relevance).
 *  [FG]    "Model Tells You What to Discard: Adaptive KV Cache Compression
 *          for LLMs" (review page), Figure 2 caption: the fixed
 *          "Frequency + Local" cache is the H2O policy.
 *  [SH]    "Scissorhands: Exploiting the Persistence of Importance
 *          Hypothesis for LLM KV Cache Compression at Test Time", abstract:
 *          the KV cache is held at a fixed budget.
 *  [HE]    "HashEvict: A Pre-Attention KV Cache Eviction Strategy using
 *          Locality-Sensitive Hashing", abstract: Hamming distance between
 *          binarised Gaussian projections of the current query and the
 *          cached keys, projection length far below the head dimension,
 *          decided before attention; at every decode step the new token's
 *          key and value replace the cached token expected to receive the
 *          lowest attention score.
 *
 * Where the pages leave a step open the oracle takes these readings (each is
 * listed, with its reason, in the design notes of the repository):
 *  - the new token attends to itself and to the n live slots (n+1 keys);
 *  - this step's probabilities are added to the scores before the victim is
 *    chosen; the new token starts with its own probability as its score;
 *  - the recent window after decoding position p is p-r+1..p, so the
 *    eviction candidates are the slots holding positions <= p-r;
 *  - ties go to the lowest slot index (eviction) and to the lower position
 *    (prompt top-k);
 *  - after the prompt, kept positions occupy slots 0..n-1 in ascending
 *    position order; empty slots hold position -1 and score 0;
 *  - scores are a plain running sum (no decay);
 *  - LSH bit j is 1 iff the fp32 projection onto column j of W is > 0;
 *  - the LSH cache is built from the prompt by replaying the decode
 *    replacement rule token by token; the LSH step evicts and inserts
 *    first and then attends over the budget (the victim is not attended);
 *  - if no slot is an eviction candidate (possible only for a state that
 *    breaks the recent-window invariant), every live slot is a candidate;
 *  - grouped-query attention (an optional mode): a cache unit shared by G
 *    query heads accumulates the sum of their probabilities per slot;
 *  - int8 cache slots (an optional mode): each stored K or V row keeps int8
 *    codes and one fp32 scale, amax/127, with codes rint(x * (127/amax))
 *    in fp32, half to even; a step attends to its own new token at full
 *    precision and stores it quantised (the quantiser is below; the mode's
 *    bookkeeping is in the Python wrapper); 4-bit slots are the same with
 *    codes in [-7, 7], scale amax/7 and codes rint((7/amax) * x);
 *  - the persistence-of-importance rule (an optional cache kind, [SH]): a
 *    token is pivotal at a step when its attention probability exceeds
 *    the uniform share 1/m over the m tokens attended that step; each
 *    token keeps its pivotal flags of the last 32 steps (prompt rows count
 *    as steps); its importance is the number of flags set; the victim is
 *    the candidate with the lowest importance, then the oldest position;
 *    the prompt keeps the recent window and the H most important earlier
 *    tokens, ties to the newer position;
 *  - the per-head policy (an optional profile, [FG]): a policy's recovery
 *    is the average over the prompt's rows of the attention mass it keeps
 *    at that row; the first of local, frequency + local and full cache
 *    whose recovery reaches the threshold is the head's policy.
 *
 * parity unpinned: the readings above that have no printed example on the
 * pages (self-attention of the new token, accumulate-before-evict order,
 * slot order after the prompt, the LSH prompt replay and attend-after-evict,
 * the grouped-query sum, the whole persistence-of-importance rule) are
 * pinned only through the invariants and closed forms the tests check, not
 * against a value the pages print.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* threads (the oracle parallelises only over independent units)       */
/* ------------------------------------------------------------------ */
void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static double dot(const double* a, const double* b, int d)
{
    double s = 0.0;
    for (int e = 0; e < d; ++e) s += a[e] * b[e];
    return s;
}

/* ------------------------------------------------------------------ */
/* Prompt statistics [H2O 提案手法]: the accumulated attention a prompt  */
/* token receives from every later prompt row under causal softmax.    */
/*   z_ij = scale * q_i . k_j            (j <= i)                        */
/*   m_i  = max_j z_ij,  l_i = sum_j exp(z_ij - m_i)                    */
/*   c_j  = sum_{i >= j} exp(z_ij - m_i) / l_i                          */
/* One row at a time, exactly as defined; Q, K are [U][T][d].           */
/* ------------------------------------------------------------------ */
void oracle_prefill_scores(int U, int T, int d, double scale,
                           const double* Q, const double* K,
                           double* m, double* l, double* c)
{
    #pragma omp parallel for schedule(dynamic, 1)
    for (int u = 0; u < U; ++u) {
        const double* Qu = Q + (size_t)u * T * d;
        const double* Ku = K + (size_t)u * T * d;
        double* mu = m + (size_t)u * T;
        double* lu = l + (size_t)u * T;
        double* cu = c + (size_t)u * T;
        double* z = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
        for (int j = 0; j < T; ++j) cu[j] = 0.0;
        for (int i = 0; i < T; ++i) {
            double mi = -INFINITY;
            for (int j = 0; j <= i; ++j) {
                z[j] = scale * dot(Qu + (size_t)i * d, Ku + (size_t)j * d, d);
                if (z[j] > mi) mi = z[j];
            }
            double li = 0.0;
            for (int j = 0; j <= i; ++j) li += exp(z[j] - mi);
            for (int j = 0; j <= i; ++j) cu[j] += exp(z[j] - mi) / li;
            mu[i] = mi;
            lu[i] = li;
        }
        free(z);
    }
}

/* ------------------------------------------------------------------ */
/* Initial cache selection [H2O 提案手法, FG Figure 2]: keep the recent  */
/* window T-r..T-1 plus the H prompt tokens with the largest column     */
/* sums among positions 0..T-r-1 (ties to the lower position).  When    */
/* T <= B every prompt token is kept.  kept[] receives the kept         */
/* positions in ascending order; the return value is their count.      */
/* margin (nullable) receives the relative gap between the H-th and     */
/* the (H+1)-th candidate score, +inf when no choice was made.          */
/* ------------------------------------------------------------------ */
typedef struct { double c; int j; } cand_t;

static int cand_cmp(const void* a, const void* b)
{
    const cand_t* x = (const cand_t*)a;
    const cand_t* y = (const cand_t*)b;
    if (x->c > y->c) return -1;
    if (x->c < y->c) return 1;
    return (x->j < y->j) ? -1 : (x->j > y->j);
}

int oracle_select(int T, int B, int H, int r, const double* c,
                  int* kept, double* margin)
{
    if (margin) *margin = INFINITY;
    if (T <= B) {
        for (int j = 0; j < T; ++j) kept[j] = j;
        return T;
    }
    int ncand = T - r;
    char* keep = (char*)calloc((size_t)T, 1);
    for (int j = ncand; j < T; ++j) keep[j] = 1;
    cand_t* cs = (cand_t*)malloc(sizeof(cand_t) * (size_t)(ncand > 0 ? ncand : 1));
    for (int j = 0; j < ncand; ++j) { cs[j].c = c[j]; cs[j].j = j; }
    qsort(cs, (size_t)ncand, sizeof(cand_t), cand_cmp);
    int h = H < ncand ? H : ncand;
    for (int t = 0; t < h; ++t) keep[cs[t].j] = 1;
    if (margin && h >= 1 && h < ncand) {
        double a = cs[h - 1].c, b2 = cs[h].c;
        double den = fabs(a) > 1e-30 ? fabs(a) : 1e-30;
        *margin = (a - b2) / den;
    }
    int n = 0;
    for (int j = 0; j < T; ++j) if (keep[j]) kept[n++] = j;
    free(cs);
    free(keep);
    return n;
}

/* Fill one unit's cache from the kept prompt positions (ascending):     */
/* slot s holds position kept[s], its K/V row and score c[kept[s]].      */
static void build_unit(int T, int d, int B, int n, const int* kept,
                       const double* c, const double* K, const double* V,
                       double* cK, double* cV, double* score, int* pos)
{
    (void)T;
    for (int s = 0; s < B; ++s) {
        if (s < n) {
            int j = kept[s];
            memcpy(cK + (size_t)s * d, K + (size_t)j * d, sizeof(double) * d);
            memcpy(cV + (size_t)s * d, V + (size_t)j * d, sizeof(double) * d);
            if (score) score[s] = c[j];
            pos[s] = j;
        } else {
            memset(cK + (size_t)s * d, 0, sizeof(double) * d);
            memset(cV + (size_t)s * d, 0, sizeof(double) * d);
            if (score) score[s] = 0.0;
            pos[s] = -1;
        }
    }
}

/* Build U caches from kept position lists given by the caller ([U][B],  */
/* counts nkept[U]); used to align the oracle with a near-tie choice.    */
void oracle_build_cache(int U, int T, int d, int B, const int* kept, const int* nkept,
                        const double* c, const double* K, const double* V,
                        double* cK, double* cV, double* score, int* pos, int* occ)
{
    for (int u = 0; u < U; ++u) {
        build_unit(T, d, B, nkept[u], kept + (size_t)u * B, c + (size_t)u * T,
                   K + (size_t)u * T * d, V + (size_t)u * T * d,
                   cK + (size_t)u * B * d, cV + (size_t)u * B * d,
                   score + (size_t)u * B, pos + (size_t)u * B);
        occ[u] = nkept[u];
    }
}

/* Whole H2O prompt phase for U units: statistics, selection, cache.     */
/* c (nullable, [U][T]) receives the column sums; kept ([U][B]) and      */
/* margin ([U]) are nullable.                                            */
void oracle_h2o_prefill(int U, int T, int d, int B, int H, int r, double scale,
                        const double* Q, const double* K, const double* V,
                        double* cK, double* cV, double* score, int* pos, int* occ,
                        double* c_out, int* kept_out, double* margin)
{
    double* m = (double*)malloc(sizeof(double) * (size_t)U * T);
    double* l = (double*)malloc(sizeof(double) * (size_t)U * T);
    double* c = c_out ? c_out : (double*)malloc(sizeof(double) * (size_t)U * T);
    oracle_prefill_scores(U, T, d, scale, Q, K, m, l, c);
    #pragma omp parallel for schedule(dynamic, 1)
    for (int u = 0; u < U; ++u) {
        int* kept = (int*)malloc(sizeof(int) * (size_t)(T > 0 ? T : 1));
        double mg;
        int n = oracle_select(T, B, H, r, c + (size_t)u * T, kept, &mg);
        build_unit(T, d, B, n, kept, c + (size_t)u * T,
                   K + (size_t)u * T * d, V + (size_t)u * T * d,
                   cK + (size_t)u * B * d, cV + (size_t)u * B * d,
                   score + (size_t)u * B, pos + (size_t)u * B);
        occ[u] = n;
        if (margin) margin[u] = mg;
        if (kept_out)
            for (int s = 0; s < B; ++s) kept_out[(size_t)u * B + s] = s < n ? kept[s] : -1;
        free(kept);
    }
    if (!c_out) free(c);
    free(l);
    free(m);
}

/* ------------------------------------------------------------------ */
/* One H2O decode step at position p for U units [H2O 提案手法]:        */
/*  1. attend: z_s = scale q.k_s over the n live slots and the new key; */
/*     P = softmax(z); out = sum_s P_s v_s (+ P_new v_new);             */
/*  2. accumulate: score_s += P_s;                                      */
/*  3. evict: if n < B the new token takes slot n; otherwise the victim */
/*     is the candidate (pos <= p - r) with the smallest score, lowest  */
/*     slot on ties;                                                    */
/*  4. insert: the victim slot gets (k, v, P_new, p).                   */
/* victim[u] = -1 on append.  margin[u] = relative gap between the two  */
/* smallest candidate scores (+inf with fewer than two candidates or on */
/* append).  evicted[u] = the score that left the cache (0 on append).  */
/* forced (nullable): forced[u] >= 0 overrides the victim choice.       */
/* ------------------------------------------------------------------ */
void oracle_h2o_decode_step(int U, int d, int B, int r, double scale, int p,
                            double* cK, double* cV, double* score, int* pos, int* occ,
                            const double* q, const double* k, const double* v,
                            double* out, int* victim, double* margin, double* evicted,
                            const int* forced)
{
    #pragma omp parallel for schedule(dynamic, 4)
    for (int u = 0; u < U; ++u) {
        double* Ku = cK + (size_t)u * B * d;
        double* Vu = cV + (size_t)u * B * d;
        double* su = score + (size_t)u * B;
        int* pu = pos + (size_t)u * B;
        const double* qu = q + (size_t)u * d;
        const double* ku = k + (size_t)u * d;
        const double* vu = v + (size_t)u * d;
        double* ou = out + (size_t)u * d;
        int n = occ[u];
        double* z = (double*)malloc(sizeof(double) * (size_t)(n + 1));

        /* 1. attend over the n live slots plus the new token (index n) */
        double mx = -INFINITY;
        for (int s = 0; s < n; ++s) {
            z[s] = scale * dot(qu, Ku + (size_t)s * d, d);
            if (z[s] > mx) mx = z[s];
        }
        z[n] = scale * dot(qu, ku, d);
        if (z[n] > mx) mx = z[n];
        double lsum = 0.0;
        for (int s = 0; s <= n; ++s) lsum += exp(z[s] - mx);
        for (int e = 0; e < d; ++e) ou[e] = 0.0;
        for (int s = 0; s <= n; ++s) {
            double P = exp(z[s] - mx) / lsum;
            const double* vs = (s < n) ? Vu + (size_t)s * d : vu;
            for (int e = 0; e < d; ++e) ou[e] += P * vs[e];
        }
        double P_new = exp(z[n] - mx) / lsum;

        /* 2. accumulate this step's attention into the live slots */
        for (int s = 0; s < n; ++s) su[s] += exp(z[s] - mx) / lsum;

        /* 3. evict */
        int slot;
        double mg = INFINITY, ev = 0.0;
        if (n < B) {
            slot = n;
            occ[u] = n + 1;
            if (victim) victim[u] = -1;
        } else {
            int ncand = 0;
            for (int s = 0; s < n; ++s) if (pu[s] <= p - r) ++ncand;
            int best = -1, second = -1;
            for (int s = 0; s < n; ++s) {
                if (ncand > 0 && !(pu[s] <= p - r)) continue;
                if (best < 0 || su[s] < su[best]) { second = best; best = s; }
                else if (second < 0 || su[s] < su[second]) second = s;
            }
            if (second >= 0) {
                double den = fabs(su[best]) > 1e-30 ? fabs(su[best]) : 1e-30;
                mg = (su[second] - su[best]) / den;
            }
            slot = (forced && forced[u] >= 0) ? forced[u] : best;
            ev = su[slot];
            if (victim) victim[u] = slot;
        }
        if (margin) margin[u] = mg;
        if (evicted) evicted[u] = ev;

        /* 4. insert */
        memcpy(Ku + (size_t)slot * d, ku, sizeof(double) * d);
        memcpy(Vu + (size_t)slot * d, vu, sizeof(double) * d);
        su[slot] = P_new;
        pu[slot] = p;
        free(z);
    }
}

/* ------------------------------------------------------------------ */
/* H2O decode step for U cache units, each shared by G query heads      */
/* (grouped-query attention; the cache is that of a key/value head).    */
/* Every head attends with its own softmax over the unit's n live slots */
/* and the new token; a slot's accumulated score grows by the sum of    */
/* the G heads' probabilities this step (the reading of "accumulated   */
/* attention" for a shared slot), and the new token's score is the sum  */
/* of its G probabilities.  Eviction and insertion follow the one-head  */
/* step.  q, out: [U][G][d]; k, v: [U][d].  Outputs as in the one-head  */
/* step.                                                                */
/* ------------------------------------------------------------------ */
void oracle_h2o_decode_step_gqa(int U, int G, int d, int B, int r, double scale, int p,
                                double* cK, double* cV, double* score, int* pos, int* occ,
                                const double* q, const double* k, const double* v,
                                double* out, int* victim, double* margin, double* evicted,
                                const int* forced)
{
    #pragma omp parallel for schedule(dynamic, 4)
    for (int u = 0; u < U; ++u) {
        double* Ku = cK + (size_t)u * B * d;
        double* Vu = cV + (size_t)u * B * d;
        double* su = score + (size_t)u * B;
        int* pu = pos + (size_t)u * B;
        const double* ku = k + (size_t)u * d;
        const double* vu = v + (size_t)u * d;
        const int n = occ[u];
        double* z = (double*)malloc(sizeof(double) * (size_t)(n + 1));
        double* add = (double*)calloc((size_t)(n + 1), sizeof(double));
        for (int g = 0; g < G; ++g) {
            const double* qg = q + ((size_t)u * G + g) * d;
            double* og = out + ((size_t)u * G + g) * d;
            double mx = -INFINITY;
            for (int s = 0; s < n; ++s) {
                z[s] = scale * dot(qg, Ku + (size_t)s * d, d);
                if (z[s] > mx) mx = z[s];
            }
            z[n] = scale * dot(qg, ku, d);
            if (z[n] > mx) mx = z[n];
            double lsum = 0.0;
            for (int s = 0; s <= n; ++s) lsum += exp(z[s] - mx);
            for (int e = 0; e < d; ++e) og[e] = 0.0;
            for (int s = 0; s <= n; ++s) {
                const double P = exp(z[s] - mx) / lsum;
                const double* vs = (s < n) ? Vu + (size_t)s * d : vu;
                for (int e = 0; e < d; ++e) og[e] += P * vs[e];
                add[s] += P;                          /* heads in order g = 0..G-1 */
            }
        }
        for (int s = 0; s < n; ++s) su[s] += add[s];
        const double P_new = add[n];
        int slot;
        double mg = INFINITY, ev = 0.0;
        if (n < B) {
            slot = n;
            occ[u] = n + 1;
            if (victim) victim[u] = -1;
        } else {
            int ncand = 0;
            for (int s = 0; s < n; ++s) if (pu[s] <= p - r) ++ncand;
            int best = -1, second = -1;
            for (int s = 0; s < n; ++s) {
                if (ncand > 0 && !(pu[s] <= p - r)) continue;
                if (best < 0 || su[s] < su[best]) { second = best; best = s; }
                else if (second < 0 || su[s] < su[second]) second = s;
            }
            if (second >= 0) {
                const double den = fabs(su[best]) > 1e-30 ? fabs(su[best]) : 1e-30;
                mg = (su[second] - su[best]) / den;
            }
            slot = (forced && forced[u] >= 0) ? forced[u] : best;
            ev = su[slot];
            if (victim) victim[u] = slot;
        }
        if (margin) margin[u] = mg;
        if (evicted) evicted[u] = ev;
        memcpy(Ku + (size_t)slot * d, ku, sizeof(double) * d);
        memcpy(Vu + (size_t)slot * d, vu, sizeof(double) * d);
        su[slot] = P_new;
        pu[slot] = p;
        free(add);
        free(z);
    }
}

/* ------------------------------------------------------------------ */
/* int8 cache slots with one fp32 scale per row [SH abstract: a        */
/* budgeted cache combines with 4-bit quantisation of its entries; the  */
/* int8 form and its rounding are readings, listed in the design notes]:*/
/*   amax = max_e |x_e|                                  (exact, fp32)   */
/*   amax == 0:  scale = 0 and every code is 0                           */
/*   otherwise:  inv = 127 / amax                     (fp32, rounded)   */
/*               code_e = rint(x_e * inv), clamped to [-127, 127]        */
/*                        (fp32 product; rint rounds half to even)       */
/*               scale = amax / 127                    (fp32, rounded)   */
/* A stored row reads back as code_e * scale.  X holds n rows of d      */
/* values, each exactly representable in fp32.                          */
/* ------------------------------------------------------------------ */
void oracle_quantize_rows(int n, int d, const double* X, signed char* code, float* scale)
{
    for (int t = 0; t < n; ++t) {
        const double* x = X + (size_t)t * d;
        signed char* c = code + (size_t)t * d;
        float amax = 0.0f;
        for (int e = 0; e < d; ++e) {
            float a = fabsf((float)x[e]);
            if (a > amax) amax = a;
        }
        if (amax == 0.0f) {
            for (int e = 0; e < d; ++e) c[e] = 0;
            scale[t] = 0.0f;
            continue;
        }
        float inv = 127.0f / amax;
        for (int e = 0; e < d; ++e) {
            float y = rintf((float)x[e] * inv);
            if (y > 127.0f) y = 127.0f;
            if (y < -127.0f) y = -127.0f;
            c[e] = (signed char)y;
        }
        scale[t] = amax / 127.0f;
    }
}

/* ------------------------------------------------------------------ */
/* 4-bit cache rows [Scissorhands abstract: a budgeted cache combines  */
/* with quantisation of its entries, down to 4 bits; the form is this  */
/* library's reading]: per row amax = max |x_e| (fp32), code_e =       */
/* rint(x_e * (7 / amax)) in fp32 (half to even), clamped to +-7, and  */
/* scale = amax / 7; all codes 0 and scale 0 when amax = 0.  The row   */
/* reads back as code_e * scale.  Codes are returned one per byte.      */
/* ------------------------------------------------------------------ */
void oracle_quantize_rows4(int n, int d, const double* X, signed char* code, float* scale)
{
    for (int t = 0; t < n; ++t) {
        const double* x = X + (size_t)t * d;
        signed char* c = code + (size_t)t * d;
        float amax = 0.0f;
        for (int e = 0; e < d; ++e) {
            float a = fabsf((float)x[e]);
            if (a > amax) amax = a;
        }
        if (amax == 0.0f) {
            for (int e = 0; e < d; ++e) c[e] = 0;
            scale[t] = 0.0f;
            continue;
        }
        float inv = 7.0f / amax;
        for (int e = 0; e < d; ++e) {
            float y = rintf(inv * (float)x[e]);
            if (y > 7.0f) y = 7.0f;
            if (y < -7.0f) y = -7.0f;
            c[e] = (signed char)y;
        }
        scale[t] = amax / 7.0f;
    }
}

/* ------------------------------------------------------------------ */
/* HashEvict sign projection [HE abstract]: bit j of the code is set    */
/* iff the fp32 projection of x onto column j of W (W is [d][32],       */
/* row-major) is positive; the projection is the fused multiply-add     */
/* chain acc = fmaf(x_i, W[i][j], acc) for i = 0..d-1 from acc = 0.     */
/* ------------------------------------------------------------------ */
uint32_t oracle_lsh_code(int d, const double* x, const float* W)
{
    uint32_t code = 0u;
    for (int j = 0; j < 32; ++j) {
        float acc = 0.0f;
        for (int i = 0; i < d; ++i) acc = fmaf((float)x[i], W[(size_t)i * 32 + j], acc);
        if (acc > 0.0f) code |= (1u << j);
    }
    return code;
}

void oracle_lsh_codes(int n, int d, const double* X, const float* W, uint32_t* codes)
{
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < n; ++t) codes[t] = oracle_lsh_code(d, X + (size_t)t * d, W);
}

static int hamming(uint32_t a, uint32_t b)
{
    uint32_t x = a ^ b;
    int cnt = 0;
    while (x) { cnt += (int)(x & 1u); x >>= 1; }
    return cnt;
}

/* HashEvict replacement rule for one unit at position p: the slot to     */
/* overwrite (append slot n when not full; otherwise the candidate with    */
/* the largest Hamming distance to code_q, lowest slot on ties).           */
static int lsh_victim(int B, int r, int p, int n, const uint32_t* code, const int* pos,
                      uint32_t code_q, int* is_append)
{
    if (n < B) { *is_append = 1; return n; }
    *is_append = 0;
    int ncand = 0;
    for (int s = 0; s < n; ++s) if (pos[s] <= p - r) ++ncand;
    int best = -1, bestd = -1;
    for (int s = 0; s < n; ++s) {
        if (ncand > 0 && !(pos[s] <= p - r)) continue;
        int dist = hamming(code_q, code[s]);
        if (dist > bestd) { bestd = dist; best = s; }
    }
    return best;
}

/* LSH prompt phase: tokens 0..T-1 enter one at a time under the decode   */
/* replacement rule (no attention output).                                */
void oracle_lsh_prefill(int U, int T, int d, int B, int r,
                        const double* Q, const double* K, const double* V, const float* W,
                        double* cK, double* cV, uint32_t* code, int* pos, int* occ)
{
    #pragma omp parallel for schedule(dynamic, 1)
    for (int u = 0; u < U; ++u) {
        const double* Qu = Q + (size_t)u * T * d;
        const double* Ku = K + (size_t)u * T * d;
        const double* Vu = V + (size_t)u * T * d;
        double* cKu = cK + (size_t)u * B * d;
        double* cVu = cV + (size_t)u * B * d;
        uint32_t* cu = code + (size_t)u * B;
        int* pu = pos + (size_t)u * B;
        for (int s = 0; s < B; ++s) {
            memset(cKu + (size_t)s * d, 0, sizeof(double) * d);
            memset(cVu + (size_t)s * d, 0, sizeof(double) * d);
            cu[s] = 0u;
            pu[s] = -1;
        }
        int n = 0;
        for (int t = 0; t < T; ++t) {
            int app;
            uint32_t cq = (n < B) ? 0u : oracle_lsh_code(d, Qu + (size_t)t * d, W);
            int slot = lsh_victim(B, r, t, n, cu, pu, cq, &app);
            if (app) ++n;
            memcpy(cKu + (size_t)slot * d, Ku + (size_t)t * d, sizeof(double) * d);
            memcpy(cVu + (size_t)slot * d, Vu + (size_t)t * d, sizeof(double) * d);
            cu[slot] = oracle_lsh_code(d, Ku + (size_t)t * d, W);
            pu[slot] = t;
        }
        occ[u] = n;
    }
}

/* One HashEvict decode step at position p [HE abstract]: choose the     */
/* victim before attention, put (k, v, code(k), p) in its slot, then     */
/* attend over the live slots (the new token included, the victim not).  */
void oracle_lsh_decode_step(int U, int d, int B, int r, double scale, int p,
                            double* cK, double* cV, uint32_t* code, int* pos, int* occ,
                            const double* q, const double* k, const double* v,
                            const float* W, double* out, int* victim)
{
    #pragma omp parallel for schedule(dynamic, 4)
    for (int u = 0; u < U; ++u) {
        double* Ku = cK + (size_t)u * B * d;
        double* Vu = cV + (size_t)u * B * d;
        uint32_t* cu = code + (size_t)u * B;
        int* pu = pos + (size_t)u * B;
        const double* qu = q + (size_t)u * d;
        const double* ku = k + (size_t)u * d;
        const double* vu = v + (size_t)u * d;
        double* ou = out + (size_t)u * d;
        int n = occ[u];
        uint32_t cq = oracle_lsh_code(d, qu, W);
        int app;
        int slot = lsh_victim(B, r, p, n, cu, pu, cq, &app);
        if (app) { ++n; occ[u] = n; }
        if (victim) victim[u] = app ? -1 : slot;
        memcpy(Ku + (size_t)slot * d, ku, sizeof(double) * d);
        memcpy(Vu + (size_t)slot * d, vu, sizeof(double) * d);
        cu[slot] = oracle_lsh_code(d, ku, W);
        pu[slot] = p;

        double* z = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        double mx = -INFINITY;
        for (int s = 0; s < n; ++s) {
            z[s] = scale * dot(qu, Ku + (size_t)s * d, d);
            if (z[s] > mx) mx = z[s];
        }
        double lsum = 0.0;
        for (int s = 0; s < n; ++s) lsum += exp(z[s] - mx);
        for (int e = 0; e < d; ++e) ou[e] = 0.0;
        for (int s = 0; s < n; ++s) {
            double P = exp(z[s] - mx) / lsum;
            for (int e = 0; e < d; ++e) ou[e] += P * Vu[(size_t)s * d + e];
        }
        free(z);
    }
}

/* ------------------------------------------------------------------ */
/* Persistence of importance [SH abstract: only tokens that were        */
/* pivotal -- had a substantial influence -- at some step keep          */
/* influencing later steps; the fixed-budget cache stores the pivotal   */
/* tokens preferentially].  The reading (listed in the design notes):   */
/*   pivotal at a step:  P_j > 1/m, m = tokens attended that step,      */
/*                       tested as P_j * m > 1 in fp64;                 */
/*   history:            a 32-bit word per token, bit 0 = the latest    */
/*                       step; each step shifts it left by one and puts */
/*                       the new flag in bit 0 (older flags fall out);  */
/*   importance:         the number of set bits;                        */
/*   victim:             among slots with position <= p - r (every live */
/*                       slot if none), the lowest importance, then the */
/*                       lowest position.                               */
/* `margin` reports min |P_j * m - 1| over the flags a call decided     */
/* with m > 1, so that a caller can tell a decision that fp32 rounding  */
/* could flip (with m = 1, P = 1 exactly and the flag is 0).            */
/* ------------------------------------------------------------------ */
static int bits_set(uint32_t x)
{
    int n = 0;
    for (int b = 0; b < 32; ++b) n += (int)((x >> b) & 1u);
    return n;
}

/* Prompt flags: row i (query i, keys 0..i, m = i + 1 tokens) is a step;   */
/* the last 32 rows T-32..T-1 set bit T-1-i of mask[j] for every pivotal */
/* key j <= i.  mask: [U][T]; margin: [U]; tval: NULL or [U][32][T], the    */
/* value P_ij * m of row i = T-32+w (w = 0..31, clipped at 0) in row w     */
/* (0 where j > i).                                                        */
void oracle_sh_prompt_masks(int U, int T, int d, double scale, const double* Q, const double* K,
                            uint32_t* mask, double* margin, double* tval)
{
    #pragma omp parallel for schedule(dynamic, 1)
    for (int u = 0; u < U; ++u) {
        const double* Qu = Q + (size_t)u * T * d;
        const double* Ku = K + (size_t)u * T * d;
        uint32_t* mu = mask + (size_t)u * T;
        double* z = (double*)malloc(sizeof(double) * (size_t)T);
        double mg = INFINITY;
        for (int j = 0; j < T; ++j) mu[j] = 0u;
        const int i0 = T > 32 ? T - 32 : 0;
        if (tval)
            for (size_t x = 0; x < (size_t)32 * T; ++x) tval[(size_t)u * 32 * T + x] = 0.0;
        for (int i = i0; i < T; ++i) {
            double mx = -INFINITY;
            for (int j = 0; j <= i; ++j) {
                z[j] = scale * dot(Qu + (size_t)i * d, Ku + (size_t)j * d, d);
                if (z[j] > mx) mx = z[j];
            }
            double l = 0.0;
            for (int j = 0; j <= i; ++j) l += exp(z[j] - mx);
            for (int j = 0; j <= i; ++j) {
                const double t = exp(z[j] - mx) / l * (double)(i + 1);
                if (t > 1.0) mu[j] |= 1u << (T - 1 - i);
                if (tval) tval[((size_t)u * 32 + (i - i0)) * T + j] = t;
                if (i > 0 && fabs(t - 1.0) < mg) mg = fabs(t - 1.0);   /* m = 1: P = 1 exactly */
            }
        }
        margin[u] = mg;
        free(z);
    }
}

/* Prompt selection: all T tokens when T <= B; otherwise the recent window  */
/* T-r..T-1 and the H tokens among 0..T-r-1 with the most set bits, ties to */
/* the newer position.  kept: [B] ascending positions, -1 padded; returns   */
/* the number kept.                                                         */
int oracle_sh_select(int T, int B, int H, int r, const uint32_t* mask, int* kept)
{
    for (int s = 0; s < B; ++s) kept[s] = -1;
    if (T <= B) {
        for (int j = 0; j < T; ++j) kept[j] = j;
        return T;
    }
    const int ncand = T - r;
    char* keep = (char*)calloc((size_t)T, 1);
    for (int j = ncand; j < T; ++j) keep[j] = 1;
    for (int h = 0; h < H && h < ncand; ++h) {
        int best = -1;
        for (int j = ncand - 1; j >= 0; --j) {        /* newest first: ties stay with the newer */
            if (keep[j]) continue;
            if (best < 0 || bits_set(mask[j]) > bits_set(mask[best])) best = j;
        }
        if (best < 0) break;                           /* cannot happen: h < ncand */
        keep[best] = 1;
    }
    int n = 0;
    for (int j = 0; j < T; ++j)
        if (keep[j]) kept[n++] = j;
    free(keep);
    return n;
}

/* One decode step for U units (new token at position p): attend over the  */
/* n live slots and the new token, shift every live slot's history and set  */
/* this step's flag, evict (when full) by the rule above, insert the new   */
/* token with its own flag as its history.  K, V: [U][B][d]; mask, pos:     */
/* [U][B]; occ: [U]; q, k, v: [U][d]; out: [U][d]; victim: [U] (-1 when     */
/* appended); margin: [U]; forced: [U] or NULL (a slot >= 0 replaces the     */
/* rule's choice); tval: NULL or [U][B+1], P * m of slot s (s < n) and of   */
/* the new token (index B).                                                 */
void oracle_sh_decode_step(int U, int d, int B, int r, double scale, int p,
                           double* cK, double* cV, uint32_t* mask, int* pos, int* occ,
                           const double* q, const double* k, const double* v,
                           double* out, int* victim, double* margin, const int* forced,
                           double* tval)
{
    #pragma omp parallel for schedule(dynamic, 4)
    for (int u = 0; u < U; ++u) {
        double* Ku = cK + (size_t)u * B * d;
        double* Vu = cV + (size_t)u * B * d;
        uint32_t* mu = mask + (size_t)u * B;
        int* pu = pos + (size_t)u * B;
        const double* qu = q + (size_t)u * d;
        const double* ku = k + (size_t)u * d;
        const double* vu = v + (size_t)u * d;
        double* ou = out + (size_t)u * d;
        const int n = occ[u];
        double* z = (double*)malloc(sizeof(double) * (size_t)(n + 1));
        double mx = -INFINITY;
        for (int s = 0; s < n; ++s) {
            z[s] = scale * dot(qu, Ku + (size_t)s * d, d);
            if (z[s] > mx) mx = z[s];
        }
        z[n] = scale * dot(qu, ku, d);
        if (z[n] > mx) mx = z[n];
        double l = 0.0;
        for (int s = 0; s <= n; ++s) l += exp(z[s] - mx);
        for (int e = 0; e < d; ++e) ou[e] = 0.0;
        double mg = INFINITY;
        uint32_t flag_new = 0u;
        for (int s = 0; s <= n; ++s) {
            const double P = exp(z[s] - mx) / l;
            const double* vs = (s < n) ? Vu + (size_t)s * d : vu;
            for (int e = 0; e < d; ++e) ou[e] += P * vs[e];
            const double t = P * (double)(n + 1);
            const uint32_t f = t > 1.0 ? 1u : 0u;
            if (n > 0 && fabs(t - 1.0) < mg) mg = fabs(t - 1.0);        /* m = 1: P = 1 exactly */
            if (tval) tval[(size_t)u * (B + 1) + (s < n ? s : B)] = t;
            if (s < n) mu[s] = (mu[s] << 1) | f;
            else flag_new = f;
        }
        int slot;
        if (n < B) {
            slot = n;
            occ[u] = n + 1;
            if (victim) victim[u] = -1;
        } else {
            int ncand = 0;
            for (int s = 0; s < n; ++s) if (pu[s] <= p - r) ++ncand;
            int best = -1;
            for (int s = 0; s < n; ++s) {
                if (ncand > 0 && !(pu[s] <= p - r)) continue;
                if (best < 0) { best = s; continue; }
                const int a = bits_set(mu[s]), b = bits_set(mu[best]);
                if (a < b || (a == b && pu[s] < pu[best])) best = s;
            }
            slot = (forced && forced[u] >= 0) ? forced[u] : best;
            if (victim) victim[u] = slot;
        }
        if (margin) margin[u] = mg;
        memcpy(Ku + (size_t)slot * d, ku, sizeof(double) * d);
        memcpy(Vu + (size_t)slot * d, vu, sizeof(double) * d);
        mu[slot] = flag_new;
        pu[slot] = p;
        free(z);
    }
}

/* ------------------------------------------------------------------ */
/* Per-head cache policy from the prompt's attention [FG abstract:      */
/* profile the attention heads; evict long-range context on heads that  */
/* attend locally, keep the frequent tokens on heads that attend to a   */
/* few of them, keep the standard cache on heads that attend broadly;   */
/* FG Figure 2: "Frequency + Local" is the fixed H2O cache.  The        */
/* recovery test is this library's reading]:                            */
/*   A_ij = exp(z_ij - m_i) / l_i over keys j <= i (prompt rows);        */
/*   local:      row i keeps keys i-B+1 .. i;                            */
/*   frequency:  row i keeps keys i-r+1 .. i and the heavy keys j <= i-r,*/
/*               heavy = the H largest column sums among j < T-r (ties  */
/*               to the lower j, as the prompt selection);              */
/*   recovery = (1/T) sum_i sum_{j kept at row i} A_ij;                 */
/*   policy 0 (local) if recovery(local) >= tau, else 1 (frequency +    */
/*   local) if recovery(frequency) >= tau, else 2 (full cache).         */
/* policy, rec_local, rec_freq: [U].                                     */
/* ------------------------------------------------------------------ */
void oracle_fg_profile(int U, int T, int d, int B, int H, int r, double scale, double tau,
                       const double* Q, const double* K, int* policy, double* rec_local, double* rec_freq)
{
    #pragma omp parallel for schedule(dynamic, 1)
    for (int u = 0; u < U; ++u) {
        const double* Qu = Q + (size_t)u * T * d;
        const double* Ku = K + (size_t)u * T * d;
        double* z = (double*)malloc(sizeof(double) * (size_t)T);
        double* c = (double*)calloc((size_t)T, sizeof(double));
        char* heavy = (char*)calloc((size_t)T, 1);
        /* pass 1: column sums, then the heavy keys */
        for (int pass = 0; pass < 2; ++pass) {
            double keep_l = 0.0, keep_f = 0.0;
            for (int i = 0; i < T; ++i) {
                double mi = -INFINITY;
                for (int j = 0; j <= i; ++j) {
                    z[j] = scale * dot(Qu + (size_t)i * d, Ku + (size_t)j * d, d);
                    if (z[j] > mi) mi = z[j];
                }
                double li = 0.0;
                for (int j = 0; j <= i; ++j) li += exp(z[j] - mi);
                for (int j = 0; j <= i; ++j) {
                    const double a = exp(z[j] - mi) / li;
                    if (pass == 0) {
                        c[j] += a;
                    } else {
                        if (j >= i - B + 1) keep_l += a;
                        if (j >= i - r + 1 || (heavy[j] && j <= i - r)) keep_f += a;
                    }
                }
            }
            if (pass == 0) {
                const int ncand = T - r;
                if (T <= B) {
                    /* the H2O prompt rule keeps every token of a prompt that
                       fits the budget, so the frequency + local cache holds
                       them all */
                    for (int j = 0; j < T; ++j) heavy[j] = 1;
                } else if (ncand > 0) {
                    cand_t* cs = (cand_t*)malloc(sizeof(cand_t) * (size_t)ncand);
                    for (int j = 0; j < ncand; ++j) { cs[j].c = c[j]; cs[j].j = j; }
                    qsort(cs, (size_t)ncand, sizeof(cand_t), cand_cmp);
                    for (int t = 0; t < H && t < ncand; ++t) heavy[cs[t].j] = 1;
                    free(cs);
                }
            } else {
                rec_local[u] = keep_l / (double)T;
                rec_freq[u] = keep_f / (double)T;
                policy[u] = rec_local[u] >= tau ? 0 : (rec_freq[u] >= tau ? 1 : 2);
            }
        }
        free(heavy);
        free(c);
        free(z);
    }
}
