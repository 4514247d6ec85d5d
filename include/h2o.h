/*
 * h2o.h -- C ABI of libh2o_gb300.so: budgeted-KV-cache decode attention with
 * heavy-hitter (H2O) eviction and the HashEvict LSH variant, on one GB300
 * (sm_103a).
 *
 * The operations follow these pages (cited by title and section):
 *  [H2O] "H2O: Heavy-Hitter Oracle for Efficient Generative Inference of Large
 *        Language Models" (review page), 提案手法 (method) and 研究の動機と目的
 *        (motivation) sections: heavy hitters are the tokens that accumulate
 *        the most attention; a greedy per-decode-step rule driven by local
 *        attention statistics evicts, balancing recency against relevance.
 *  [FG]  "Model Tells You What to Discard: Adaptive KV Cache Compression for
 *        LLMs" (review page), Figure 2 caption: the fixed "Frequency + Local"
 *        cache, i.e. heavy hitters plus a recent window.
 *  [SH]  "Scissorhands: Exploiting the Persistence of Importance Hypothesis
 *        for LLM KV Cache Compression at Test Time", abstract: the cache is
 *        held at a fixed budget.
 *  [HE]  "HashEvict: A Pre-Attention KV Cache Eviction Strategy using
 *        Locality-Sensitive Hashing", abstract: Hamming distance between
 *        binarised Gaussian projections of the query and the cached keys,
 *        decided before attention; the new token replaces the cached token
 *        expected to receive the least attention; a compact binary structure
 *        is kept in GPU memory.
 *
 * Conventions shared by every call
 *  - U = batch * heads independent (batch, head) units; the unit index is
 *    b * heads + h.  d = head_dim (64 or 128).  Element type is fp32
 *    (H2O_F32) or bf16 (H2O_BF16) for every Q/K/V/q/k/v buffer of a handle.
 *    A grouped-query handle (h2o_init_gqa) has U = batch * kv_heads cache
 *    units and G query heads per unit: its Q, q and out have U * G rows.
 *  - Four handle kinds: H2O (h2o_init, h2o_init_gqa; h2o_* calls),
 *    HashEvict (lsh_init; lsh_* calls), persistence of importance
 *    (sh_init; sh_* calls) and per-head policies (fg_init; fg_* calls).  State, sync, stream and destroy calls (h2o_*)
 *    take any kind; a prefill or decode call of another kind is
 *    H2O_ERR_STATE.
 *  - Pointers named "device" must point to device memory of the current
 *    device, C-contiguous, 16-byte aligned.  The caller owns them.
 *  - The library owns the cache (K, V [U][B][d]), the scores (fp64
 *    [U][B]), the slot positions (int32 [U][B], -1 = empty), the LSH codes
 *    (uint32 [U][B]), the per-unit occupancy and next position, and the
 *    prompt scratch.  The cache is allocated by *_init; the prompt scratch
 *    by the first *_prefill with a given or larger prompt length (so that
 *    call must not be inside a CUDA stream capture).
 *  - Calls enqueue work on the handle's stream and return without waiting.
 *    Argument and state errors are returned synchronously; a device-side
 *    error (a bounded wait that ran out) is reported by h2o_sync.
 *  - Decode steps use programmatic dependent launch: a step may start while
 *    the previous kernel in its stream drains.  It reads q, k, v only after
 *    that kernel has completed; it reads its own cache earlier only when the
 *    last cache this library wrote on the stream belongs to another handle.
 *    So nothing but this API may write a handle's cache (it is private).
 *  - Every int-returning call returns H2O_OK (0) or a negative h2o_status;
 *    h2o_last_error() then describes the failure (thread-local).
 *  - Positions are 0-based.  After a prompt of T tokens the next decoded
 *    token has position T, then T+1, ...
 *  - Argument types chosen for the host side: the softmax scale is a
 *    double; accumulated scores cross the boundary as fp64 (the device keeps
 *    each as an unevaluated pair of fp32 values, about 48 significant bits);
 *    occupancy and next position are per-unit arrays, since every unit
 *    advances on its own once a state is loaded by hand.
 *  - The library keeps per-device set-up (kernel attributes, device
 *    addresses of its fixed arrays) for the life of the process, and a
 *    handle's buffers live in the device's context: after cudaDeviceReset
 *    on a device, no handle created before it and no call of this library
 *    may be used on that device again in the process.
 */
#ifndef H2O_GB300_H
#define H2O_GB300_H

#ifdef __cplusplus
extern "C" {
#endif

typedef struct h2o_ctx* h2o_handle;

typedef enum {
    H2O_OK = 0,
    H2O_ERR_ARG = -1,             /* bad argument (null, size, alignment)      */
    H2O_ERR_STATE = -2,           /* wrong call order or wrong handle kind     */
    H2O_ERR_ALLOC = -3,           /* device allocation failed                  */
    H2O_ERR_CUDA = -4,            /* a CUDA runtime call failed                */
    H2O_ERR_DEVICE_TIMEOUT = -5,  /* a kernel's bounded wait ran out           */
    H2O_ERR_UNSUPPORTED = -6      /* not supported on this device / dtype      */
} h2o_status;

enum { H2O_F32 = 0, H2O_BF16 = 1 };

/*
 * H2O_KV8 -- OR into dtype (H2O_BF16 | H2O_KV8, H2O_F32 | H2O_KV8) to store
 * the cache's K and V rows as int8 codes with one fp32 scale per row
 * [SH abstract: a budgeted cache combines with quantisation of its
 * entries; the int8 form is this library's reading].  Inputs keep their
 * type.  A row x is stored as amax = max|x_e|, scale = amax / 127 and
 * code_e = rint(x_e * (127 / amax)) (fp32 arithmetic, half to even, within
 * +-127; all zero when amax = 0), and reads back as code_e * scale.  A
 * decode step attends to its own new token at full precision and then
 * stores it quantised.  Eviction, scores and codes follow the same rules
 * as without the flag.  The paper has no counterpart for the flag itself.
 */
enum { H2O_KV8 = 2 };

/*
 * H2O_KV4 -- OR into dtype instead of H2O_KV8 to store the rows as 4-bit
 * codes with one fp32 scale per row [SH abstract: quantisation of the
 * entries down to 4 bits; the form is this library's reading]:
 * scale = amax / 7, code_e = rint(x_e * (7 / amax)) (fp32, half to even,
 * within +-7; all zero when amax = 0).  A row of d codes takes d/2 bytes:
 * byte i holds element 2i in its low nibble and element 2i+1 in its high
 * nibble, each in offset binary (code + 8).  Everything else as H2O_KV8;
 * the two flags are exclusive.
 */
enum { H2O_KV4 = 4 };

/*
 * h2o_init -- create an H2O cache handle [H2O 提案手法; FG Figure 2; SH].
 *   budget = B slots per unit (>= 1), heavy = H heavy-hitter slots,
 *   recent = r recent-window slots; heavy + recent must equal budget.
 *   batch, heads >= 1; head_dim in {64, 128}; dtype H2O_F32 or H2O_BF16,
 *   optionally | H2O_KV8 or | H2O_KV4;
 *   scale > 0 is the softmax scale (usually 1/sqrt(head_dim)).
 *   cuda_stream: the cudaStream_t to enqueue on (NULL = legacy stream).
 * On success *out holds the handle; destroy it with h2o_destroy.
 */
int h2o_init(h2o_handle* out, int budget, int heavy, int recent, int batch, int heads,
             int head_dim, int dtype, double scale, void* cuda_stream);

/*
 * h2o_init_gqa -- create an H2O handle whose caches are shared by groups
 * of query heads (grouped-query attention) [H2O 提案手法: a slot's score
 * is the attention it accumulates; the grouped form is this library's
 * reading].  U = batch * kv_heads cache units (unit index b * kv_heads +
 * h); each is shared by `groups` = G query heads (1 <= G <= 16), query head
 * g of unit u being row u * G + g of Q, q and out.  Every head attends with
 * its own softmax; a slot's score grows by the sum of its G heads'
 * probabilities (added in head order), a prompt token's c_j is the sum of
 * its G heads' column sums, and the new token's score is the sum of its G
 * own probabilities.  Eviction and insertion are as for one head.
 *   budget <= 1024 when G > 1.  Other arguments as h2o_init; G = 1 is
 *   exactly h2o_init.
 * h2o_prefill then takes Q [U*G][T][d] and K, V [U][T][d];
 * h2o_decode_step takes q [U*G][d], k, v [U][d], out [U*G][d] and
 * victim_out [U]; h2o_get_prefill_stats returns m and l [U*G][T] and the
 * unit sums c [U][T].  State calls work on the U cache units.
 */
int h2o_init_gqa(h2o_handle* out, int budget, int heavy, int recent, int batch, int kv_heads, int groups,
                 int head_dim, int dtype, double scale, void* cuda_stream);

/*
 * h2o_prefill -- build the initial cache from a prompt of T >= 1 tokens
 * [H2O 提案手法]: the accumulated attention of prompt token j is
 *   c_j = sum_{i>=j} exp(z_ij - m_i) / l_i,  z_ij = scale q_i.k_j,
 *   m_i = max_{j<=i} z_ij,  l_i = sum_{j<=i} exp(z_ij - m_i);
 * if T <= B every token is kept, otherwise the recent window T-r..T-1 and
 * the H largest c_j among j < T-r (ties to the lower j).  Kept tokens fill
 * slots 0..n-1 in ascending position; each slot's score starts at c_j.
 *   Q, K, V: device [U][T][d] of the handle's dtype.
 * Resets the handle's decode position to T.  Allocates the prompt scratch
 * (20 bytes per unit per token: row max, normaliser and bias, column sums;
 * per query head on a grouped-query handle, plus 8 per cache unit per token)
 * when T exceeds the largest T seen so far.
 */
int h2o_prefill(h2o_handle h, const void* Q, const void* K, const void* V, int T);

/*
 * h2o_decode_step -- one decode step for all U units [H2O 提案手法]:
 *   attend:     out = softmax(scale q.K) V over the live slots and the new
 *               token itself;
 *   accumulate: every live slot's score += its probability this step;
 *   evict:      if the cache is full, the victim is the slot with the
 *               smallest score among slots whose position is <= p - r
 *               (p = this token's position), lowest slot on ties;
 *               otherwise the next empty slot;
 *   insert:     the victim slot takes (k, v), score = the new token's own
 *               probability, position p.
 *   q, k, v: device [U][d] of the handle's dtype; out: device fp32 [U][d];
 *   victim_out: device int32 [U] or NULL, receives the evicted slot or -1
 *   when the token was appended.
 * Requires a prior h2o_prefill (or h2o_set_state) on an H2O handle.
 */
int h2o_decode_step(h2o_handle h, const void* q, const void* k, const void* v,
                    float* out, int* victim_out);

/*
 * sh_init -- create a persistence-of-importance cache handle [SH abstract:
 * tokens that were pivotal -- had a substantial influence -- at a step keep
 * influencing later steps, so a fixed-budget cache keeps them; the exact
 * rule is this library's reading]:
 *   pivotal:    at a step that attends to m tokens, a token whose
 *               probability exceeds the uniform share, P * m > 1;
 *   history:    each slot keeps the flags of its last 32 steps, a uint32
 *               with bit 0 = the latest step; importance = its set bits;
 *   evict:      when full, among slots with position <= p - r (every live
 *               slot if none) the lowest importance, then the lowest
 *               position;
 *   insert:     the new token's history is its own flag this step.
 *   Arguments as h2o_init (heavy + recent = budget); H2O_KV8 and H2O_KV4
 *   are not supported (H2O_ERR_UNSUPPORTED).
 */
int sh_init(h2o_handle* out, int budget, int heavy, int recent, int batch, int heads, int head_dim,
            int dtype, double scale, void* cuda_stream);

/*
 * sh_prefill -- initial cache from a prompt of T >= 1 tokens [SH]: the last
 * min(T, 32) prompt rows are steps (row i attends to keys 0..i, m = i + 1);
 * a token's history has bit T-1-i set when it was pivotal for row i.  Keeps
 * every token when T <= B, otherwise the recent window T-r..T-1 and the H
 * tokens among 0..T-r-1 with the most set bits (ties to the newer
 * position); slots 0..n-1 in ascending position with their histories.
 *   Q, K, V: device [U][T][d] of the handle's dtype.  Allocates prompt
 *   scratch (20 bytes per unit per token) when T exceeds the largest T seen.
 */
int sh_prefill(h2o_handle h, const void* Q, const void* K, const void* V, int T);

/*
 * sh_decode_step -- one decode step for all U units [SH]: attend as
 * h2o_decode_step (live slots and the new token itself), shift every live
 * slot's history and set this step's flag, evict by the rule of sh_init
 * when full, insert (k, v) with position p.  Arguments as h2o_decode_step.
 * h2o_get_state / h2o_set_state carry the histories in `code` (scores 0).
 */
int sh_decode_step(h2o_handle h, const void* q, const void* k, const void* v,
                   float* out, int* victim_out);

/*
 * fg_init -- create a per-head policy cache handle [FG, method section:
 * each attention head is profiled on the prompt and given its own cache
 * policy, the first that recovers enough of its attention; Figure 2
 * caption: the fixed "Frequency + Local" policy is the H2O cache].  Three
 * policies, tried in this order (special-token and punctuation policies
 * need token ids and are not offered):
 *   0 local:              the newest `budget` tokens (H2O with heavy 0,
 *                         recent = budget: a sliding window);
 *   1 frequency + local:  the H2O cache (budget, heavy, recent);
 *   2 full:               every token up to `full_budget` (H2O with heavy 0,
 *                         recent = full_budget);
 * and a head takes the first whose recovery -- the attention mass its kept
 * set holds at each prompt row, averaged over the rows -- reaches tau.  The
 * recovery test and the order are this library's reading of the page.
 *   budget = heavy + recent as h2o_init; full_budget >= 1 (usually the
 *   prompt plus the decode steps); 0 < tau <= 1.  H2O_KV8 and H2O_KV4 are not
 *   supported.
 *   Every unit holds max(budget, full_budget) slots; a unit of policy 0 or 1
 *   uses `budget` of them.  State calls see that many slots per unit.
 */
int fg_init(h2o_handle* out, int budget, int heavy, int recent, int full_budget, double tau, int batch, int heads,
            int head_dim, int dtype, double scale, void* cuda_stream);

/*
 * fg_prefill -- profile every head on a prompt of T >= 1 tokens and build
 * its cache by its policy [FG method section; H2O 提案手法]:
 *   local recovery     = (1/T) sum_i sum_{j = i-budget+1 .. i} P_ij,
 *   frequency + local  = (1/T) sum_i sum_{j = i-recent+1 .. i, or j heavy
 *                        and j <= i-recent} P_ij, the heavy keys being the
 *                        H2O prompt selection's (all kept tokens when
 *                        T <= budget),
 * with P_ij the causal softmax of the prompt (as h2o_prefill); then the
 * unit's cache is built by the H2O prompt rule with its policy's budget,
 * heavy count and window.  Q, K, V: device [U][T][d].  Allocates prompt
 * scratch (36 bytes per unit per token) when T exceeds the largest T seen.
 */
int fg_prefill(h2o_handle h, const void* Q, const void* K, const void* V, int T);

/*
 * fg_decode_step -- one decode step of every unit by the H2O rule
 * (h2o_decode_step) with its own policy's budget and recent window: two
 * launches, one over the units on a compressed policy and one over the
 * units on the full cache (lists built by fg_prefill).  Arguments as
 * h2o_decode_step.
 */
int fg_decode_step(h2o_handle h, const void* q, const void* k, const void* v, float* out, int* victim_out);

/*
 * fg_get_policy -- copy the last fg_prefill's choice to HOST buffers [U]
 * (any may be NULL): policy (0 local, 1 frequency + local, 2 full) and the
 * two recoveries.  Before any fg_prefill every unit reads policy 1 with
 * recoveries 0.  Waits for the handle's stream.
 */
int fg_get_policy(h2o_handle h, int* policy, double* rec_local, double* rec_freq);

/*
 * lsh_init -- create a HashEvict cache handle [HE abstract].
 *   budget = B slots, recent = r slots never evicted (0 <= r <= B);
 *   W: device fp32 [d][32], the Gaussian projection matrix, copied at init.
 *   Other arguments as h2o_init.
 * Code of a vector x: bit j is 1 iff the fp32 fused multiply-add chain
 *   acc = fmaf(x_i, W[i][j], acc), i = 0..d-1, from acc = 0, ends > 0.
 */
int lsh_init(h2o_handle* out, int budget, int recent, int batch, int heads, int head_dim,
             int dtype, double scale, const float* W, void* cuda_stream);

/*
 * lsh_prefill -- build the initial HashEvict cache from a prompt of T >= 1
 * tokens by replaying the decode replacement rule token by token: tokens
 * enter empty slots while there are any; afterwards token t replaces the
 * slot with the largest Hamming distance between code(q_t) and the slot's
 * key code among slots with position <= t - r (lowest slot on ties).
 *   Q, K, V: device [U][T][d].  Scratch: 8 bytes per unit per token.
 */
int lsh_prefill(h2o_handle h, const void* Q, const void* K, const void* V, int T);

/*
 * lsh_decode_step -- one HashEvict step [HE abstract]: the victim is chosen
 * before attention (largest Hamming distance between code(q) and the
 * cached key codes among slots with position <= p - r, lowest slot on ties;
 * the next empty slot while the cache is not full), the new (k, v, code(k),
 * p) is written into it, and out = softmax(scale q.K) V over the live slots,
 * which now hold the new token and no longer the victim.
 *   Arguments as h2o_decode_step.  Requires lsh_prefill on an LSH handle.
 */
int lsh_decode_step(h2o_handle h, const void* q, const void* k, const void* v,
                    float* out, int* victim_out);

/*
 * h2o_get_state -- copy the cache to HOST buffers (any pointer may be NULL):
 *   K, V [U][B][d] of the handle's dtype (int8 codes for H2O_KV8 handles;
 *   [U][B][d/2] bytes of packed codes for H2O_KV4 handles; the scales of
 *   both from h2o_get_kv_scales); score fp64 [U][B] (H2O handles;
 *   zeros for LSH); pos int32 [U][B]; code uint32 [U][B] (LSH handles;
 *   zeros for H2O); occupancy int32 [U]; next_pos int32 [U].
 * Waits for the handle's stream.
 */
int h2o_get_state(h2o_handle h, void* K, void* V, double* score, int* pos, unsigned* code,
                  int* occupancy, int* next_pos);

/*
 * h2o_set_state -- overwrite the cache from HOST buffers laid out as in
 * h2o_get_state (NULL leaves that part unchanged).  Marks the handle ready
 * for decode.  Waits for the handle's stream.
 */
int h2o_set_state(h2o_handle h, const void* K, const void* V, const double* score,
                  const int* pos, const unsigned* code, const int* occupancy,
                  const int* next_pos);

/*
 * h2o_get_kv_scales / h2o_set_kv_scales -- the fp32 K and V row scales
 * [U][B] of an H2O_KV8 or H2O_KV4 handle, to / from HOST buffers (get:
 * either may be NULL; set: both required).  H2O_ERR_STATE on a handle
 * with neither flag.  Both wait for the handle's stream.  The quantised
 * caches are this library's reading of the quantised budgeted cache (see
 * H2O_KV8, H2O_KV4).
 */
int h2o_get_kv_scales(h2o_handle h, float* kscale, float* vscale);
int h2o_set_kv_scales(h2o_handle h, const float* kscale, const float* vscale);

/*
 * h2o_get_prefill_stats -- copy the last h2o_prefill's (or fg_prefill's) prompt statistics to
 * HOST buffers [U][T] (any may be NULL): m (row max of z, natural-log
 * units), l (row normaliser) and c (column sums, fp64).  Waits.  On a
 * grouped-query handle m and l are [U*G][T] (per query head) and c is
 * [U][T] (per cache unit, the sum over its heads).
 */
int h2o_get_prefill_stats(h2o_handle h, float* m, float* l, double* c);

/* Replace the stream later calls enqueue on. */
int h2o_set_stream(h2o_handle h, void* cuda_stream);

/*
 * h2o_set_decode_split -- CTAs (1..16) that share one unit's slots in the
 * decode kernels (a thread-block cluster); 0 restores the automatic choice.
 * Affects performance only, never results.  H2O_ERR_ARG below
 * ceil(budget / 1024); on a per-head-policy handle the bound is the
 * compressed policies' budget, and the units on the full cache take at
 * least ceil(full_budget / 1024) CTAs whatever is set.  H2O_ERR_STATE on a
 * grouped-query handle (G > 1), whose cluster is always its G query heads.
 */
int h2o_set_decode_split(h2o_handle h, int ctas_per_unit);

/*
 * h2o_sync -- wait for the handle's stream; returns H2O_ERR_DEVICE_TIMEOUT
 * if a kernel reported a bounded wait that ran out (the error word is then
 * cleared), H2O_ERR_CUDA on a CUDA error.
 */
int h2o_sync(h2o_handle h);

/* Free every library-owned buffer of the handle; NULL is a no-op. */
void h2o_destroy(h2o_handle h);

/*
 * h2o_prompt_scores_noalloc -- the prompt column sums c [U][T] (fp64) that
 * h2o_prefill ranks prompt tokens by, computed without allocating device
 * memory.  The pages have no counterpart: this is a variant of the prompt
 * scorer for callers that cannot call cudaMalloc -- serving runtimes that
 * reserve all device memory for their own pool at start-up and forbid
 * allocations afterwards, and hosts whose allocation calls may synchronise
 * the device in the middle of their own streams' work.
 *
 * The scorer's scratch (row max, normaliser and bias, 12 bytes per unit per
 * token) is a fixed device array inside the library of H2O_NOALLOC_MAX_TOKENS
 * unit-tokens (12 MiB), present on every device that loads the library until
 * the process exits.  The call allocates nothing.
 *   Q, K:  device [batch*heads][T][head_dim] of dtype, 16-byte aligned;
 *   c:     device fp64 [batch*heads][T], written in full;
 *   batch, heads, T >= 1 with batch*heads*T <= H2O_NOALLOC_MAX_TOKENS,
 *   otherwise H2O_ERR_ARG; head_dim in {64, 128}; scale > 0;
 *   cuda_stream: the stream to enqueue on (NULL = legacy stream).
 * The first call on each device looks up the array's device address (a
 * set-up step, not an allocation); make that first call before any stream
 * capture.  All calls share the one array and nothing in it carries over
 * between calls, but calls whose work overlaps on the GPU (other streams,
 * other host threads) race on it: the caller must serialise them.
 * There is no handle and so no h2o_sync for this call: if one of the
 * scorer's bounded waits runs out on the device (about a second), the
 * column sums it could not finish are written as NaN instead, so a caller
 * that checks c for NaN sees the failure.
 */
#define H2O_NOALLOC_MAX_TOKENS (1 << 20)
int h2o_prompt_scores_noalloc(const void* Q, const void* K, int batch, int heads, int T,
                              int head_dim, int dtype, double scale, double* c,
                              void* cuda_stream);

/*
 * h2o_selftest_wait_timeout -- enqueue one small kernel that waits, through
 * the same bounded mbarrier wait every kernel of this library uses, on a
 * barrier nothing ever completes.  The wait gives up after about a second
 * of GPU clock, sets the handle's device error word and the kernel returns;
 * the next h2o_sync then reports H2O_ERR_DEVICE_TIMEOUT and clears the word,
 * and the handle stays usable.  The pages have no counterpart: this checks
 * the failure-detection path without faulting or hanging the GPU.
 */
int h2o_selftest_wait_timeout(h2o_handle h);

/* Thread-local description of the last failure in this thread ("" if none). */
const char* h2o_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* H2O_GB300_H */
