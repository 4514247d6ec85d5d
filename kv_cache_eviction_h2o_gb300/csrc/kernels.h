// kernels.h -- launchers between the C ABI (h2o_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace h2o {

// One handle's device-resident cache.
struct CacheView {
    void* K;            // [U][B][D] element type per dtype; int8 codes when qbits 8, [U][B][D/2] bytes of 4-bit codes when qbits 4
    void* V;            // [U][B][D]
    float2* kvs;        // qbits: [U][Bp] {K scale, V scale} of every slot, else nullptr
    int qbits, Bp;      // rows stored as codes of 8 or 4 bits (0: the input type); Bp = B rounded up to even
    float2* score;      // [U][B] accumulated attention (H2O) as an unevaluated fp32 pair hi + lo
    int* pos;           // [U][B] token position per slot, -1 = empty
    uint32_t* code;     // [U][B] key codes (LSH); pivotal histories (persistence of importance)
    int2* ustate;       // [U] {occupancy, position of the next token}
    int* err;           // device error word (DeviceError bits)
    const int4* upol;   // per-unit {budget, heavy, recent, policy} (per-head policies), else nullptr:
                        // unit u then holds at most upol[u].x of its B slots
    int U, B, D, dtype, r;
    float qscale;       // softmax scale * log2(e): logits are kept in base 2
};

struct DecodeArgs {
    CacheView c;
    const void* q;      // [U][D] ([U * G][D] for a grouped-query cache)
    const void* k;      // [U][D]
    const void* v;      // [U][D]
    float* out;         // [U][D] ([U * G][D])
    int* victim_out;    // [U] or nullptr
    const float* W;     // [D][32] (LSH)
    int early;          // 1: the previous kernel in the stream does not write this
                        // cache, so the cache may be read before the dependency wait
    int G;              // H2O: query heads sharing each cache unit (0 or 1: one);
                        // q and out then hold U * G rows, head g of unit u in row u * G + g
    int num_sms;        // the device's SM count (selects the tile)
    const int* ulist;   // or nullptr: CTA group g takes unit ulist[g] for g < *ucount and exits beyond
    const int* ucount;  // (written by earlier kernels of the handle: read after the dependency wait)
};

struct PromptArgs {
    const void* Q;      // [U][T][D]
    const void* K;
    const void* V;
    int T;
    int H;              // heavy-hitter slots (H2O)
    float* m2;          // [U][T] row max, base-2 logit units
    float* l;           // [U][T] row normaliser
    float* nb;          // [U][T] row bias -(m2 + log2 l), written by the tensor-core pass 1 for its pass 2
    double* c;          // [U][T] column sums
    uint32_t* cq;       // [U][T] query codes (LSH)
    uint32_t* ck;       // [U][T] key codes (LSH)
    int G;              // prompt scorer: query heads per key row set (0 or 1: one);
                        // query unit u reads the keys of unit u / G
    int budget;         // selection budget (0: the cache's B)
    double* bandB;      // [U][T] or nullptr: per key j, the probabilities of rows j .. j+wB-1
    double* bandr;      // [U][T] or nullptr: the same for rows j .. j+wr-1
    int wB, wr;
};

// Per-head policy profile [the "Model Tells You What to Discard" review
// page, method section]: per unit, the recoveries of the local and the
// frequency + local caches and the first policy reaching tau.
struct FgArgs {
    int4* upol;         // out: [U] {budget, heavy, recent, policy}
    double2* rec;       // out: [U] {local recovery, frequency + local recovery}
    double tau;
    int B, H, r;        // frequency + local (H2O) parameters; local is (B, 0, B)
    int B_full;         // full cache: (B_full, 0, B_full)
};

cudaError_t launch_h2o_decode(const DecodeArgs& a, int split, cudaStream_t st);
// one-head H2O step over many units, one warp per unit; *used = false
// (nothing launched) when it does not apply
cudaError_t launch_h2o_decode_warps(const DecodeArgs& a, cudaStream_t st, bool* used);
cudaError_t launch_lsh_decode(const DecodeArgs& a, int split, cudaStream_t st);
// persistence-of-importance step (histories in CacheView::code)
cudaError_t launch_sh_decode(const DecodeArgs& a, int split, cudaStream_t st);
int auto_decode_split(int U, int B, int num_sms);
// split of a bf16, head_dim 128 one-head H2O / HashEvict cache with U < SMs
// (qbits: 8 or 4 for quantised rows, else 0)
int few_units_split(int U, int B, int num_sms, bool lsh, int qbits);
int max_decode_split();

cudaError_t launch_prompt_stats(const CacheView& c, const PromptArgs& p, cudaStream_t st);
// tensor-core prompt scorer (bf16, head_dim 128)
bool prompt_tc_supported(const CacheView& c);
cudaError_t launch_prompt_stats_tc(const CacheView& c, const PromptArgs& p, cudaStream_t st);
cudaError_t launch_select(const CacheView& c, const PromptArgs& p, cudaStream_t st);
// ckv[u][j] = sum over g = 0..G-1 of c[u * G + g][j], u < U, j < T
cudaError_t launch_group_sum(const double* c, double* ckv, int U, int G, int T, cudaStream_t st);
// persistence-of-importance prompt: histories into p.ck, selection keys into
// p.c, then the selection and the gather (histories copied into c.code)
cudaError_t launch_sh_prompt(const CacheView& c, const PromptArgs& p, cudaStream_t st);
// its tensor-core history pass (bf16, head_dim 128; needs p.m2, p.l scratch)
cudaError_t launch_sh_flags_tc(const CacheView& c, const PromptArgs& p, cudaStream_t st);
cudaError_t launch_gather(const CacheView& c, const PromptArgs& p, bool with_codes, cudaStream_t st);
// the selection and the kept rows' copy in one kernel where the prompt allows (H2O)
cudaError_t launch_select_gather(const CacheView& c, const PromptArgs& p, cudaStream_t st);
// per-head policies: recoveries from the column and band sums and the H2O
// selection already made, the policy, and the kept set of local and full
// units rewritten (the gather follows)
cudaError_t launch_fg_policy(const CacheView& c, const PromptArgs& p, const FgArgs& f, cudaStream_t st);
// per-head policies: the units of policy 0 or 1 into lists[0 ..), those of
// policy 2 into lists[U ..), in unit order; counts[0], counts[1]
cudaError_t launch_fg_lists(const int4* upol, int U, int* lists, int* counts, cudaStream_t st);
// One CTA whose bounded wait on a barrier nobody completes must run out and
// set *err.
cudaError_t launch_wait_selftest(int* err, cudaStream_t st);

// Record a failure for h2o_last_error() and return `code`.
int set_last_error(int code, const char* fmt, ...);

// W: the projection [D][32] on the device; W_host: the same values in host
// memory (the sign-code kernel takes them as a launch parameter).
cudaError_t launch_lsh_prompt(const CacheView& c, const PromptArgs& p, const float* W,
                              const float* W_host, cudaStream_t st);

}  // namespace h2o
