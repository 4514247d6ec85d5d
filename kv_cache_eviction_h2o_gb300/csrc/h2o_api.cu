// h2o_api.cu -- the C ABI declared in include/h2o.h: argument checks, device
// buffers owned by a handle, and the launch sequence of each call.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "h2o.h"
#include "kernels.h"

using namespace h2o;

namespace {

thread_local char g_err[512] = "";

}  // namespace

int h2o::set_last_error(int code, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

namespace {

int fail(int code, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* where)
{
    return fail(H2O_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

// Host-side fault injection for the failure-path tests: H2O_FAULT=alloc makes
// the next device allocation fail, H2O_FAULT=launch the next launch.
bool inject(const char* what)
{
    const char* f = getenv("H2O_FAULT");
    return f && strcmp(f, what) == 0;
}

enum Kind { kH2O = 0, kLSH = 1, kSH = 2, kFG = 3 };

const char* kind_name(int k)
{
    return k == kH2O ? "H2O" : k == kLSH ? "LSH" : k == kSH ? "persistence-of-importance" : "per-head policy";
}

// The handle whose cache the library last wrote on each (device, stream).
// A decode kernel may read its own cache before its programmatic-launch
// dependency wait only when the work queued just before it on the stream
// did not write that cache.  That holds when the last cache this library
// wrote on the stream belongs to another handle: every kernel of the library
// launched with programmatic serialisation waits for its predecessor before
// it lets its own dependents start, so everything queued before that other
// handle's work has completed by the time this kernel starts, and kernels
// of the caller never write a cache (it is private to the handle).  A stream
// with no record is treated as unsafe.
struct LastWrite {
    int device;
    cudaStream_t stream;
    const void* h;
};
constexpr int kLastWrites = 64;
std::mutex g_lw_mu;
LastWrite g_lw[kLastWrites];
int g_lw_n = 0, g_lw_next = 0;

// Record that `h` writes its cache on (device, stream); return true when the
// previous record for that stream names another handle.
bool note_cache_write(int device, cudaStream_t stream, const void* h)
{
    std::lock_guard<std::mutex> lock(g_lw_mu);
    for (int i = 0; i < g_lw_n; ++i) {
        if (g_lw[i].device == device && g_lw[i].stream == stream) {
            const bool other = g_lw[i].h != h;
            g_lw[i].h = h;
            return other;
        }
    }
    const int i = g_lw_n < kLastWrites ? g_lw_n++ : (g_lw_next++ % kLastWrites);
    g_lw[i] = LastWrite{device, stream, h};
    return false;
}

void forget_cache_writes(const void* h)
{
    std::lock_guard<std::mutex> lock(g_lw_mu);
    for (int i = 0; i < g_lw_n; ++i)
        if (g_lw[i].h == h) g_lw[i].h = nullptr;
}

}  // namespace

struct h2o_ctx {
    int kind;
    int B, H, r, batch, heads, D, dtype, U;
    int G;                     // query heads per cache unit (H2O grouped-query cache)
    double scale;
    cudaStream_t stream;
    int device;
    int num_sms;
    int split;                 // 0 = automatic
    // cache
    void* K;
    void* V;
    float2* score;             // hi + lo fp32 pairs
    float2* kvs;               // quantised cache: {K scale, V scale} per slot, [U][Bp]
    int qbits, Bp;             // 8 / 4: rows stored as int8 / 4-bit codes; 0: the input type
    int* pos;
    uint32_t* code;
    int2* ustate;
    int* err;
    float* W;
    float* W_host;             // host copy of W (launch parameter of the prompt codes)
    // prompt scratch
    int T_cap;
    float* m2;
    float* nb;                 // row biases for the scorer's second pass: the second half of l's allocation
    float* l;
    double* c;                 // per query head
    double* ckv;               // per cache unit (G > 1): the sum over its heads
    uint32_t* cq;
    uint32_t* ck;
    int last_T;
    int ready;                 // 1 once a prompt or a state was loaded
    // per-head policies (kind kFG): B above is the slot stride max(B_sel, B_full)
    int B_sel, B_full;         // frequency + local budget; full-cache budget
    double tau;
    int4* upol;                // [U] {budget, heavy, recent, policy}
    double2* rec;              // [U] {local, frequency + local} recoveries
    double* bandB;             // prompt scratch [U][T]: band sums of width B_sel and r
    double* bandr;
    int* ulists;               // [2U + 2]: units of policy 0/1, of policy 2, then the two counts
};

namespace {

size_t elem_size(int dtype) { return dtype == H2O_BF16 ? 2 : 4; }

// Bytes of one stored K or V row: the input type, int8 codes, or packed
// 4-bit codes.
size_t row_bytes(const h2o_ctx* h)
{
    if (h->qbits == 8) return (size_t)h->D;
    if (h->qbits == 4) return (size_t)h->D / 2;
    return (size_t)h->D * elem_size(h->dtype);
}

int dev_alloc(void** p, size_t bytes, const char* what)
{
    *p = nullptr;
    if (inject("alloc")) return fail(H2O_ERR_ALLOC, "allocation of %s failed (injected)", what);
    if (bytes == 0) bytes = 16;
    cudaError_t e = cudaMalloc(p, bytes);
    if (e != cudaSuccess) {
        *p = nullptr;
        cudaGetLastError();
        return fail(H2O_ERR_ALLOC, "cudaMalloc(%zu) for %s: %s", bytes, what, cudaGetErrorString(e));
    }
    return H2O_OK;
}

void free_prompt(h2o_ctx* h)
{
    cudaFree(h->m2); cudaFree(h->l); cudaFree(h->c); cudaFree(h->ckv); cudaFree(h->cq); cudaFree(h->ck);
    cudaFree(h->bandB); cudaFree(h->bandr);
    h->m2 = nullptr; h->l = nullptr; h->c = nullptr; h->ckv = nullptr; h->cq = nullptr; h->ck = nullptr;
    h->nb = nullptr;
    h->bandB = nullptr; h->bandr = nullptr;
    h->T_cap = 0;
}

void free_all(h2o_ctx* h)
{
    free_prompt(h);
    cudaFree(h->ulists);
    cudaFree(h->K); cudaFree(h->V); cudaFree(h->score); cudaFree(h->pos); cudaFree(h->code);
    cudaFree(h->ustate); cudaFree(h->err); cudaFree(h->W); cudaFree(h->kvs); cudaFree(h->upol); cudaFree(h->rec);
    free(h->W_host);
    h->W_host = nullptr;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// the per-unit policy arrays of a per-head policy handle
int rc0_alloc(h2o_ctx* h, size_t U)
{
    int rc;
    if ((rc = dev_alloc((void**)&h->upol, U * sizeof(int4), "unit policies")) ||
        (rc = dev_alloc((void**)&h->rec, U * sizeof(double2), "policy recoveries")) ||
        (rc = dev_alloc((void**)&h->ulists, (2 * U + 2) * sizeof(int), "policy unit lists")))
        return rc;
    return H2O_OK;
}

CacheView view(const h2o_ctx* h)
{
    CacheView v;
    v.K = h->K; v.V = h->V; v.score = h->score; v.pos = h->pos; v.code = h->code;
    v.kvs = h->kvs; v.qbits = h->qbits; v.Bp = h->Bp;
    v.ustate = h->ustate; v.err = h->err;
    v.U = h->U; v.B = h->B; v.D = h->D; v.dtype = h->dtype; v.r = h->r;
    v.upol = h->upol;
    v.qscale = (float)(h->scale * 1.4426950408889634);
    return v;
}

int create(h2o_handle* out, int kind, int budget, int heavy, int recent, int batch, int heads,
           int head_dim, int dtype, double scale, const float* W, void* stream, int groups = 1,
           int full_budget = 0, double tau = 0.0)
{
    if (!out) return fail(H2O_ERR_ARG, "out handle pointer is NULL");
    *out = nullptr;
    if (groups < 1 || groups > max_decode_split())
        return fail(H2O_ERR_ARG, "groups must be in [1, %d] (got %d)", max_decode_split(), groups);
    if (groups > 1 && budget > 1024)
        return fail(H2O_ERR_ARG, "a grouped-query cache holds at most 1024 slots (got %d)", budget);
    if (budget < 1) return fail(H2O_ERR_ARG, "budget must be >= 1 (got %d)", budget);
    if (recent < 0 || recent > budget) return fail(H2O_ERR_ARG, "recent must be in [0, budget] (got %d)", recent);
    if ((kind == kH2O || kind == kSH || kind == kFG) && (heavy < 0 || heavy + recent != budget))
        return fail(H2O_ERR_ARG, "heavy + recent must equal budget (%d + %d != %d)", heavy, recent, budget);
    if (batch < 1 || heads < 1) return fail(H2O_ERR_ARG, "batch and heads must be >= 1");
    if ((long long)batch * heads * groups > (1LL << 24)) return fail(H2O_ERR_ARG, "batch * heads too large");
    if (head_dim != 64 && head_dim != 128) return fail(H2O_ERR_ARG, "head_dim must be 64 or 128 (got %d)", head_dim);
    if ((dtype & ~(H2O_BF16 | H2O_KV8 | H2O_KV4)) != 0 || (dtype & (H2O_KV8 | H2O_KV4)) == (H2O_KV8 | H2O_KV4))
        return fail(H2O_ERR_ARG, "dtype must be H2O_F32 or H2O_BF16, optionally | H2O_KV8 or | H2O_KV4");
    const int qbits = (dtype & H2O_KV8) ? 8 : (dtype & H2O_KV4) ? 4 : 0;
    if (kind == kSH && qbits)
        return fail(H2O_ERR_UNSUPPORTED, "H2O_KV8 / H2O_KV4 are not supported on persistence-of-importance handles");
    if (kind == kFG && qbits)
        return fail(H2O_ERR_UNSUPPORTED, "H2O_KV8 / H2O_KV4 are not supported on per-head policy handles");
    if (kind == kFG && (full_budget < 1 || full_budget >= (1 << 20)))
        return fail(H2O_ERR_ARG, "full_budget must be in [1, 2^20) (got %d)", full_budget);
    if (kind == kFG && !(tau > 0.0 && tau <= 1.0)) return fail(H2O_ERR_ARG, "tau must be in (0, 1]");
    dtype &= H2O_BF16;
    if (!(scale > 0.0) || !std::isfinite(scale)) return fail(H2O_ERR_ARG, "scale must be finite and > 0");
    if ((long long)budget >= (1LL << 20)) return fail(H2O_ERR_ARG, "budget must be below 2^20");
    if (kind == kLSH && budget > 28 * 1024)
        return fail(H2O_ERR_ARG, "HashEvict budget must be <= %d (its prompt replay keeps the slots in shared memory)", 28 * 1024);
    if (kind == kLSH && !W) return fail(H2O_ERR_ARG, "W is NULL");
    if (kind == kLSH && !aligned16(W)) return fail(H2O_ERR_ARG, "W must be 16-byte aligned");

    h2o_ctx* h = new (std::nothrow) h2o_ctx();
    if (!h) return fail(H2O_ERR_ALLOC, "host allocation failed");
    memset(h, 0, sizeof(*h));
    h->kind = kind; h->B = budget; h->H = heavy; h->r = recent; h->batch = batch; h->heads = heads;
    h->D = head_dim; h->dtype = dtype; h->U = batch * heads; h->G = groups; h->scale = scale;
    h->qbits = qbits; h->Bp = (budget + 1) & ~1;
    if (kind == kFG) {
        h->B_sel = budget;
        h->B_full = full_budget;
        h->tau = tau;
        h->B = budget > full_budget ? budget : full_budget;   // slot stride
    }
    h->stream = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaGetDevice(&h->device);
    if (e != cudaSuccess) { delete h; cudaGetLastError(); return cuda_fail(e, "cudaGetDevice"); }
    e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
    if (e != cudaSuccess) { delete h; cudaGetLastError(); return cuda_fail(e, "cudaDeviceGetAttribute"); }
    int major = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, h->device);
    if (major < 10) { delete h; return fail(H2O_ERR_UNSUPPORTED, "device compute capability %d.x is not sm_103", major); }

    const size_t U = (size_t)h->U, B = (size_t)h->B, row = row_bytes(h);
    if (kind == kFG && ((rc0_alloc(h, U) != H2O_OK))) { free_all(h); delete h; return H2O_ERR_ALLOC; }
    int rc = H2O_OK;
    if ((rc = dev_alloc(&h->K, U * B * row, "cache K")) ||
        (rc = dev_alloc(&h->V, U * B * row, "cache V")) ||
        (rc = dev_alloc((void**)&h->pos, U * B * sizeof(int), "positions")) ||
        (rc = dev_alloc((void**)&h->ustate, U * sizeof(int2), "unit state")) ||
        (rc = dev_alloc((void**)&h->err, sizeof(int), "error word"))) {
        free_all(h); delete h; return rc;
    }
    if (qbits && (rc = dev_alloc((void**)&h->kvs, U * (size_t)h->Bp * sizeof(float2), "slot scales"))) {
        free_all(h); delete h; return rc;
    }
    if (kind == kH2O || kind == kFG) {
        if ((rc = dev_alloc((void**)&h->score, U * B * sizeof(float2), "scores"))) { free_all(h); delete h; return rc; }
    } else if (kind == kSH) {
        if ((rc = dev_alloc((void**)&h->code, U * B * sizeof(uint32_t), "pivotal histories"))) { free_all(h); delete h; return rc; }
    } else {
        if ((rc = dev_alloc((void**)&h->code, U * B * sizeof(uint32_t), "codes")) ||
            (rc = dev_alloc((void**)&h->W, (size_t)head_dim * 32 * sizeof(float), "projection"))) {
            free_all(h); delete h; return rc;
        }
        e = cudaMemcpyAsync(h->W, W, (size_t)head_dim * 32 * sizeof(float), cudaMemcpyDeviceToDevice, h->stream);
        if (e != cudaSuccess) { free_all(h); delete h; return cuda_fail(e, "copy W"); }
        h->W_host = static_cast<float*>(malloc((size_t)head_dim * 32 * sizeof(float)));
        if (!h->W_host) { free_all(h); delete h; return fail(H2O_ERR_ALLOC, "host allocation failed"); }
        e = cudaMemcpyAsync(h->W_host, W, (size_t)head_dim * 32 * sizeof(float), cudaMemcpyDeviceToHost, h->stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
        if (e != cudaSuccess) { free_all(h); delete h; return cuda_fail(e, "copy W to the host"); }
    }
    e = cudaMemsetAsync(h->err, 0, sizeof(int), h->stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->ustate, 0, U * sizeof(int2), h->stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->pos, 0xff, U * B * sizeof(int), h->stream);
    if (e == cudaSuccess && qbits) e = cudaMemsetAsync(h->kvs, 0, U * (size_t)h->Bp * sizeof(float2), h->stream);
    if (e == cudaSuccess && kind == kFG) {
        int4* init = static_cast<int4*>(malloc(U * sizeof(int4)));
        if (!init) { free_all(h); delete h; return fail(H2O_ERR_ALLOC, "host allocation failed"); }
        for (size_t u = 0; u < U; ++u) init[u] = make_int4(budget, heavy, recent, 1);
        e = cudaMemcpyAsync(h->upol, init, U * sizeof(int4), cudaMemcpyHostToDevice, h->stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(h->rec, 0, U * sizeof(double2), h->stream);
        // every unit on policy 1 until a prompt is profiled
        int* lists = static_cast<int*>(malloc((2 * U + 2) * sizeof(int)));
        if (!lists) { free(init); free_all(h); delete h; return fail(H2O_ERR_ALLOC, "host allocation failed"); }
        for (size_t u = 0; u < U; ++u) { lists[u] = (int)u; lists[U + u] = 0; }
        lists[2 * U] = (int)U;
        lists[2 * U + 1] = 0;
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(h->ulists, lists, (2 * U + 2) * sizeof(int), cudaMemcpyHostToDevice, h->stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
        free(lists);
        free(init);
    }
    if (e != cudaSuccess) { free_all(h); delete h; return cuda_fail(e, "initialise state"); }
    note_cache_write(h->device, h->stream, h);
    *out = h;
    return H2O_OK;
}

int ensure_prompt_scratch(h2o_ctx* h, int T)
{
    if (T <= h->T_cap) return H2O_OK;
    // the old buffers may still be read by queued work
    cudaError_t e = cudaStreamSynchronize(h->stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    free_prompt(h);
    const size_t n = (size_t)h->U * (size_t)T, nq = n * (size_t)h->G;
    int rc;
    if (h->kind == kFG) {
        if ((rc = dev_alloc((void**)&h->m2, n * sizeof(float), "row max")) ||
            (rc = dev_alloc((void**)&h->l, (2 * n + 4) * sizeof(float), "row normaliser and bias")) ||
            (rc = dev_alloc((void**)&h->c, n * sizeof(double), "column sums")) ||
            (rc = dev_alloc((void**)&h->bandB, n * sizeof(double), "band sums (budget)")) ||
            (rc = dev_alloc((void**)&h->bandr, n * sizeof(double), "band sums (window)"))) {
            free_prompt(h); return rc;
        }
    } else if (h->kind == kH2O) {
        if ((rc = dev_alloc((void**)&h->m2, nq * sizeof(float), "row max")) ||
            (rc = dev_alloc((void**)&h->l, (2 * nq + 4) * sizeof(float), "row normaliser and bias")) ||
            (rc = dev_alloc((void**)&h->c, nq * sizeof(double), "column sums"))) {
            free_prompt(h); return rc;
        }
        if (h->G > 1 && (rc = dev_alloc((void**)&h->ckv, n * sizeof(double), "cache unit column sums"))) {
            free_prompt(h); return rc;
        }
    } else if (h->kind == kSH) {
        if ((rc = dev_alloc((void**)&h->m2, n * sizeof(float), "row max")) ||
            (rc = dev_alloc((void**)&h->l, n * sizeof(float), "row normaliser")) ||
            (rc = dev_alloc((void**)&h->c, n * sizeof(double), "selection keys")) ||
            (rc = dev_alloc((void**)&h->ck, n * sizeof(uint32_t), "prompt histories"))) {
            free_prompt(h); return rc;
        }
    } else {
        if ((rc = dev_alloc((void**)&h->cq, n * sizeof(uint32_t), "query codes")) ||
            (rc = dev_alloc((void**)&h->ck, n * sizeof(uint32_t), "key codes"))) {
            free_prompt(h); return rc;
        }
    }
    // the row biases follow the normalisers in the same allocation, from a
    // 16-byte boundary (the persistence-of-importance and hashing handles
    // have no second pass)
    const size_t nl = (h->kind == kFG) ? n : nq;
    h->nb = (h->kind == kFG || h->kind == kH2O) ? h->l + ((nl + 3) & ~(size_t)3) : nullptr;
    h->T_cap = T;
    return H2O_OK;
}

int check_prompt(h2o_ctx* h, int kind, const void* Q, const void* K, const void* V, int T)
{
    if (!h) return fail(H2O_ERR_ARG, "handle is NULL");
    if (h->kind != kind)
        return fail(H2O_ERR_STATE, "%s called on a %s handle",
                    kind == kH2O ? "h2o_prefill" : kind == kLSH ? "lsh_prefill" : kind == kSH ? "sh_prefill" : "fg_prefill",
                    kind_name(h->kind));
    if (!Q || !K || !V) return fail(H2O_ERR_ARG, "Q, K and V must be non-NULL");
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V)) return fail(H2O_ERR_ARG, "Q, K, V must be 16-byte aligned");
    if (T < 1) return fail(H2O_ERR_ARG, "prompt length must be >= 1 (got %d)", T);
    if ((long long)T * h->U * h->G > (1LL << 31) / 4) return fail(H2O_ERR_ARG, "prompt too long for this batch");
    if ((kind == kH2O || kind == kSH || kind == kFG) && T >= (1 << 24)) return fail(H2O_ERR_ARG, "prompt too long");
    return H2O_OK;
}

int check_step(h2o_ctx* h, int kind, const void* q, const void* k, const void* v, const float* out)
{
    if (!h) return fail(H2O_ERR_ARG, "handle is NULL");
    if (h->kind != kind)
        return fail(H2O_ERR_STATE, "%s called on a %s handle",
                    kind == kH2O ? "h2o_decode_step" : kind == kLSH ? "lsh_decode_step"
                                     : kind == kSH ? "sh_decode_step" : "fg_decode_step",
                    kind_name(h->kind));
    if (!h->ready) return fail(H2O_ERR_STATE, "decode before prefill");
    if (!q || !k || !v || !out) return fail(H2O_ERR_ARG, "q, k, v and out must be non-NULL");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return fail(H2O_ERR_ARG, "q, k, v, out must be 16-byte aligned");
    return H2O_OK;
}

int decode_split(const h2o_ctx* h)
{
    int s;
    if (h->split > 0)
        s = h->split;
    else if (h->dtype == H2O_BF16 && h->D == 128 && h->G == 1 && (h->kind == kH2O || h->kind == kLSH) &&
             h->U < h->num_sms)
        s = few_units_split(h->U, h->B, h->num_sms, h->kind == kLSH, h->qbits);
    else
        s = auto_decode_split(h->U, h->B, h->num_sms);
    const int lo = (h->B + 1023) / 1024;
    if (s < lo) s = lo;
    if (s > max_decode_split()) s = max_decode_split();
    return s;
}

}  // namespace

extern "C" {

int h2o_init(h2o_handle* out, int budget, int heavy, int recent, int batch, int heads, int head_dim,
             int dtype, double scale, void* cuda_stream)
{
    return create(out, kH2O, budget, heavy, recent, batch, heads, head_dim, dtype, scale, nullptr, cuda_stream);
}

int h2o_init_gqa(h2o_handle* out, int budget, int heavy, int recent, int batch, int kv_heads, int groups,
                 int head_dim, int dtype, double scale, void* cuda_stream)
{
    return create(out, kH2O, budget, heavy, recent, batch, kv_heads, head_dim, dtype, scale, nullptr, cuda_stream,
                  groups);
}

int sh_init(h2o_handle* out, int budget, int heavy, int recent, int batch, int heads, int head_dim, int dtype,
            double scale, void* cuda_stream)
{
    return create(out, kSH, budget, heavy, recent, batch, heads, head_dim, dtype, scale, nullptr, cuda_stream);
}

int lsh_init(h2o_handle* out, int budget, int recent, int batch, int heads, int head_dim, int dtype,
             double scale, const float* W, void* cuda_stream)
{
    return create(out, kLSH, budget, budget - recent, recent, batch, heads, head_dim, dtype, scale, W,
                  cuda_stream);
}

int h2o_prefill(h2o_handle h, const void* Q, const void* K, const void* V, int T)
{
    int rc = check_prompt(h, kH2O, Q, K, V, T);
    if (rc) return rc;
    if ((rc = ensure_prompt_scratch(h, T))) return rc;
    if (inject("launch")) return fail(H2O_ERR_CUDA, "kernel launch failed (injected)");
    CacheView cv = view(h);
    PromptArgs pa = {};
    pa.Q = Q; pa.K = K; pa.V = V; pa.T = T; pa.H = h->H;
    pa.m2 = h->m2; pa.l = h->l; pa.nb = h->nb; pa.c = h->c; pa.G = h->G;
    note_cache_write(h->device, h->stream, h);
    cudaError_t e;
    if (h->G > 1) {
        // column sums per query head, then per cache unit
        CacheView qv = cv;
        qv.U = h->U * h->G;
        e = launch_prompt_stats(qv, pa, h->stream);
        if (e == cudaSuccess) e = launch_group_sum(h->c, h->ckv, h->U, h->G, T, h->stream);
        pa.c = h->ckv;
    } else {
        e = launch_prompt_stats(cv, pa, h->stream);
    }
    if (e == cudaSuccess) e = launch_select_gather(cv, pa, h->stream);
    if (e != cudaSuccess) return cuda_fail(e, "h2o_prefill launch");
    h->last_T = T;
    h->ready = 1;
    return H2O_OK;
}

int lsh_prefill(h2o_handle h, const void* Q, const void* K, const void* V, int T)
{
    int rc = check_prompt(h, kLSH, Q, K, V, T);
    if (rc) return rc;
    if ((rc = ensure_prompt_scratch(h, T))) return rc;
    if (inject("launch")) return fail(H2O_ERR_CUDA, "kernel launch failed (injected)");
    CacheView cv = view(h);
    PromptArgs pa = {};
    pa.Q = Q; pa.K = K; pa.V = V; pa.T = T;
    pa.cq = h->cq; pa.ck = h->ck;
    note_cache_write(h->device, h->stream, h);
    cudaError_t e = launch_lsh_prompt(cv, pa, h->W, h->W_host, h->stream);
    if (e != cudaSuccess) return cuda_fail(e, "lsh_prefill launch");
    h->last_T = T;
    h->ready = 1;
    return H2O_OK;
}

int sh_prefill(h2o_handle h, const void* Q, const void* K, const void* V, int T)
{
    int rc = check_prompt(h, kSH, Q, K, V, T);
    if (rc) return rc;
    if ((rc = ensure_prompt_scratch(h, T))) return rc;
    if (inject("launch")) return fail(H2O_ERR_CUDA, "kernel launch failed (injected)");
    CacheView cv = view(h);
    PromptArgs pa = {};
    pa.Q = Q; pa.K = K; pa.V = V; pa.T = T; pa.H = h->H;
    pa.c = h->c; pa.ck = h->ck; pa.m2 = h->m2; pa.l = h->l;
    note_cache_write(h->device, h->stream, h);
    cudaError_t e = launch_sh_prompt(cv, pa, h->stream);
    if (e != cudaSuccess) return cuda_fail(e, "sh_prefill launch");
    h->last_T = T;
    h->ready = 1;
    return H2O_OK;
}

int sh_decode_step(h2o_handle h, const void* q, const void* k, const void* v, float* out, int* victim_out)
{
    int rc = check_step(h, kSH, q, k, v, out);
    if (rc) return rc;
    if (inject("launch")) return fail(H2O_ERR_CUDA, "kernel launch failed (injected)");
    DecodeArgs a = {};
    a.c = view(h); a.q = q; a.k = k; a.v = v; a.out = out; a.victim_out = victim_out;
    a.early = note_cache_write(h->device, h->stream, h) ? 1 : 0;
    a.num_sms = h->num_sms;
    cudaError_t e = launch_sh_decode(a, decode_split(h), h->stream);
    if (e != cudaSuccess) return cuda_fail(e, "sh_decode_step launch");
    return H2O_OK;
}

int h2o_decode_step(h2o_handle h, const void* q, const void* k, const void* v, float* out, int* victim_out)
{
    int rc = check_step(h, kH2O, q, k, v, out);
    if (rc) return rc;
    if (inject("launch")) return fail(H2O_ERR_CUDA, "kernel launch failed (injected)");
    DecodeArgs a = {};
    a.c = view(h); a.q = q; a.k = k; a.v = v; a.out = out; a.victim_out = victim_out; a.G = h->G;
    a.early = note_cache_write(h->device, h->stream, h) ? 1 : 0;
    a.num_sms = h->num_sms;
    cudaError_t e = launch_h2o_decode(a, decode_split(h), h->stream);
    if (e != cudaSuccess) return cuda_fail(e, "h2o_decode_step launch");
    return H2O_OK;
}

int lsh_decode_step(h2o_handle h, const void* q, const void* k, const void* v, float* out, int* victim_out)
{
    int rc = check_step(h, kLSH, q, k, v, out);
    if (rc) return rc;
    if (inject("launch")) return fail(H2O_ERR_CUDA, "kernel launch failed (injected)");
    DecodeArgs a = {};
    a.c = view(h); a.q = q; a.k = k; a.v = v; a.out = out; a.victim_out = victim_out; a.W = h->W;
    a.early = note_cache_write(h->device, h->stream, h) ? 1 : 0;
    a.num_sms = h->num_sms;
    cudaError_t e = launch_lsh_decode(a, decode_split(h), h->stream);
    if (e != cudaSuccess) return cuda_fail(e, "lsh_decode_step launch");
    return H2O_OK;
}

int fg_init(h2o_handle* out, int budget, int heavy, int recent, int full_budget, double tau, int batch, int heads,
            int head_dim, int dtype, double scale, void* cuda_stream)
{
    return create(out, kFG, budget, heavy, recent, batch, heads, head_dim, dtype, scale, nullptr, cuda_stream, 1,
                  full_budget, tau);
}

int fg_prefill(h2o_handle h, const void* Q, const void* K, const void* V, int T)
{
    int rc = check_prompt(h, kFG, Q, K, V, T);
    if (rc) return rc;
    if ((rc = ensure_prompt_scratch(h, T))) return rc;
    if (inject("launch")) return fail(H2O_ERR_CUDA, "kernel launch failed (injected)");
    CacheView cv = view(h);
    PromptArgs pa = {};
    pa.Q = Q; pa.K = K; pa.V = V; pa.T = T; pa.H = h->H; pa.G = 1;
    pa.m2 = h->m2; pa.l = h->l; pa.nb = h->nb; pa.c = h->c;
    pa.budget = h->B_sel;
    pa.bandB = h->bandB; pa.bandr = h->bandr; pa.wB = h->B_sel; pa.wr = h->r;
    FgArgs fa = {};
    fa.upol = h->upol; fa.rec = h->rec; fa.tau = h->tau;
    fa.B = h->B_sel; fa.H = h->H; fa.r = h->r; fa.B_full = h->B_full;
    note_cache_write(h->device, h->stream, h);
    cudaError_t e = launch_prompt_stats(cv, pa, h->stream);
    if (e == cudaSuccess) e = launch_select(cv, pa, h->stream);
    if (e == cudaSuccess) e = launch_fg_policy(cv, pa, fa, h->stream);
    if (e == cudaSuccess) e = launch_fg_lists(h->upol, h->U, h->ulists, h->ulists + 2 * h->U, h->stream);
    if (e == cudaSuccess) e = launch_gather(cv, pa, false, h->stream);
    if (e != cudaSuccess) return cuda_fail(e, "fg_prefill launch");
    h->last_T = T;
    h->ready = 1;
    return H2O_OK;
}

int fg_decode_step(h2o_handle h, const void* q, const void* k, const void* v, float* out, int* victim_out)
{
    int rc = check_step(h, kFG, q, k, v, out);
    if (rc) return rc;
    if (inject("launch")) return fail(H2O_ERR_CUDA, "kernel launch failed (injected)");
    // two launches over the units' lists: the compressed policies (budget
    // B_sel) with their own split, then the full caches (B_full) with theirs;
    // a unit's CTAs exist in one of them only, so the second may read its
    // units' caches while the first drains
    DecodeArgs a = {};
    a.c = view(h); a.q = q; a.k = k; a.v = v; a.out = out; a.victim_out = victim_out; a.G = 1;
    a.early = note_cache_write(h->device, h->stream, h) ? 1 : 0;
    a.num_sms = h->num_sms;
    const int* counts = h->ulists + 2 * h->U;
    int s_small = h->split > 0 ? h->split : auto_decode_split(h->U, h->B_sel, h->num_sms);
    int s_full = h->split > 0 ? h->split : auto_decode_split(h->U, h->B_full, h->num_sms);
    s_small = std::max(s_small, (h->B_sel + 1023) / 1024);
    s_full = std::max(s_full, (h->B_full + 1023) / 1024);
    s_small = std::min(s_small, max_decode_split());
    s_full = std::min(s_full, max_decode_split());
    a.ulist = h->ulists;
    a.ucount = counts;
    cudaError_t e = launch_h2o_decode(a, s_small, h->stream);
    if (e == cudaSuccess) {
        a.ulist = h->ulists + h->U;
        a.ucount = counts + 1;
        a.early = 1;
        e = launch_h2o_decode(a, s_full, h->stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "fg_decode_step launch");
    return H2O_OK;
}

int fg_get_policy(h2o_handle h, int* policy, double* rec_local, double* rec_freq)
{
    if (!h) return fail(H2O_ERR_ARG, "handle is NULL");
    if (h->kind != kFG) return fail(H2O_ERR_STATE, "fg_get_policy called on a %s handle", kind_name(h->kind));
    const size_t U = (size_t)h->U;
    int4* pp = static_cast<int4*>(malloc(U * sizeof(int4)));
    double2* rr = static_cast<double2*>(malloc(U * sizeof(double2)));
    if (!pp || !rr) { free(pp); free(rr); return fail(H2O_ERR_ALLOC, "host allocation failed"); }
    cudaError_t e = cudaMemcpyAsync(pp, h->upol, U * sizeof(int4), cudaMemcpyDeviceToHost, h->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(rr, h->rec, U * sizeof(double2), cudaMemcpyDeviceToHost, h->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
    if (e == cudaSuccess) {
        for (size_t u = 0; u < U; ++u) {
            if (policy) policy[u] = pp[u].w;
            if (rec_local) rec_local[u] = rr[u].x;
            if (rec_freq) rec_freq[u] = rr[u].y;
        }
    }
    free(pp);
    free(rr);
    if (e != cudaSuccess) return cuda_fail(e, "fg_get_policy");
    return H2O_OK;
}

int h2o_get_state(h2o_handle h, void* K, void* V, double* score, int* pos, unsigned* code, int* occupancy,
                  int* next_pos)
{
    if (!h) return fail(H2O_ERR_ARG, "handle is NULL");
    const size_t UB = (size_t)h->U * h->B, row = row_bytes(h);
    cudaError_t e = cudaSuccess;
    if (K && e == cudaSuccess) e = cudaMemcpyAsync(K, h->K, UB * row, cudaMemcpyDeviceToHost, h->stream);
    if (V && e == cudaSuccess) e = cudaMemcpyAsync(V, h->V, UB * row, cudaMemcpyDeviceToHost, h->stream);
    if (pos && e == cudaSuccess) e = cudaMemcpyAsync(pos, h->pos, UB * sizeof(int), cudaMemcpyDeviceToHost, h->stream);
    float2* pairs = nullptr;
    if (score && e == cudaSuccess) {
        if (h->score) {
            pairs = static_cast<float2*>(malloc(UB * sizeof(float2)));
            if (!pairs) return fail(H2O_ERR_ALLOC, "host allocation failed");
            e = cudaMemcpyAsync(pairs, h->score, UB * sizeof(float2), cudaMemcpyDeviceToHost, h->stream);
        } else {
            memset(score, 0, UB * sizeof(double));
        }
    }
    if (code && e == cudaSuccess) {
        if (h->code) e = cudaMemcpyAsync(code, h->code, UB * sizeof(uint32_t), cudaMemcpyDeviceToHost, h->stream);
        else memset(code, 0, UB * sizeof(uint32_t));
    }
    int2* us = nullptr;
    if ((occupancy || next_pos) && e == cudaSuccess) {
        us = static_cast<int2*>(malloc((size_t)h->U * sizeof(int2)));
        if (!us) return fail(H2O_ERR_ALLOC, "host allocation failed");
        e = cudaMemcpyAsync(us, h->ustate, (size_t)h->U * sizeof(int2), cudaMemcpyDeviceToHost, h->stream);
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
    if (e == cudaSuccess && us) {
        for (int u = 0; u < h->U; ++u) {
            if (occupancy) occupancy[u] = us[u].x;
            if (next_pos) next_pos[u] = us[u].y;
        }
    }
    if (e == cudaSuccess && pairs)
        for (size_t i = 0; i < UB; ++i) score[i] = (double)pairs[i].x + (double)pairs[i].y;
    free(us);
    free(pairs);
    if (e != cudaSuccess) return cuda_fail(e, "h2o_get_state");
    return H2O_OK;
}

int h2o_set_state(h2o_handle h, const void* K, const void* V, const double* score, const int* pos,
                  const unsigned* code, const int* occupancy, const int* next_pos)
{
    if (!h) return fail(H2O_ERR_ARG, "handle is NULL");
    const size_t UB = (size_t)h->U * h->B, row = row_bytes(h);
    if (occupancy)
        for (int u = 0; u < h->U; ++u)
            if (occupancy[u] < 0 || occupancy[u] > h->B) return fail(H2O_ERR_ARG, "occupancy out of range");
    cudaError_t e = cudaStreamSynchronize(h->stream);
    note_cache_write(h->device, h->stream, h);
    if (K && e == cudaSuccess) e = cudaMemcpyAsync(h->K, K, UB * row, cudaMemcpyHostToDevice, h->stream);
    if (V && e == cudaSuccess) e = cudaMemcpyAsync(h->V, V, UB * row, cudaMemcpyHostToDevice, h->stream);
    if (pos && e == cudaSuccess) e = cudaMemcpyAsync(h->pos, pos, UB * sizeof(int), cudaMemcpyHostToDevice, h->stream);
    float2* pairs = nullptr;
    if (score && h->score && e == cudaSuccess) {
        pairs = static_cast<float2*>(malloc(UB * sizeof(float2)));
        if (!pairs) return fail(H2O_ERR_ALLOC, "host allocation failed");
        for (size_t i = 0; i < UB; ++i) {
            const float hi = (float)score[i];
            pairs[i] = make_float2(hi, (float)(score[i] - (double)hi));
        }
        e = cudaMemcpyAsync(h->score, pairs, UB * sizeof(float2), cudaMemcpyHostToDevice, h->stream);
    }
    if (code && h->code && e == cudaSuccess)
        e = cudaMemcpyAsync(h->code, code, UB * sizeof(uint32_t), cudaMemcpyHostToDevice, h->stream);
    int2* us = nullptr;
    if ((occupancy || next_pos) && e == cudaSuccess) {
        us = static_cast<int2*>(malloc((size_t)h->U * sizeof(int2)));
        if (!us) return fail(H2O_ERR_ALLOC, "host allocation failed");
        e = cudaMemcpyAsync(us, h->ustate, (size_t)h->U * sizeof(int2), cudaMemcpyDeviceToHost, h->stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
        if (e == cudaSuccess) {
            for (int u = 0; u < h->U; ++u) {
                if (occupancy) us[u].x = occupancy[u];
                if (next_pos) us[u].y = next_pos[u];
            }
            e = cudaMemcpyAsync(h->ustate, us, (size_t)h->U * sizeof(int2), cudaMemcpyHostToDevice, h->stream);
        }
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
    free(us);
    free(pairs);
    if (e != cudaSuccess) return cuda_fail(e, "h2o_set_state");
    h->ready = 1;
    return H2O_OK;
}

int h2o_get_kv_scales(h2o_handle h, float* kscale, float* vscale)
{
    if (!h) return fail(H2O_ERR_ARG, "handle is NULL");
    if (!h->qbits) return fail(H2O_ERR_STATE, "the handle's cache is not quantised (H2O_KV8 or H2O_KV4)");
    const size_t n = (size_t)h->U * h->Bp;
    float2* s = static_cast<float2*>(malloc(n * sizeof(float2)));
    if (!s) return fail(H2O_ERR_ALLOC, "host allocation failed");
    cudaError_t e = cudaMemcpyAsync(s, h->kvs, n * sizeof(float2), cudaMemcpyDeviceToHost, h->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
    if (e == cudaSuccess) {
        for (int u = 0; u < h->U; ++u)
            for (int b = 0; b < h->B; ++b) {
                const float2 x = s[(size_t)u * h->Bp + b];
                if (kscale) kscale[(size_t)u * h->B + b] = x.x;
                if (vscale) vscale[(size_t)u * h->B + b] = x.y;
            }
    }
    free(s);
    if (e != cudaSuccess) return cuda_fail(e, "h2o_get_kv_scales");
    return H2O_OK;
}

int h2o_set_kv_scales(h2o_handle h, const float* kscale, const float* vscale)
{
    if (!h) return fail(H2O_ERR_ARG, "handle is NULL");
    if (!h->qbits) return fail(H2O_ERR_STATE, "the handle's cache is not quantised (H2O_KV8 or H2O_KV4)");
    if (!kscale || !vscale) return fail(H2O_ERR_ARG, "kscale and vscale must be non-NULL");
    const size_t n = (size_t)h->U * h->Bp;
    float2* s = static_cast<float2*>(calloc(n, sizeof(float2)));
    if (!s) return fail(H2O_ERR_ALLOC, "host allocation failed");
    for (int u = 0; u < h->U; ++u)
        for (int b = 0; b < h->B; ++b)
            s[(size_t)u * h->Bp + b] = make_float2(kscale[(size_t)u * h->B + b], vscale[(size_t)u * h->B + b]);
    cudaError_t e = cudaStreamSynchronize(h->stream);
    note_cache_write(h->device, h->stream, h);
    if (e == cudaSuccess) e = cudaMemcpyAsync(h->kvs, s, n * sizeof(float2), cudaMemcpyHostToDevice, h->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
    free(s);
    if (e != cudaSuccess) return cuda_fail(e, "h2o_set_kv_scales");
    return H2O_OK;
}

int h2o_get_prefill_stats(h2o_handle h, float* m, float* l, double* c)
{
    if (!h) return fail(H2O_ERR_ARG, "handle is NULL");
    if (h->kind != kH2O && h->kind != kFG)
        return fail(H2O_ERR_STATE, "prompt statistics exist only on H2O and per-head policy handles");
    if (!h->last_T) return fail(H2O_ERR_STATE, "no prompt has been processed");
    const size_t n = (size_t)h->U * h->last_T, nq = n * (size_t)h->G;
    const double* cu = h->G > 1 ? h->ckv : h->c;
    cudaError_t e = cudaSuccess;
    if (m) e = cudaMemcpyAsync(m, h->m2, nq * sizeof(float), cudaMemcpyDeviceToHost, h->stream);
    if (l && e == cudaSuccess) e = cudaMemcpyAsync(l, h->l, nq * sizeof(float), cudaMemcpyDeviceToHost, h->stream);
    if (c && e == cudaSuccess) e = cudaMemcpyAsync(c, cu, n * sizeof(double), cudaMemcpyDeviceToHost, h->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
    if (e != cudaSuccess) return cuda_fail(e, "h2o_get_prefill_stats");
    if (m)
        for (size_t i = 0; i < nq; ++i) m[i] = (float)((double)m[i] * 0.6931471805599453);
    return H2O_OK;
}

int h2o_set_stream(h2o_handle h, void* cuda_stream)
{
    if (!h) return fail(H2O_ERR_ARG, "handle is NULL");
    h->stream = reinterpret_cast<cudaStream_t>(cuda_stream);
    return H2O_OK;
}

int h2o_set_decode_split(h2o_handle h, int ctas_per_unit)
{
    if (!h) return fail(H2O_ERR_ARG, "handle is NULL");
    if (h->G > 1)
        return fail(H2O_ERR_STATE, "a grouped-query handle runs one CTA per query head; its split is not settable");
    if (ctas_per_unit < 0 || ctas_per_unit > max_decode_split())
        return fail(H2O_ERR_ARG, "ctas_per_unit must be in [0, %d]", max_decode_split());
    // per-head policies: the compressed policies' budget bounds the split;
    // the full caches' launch raises it to what their budget needs
    const int Bmin = h->kind == kFG ? h->B_sel : h->B;
    if (ctas_per_unit > 0 && ctas_per_unit < (Bmin + 1023) / 1024)
        return fail(H2O_ERR_ARG, "ctas_per_unit must be >= %d for budget %d", (Bmin + 1023) / 1024, Bmin);
    h->split = ctas_per_unit;
    return H2O_OK;
}

int h2o_sync(h2o_handle h)
{
    if (!h) return fail(H2O_ERR_ARG, "handle is NULL");
    cudaError_t e = cudaStreamSynchronize(h->stream);
    if (e != cudaSuccess) return cuda_fail(e, "h2o_sync");
    int word = 0;
    e = cudaMemcpy(&word, h->err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "h2o_sync read error word");
    if (word) {
        cudaMemset(h->err, 0, sizeof(int));
        return fail(H2O_ERR_DEVICE_TIMEOUT, "a kernel's bounded wait ran out (error word 0x%x)", word);
    }
    return H2O_OK;
}

int h2o_selftest_wait_timeout(h2o_handle h)
{
    if (!h) return fail(H2O_ERR_ARG, "handle is NULL");
    note_cache_write(h->device, h->stream, h);
    cudaError_t e = launch_wait_selftest(h->err, h->stream);
    if (e != cudaSuccess) return cuda_fail(e, "h2o_selftest_wait_timeout launch");
    return H2O_OK;
}

void h2o_destroy(h2o_handle h)
{
    if (!h) return;
    cudaStreamSynchronize(h->stream);
    forget_cache_writes(h);
    free_all(h);
    delete h;
}

const char* h2o_last_error(void) { return g_err; }

}  // extern "C"
