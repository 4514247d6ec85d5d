// noalloc.cu -- the prompt scorer without any device allocation.
//
// Some callers cannot call cudaMalloc: serving runtimes that reserve all
// device memory for their own pool at start-up and forbid allocations
// afterwards, and hosts whose allocation calls may synchronise the device in
// the middle of their own streams' work.  This entry point computes the
// same prompt column sums as h2o_prefill, with the scorer's scratch (per-row
// max, normaliser and bias, 12 bytes per unit per token) held in a fixed device
// array inside the library instead of memory it allocates.  The array
// occupies kNoallocTokens * 12 bytes (12 MiB) on every device that loads the
// library, until the process exits.  With no handle there is no error word
// to sync on: a scorer CTA whose bounded wait runs out writes NaN into the
// statistics it owns, so the failure shows in the column sums.
#include <mutex>

#include "h2o.h"
#include "kernels.h"

namespace {

constexpr long long kNoallocTokens = H2O_NOALLOC_MAX_TOKENS;

// row max (base-2 logits) in [0, kNoallocTokens), row normaliser after it,
// then the row bias of the scorer's second pass
static __device__ __align__(256) float g_noalloc_scratch[3 * kNoallocTokens];

std::mutex g_mu;
void* g_addr[64];   // device address of g_noalloc_scratch, per device

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int h2o_prompt_scores_noalloc(const void* Q, const void* K, int batch, int heads, int T,
                                         int head_dim, int dtype, double scale, double* c,
                                         void* cuda_stream)
{
    using namespace h2o;
    if (!Q || !K || !c) return set_last_error(H2O_ERR_ARG, "Q, K and c must be non-NULL");
    if (!aligned16(Q) || !aligned16(K) || !aligned16(c))
        return set_last_error(H2O_ERR_ARG, "Q, K and c must be 16-byte aligned");
    if (batch < 1 || heads < 1 || T < 1) return set_last_error(H2O_ERR_ARG, "batch, heads and T must be >= 1");
    if (head_dim != 64 && head_dim != 128)
        return set_last_error(H2O_ERR_ARG, "head_dim must be 64 or 128 (got %d)", head_dim);
    if (dtype != H2O_F32 && dtype != H2O_BF16) return set_last_error(H2O_ERR_ARG, "dtype must be H2O_F32 or H2O_BF16");
    if (!(scale > 0.0)) return set_last_error(H2O_ERR_ARG, "scale must be > 0");
    const long long tokens = (long long)batch * heads * T;
    if (tokens > kNoallocTokens)
        return set_last_error(H2O_ERR_ARG,
                              "batch * heads * T = %lld exceeds the fixed scratch of %lld unit-tokens",
                              tokens, kNoallocTokens);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_last_error(H2O_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return set_last_error(H2O_ERR_UNSUPPORTED, "device index %d out of range", dev);
    void* base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_addr[dev]) {
            // one-time set-up on this device (the device is current here)
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || !p)
                return set_last_error(H2O_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
            g_addr[dev] = p;
        }
        base = g_addr[dev];
    }
    CacheView cv = {};
    cv.U = batch * heads;
    cv.D = head_dim;
    cv.dtype = dtype;
    cv.qscale = (float)(scale * 1.4426950408889634);
    PromptArgs pa = {};
    pa.Q = Q;
    pa.K = K;
    pa.T = T;
    pa.m2 = static_cast<float*>(base);
    pa.l = static_cast<float*>(base) + kNoallocTokens;
    pa.nb = static_cast<float*>(base) + 2 * kNoallocTokens;
    pa.c = c;
    e = launch_prompt_stats(cv, pa, reinterpret_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) return set_last_error(H2O_ERR_CUDA, "h2o_prompt_scores_noalloc launch: %s", cudaGetErrorString(e));
    return H2O_OK;
}
