// decode_warp.cu -- the H2O decode step over many one-head units, one warp
// per unit.
//
// The step [H2O review page, 提案手法: attend over the live slots and the
// new token, add each slot's probability to its score, evict the
// lowest-score slot outside the recent window (lowest slot on ties), write
// the new token there] is the one decode.cu computes; only the parallel plan
// differs.
//
// With thousands of units, splitting one unit's stages over the warps of a
// CTA costs a CTA-wide merge, several CTA barriers and a per-warp copy of q
// for every unit, and leaves about two warps per scheduler.  Here every warp
// owns whole units: it streams all of a unit's 16-slot stages through its own
// ring of shared-memory buffers (1-D bulk copies on mbarriers), keeps the
// online softmax alone, then runs the score pass, the arg-min and the write
// of the new token itself.  The warps of a CTA never wait for one another,
// so a dozen independent warps per SM hide each other's latencies.  A warp
// takes units w, w + W, w + 2W, ... (W = warps in the grid) and its ring runs
// on from one unit into the next, so the next unit's rows are in flight while
// this unit's epilogue runs.  Every wait is bounded; a wait that runs out
// sets the handle's error word.
#include <algorithm>
#include <mutex>

#include "decode_common.cuh"

namespace h2o {

namespace {

constexpr int kWarpsPerCta = 4;

// One warp's private shared memory.
template <typename T, int D, int QB, int NBUF>
struct WarpSlice {
    CacheElem<T, QB> kbuf[NBUF][kStage * RowElems<D, QB>];
    CacheElem<T, QB> vbuf[NBUF][kStage * RowElems<D, QB>];
    alignas(16) float2 sbuf[QB ? NBUF : 1][kStage];     // quantised rows: {K scale, V scale} per slot
    alignas(16) unsigned char in[3][D * sizeof(T)];     // this unit's q, k, v rows
    alignas(16) float e[kStage];                        // a stage's weights
    alignas(16) unsigned char qpl[QB ? 3 * D : 16];     // quantised rows: byte planes of q
    uint64_t bar[NBUF];
};

// Stage buffers per warp: about as many bytes in flight per warp for every
// row form.
template <int QB>
constexpr int warp_nbuf() { return QB == 4 ? 4 : QB == 8 ? 3 : 2; }

// Slots each warp keeps logits for, rounded to 16 bytes.
__host__ __device__ inline int z_stride(int B) { return (B + 3) & ~3; }

template <typename T, int D, int QB, int NBUF>
size_t warp_smem_bytes(int B)
{
    return kWarpsPerCta * (sizeof(WarpSlice<T, D, QB, NBUF>) + (size_t)z_stride(B) * sizeof(float));
}

// The new token's row (at src, in shared memory) into cache row dst: lanes
// below NV = D * sizeof(T) / 16 take one 16-byte piece each; a quantised row
// gets its scale from the max magnitude over those lanes.
template <int QB, typename T, int D>
__device__ __forceinline__ void store_row_warp(const unsigned char* src, CacheElem<T, QB>* dst, float* scale_dst,
                                               int lane)
{
    constexpr int NV = D * (int)sizeof(T) / 16, VE = 16 / (int)sizeof(T);
    static_assert(NV <= 32 && (NV & (NV - 1)) == 0, "a row's pieces fit one warp");
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (lane < NV) w = reinterpret_cast<const uint4*>(src)[lane];
    if constexpr (QB == 0) {
        if (lane < NV) reinterpret_cast<uint4*>(dst)[lane] = w;
    } else {
        float x[VE];
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (sizeof(T) == 2) {
                x[2 * i] = __uint_as_float(u[i] << 16);
                x[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
            } else {
                x[i] = __uint_as_float(u[i]);
            }
        }
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < VE; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
        for (int o = NV / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
        if constexpr (QB == 8) {
            const float inv = q8_inv(amax);
            if (lane < NV) {
                int8_t* d8 = reinterpret_cast<int8_t*>(dst) + lane * VE;
                if constexpr (VE == 8) *reinterpret_cast<uint2*>(d8) = make_uint2(q8_pack4(&x[0], inv), q8_pack4(&x[4], inv));
                else *reinterpret_cast<uint32_t*>(d8) = q8_pack4(&x[0], inv);
            }
            if (lane == 0) *scale_dst = q8_scale(amax);
        } else {
            const float inv = q4_inv(amax);
            if (lane < NV) {
                uint8_t* d4 = reinterpret_cast<uint8_t*>(dst) + lane * (VE / 2);
                if constexpr (VE == 8) *reinterpret_cast<uint32_t*>(d4) = q4_pack<4>(x, inv);
                else *reinterpret_cast<uint16_t*>(d4) = (uint16_t)q4_pack<2>(x, inv);
            }
            if (lane == 0) *scale_dst = q4_scale(amax);
        }
    }
}

template <typename T, int D, int QB, int NBUF, int MINB>
__global__ void __launch_bounds__(32 * kWarpsPerCta, MINB) h2o_warp_kernel(const DecodeArgs a)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    using Slice = WarpSlice<T, D, QB, NBUF>;
    using CE = CacheElem<T, QB>;
    constexpr int EPL = D / 32;
    constexpr int NV = D * (int)sizeof(T) / 16;                  // 16-byte pieces per row
    constexpr int RE = RowElems<D, QB>;
    constexpr int PL = (3 * NV + 31) / 32;                       // q, k, v pieces per lane
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const CacheView& c = a.c;
    const int B = c.B, U = c.U;
    Slice& W = reinterpret_cast<Slice*>(smem_raw)[warp];
    float* z = reinterpret_cast<float*>(smem_raw + kWarpsPerCta * sizeof(Slice)) + warp * z_stride(B);
    const int GW = (int)gridDim.x * kWarpsPerCta;                // warps in the grid
    const int w0 = (int)blockIdx.x * kWarpsPerCta + warp;        // this warp's first unit
    const int nst = (B + kStage - 1) / kStage;                   // stages of a unit

    // ring item k: stage k % nst of this warp's unit k / nst, into buffer
    // k % NBUF (nothing past the last unit)
    auto issue_item = [&](int k) {
        const int j = k / nst;
        const int u = w0 + j * GW;
        if (u >= U) return;
        const size_t ub = (size_t)u * B;
        const int s = (k - j * nst) * kStage;
        const int b = k % NBUF;
        const int rows = min(kStage, B - s);
        const uint32_t bytes = (uint32_t)(rows * RE * sizeof(CE));
        const uint32_t sbytes = QB ? (uint32_t)(((rows + 1) & ~1) * sizeof(float2)) : 0u;
        mbar_arrive_expect_tx(&W.bar[b], 2 * bytes + sbytes);
        bulk_g2s(W.kbuf[b], reinterpret_cast<const CE*>(c.K) + (ub + s) * RE, bytes, &W.bar[b]);
        bulk_g2s(W.vbuf[b], reinterpret_cast<const CE*>(c.V) + (ub + s) * RE, bytes, &W.bar[b]);
        if constexpr (QB != 0) bulk_g2s(W.sbuf[b], c.kvs + (size_t)u * c.Bp + s, sbytes, &W.bar[b]);
    };
    if (lane == 0) {
#pragma unroll
        for (int b = 0; b < NBUF; ++b) mbar_init(&W.bar[b], 1);
        fence_proxy_async_smem();
    }
    __syncwarp();
    auto prime = [&]() {
        if (lane == 0)
            for (int k = 0; k < NBUF; ++k) issue_item(k);
    };
    // a unit's q, k, v rows as 16-byte pieces, PL per lane
    auto load_rows = [&](int u, uint4 (&w)[PL]) {
#pragma unroll
        for (int i = 0; i < PL; ++i) {
            const int t = lane + 32 * i;
            w[i] = make_uint4(0u, 0u, 0u, 0u);
            if (t < 3 * NV) {
                const int r = t / NV;
                const T* row = reinterpret_cast<const T*>(r == 0 ? a.q : r == 1 ? a.k : a.v) + (size_t)u * D;
                w[i] = reinterpret_cast<const uint4*>(row)[t - r * NV];
            }
        }
    };
    auto store_rows = [&](const uint4 (&w)[PL]) {
#pragma unroll
        for (int i = 0; i < PL; ++i) {
            const int t = lane + 32 * i;
            if (t < 3 * NV) reinterpret_cast<uint4*>(W.in[t / NV])[t % NV] = w[i];
        }
    };

    // the cache of this handle may be read before the dependency wait when
    // the previous kernel in the stream cannot have written it
    if (a.early) prime();
    grid_dependency_wait();
    grid_launch_dependents();
    if (w0 >= U) return;
    if (!a.early) prime();
    int2 us = c.ustate[w0];
    {
        uint4 w[PL];
        load_rows(w0, w);
        store_rows(w);
    }
    __syncwarp();

    bool timed_out = false;
    int k_it = 0;                                                // this warp's next ring item
    for (int u = w0; u < U; u += GW) {
        const size_t ub = (size_t)u * B;
        const int n = us.x, p = us.y;
        const bool full = (n >= B);
        // this unit's scores and positions, wanted after the stages, on
        // their way to L2 meanwhile
        for (int s = lane * 16; s < n; s += 32 * 16)           // 16 score pairs per 128-byte line
            asm volatile("prefetch.global.L2 [%0];" ::"l"(c.score + ub + s));
        for (int s = lane * 32; s < n; s += 32 * 32)           // 32 positions per line
            asm volatile("prefetch.global.L2 [%0];" ::"l"(c.pos + ub + s));
        const T* qs = reinterpret_cast<const T*>(W.in[0]);
        const T* ks = reinterpret_cast<const T*>(W.in[1]);
        const T* vs = reinterpret_cast<const T*>(W.in[2]);
        QVec<T, D, QB> qv;
        load_qvec<QB, T, D>(qs, c.qscale, lane, QB ? W.qpl : nullptr, qv);
        // the new token attends to itself
        const float zn = new_logit<QB, T, D>(qs, ks, c.qscale, qv, lane);
        float m_run = zn, l_run = lane == 0 ? 1.f : 0.f, o[EPL], o2[EPL];
        load_vec<T, EPL>(vs + lane * EPL, o);
#pragma unroll
        for (int e = 0; e < EPL; ++e) o2[e] = 0.f;

        // every stage of the unit; each consumed buffer is refilled with the
        // item NBUF ahead, which runs into the next units
        for (int g = 0; g < nst; ++g, ++k_it) {
            const int b = k_it % NBUF;
            if (!mbar_wait(&W.bar[b], (uint32_t)(k_it / NBUF) & 1u)) {
                if (!timed_out && lane == 0) atomicOr(c.err, kErrWaitTimeout);
                timed_out = true;
            }
            const int gl = max(0, min(kStage, n - g * kStage));
            if (gl > 0)
                attend_rows<T, D, QB>(W.kbuf[b], W.vbuf[b], QB ? W.sbuf[b] : nullptr, W.e, z + g * kStage, gl, -1,
                                      qv, m_run, l_run, o, o2);
            __syncwarp();                                        // every lane is past the wait and the buffer
            if (lane == 0) issue_item(k_it + NBUF);
        }
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] += o2[e];

        // the next unit's rows and occupancy, requested before the epilogue
        const int un = u + GW;
        uint4 wn[PL];
        int2 us_next = make_int2(0, 0);
        if (un < U) {
            load_rows(un, wn);
            us_next = c.ustate[un];
        }

        const float M = m_run;
        const float invL = 1.f / warp_sum(l_run);
        {
            float* dst = a.out + (size_t)u * D + lane * EPL;
#pragma unroll
            for (int e = 0; e < EPL; ++e) dst[e] = o[e] * invL;
        }
        const float P_new = ex2_approx(zn - M) * invL;

        // accumulate this step's probabilities; arg-min over candidates
        // (slots whose position is at most p - r)
        ArgMin best = argmin_none();
        const int c1 = min(n, B);
        for (int s0 = 0; s0 < c1; s0 += 4 * 32) {
            float2 so[4];
            int po[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int s = s0 + 32 * t + lane;
                so[t] = make_float2(0.f, 0.f);
                po[t] = 0;
                if (s < c1) {
                    so[t] = c.score[ub + s];
                    po[t] = c.pos[ub + s];
                }
            }
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int s = s0 + 32 * t + lane;
                if (s < c1) {
                    const float Pr = ex2_approx(z[s] - M) * invL;
                    const float2 ns = pair_add(so[t], Pr);
                    c.score[ub + s] = ns;
                    if (full && po[t] <= p - c.r) argmin_take(best, ArgMin{ord_key(ns.x), ord_key(ns.y), (unsigned)s});
                }
            }
        }
        int victim = n;
        if (full) {
            best = warp_argmin(best);
            if (best.slot == 0xffffffffu) {
                // no candidate (possible only for loaded states): every live
                // slot competes, its new score re-read (written above by
                // this warp)
                __syncwarp();
                ArgMin al = argmin_none();
                for (int s = lane; s < n; s += 32) {
                    const float2 sc = c.score[ub + s];
                    argmin_take(al, ArgMin{ord_key(sc.x), ord_key(sc.y), (unsigned)s});
                }
                best = warp_argmin(al);
            }
            victim = (int)best.slot;
        }
        if (victim < 0 || victim >= B) victim = 0;            // n == 0 with B == 0 cannot happen
        __syncwarp();
        if (lane == 0) {
            c.score[ub + victim] = make_float2(P_new, 0.f);
            c.pos[ub + victim] = p;
            c.ustate[u] = make_int2(min(n + 1, B), p + 1);
            if (a.victim_out) a.victim_out[u] = full ? victim : -1;
        }
        float2* sc_pair = QB ? c.kvs + (size_t)u * c.Bp + victim : nullptr;
        store_row_warp<QB, T, D>(W.in[1], reinterpret_cast<CE*>(c.K) + (ub + victim) * RE,
                                 QB ? reinterpret_cast<float*>(sc_pair) : nullptr, lane);
        store_row_warp<QB, T, D>(W.in[2], reinterpret_cast<CE*>(c.V) + (ub + victim) * RE,
                                 QB ? reinterpret_cast<float*>(sc_pair) + 1 : nullptr, lane);

        us = us_next;
        __syncwarp();                                            // W.in and z are free again
        if (un < U) store_rows(wn);
        __syncwarp();
    }
}

// Resident CTAs per SM for budget B (0 on error), cached per device and B.
template <typename T, int D, int QB, int NBUF, int MINB>
int warp_ctas_per_sm(int dev, int B)
{
    struct Entry { int dev, B, n; };
    static Entry cache[32];
    static int n_cache = 0;
    static std::mutex mu;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < n_cache; ++i)
            if (cache[i].dev == dev && cache[i].B == B) return cache[i].n;
    }
    void (*kern)(const DecodeArgs) = h2o_warp_kernel<T, D, QB, NBUF, MINB>;
    const size_t smem = warp_smem_bytes<T, D, QB, NBUF>(B);
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 32 * kWarpsPerCta, smem) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (n_cache < 32) cache[n_cache++] = Entry{dev, B, n};
    return n;
}

template <typename T, int D, int QB>
cudaError_t launch_warp_t(const DecodeArgs& a, cudaStream_t st)
{
    constexpr int NBUF = warp_nbuf<QB>();
    constexpr int MINB = 3;                     // 12 warps per SM (16 measured slower for 4-bit rows)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int per_sm = warp_ctas_per_sm<T, D, QB, NBUF, MINB>(dev, a.c.B);
    if (per_sm <= 0) return cudaErrorInvalidConfiguration;
    const long long need = (a.c.U + kWarpsPerCta - 1) / kWarpsPerCta;
    const long long grid = std::min<long long>(need, (long long)per_sm * a.num_sms);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(32 * kWarpsPerCta, 1, 1);
    cfg.dynamicSmemBytes = warp_smem_bytes<T, D, QB, NBUF>(a.c.B);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, h2o_warp_kernel<T, D, QB, NBUF, MINB>, a);
}

template <int QB>
cudaError_t warp_form(const DecodeArgs& a, cudaStream_t st)
{
    const bool bf = a.c.dtype == 1;
    if (a.c.D == 128)
        return bf ? launch_warp_t<__nv_bfloat16, 128, QB>(a, st) : launch_warp_t<float, 128, QB>(a, st);
    if (a.c.D == 64)
        return bf ? launch_warp_t<__nv_bfloat16, 64, QB>(a, st) : launch_warp_t<float, 64, QB>(a, st);
    return cudaErrorInvalidValue;
}

// Units from which the warp-per-unit kernel runs, H2O_WARP_UNITS to override
// (for comparisons): by default eight per SM, which keeps about eight
// independent warps on every SM.
long long warp_units_min(int num_sms)
{
    static long long v = -2;
    if (v == -2) {
        const char* e = getenv("H2O_WARP_UNITS");
        v = e ? atoll(e) : -1;
    }
    return v >= 0 ? v : 8LL * num_sms;
}

}  // namespace

cudaError_t launch_h2o_decode_warps(const DecodeArgs& a, cudaStream_t st, bool* used)
{
    *used = false;
    // one-head caches with the cache's own budget; a unit's logits fit the
    // warp's buffer (one CTA's limit); fp32 rows of 128 stay on the CTA path
    // (two of their stages fill a quarter of an SM's shared memory)
    if (a.num_sms <= 0 || a.G > 1 || a.c.upol || a.c.B > kMaxChunk) return cudaSuccess;
    if (a.c.U < warp_units_min(a.num_sms)) return cudaSuccess;
    if (a.c.qbits == 0 && a.c.dtype != 1 && a.c.D == 128) return cudaSuccess;
    *used = true;
    if (a.c.qbits == 8) return warp_form<8>(a, st);
    if (a.c.qbits == 4) return warp_form<4>(a, st);
    return warp_form<0>(a, st);
}

}  // namespace h2o
