// prompt.cu -- building the initial cache from a prompt.
//
// H2O [H2O review page, 提案手法; Model Tells You What to Discard review page,
// Figure 2 caption]: the accumulated attention of prompt token j is
//   c_j = sum_{i >= j} exp(z_ij - m_i) / l_i,  z_ij = scale q_i . k_j,
// with m_i, l_i the causal row max and normaliser.  Two passes over the
// causal score tiles (row statistics, then column sums with the statistics
// known), a per-unit radix select of the H largest c_j outside the recent
// window (ties to the lower position), and a row gather into the slots.
//
// HashEvict [HashEvict abstract]: sign codes of every prompt query and key,
// then a per-unit replay of the decode replacement rule over the prompt.
//
// The score passes here run on the CUDA cores in fp32 with fp64 running
// sums; logits are kept in base 2 (q is pre-multiplied by scale * log2 e).
#include <cfloat>
#include <climits>
#include <cstdlib>

#include "common.cuh"
#include "kernels.h"

namespace h2o {

namespace {

constexpr int kTile = 64;          // rows / columns per score tile
constexpr int kPad = 4;
constexpr unsigned kFull = 0xffffffffu;

// H2O_PROMPT_CUDA_CORES=1 selects the CUDA-core scorer for bf16 / d 128 too
// (used to compare the two implementations)
bool getenv_flag(const char* name)
{
    const char* e = getenv(name);
    return e && e[0] == '1';
}

// Load rows [r0, r0 + 64) of X [T][D] into Xs[D][64 + pad] transposed and
// scaled; rows past T are zero.  Thread t handles row t % 64.
template <typename T, int D>
__device__ __forceinline__ void load_tile_t(float (*Xs)[kTile + kPad], const T* X, int r0, int T_,
                                            float scale)
{
    constexpr int VE = 16 / (int)sizeof(T);      // elements per 16-byte vector
    constexpr int NVEC = D / VE;                 // vectors per row
    const int r = threadIdx.x % kTile;
    const int row = r0 + r;
    for (int v = threadIdx.x / kTile; v < NVEC; v += blockDim.x / kTile) {
        float f[VE];
        if (row < T_) {
            load_vec<T, VE>(X + (size_t)row * D + v * VE, f);
        } else {
#pragma unroll
            for (int e = 0; e < VE; ++e) f[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < VE; ++e) Xs[v * VE + e][r] = f[e] * scale;
    }
}

// 64 x 64 tile product: acc[a][b] = sum_k A[k][ty*4+a] * Bm[k][tx*4+b]
template <int D>
__device__ __forceinline__ void tile_mma(const float (*A)[kTile + kPad], const float (*Bm)[kTile + kPad],
                                         int ty, int tx, float (&acc)[4][4])
{
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 8
    for (int k = 0; k < D; ++k) {
        const float4 av = *reinterpret_cast<const float4*>(&A[k][ty * 4]);
        const float4 bv = *reinterpret_cast<const float4*>(&Bm[k][tx * 4]);
        const float ar[4] = {av.x, av.y, av.z, av.w};
        const float br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(ar[a], br[b], acc[a][b]);
    }
}

__device__ __forceinline__ float red16_max(float v)
{
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}
__device__ __forceinline__ float red16_sum(float v)
{
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// Pass 1: causal row max m2_i (base 2) and normaliser l_i.  One CTA per
// 64-row block; the row's 64-column tiles are swept left to right.
template <typename T, int D>
__global__ void __launch_bounds__(256) rowstats_kernel(const T* __restrict__ Q, const T* __restrict__ K,
                                                      int T_, float qscale, float* __restrict__ m2,
                                                      float* __restrict__ lout)
{
    extern __shared__ __align__(16) float tiles[];
    float (*Qs)[kTile + kPad] = reinterpret_cast<float (*)[kTile + kPad]>(tiles);
    float (*Ks)[kTile + kPad] = Qs + D;
    const int unit = blockIdx.y, ib = blockIdx.x;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const T* Qu = Q + (size_t)unit * T_ * D;
    const T* Ku = K + (size_t)unit * T_ * D;
    load_tile_t<T, D>(Qs, Qu, ib * kTile, T_, qscale);
    float m[4];
    double l[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) { m[a] = -INFINITY; l[a] = 0.0; }
    for (int jb = 0; jb <= ib; ++jb) {
        __syncthreads();
        load_tile_t<T, D>(Ks, Ku, jb * kTile, T_, 1.f);
        __syncthreads();
        float acc[4][4];
        tile_mma<D>(Qs, Ks, ty, tx, acc);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int i = ib * kTile + ty * 4 + a;
            float v[4];
            float tmax = -INFINITY;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int j = jb * kTile + tx * 4 + b;
                v[b] = (j <= i && i < T_) ? acc[a][b] : -INFINITY;
                tmax = fmaxf(tmax, v[b]);
            }
            tmax = red16_max(tmax);
            const float m_new = fmaxf(m[a], tmax);
            float s = 0.f;
#pragma unroll
            for (int b = 0; b < 4; ++b) s += (v[b] == -INFINITY) ? 0.f : exp2f(v[b] - m_new);
            s = red16_sum(s);
            if (m_new != -INFINITY) {
                const double alpha = (m[a] == -INFINITY) ? 0.0 : (double)exp2f(m[a] - m_new);
                l[a] = l[a] * alpha + (double)s;
                m[a] = m_new;
            }
        }
    }
    if (tx == 0) {
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int i = ib * kTile + ty * 4 + a;
            if (i < T_) {
                m2[(size_t)unit * T_ + i] = m[a];
                lout[(size_t)unit * T_ + i] = (float)l[a];
            }
        }
    }
}

// Pass 2: column sums c_j = sum_{i >= j} 2^(s_ij - m2_i) / l_i.  One CTA per
// 64-key block sweeps the query blocks at and below the diagonal in order,
// so every c_j is summed in a fixed order (fp32 within a tile, fp64 across).
template <typename T, int D>
__global__ void __launch_bounds__(256) colsum_kernel(const T* __restrict__ Q, const T* __restrict__ K,
                                                    int T_, float qscale, const float* __restrict__ m2,
                                                    const float* __restrict__ lin, double* __restrict__ cout)
{
    extern __shared__ __align__(16) float tiles[];
    float (*Ks)[kTile + kPad] = reinterpret_cast<float (*)[kTile + kPad]>(tiles);
    float (*Qs)[kTile + kPad] = Ks + D;
    __shared__ float ms[kTile], il[kTile];
    const int unit = blockIdx.y, jb = blockIdx.x;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int nb = (T_ + kTile - 1) / kTile;
    const T* Qu = Q + (size_t)unit * T_ * D;
    const T* Ku = K + (size_t)unit * T_ * D;
    load_tile_t<T, D>(Ks, Ku, jb * kTile, T_, 1.f);
    double csum[4] = {0.0, 0.0, 0.0, 0.0};
    for (int ib = jb; ib < nb; ++ib) {
        __syncthreads();
        load_tile_t<T, D>(Qs, Qu, ib * kTile, T_, qscale);
        if (threadIdx.x < kTile) {
            const int i = ib * kTile + threadIdx.x;
            ms[threadIdx.x] = i < T_ ? m2[(size_t)unit * T_ + i] : 0.f;
            il[threadIdx.x] = i < T_ ? 1.f / lin[(size_t)unit * T_ + i] : 0.f;
        }
        __syncthreads();
        float acc[4][4];
        tile_mma<D>(Ks, Qs, ty, tx, acc);       // acc[a][b]: key ty*4+a, query tx*4+b
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int j = jb * kTile + ty * 4 + a;
            float part = 0.f;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int i = ib * kTile + tx * 4 + b;
                if (i >= j && i < T_) part += exp2f(acc[a][b] - ms[tx * 4 + b]) * il[tx * 4 + b];
            }
            part = red16_sum(part);
            csum[a] += (double)part;
        }
    }
    if (tx == 0) {
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int j = jb * kTile + ty * 4 + a;
            if (j < T_) cout[(size_t)unit * T_ + j] = csum[a];
        }
    }
}

// ------------------------------------------------------------ block scan

constexpr int kSelThreads = 1024;

// exclusive prefix sum of one int per thread over the block; returns the
// thread's offset, *total receives the block sum
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, w, o);
            if (lane >= o) w += y;
        }
        warp_tot[lane] = w;     // inclusive
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_tot[warp - 1] : 0) + x - v;
    const int tot = warp_tot[(blockDim.x >> 5) - 1];
    __syncthreads();
    *total = tot;
    return before;
}

// Per unit: the H largest column sums among positions [0, T - r) (radix
// select on the fp64 bit patterns, which order like the values because
// every c_j >= 0; ties to the lower position), plus the recent window; kept
// positions go to slots 0.. in ascending order with their scores.
__global__ void __launch_bounds__(kSelThreads) select_kernel(CacheView cv, PromptArgs pa)
{
    __shared__ unsigned hist[256];
    __shared__ int warp_tot[32];
    __shared__ unsigned long long s_prefix;
    __shared__ int s_need;
    const int unit = blockIdx.x;
    const int T_ = pa.T, B = cv.B, r = cv.r;
    const double* cu = pa.c + (size_t)unit * T_;
    const size_t ub = (size_t)unit * B;
    const int tid = threadIdx.x;
    const int per = (T_ + kSelThreads - 1) / kSelThreads;   // contiguous positions per thread
    const int j0 = tid * per, j1 = min(T_, j0 + per);

    const bool keep_all = T_ <= B;
    const int ncand = keep_all ? 0 : T_ - r;
    const int H = keep_all ? 0 : min(pa.H, ncand);

    unsigned long long thr = 0ull;      // bit pattern of the H-th largest candidate
    int need = 0;                       // how many candidates equal to thr are kept
    if (H > 0) {
        unsigned long long prefix = 0ull, mask = 0ull;
        int remaining = H;
        for (int shift = 56; shift >= 0; shift -= 8) {
            for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0u;
            __syncthreads();
            for (int j = tid; j < ncand; j += kSelThreads) {
                const unsigned long long key = (unsigned long long)__double_as_longlong(cu[j]);
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255ull], 1u);
            }
            __syncthreads();
            if (tid == 0) {
                int cum = 0;
                int dig = 0;
                for (int d = 255; d >= 0; --d) {
                    if (cum + (int)hist[d] >= remaining) { dig = d; break; }
                    cum += (int)hist[d];
                }
                remaining -= cum;
                s_prefix = prefix | ((unsigned long long)dig << shift);
                s_need = remaining;
            }
            __syncthreads();
            prefix = s_prefix;
            remaining = s_need;
            mask |= 255ull << shift;
            __syncthreads();
        }
        thr = prefix;
        need = remaining;
    }

    // rank of equal-to-threshold candidates, in ascending position
    int my_eq = 0;
    if (H > 0) {
        for (int j = j0; j < j1; ++j)
            if (j < ncand && (unsigned long long)__double_as_longlong(cu[j]) == thr) ++my_eq;
    }
    int tot;
    int eq_before = block_exclusive_scan(my_eq, warp_tot, &tot);

    // kept flags and slot offsets
    int my_keep = 0;
    {
        int eq = eq_before;
        for (int j = j0; j < j1; ++j) {
            bool k;
            if (keep_all || j >= ncand) {
                k = true;
            } else if (H == 0) {
                k = false;
            } else {
                const unsigned long long key = (unsigned long long)__double_as_longlong(cu[j]);
                if (key > thr) k = true;
                else if (key == thr) { k = eq < need; ++eq; }
                else k = false;
            }
            my_keep += k ? 1 : 0;
        }
    }
    int nkept;
    int slot = block_exclusive_scan(my_keep, warp_tot, &nkept);
    {
        int eq = eq_before;
        for (int j = j0; j < j1; ++j) {
            bool k;
            if (keep_all || j >= ncand) {
                k = true;
            } else if (H == 0) {
                k = false;
            } else {
                const unsigned long long key = (unsigned long long)__double_as_longlong(cu[j]);
                if (key > thr) k = true;
                else if (key == thr) { k = eq < need; ++eq; }
                else k = false;
            }
            if (k) {
                cv.pos[ub + slot] = j;
                if (cv.score) {
                    const float hi = __double2float_rn(cu[j]);
                    cv.score[ub + slot] = make_float2(hi, __double2float_rn(cu[j] - (double)hi));
                }
                ++slot;
            }
        }
    }
    for (int s = nkept + tid; s < B; s += kSelThreads) {
        cv.pos[ub + s] = -1;
        if (cv.score) cv.score[ub + s] = make_float2(0.f, 0.f);
    }
    if (tid == 0) cv.ustate[unit] = make_int2(nkept, T_);
}

// Copy the prompt rows named by pos[] into the slots (zero for empty slots);
// one warp per slot: lanes 0..15 move K, 16..31 move V (16 bytes each).
template <typename T, int D>
__global__ void __launch_bounds__(256) gather_kernel(CacheView cv, PromptArgs pa, int with_codes)
{
    constexpr int NV = D * (int)sizeof(T) / 16;   // 16-byte vectors per row
    const int lane = threadIdx.x & 31;
    const long long total = (long long)cv.U * cv.B;
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long slot = wid; slot < total; slot += nw) {
        const int unit = (int)(slot / cv.B);
        const int p = cv.pos[slot];
        const int half = lane >> 4, l16 = lane & 15;
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<T*>(half ? cv.V : cv.K) + (size_t)slot * D);
        const T* srcbase = reinterpret_cast<const T*>(half ? pa.V : pa.K) + ((size_t)unit * pa.T) * D;
        for (int v = l16; v < NV; v += 16) {
            uint4 w = make_uint4(0u, 0u, 0u, 0u);
            if (p >= 0) w = reinterpret_cast<const uint4*>(srcbase + (size_t)p * D)[v];
            dst[v] = w;
        }
        if (with_codes && lane == 0) cv.code[slot] = p >= 0 ? pa.ck[(size_t)unit * pa.T + p] : 0u;
    }
}

// Sign codes of every prompt query and key.  Lane j of a warp keeps column j
// of W in registers and owns bit j.  The warp hashes kCodeTok tokens per
// pass (2 * kCodeTok independent fp32 fused multiply-add chains, each in
// index order from 0); the next pass's rows are fetched into registers
// while the current chains run, then staged in shared memory.
constexpr int kCodeWarps = 8;
constexpr int kCodeTok = 4;

template <typename T, int D>
__global__ void __launch_bounds__(32 * kCodeWarps) lsh_codes_kernel(const T* __restrict__ Q, const T* __restrict__ K,
                                                                    const float* __restrict__ W, long long ntok,
                                                                    uint32_t* __restrict__ cq,
                                                                    uint32_t* __restrict__ ck)
{
    constexpr int EPL = D / 32;                       // elements of a row per lane
    __shared__ __align__(16) float xs[kCodeWarps][2 * kCodeTok][D];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float w[D];
#pragma unroll
    for (int i = 0; i < D; ++i) w[i] = __ldg(W + i * 32 + lane);
    const long long step = (long long)gridDim.x * kCodeWarps * kCodeTok;
    long long tok0 = ((long long)blockIdx.x * kCodeWarps + warp) * kCodeTok;
    float pre[2 * kCodeTok][EPL];
    auto fetch = [&](long long t0) {
#pragma unroll
        for (int k = 0; k < kCodeTok; ++k) {
            const long long t = t0 + k;
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                pre[2 * k][e] = t < ntok ? Elem<T>::to_f(Q[t * D + lane * EPL + e]) : 0.f;
                pre[2 * k + 1][e] = t < ntok ? Elem<T>::to_f(K[t * D + lane * EPL + e]) : 0.f;
            }
        }
    };
    fetch(tok0);
    for (; tok0 < ntok; tok0 += step) {
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 2 * kCodeTok; ++r)
#pragma unroll
            for (int e = 0; e < EPL; ++e) xs[warp][r][lane * EPL + e] = pre[r][e];
        __syncwarp();
        fetch(tok0 + step);
        float acc[2 * kCodeTok];
#pragma unroll
        for (int r = 0; r < 2 * kCodeTok; ++r) acc[r] = 0.f;
#pragma unroll
        for (int i = 0; i < D; i += 4) {
#pragma unroll
            for (int r = 0; r < 2 * kCodeTok; ++r) {
                const float4 x4 = *reinterpret_cast<const float4*>(&xs[warp][r][i]);
                acc[r] = __fmaf_rn(x4.x, w[i], acc[r]);
                acc[r] = __fmaf_rn(x4.y, w[i + 1], acc[r]);
                acc[r] = __fmaf_rn(x4.z, w[i + 2], acc[r]);
                acc[r] = __fmaf_rn(x4.w, w[i + 3], acc[r]);
            }
        }
#pragma unroll
        for (int k = 0; k < kCodeTok; ++k) {
            const unsigned bq = __ballot_sync(kFull, acc[2 * k] > 0.f);
            const unsigned bk = __ballot_sync(kFull, acc[2 * k + 1] > 0.f);
            if (lane == 0 && tok0 + k < ntok) { cq[tok0 + k] = bq; ck[tok0 + k] = bk; }
        }
    }
}

// The same replay with each lane's slots (s = lane + 32 i) held in registers,
// for budgets up to 32 * kRegSlots: no shared-memory round trip per step.
constexpr int kRegSlots = 16;

__global__ void __launch_bounds__(64) lsh_replay_reg_kernel(CacheView cv, PromptArgs pa)
{
    const int B = cv.B, T_ = pa.T, r = cv.r;
    const int lane = threadIdx.x & 31;
    const int unit = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (unit >= cv.U) return;
    const uint32_t* cq = pa.cq + (size_t)unit * T_;
    const uint32_t* ck = pa.ck + (size_t)unit * T_;
    const int n0 = min(T_, B);
    uint32_t code[kRegSlots];
    int pos[kRegSlots];
#pragma unroll
    for (int i = 0; i < kRegSlots; ++i) {
        const int s = lane + 32 * i;
        pos[i] = s < n0 ? s : -1;
        code[i] = s < n0 ? ck[s] : 0u;
    }
    uint32_t qb = 0u, kb = 0u;
    for (int t = B; t < T_; ++t) {
        const int o = (t - B) & 31;
        if (o == 0) {
            const int tt = t + lane;
            qb = tt < T_ ? cq[tt] : 0u;
            kb = tt < T_ ? ck[tt] : 0u;
        }
        const uint32_t q = __shfl_sync(kFull, qb, o);
        const uint32_t knew = __shfl_sync(kFull, kb, o);
        unsigned b0 = 0u, b1 = 0u;           // two chains over even / odd register slots
#pragma unroll
        for (int i = 0; i < kRegSlots; ++i) {
            const int s = lane + 32 * i;
            const unsigned key = ((unsigned)__popc(q ^ code[i]) << 20) | (0xFFFFFu - (unsigned)s);
            if (s < B && pos[i] <= t - r) {
                if (i & 1) b1 = max(b1, key); else b0 = max(b0, key);
            }
        }
        unsigned best = __reduce_max_sync(kFull, max(b0, b1));
        if (best == 0u) {                    // no slot outside the window: every slot competes
#pragma unroll
            for (int i = 0; i < kRegSlots; ++i) {
                const int s = lane + 32 * i;
                if (s < B) best = max(best, ((unsigned)__popc(q ^ code[i]) << 20) | (0xFFFFFu - (unsigned)s));
            }
            best = __reduce_max_sync(kFull, best);
        }
        const int v = (int)(0xFFFFFu - (best & 0xFFFFFu));
        if ((v & 31) == lane) {
            const int iv = v >> 5;
#pragma unroll
            for (int i = 0; i < kRegSlots; ++i)
                if (i == iv) { code[i] = knew; pos[i] = t; }
        }
    }
    const size_t ub = (size_t)unit * B;
#pragma unroll
    for (int i = 0; i < kRegSlots; ++i) {
        const int s = lane + 32 * i;
        if (s < B) cv.pos[ub + s] = pos[i];
    }
    if (lane == 0) cv.ustate[unit] = make_int2(n0, T_);
}

// Replay the HashEvict replacement rule over the prompt, one warp per unit:
// the first B tokens fill the slots; token t >= B replaces the slot with the
// largest Hamming distance to code(q_t) among slots with position <= t - r
// (lowest slot on ties; every slot if none qualifies).  The slots' codes and
// positions live in shared memory; the arg-max is one unsigned max of
// (distance << 20) | (2^20 - 1 - slot).
__global__ void lsh_replay_kernel(CacheView cv, PromptArgs pa, int warps_per_cta)
{
    extern __shared__ __align__(16) unsigned char sm[];
    const int B = cv.B, T_ = pa.T, r = cv.r;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int unit = blockIdx.x * warps_per_cta + warp;
    if (unit >= cv.U) return;
    uint32_t* code = reinterpret_cast<uint32_t*>(sm) + (size_t)warp * 2 * B;
    int* pos = reinterpret_cast<int*>(code + B);
    const uint32_t* cq = pa.cq + (size_t)unit * T_;
    const uint32_t* ck = pa.ck + (size_t)unit * T_;
    const int n0 = min(T_, B);
    for (int s = lane; s < B; s += 32) {
        pos[s] = s < n0 ? s : -1;
        code[s] = s < n0 ? ck[s] : 0u;
    }
    __syncwarp();
    uint32_t qb = 0u, kb = 0u;      // this lane's entry of the current 32-token batch
    for (int t = B; t < T_; ++t) {
        const int o = (t - B) & 31;
        if (o == 0) {
            const int tt = t + lane;
            qb = tt < T_ ? cq[tt] : 0u;
            kb = tt < T_ ? ck[tt] : 0u;
        }
        const uint32_t q = __shfl_sync(kFull, qb, o);
        const uint32_t knew = __shfl_sync(kFull, kb, o);
        unsigned best = 0u, best_all = 0u;
        for (int s = lane; s < B; s += 32) {
            const unsigned key = ((unsigned)__popc(q ^ code[s]) << 20) | (0xFFFFFu - (unsigned)s);
            if (pos[s] <= t - r) best = max(best, key);
            best_all = max(best_all, key);
        }
        best = __reduce_max_sync(kFull, best);
        best_all = __reduce_max_sync(kFull, best_all);
        const int v = (int)(0xFFFFFu - ((best ? best : best_all) & 0xFFFFFu));
        if (lane == 0) {
            code[v] = knew;
            pos[v] = t;
        }
        __syncwarp();
    }
    const size_t ub = (size_t)unit * B;
    for (int s = lane; s < B; s += 32) cv.pos[ub + s] = pos[s];
    if (lane == 0) cv.ustate[unit] = make_int2(n0, T_);
}

template <typename T, int D>
cudaError_t stats_t(const CacheView& c, const PromptArgs& p, cudaStream_t st)
{
    const int nb = (p.T + kTile - 1) / kTile;
    dim3 grid((unsigned)nb, (unsigned)c.U);
    const size_t smem = 2 * (size_t)D * (kTile + kPad) * sizeof(float);
    static bool configured[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(rowstats_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(colsum_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    rowstats_kernel<T, D><<<grid, 256, smem, st>>>(reinterpret_cast<const T*>(p.Q),
                                                 reinterpret_cast<const T*>(p.K), p.T, c.qscale, p.m2, p.l);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    colsum_kernel<T, D><<<grid, 256, smem, st>>>(reinterpret_cast<const T*>(p.Q),
                                               reinterpret_cast<const T*>(p.K), p.T, c.qscale, p.m2, p.l,
                                               p.c);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t gather_t(const CacheView& c, const PromptArgs& p, bool with_codes, cudaStream_t st)
{
    const long long warps = (long long)c.U * c.B;
    long long blocks = (warps + 7) / 8;
    if (blocks > 65535LL * 8) blocks = 65535LL * 8;
    gather_kernel<T, D><<<(unsigned)blocks, 256, 0, st>>>(c, p, with_codes ? 1 : 0);
    return cudaGetLastError();
}

// warps per CTA of the replay: how many units' slot state fits the shared
// memory chosen (H2O_REPLAY_WARPS overrides, for tuning)
int replay_warps(int B)
{
    const char* e = getenv("H2O_REPLAY_WARPS");
    int w = e ? atoi(e) : 2;
    const int fit = (int)((48 * 1024) / ((size_t)B * 8));
    if (w > fit) w = fit;
    if (w < 1) w = 1;
    return w;
}

template <typename T, int D>
cudaError_t lsh_t(const CacheView& c, const PromptArgs& p, const float* W, cudaStream_t st)
{
    const long long ntok = (long long)c.U * p.T;
    int sms = 0, dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    long long blocks = (ntok + kCodeWarps * kCodeTok - 1) / (kCodeWarps * kCodeTok);
    if (blocks > 4LL * sms) blocks = 4LL * sms;
    lsh_codes_kernel<T, D><<<(unsigned)blocks, 32 * kCodeWarps, 0, st>>>(
        reinterpret_cast<const T*>(p.Q), reinterpret_cast<const T*>(p.K), W, ntok, p.cq, p.ck);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (c.B <= 32 * kRegSlots) {
        lsh_replay_reg_kernel<<<(unsigned)((c.U + 1) / 2), 64, 0, st>>>(c, p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        return gather_t<T, D>(c, p, true, st);
    }
    const size_t per_unit = (size_t)c.B * 8;
    const int wpc = replay_warps(c.B);
    const size_t smem = per_unit * wpc;
    if (smem > 48 * 1024) {
        static size_t configured[64] = {0};
        if (configured[dev] < smem) {
            e = cudaFuncSetAttribute(lsh_replay_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            configured[dev] = smem;
        }
    }
    lsh_replay_kernel<<<(unsigned)((c.U + wpc - 1) / wpc), 32 * wpc, smem, st>>>(c, p, wpc);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return gather_t<T, D>(c, p, true, st);
}

}  // namespace

cudaError_t launch_prompt_stats(const CacheView& c, const PromptArgs& p, cudaStream_t st)
{
    if (prompt_tc_supported(c) && !getenv_flag("H2O_PROMPT_CUDA_CORES"))
        return launch_prompt_stats_tc(c, p, st);
    const bool bf = c.dtype == 1;
    if (c.D == 128) return bf ? stats_t<__nv_bfloat16, 128>(c, p, st) : stats_t<float, 128>(c, p, st);
    if (c.D == 64) return bf ? stats_t<__nv_bfloat16, 64>(c, p, st) : stats_t<float, 64>(c, p, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_select(const CacheView& c, const PromptArgs& p, cudaStream_t st)
{
    select_kernel<<<(unsigned)c.U, kSelThreads, 0, st>>>(c, p);
    return cudaGetLastError();
}

cudaError_t launch_gather(const CacheView& c, const PromptArgs& p, bool with_codes, cudaStream_t st)
{
    const bool bf = c.dtype == 1;
    if (c.D == 128)
        return bf ? gather_t<__nv_bfloat16, 128>(c, p, with_codes, st) : gather_t<float, 128>(c, p, with_codes, st);
    if (c.D == 64)
        return bf ? gather_t<__nv_bfloat16, 64>(c, p, with_codes, st) : gather_t<float, 64>(c, p, with_codes, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_lsh_prompt(const CacheView& c, const PromptArgs& p, const float* W, cudaStream_t st)
{
    const bool bf = c.dtype == 1;
    if (c.D == 128) return bf ? lsh_t<__nv_bfloat16, 128>(c, p, W, st) : lsh_t<float, 128>(c, p, W, st);
    if (c.D == 64) return bf ? lsh_t<__nv_bfloat16, 64>(c, p, W, st) : lsh_t<float, 64>(c, p, W, st);
    return cudaErrorInvalidValue;
}

}  // namespace h2o
