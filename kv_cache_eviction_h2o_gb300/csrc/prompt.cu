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
// Grouped-query caches: query unit u reads the keys of cache unit u / G, and
// a cache unit's column sums are its G heads' sums.  Persistence of
// importance [Scissorhands abstract]: the pivotal histories of the last 32
// rows (CUDA-core kernel here, tensor-core one in prompt_tc.cu) feed the same
// select and gather.
//
// The score passes here run on the CUDA cores in fp32 with fp64 running
// sums; logits are kept in base 2 (q is pre-multiplied by scale * log2 e).
#include <cfloat>
#include <climits>
#include <cstdlib>
#include <cstring>
#include <type_traits>

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
                                                      int T_, int G, float qscale, float* __restrict__ m2,
                                                      float* __restrict__ lout)
{
    extern __shared__ __align__(16) float tiles[];
    float (*Qs)[kTile + kPad] = reinterpret_cast<float (*)[kTile + kPad]>(tiles);
    float (*Ks)[kTile + kPad] = Qs + D;
    const int unit = blockIdx.y, ib = blockIdx.x;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const T* Qu = Q + (size_t)unit * T_ * D;
    const T* Ku = K + (size_t)(unit / G) * T_ * D;   // keys of this query unit
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
                                                    int T_, int G, float qscale, const float* __restrict__ m2,
                                                    const float* __restrict__ lin, double* __restrict__ cout,
                                                    double* __restrict__ bandB, double* __restrict__ bandr,
                                                    int wB, int wr)
{
    extern __shared__ __align__(16) float tiles[];
    float (*Ks)[kTile + kPad] = reinterpret_cast<float (*)[kTile + kPad]>(tiles);
    float (*Qs)[kTile + kPad] = Ks + D;
    __shared__ float ms[kTile], il[kTile];
    const int unit = blockIdx.y, jb = blockIdx.x;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int nb = (T_ + kTile - 1) / kTile;
    const T* Qu = Q + (size_t)unit * T_ * D;
    const T* Ku = K + (size_t)(unit / G) * T_ * D;   // keys of this query unit
    load_tile_t<T, D>(Ks, Ku, jb * kTile, T_, 1.f);
    double csum[4] = {0.0, 0.0, 0.0, 0.0};
    double bsum[4] = {0.0, 0.0, 0.0, 0.0}, rsum[4] = {0.0, 0.0, 0.0, 0.0};   // band sums
    const int wmax = max(wB, wr);
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
        // rows of this tile within the widest band of some key of the block
        const bool band = bandB && ib * kTile < (jb + 1) * kTile + wmax;
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int j = jb * kTile + ty * 4 + a;
            float part = 0.f, pB = 0.f, pr = 0.f;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int i = ib * kTile + tx * 4 + b;
                if (i >= j && i < T_) {
                    const float x = exp2f(acc[a][b] - ms[tx * 4 + b]) * il[tx * 4 + b];
                    part += x;
                    if (band) {
                        if (i - j < wB) pB += x;
                        if (i - j < wr) pr += x;
                    }
                }
            }
            part = red16_sum(part);
            csum[a] += (double)part;
            if (band) {
                bsum[a] += (double)red16_sum(pB);
                rsum[a] += (double)red16_sum(pr);
            }
        }
    }
    if (tx == 0) {
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int j = jb * kTile + ty * 4 + a;
            if (j < T_) {
                cout[(size_t)unit * T_ + j] = csum[a];
                if (bandB) {
                    bandB[(size_t)unit * T_ + j] = bsum[a];
                    bandr[(size_t)unit * T_ + j] = rsum[a];
                }
            }
        }
    }
}

// ------------------------------------------------------------ block scan


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
// The digit of a radix round: with hist[d] the candidates of digit d still
// in play and `remaining` of them to keep, the largest digit d such that at
// least `remaining` candidates have digit >= d, and how many of those with
// digit > d there are (cum).  One warp: each lane sums 8 bins, a suffix scan
// over the lanes and a ballot find the lane holding the digit, which then
// walks its 8 bins from the top.
__device__ __forceinline__ void radix_digit(const unsigned* hist, int remaining, int lane, int& dig, int& cum)
{
    unsigned b[8];
    unsigned tot = 0u;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        b[k] = hist[8 * lane + k];
        tot += b[k];
    }
    // inclusive suffix sum over lanes: bins of this lane and every higher one
    unsigned suf = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_down_sync(kFull, suf, o);
        if (lane + o < 32) suf += y;
    }
    const unsigned hit = __ballot_sync(kFull, suf >= (unsigned)remaining);
    const int L = hit ? 31 - __clz(hit) : 0;             // highest lane reaching the target
    const unsigned above = __shfl_sync(kFull, suf - tot, L);   // bins of the lanes above L
    int d = 8 * L, c = (int)above;
    if (lane == L) {
#pragma unroll
        for (int k = 7; k >= 0; --k) {
            if (c + (int)b[k] >= remaining) { d = 8 * L + k; break; }
            c += (int)b[k];
        }
    }
    dig = __shfl_sync(kFull, d, L);
    cum = __shfl_sync(kFull, c, L);
}

// Copy the prompt rows named by pos[] into slots s0 .. s0 + SW - 1 (those
// below `end`; zero rows for empty slots): lanes 0..15 of the warp move K,
// 16..31 move V (16 bytes each).  The warp requests all SW positions, then
// all SW rows, before it stores any, so SW rows are in flight per lane.
// Quantised slots take the half-warp's max magnitude as the row's scale.
template <typename T, int D, int SW>
__device__ __forceinline__ void gather_group(const CacheView& cv, const PromptArgs& pa, long long s0, long long end,
                                             int lane, int with_codes)
{
    constexpr int NV = D * (int)sizeof(T) / 16;   // 16-byte vectors per row
    constexpr int VE = 16 / (int)sizeof(T);       // elements per 16-byte vector
    constexpr int VPL = (NV + 15) / 16;           // vectors per lane of a half-warp
    const int half = lane >> 4, l16 = lane & 15;
    int p[SW], unit[SW];
#pragma unroll
    for (int k = 0; k < SW; ++k) {
        const long long slot = s0 + k;
        unit[k] = (int)(slot / cv.B);
        p[k] = slot < end ? cv.pos[slot] : -1;
    }
    uint4 w[SW][VPL];
#pragma unroll
    for (int k = 0; k < SW; ++k) {
        const T* src = reinterpret_cast<const T*>(half ? pa.V : pa.K) + ((size_t)unit[k] * pa.T + (size_t)max(p[k], 0)) * D;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int v = l16 + 16 * i;
            w[k][i] = make_uint4(0u, 0u, 0u, 0u);
            if (p[k] >= 0 && v < NV) w[k][i] = reinterpret_cast<const uint4*>(src)[v];
        }
    }
#pragma unroll
    for (int k = 0; k < SW; ++k) {
        const long long slot = s0 + k;
        if (slot >= end) break;
        if (!cv.qbits) {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<T*>(half ? cv.V : cv.K) + (size_t)slot * D);
#pragma unroll
            for (int i = 0; i < VPL; ++i) {
                const int v = l16 + 16 * i;
                if (v < NV) dst[v] = w[k][i];
            }
        } else {
            float x[VPL][VE];
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < VPL; ++i) {
                const uint32_t u[4] = {w[k][i].x, w[k][i].y, w[k][i].z, w[k][i].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if constexpr (sizeof(T) == 2) {
                        x[i][2 * e] = __uint_as_float(u[e] << 16);
                        x[i][2 * e + 1] = __uint_as_float(u[e] & 0xffff0000u);
                    } else {
                        x[i][e] = __uint_as_float(u[e]);
                    }
                }
#pragma unroll
                for (int e = 0; e < VE; ++e) amax = fmaxf(amax, fabsf(x[i][e]));
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
            float* scale_out =
                reinterpret_cast<float*>(cv.kvs + (size_t)unit[k] * cv.Bp + (slot - (long long)unit[k] * cv.B)) + half;
            if (cv.qbits == 8) {
                const float inv = q8_inv(amax);
                uint8_t* dst = reinterpret_cast<uint8_t*>(half ? cv.V : cv.K) + (size_t)slot * D;
#pragma unroll
                for (int i = 0; i < VPL; ++i) {
                    const int v = l16 + 16 * i;
                    if (v < NV) {
                        if constexpr (VE == 8) {
                            *reinterpret_cast<uint2*>(dst + v * VE) =
                                make_uint2(q8_pack4(&x[i][0], inv), q8_pack4(&x[i][4], inv));
                        } else {
                            *reinterpret_cast<uint32_t*>(dst + v * VE) = q8_pack4(&x[i][0], inv);
                        }
                    }
                }
                if (l16 == 0) *scale_out = q8_scale(amax);
            } else {
                // 4-bit row: D / 2 bytes, VE / 2 per 16-byte input vector
                const float inv = q4_inv(amax);
                uint8_t* dst = reinterpret_cast<uint8_t*>(half ? cv.V : cv.K) + (size_t)slot * (D / 2);
#pragma unroll
                for (int i = 0; i < VPL; ++i) {
                    const int v = l16 + 16 * i;
                    if (v < NV) {
                        if constexpr (VE == 8) *reinterpret_cast<uint32_t*>(dst + v * 4) = q4_pack<4>(&x[i][0], inv);
                        else *reinterpret_cast<uint16_t*>(dst + v * 2) = (uint16_t)q4_pack<2>(&x[i][0], inv);
                    }
                }
                if (l16 == 0) *scale_out = q4_scale(amax);
            }
        }
        if (with_codes && lane == 0) cv.code[slot] = p[k] >= 0 ? pa.ck[(size_t)unit[k] * pa.T + p[k]] : 0u;
    }
}

// Heavy set of each unit [H2O review page, 提案手法: the H tokens of largest
// accumulated attention outside the recent window] (one CTA per unit): an
// 8-bit radix select, from the top byte down, of the H-th largest
// candidate's bit pattern (the column sums are non-negative, so their fp64
// bit patterns order as the values).  The candidates' keys are held in registers across the rounds
// (PER per thread, strided by NT) when they fit, and the rounds stop as
// soon as the threshold's bucket is kept whole: every key sharing the
// prefix found so far is then kept, and no tie needs breaking.  Otherwise
// the keys equal to the full threshold are kept in ascending position up to
// the count still needed.  With a row type T (not void) the CTA then copies
// its unit's kept rows into the slots itself (the H2O prompt phase): its
// warps take 16 consecutive slots at a time, all their rows in flight.
template <int NT, int PER, typename T = void, int D = 0>
__global__ void __launch_bounds__(NT) select_kernel(CacheView cv, PromptArgs pa)
{
    __shared__ unsigned hist[256];
    __shared__ int warp_tot[32];
    __shared__ unsigned long long s_prefix;
    __shared__ int s_need, s_done;
    const int unit = blockIdx.x;
    const int T_ = pa.T, B = pa.budget > 0 ? pa.budget : cv.B, r = cv.r;
    const double* cu = pa.c + (size_t)unit * T_;
    const size_t ub = (size_t)unit * cv.B;     // slot stride: the cache's B
    const int tid = threadIdx.x;
    const int per = (T_ + NT - 1) / NT;      // contiguous positions per thread
    const int j0 = tid * per, j1 = min(T_, j0 + per);

    const bool keep_all = T_ <= B;
    const int ncand = keep_all ? 0 : T_ - r;
    const int H = keep_all ? 0 : min(pa.H, ncand);

    unsigned long long thr = 0ull;      // the threshold's bits under `mask`
    unsigned long long mask = 0ull;     // the bits the rounds have fixed
    int need = 0;                       // how many candidates matching thr under mask are kept
    if (H > 0) {
        unsigned long long prefix = 0ull;
        int remaining = H;
        const bool in_regs = ncand <= NT * PER;
        unsigned long long kr[PER];
        if (in_regs) {
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int j = tid + i * NT;
                kr[i] = j < ncand ? (unsigned long long)__double_as_longlong(cu[j]) : 0ull;
            }
        }
        // one key's digit into the histogram, warp-aggregated: one
        // shared-memory atomic per distinct digit per warp (many candidates
        // can share a digit, e.g. the zero low bytes of integer-valued keys)
        auto count = [&](bool valid, unsigned long long key, int shift) {
            int dig = -1;
            if (valid && (key & mask) == prefix) dig = (int)((key >> shift) & 255ull);
            const unsigned peers = __match_any_sync(0xffffffffu, dig);
            if (dig >= 0 && (tid & 31) == __ffs(peers) - 1) atomicAdd(&hist[dig], (unsigned)__popc(peers));
        };
        for (int shift = 56; shift >= 0; shift -= 8) {
            for (int i = tid; i < 256; i += NT) hist[i] = 0u;
            __syncthreads();
            if (in_regs) {
#pragma unroll
                for (int i = 0; i < PER; ++i) {
                    if (i * NT + (tid - (tid & 31)) >= ncand) break;      // warp-uniform
                    count(tid + i * NT < ncand, kr[i], shift);
                }
            } else {
                for (int jb = tid - (tid & 31); jb < ncand; jb += NT) {
                    const int j = jb + (tid & 31);
                    count(j < ncand, j < ncand ? (unsigned long long)__double_as_longlong(cu[j]) : 0ull, shift);
                }
            }
            __syncthreads();
            if (tid < 32) {
                int dig, cum;
                radix_digit(hist, remaining, tid, dig, cum);
                if (tid == 0) {
                    s_prefix = prefix | ((unsigned long long)dig << shift);
                    s_need = remaining - cum;
                    s_done = (remaining - cum) == (int)hist[dig];   // the bucket is kept whole
                }
            }
            __syncthreads();
            prefix = s_prefix;
            remaining = s_need;
            mask |= 255ull << shift;
            const bool done = s_done != 0;
            __syncthreads();
            if (done) break;
        }
        thr = prefix;
        need = remaining;
    }

    // rank of equal-to-threshold candidates, in ascending position
    int my_eq = 0;
    if (H > 0) {
        for (int j = j0; j < j1; ++j)
            if (j < ncand && ((unsigned long long)__double_as_longlong(cu[j]) & mask) == thr) ++my_eq;
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
                const unsigned long long key = (unsigned long long)__double_as_longlong(cu[j]) & mask;
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
                const unsigned long long key = (unsigned long long)__double_as_longlong(cu[j]) & mask;
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
    for (int s = nkept + tid; s < cv.B; s += NT) {
        cv.pos[ub + s] = -1;
        if (cv.score) cv.score[ub + s] = make_float2(0.f, 0.f);
    }
    if (tid == 0) cv.ustate[unit] = make_int2(nkept, T_);
    if constexpr (!std::is_void<T>::value) {
        constexpr int SW = 16;
        __syncthreads();                          // every slot's position is written
        const int warp = tid >> 5, lane = tid & 31;
        const long long end = (long long)ub + cv.B;
        for (long long s0 = (long long)ub + warp * SW; s0 < end; s0 += (NT / 32) * SW)
            gather_group<T, D, SW>(cv, pa, s0, end, lane, 0);
    }
}

// Per-head policy of every unit ["Model Tells You What to Discard" review
// page, method section: each head is profiled on the prompt and takes the
// first policy whose cache recovers enough of its attention; Figure 2
// caption: the frequency + local policy is the H2O cache].  Recovery of a
// policy = the attention mass its kept set holds at each prompt row,
// averaged over the rows:
//   local (the newest B keys):   sum_j bandB_j / T
//   frequency + local:           (sum_j bandr_j + sum_{j heavy} (c_j - bandr_j)) / T
// where band*_j is key j's probability mass from rows j .. j+w-1 (the rows
// whose window holds it) and the heavy keys are the H2O selection's kept
// keys older than the window (all kept keys hold, for a prompt within the
// budget).  Policy: local if its recovery reaches tau, else frequency +
// local if its does, else full.  Local and full units then keep the newest
// min(T, budget) tokens.  One CTA (256 threads) per unit, after the H2O
// selection (budget B) and before the gather.
__global__ void __launch_bounds__(256) fg_policy_kernel(CacheView cv, PromptArgs pa, FgArgs fa)
{
    __shared__ double red[3][8];
    __shared__ int s_n;
    const int unit = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T_ = pa.T;
    const size_t ub = (size_t)unit * cv.B;
    const double* cu = pa.c + (size_t)unit * T_;
    const double* bB = pa.bandB + (size_t)unit * T_;
    const double* br = pa.bandr + (size_t)unit * T_;
    double sB = 0.0, sr = 0.0, sh = 0.0;
    for (int j = tid; j < T_; j += 256) {
        sB += bB[j];
        sr += br[j];
    }
    const int n = cv.ustate[unit].x;
    for (int s = tid; s < n; s += 256) {
        const int j = cv.pos[ub + s];
        if (j >= 0 && j < T_ - fa.r) sh += cu[j] - br[j];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        sB += __shfl_xor_sync(kFull, sB, o);
        sr += __shfl_xor_sync(kFull, sr, o);
        sh += __shfl_xor_sync(kFull, sh, o);
    }
    if (lane == 0) { red[0][warp] = sB; red[1][warp] = sr; red[2][warp] = sh; }
    __syncthreads();
    if (tid == 0) {
        double a = 0.0, b = 0.0, h = 0.0;
        for (int w = 0; w < 8; ++w) { a += red[0][w]; b += red[1][w]; h += red[2][w]; }
        const double rl = a / (double)T_, rf = (b + h) / (double)T_;
        const int policy = rl >= fa.tau ? 0 : (rf >= fa.tau ? 1 : 2);
        const int4 pp = policy == 0 ? make_int4(fa.B, 0, fa.B, 0)
                      : policy == 1 ? make_int4(fa.B, fa.H, fa.r, 1)
                                    : make_int4(fa.B_full, 0, fa.B_full, 2);
        fa.upol[unit] = pp;
        fa.rec[unit] = make_double2(rl, rf);
        s_n = policy == 1 ? -1 : min(T_, pp.x);
    }
    __syncthreads();
    const int nk = s_n;
    if (nk < 0) return;                     // frequency + local: the H2O selection stands
    for (int s = tid; s < cv.B; s += 256) {
        const int j = s < nk ? T_ - nk + s : -1;
        cv.pos[ub + s] = j;
        float2 sc = make_float2(0.f, 0.f);
        if (j >= 0) {
            const float hi = __double2float_rn(cu[j]);
            sc = make_float2(hi, __double2float_rn(cu[j] - (double)hi));
        }
        cv.score[ub + s] = sc;
    }
    if (tid == 0) cv.ustate[unit] = make_int2(nk, T_);
}

// The rows of every unit's slots after a selection that pos[] records (the
// per-head policies rewrite it after the selection; HashEvict's replay
// writes it): a warp takes kGatherSlots consecutive slots per round of a
// grid-stride loop.
constexpr int kGatherSlots = 4;

template <typename T, int D>
__global__ void __launch_bounds__(256) gather_kernel(CacheView cv, PromptArgs pa, int with_codes)
{
    const int lane = threadIdx.x & 31;
    const long long total = (long long)cv.U * cv.B;
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long s0 = wid * kGatherSlots; s0 < total; s0 += nw * kGatherSlots)
        gather_group<T, D, kGatherSlots>(cv, pa, s0, total, lane, with_codes);
}

// Sign codes of every prompt query and key, one row (a query or a key) per
// thread: bit j is the sign of the fp32 fused multiply-add chain
// x[0] W[0][j] + ... + x[D-1] W[D-1][j] taken in index order from 0.  A
// thread runs its row's 32 chains side by side.  W is a launch parameter, so
// every multiply-add reads its W value from the constant bank, broadcast to
// the warp, instead of through shared memory (where delivering one value to
// 32 lanes costs a shared-memory cycle, a quarter of the SM's FMA rate; W
// staged in shared memory and read four values per broadcast load measured
// 1.5x slower than this: 331 against 220 us on the OPT-6.7B-shaped prompt;
// two rows per thread, each W value feeding both, 268 us: 128 registers
// halve the warps per SM).
constexpr int kCodeThreads = 256;

template <int D>
struct WParam {
    float w[D * 32];
};

// The fp32 values of one 16-byte chunk of T.
template <typename T>
__device__ __forceinline__ void chunk_to_f32(const uint4& w, float* out)
{
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if constexpr (sizeof(T) == 2) {
            out[2 * k] = __uint_as_float(u[k] << 16);
            out[2 * k + 1] = __uint_as_float(u[k] & 0xffff0000u);
        } else {
            out[k] = __uint_as_float(u[k]);
        }
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kCodeThreads) lsh_codes_kernel(const T* __restrict__ Q, const T* __restrict__ K,
                                                                 const __grid_constant__ WParam<D> wp,
                                                                 long long ntok, uint32_t* __restrict__ cq,
                                                                 uint32_t* __restrict__ ck)
{
    constexpr int VE = 16 / (int)sizeof(T);           // elements per 16-byte chunk
    constexpr int NCH = D / VE;                       // chunks per row
    constexpr int G = NCH < 8 ? NCH : 8;              // chunks loaded ahead
    const long long rows = 2 * ntok;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x; g < rows; g += stride) {
        const bool is_q = g < ntok;
        const long long t = is_q ? g : g - ntok;
        const uint4* row = reinterpret_cast<const uint4*>((is_q ? Q : K) + t * D);
        float acc[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] = 0.f;
#pragma unroll
        for (int c0 = 0; c0 < NCH; c0 += G) {
            uint4 ch[G];
#pragma unroll
            for (int c = 0; c < G; ++c) ch[c] = __ldg(row + c0 + c);
#pragma unroll
            for (int c = 0; c < G; ++c) {
                float xv[VE];
                chunk_to_f32<T>(ch[c], xv);
#pragma unroll
                for (int e = 0; e < VE; ++e) {
                    const int i = (c0 + c) * VE + e;
#pragma unroll
                    for (int j = 0; j < 32; ++j) acc[j] = __fmaf_rn(xv[e], wp.w[i * 32 + j], acc[j]);
                }
            }
        }
        uint32_t code = 0u;
#pragma unroll
        for (int j = 0; j < 32; ++j) code |= (acc[j] > 0.f ? 1u : 0u) << j;
        (is_q ? cq : ck)[t] = code;
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

// The same replay, software-pipelined, for a recent window r >= 2 and
// budgets up to 32 * NR.  A slot replaced at step t holds position t, which
// is no candidate at step t + 1 (t > t + 1 - r), so step t + 1's scan can run
// on registers that do not yet hold step t's replacement: each lane keeps its
// two largest candidate keys, and once step t's victim is known (its
// warp-wide max was reduced while the scan ran) a lane whose largest key
// names that slot falls back to its second.  The victim's registers are then
// updated.  Positions are 0..t-1 and distinct during the replay and B >= r,
// so some slot is always a candidate; the every-slot rule is kept anyway.
template <int NR>
__global__ void __launch_bounds__(64) lsh_replay_pipe_kernel(CacheView cv, PromptArgs pa)
{
    const int B = cv.B, T_ = pa.T, r = cv.r;
    const int lane = threadIdx.x & 31;
    const int unit = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (unit >= cv.U) return;
    const uint32_t* cq = pa.cq + (size_t)unit * T_;
    const uint32_t* ck = pa.ck + (size_t)unit * T_;
    const int n0 = min(T_, B);
    uint32_t code[NR];
    int pos[NR];
    unsigned vmask = 0u;                        // bit i: slot lane + 32 i exists
#pragma unroll
    for (int i = 0; i < NR; ++i) {
        const int s = lane + 32 * i;
        const bool ok = s < n0;
        vmask |= ok ? (1u << i) : 0u;
        pos[i] = ok ? s : INT_MAX;
        code[i] = ok ? ck[s] : 0u;
    }
    // key of register slot i: (distance << 20) | (2^20 - 1 - slot)
    auto slot_key = [&](uint32_t q, int i) -> unsigned {
        return ((unsigned)__popc(q ^ code[i]) << 20) | (0xFFFFFu - (unsigned)(lane + 32 * i));
    };
    auto every_slot_best = [&](uint32_t q) -> unsigned {
        unsigned b = 0u;
#pragma unroll
        for (int i = 0; i < NR; ++i)
            if (vmask >> i & 1u) b = max(b, slot_key(q, i));
        return __reduce_max_sync(kFull, b);
    };
    // put (kcode, p) into the slot that `key` names (selects, no branch: an
    // indexed jump per step cost more than the selects)
    auto replace = [&](unsigned key, uint32_t kcode, int p) {
        const int v = (int)(0xFFFFFu - (key & 0xFFFFFu));
        const int vl = v & 31, iv = v >> 5;
#pragma unroll
        for (int i = 0; i < NR; ++i) {
            const bool hit = (lane == vl) && (i == iv);
            code[i] = hit ? kcode : code[i];
            pos[i] = hit ? p : pos[i];
        }
    };
    // this lane's entry of the current and of the next 32-token batch
    uint32_t qb = 0u, kb = 0u, qn = 0u, kn = 0u;
    {
        const int t0 = B + lane, t1 = B + 32 + lane;
        if (t0 < T_) { qb = cq[t0]; kb = ck[t0]; }
        if (t1 < T_) { qn = cq[t1]; kn = ck[t1]; }
    }
    unsigned prev = 0u;                         // last step's largest candidate key
    uint32_t qprev = 0u, kprev = 0u;
    for (int t = B; t < T_; ++t) {
        const int o = (t - B) & 31;
        if (o == 0 && t > B) {
            qb = qn; kb = kn;
            const int tt = t + 32 + lane;
            qn = tt < T_ ? cq[tt] : 0u;
            kn = tt < T_ ? ck[tt] : 0u;
        }
        const uint32_t q = __shfl_sync(kFull, qb, o);
        const uint32_t knew = __shfl_sync(kFull, kb, o);
        const int tr = t - r;
        unsigned b1 = 0u, b2 = 0u;
#pragma unroll
        for (int i = 0; i < NR; ++i) {
            const unsigned k = pos[i] <= tr ? slot_key(q, i) : 0u;
            b2 = max(b2, min(b1, k));
            b1 = max(b1, k);
        }
        if (t > B) {
            if (prev == 0u) prev = every_slot_best(qprev);
            if ((b1 & 0xFFFFFu) == (prev & 0xFFFFFu)) b1 = b2;
            replace(prev, kprev, t - 1);
        }
        prev = __reduce_max_sync(kFull, b1);
        qprev = q;
        kprev = knew;
    }
    if (T_ > B) {
        if (prev == 0u) prev = every_slot_best(qprev);
        replace(prev, kprev, T_ - 1);
    }
    const size_t ub = (size_t)unit * B;
#pragma unroll
    for (int i = 0; i < NR; ++i) {
        const int s = lane + 32 * i;
        if (s < B) cv.pos[ub + s] = (vmask >> i & 1u) ? pos[i] : -1;
    }
    if (lane == 0) cv.ustate[unit] = make_int2(n0, T_);
}

// The pipelined replay with one CTA of WU warps per unit (recent window
// r >= 2, budgets up to 32 WU NR): thread tid owns slots tid + 32 WU i, so a
// step scans NR slots per thread instead of B / 32, and the warps' largest
// keys meet through shared memory (one buffer per step parity) and one CTA
// barrier.  Same rule, keys and pipelining as lsh_replay_pipe_kernel:
// step t + 1's scan runs before step t's victim is applied (that slot holds
// position t, no candidate at t + 1), each thread keeping its two largest
// candidate keys.
template <int NR, int WU>
__global__ void __launch_bounds__(32 * WU) lsh_replay_wide_kernel(CacheView cv, PromptArgs pa)
{
    constexpr int NT = 32 * WU;
    __shared__ unsigned red[2][WU];
    const int B = cv.B, T_ = pa.T, r = cv.r;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int unit = blockIdx.x;
    const uint32_t* cq = pa.cq + (size_t)unit * T_;
    const uint32_t* ck = pa.ck + (size_t)unit * T_;
    const int n0 = min(T_, B);
    uint32_t code[NR];
    int pos[NR];
    unsigned vmask = 0u;                        // bit i: slot tid + NT i exists
#pragma unroll
    for (int i = 0; i < NR; ++i) {
        const int s = tid + NT * i;
        const bool ok = s < n0;
        vmask |= ok ? (1u << i) : 0u;
        pos[i] = ok ? s : INT_MAX;
        code[i] = ok ? ck[s] : 0u;
    }
    auto slot_key = [&](uint32_t q, int i) -> unsigned {
        return ((unsigned)__popc(q ^ code[i]) << 20) | (0xFFFFFu - (unsigned)(tid + NT * i));
    };
    // the CTA-wide max of every thread's `v` (parity: the step's buffer)
    auto cta_max = [&](unsigned v, int parity) -> unsigned {
        v = __reduce_max_sync(kFull, v);
        if (lane == 0) red[parity][warp] = v;
        __syncthreads();
        unsigned m = red[parity][0];
#pragma unroll
        for (int w = 1; w < WU; ++w) m = max(m, red[parity][w]);
        return m;
    };
    auto every_slot_best = [&](uint32_t q, int parity) -> unsigned {
        unsigned b = 0u;
#pragma unroll
        for (int i = 0; i < NR; ++i)
            if (vmask >> i & 1u) b = max(b, slot_key(q, i));
        return cta_max(b, parity);
    };
    auto replace = [&](unsigned key, uint32_t kcode, int p) {
        const int v = (int)(0xFFFFFu - (key & 0xFFFFFu));
        const int vt = v % NT, iv = v / NT;
#pragma unroll
        for (int i = 0; i < NR; ++i) {
            const bool hit = (tid == vt) && (i == iv);
            code[i] = hit ? kcode : code[i];
            pos[i] = hit ? p : pos[i];
        }
    };
    uint32_t qb = 0u, kb = 0u, qn = 0u, kn = 0u;
    {
        const int t0 = B + lane, t1 = B + 32 + lane;
        if (t0 < T_) { qb = cq[t0]; kb = ck[t0]; }
        if (t1 < T_) { qn = cq[t1]; kn = ck[t1]; }
    }
    unsigned prev = 0u;
    uint32_t qprev = 0u, kprev = 0u;
    int par = 0;                                // parity of the reduction buffer
    for (int t = B; t < T_; ++t) {
        const int o = (t - B) & 31;
        if (o == 0 && t > B) {
            qb = qn; kb = kn;
            const int tt = t + 32 + lane;
            qn = tt < T_ ? cq[tt] : 0u;
            kn = tt < T_ ? ck[tt] : 0u;
        }
        const uint32_t q = __shfl_sync(kFull, qb, o);
        const uint32_t knew = __shfl_sync(kFull, kb, o);
        const int tr = t - r;
        unsigned b1 = 0u, b2 = 0u;
#pragma unroll
        for (int i = 0; i < NR; ++i) {
            const unsigned k = pos[i] <= tr ? slot_key(q, i) : 0u;
            b2 = max(b2, min(b1, k));
            b1 = max(b1, k);
        }
        if (t > B) {
            if (prev == 0u) {
                prev = every_slot_best(qprev, par);
                par ^= 1;
            }
            if ((b1 & 0xFFFFFu) == (prev & 0xFFFFFu)) b1 = b2;
            replace(prev, kprev, t - 1);
        }
        prev = cta_max(b1, par);
        par ^= 1;
        qprev = q;
        kprev = knew;
    }
    if (T_ > B) {
        if (prev == 0u) prev = every_slot_best(qprev, par);
        replace(prev, kprev, T_ - 1);
    }
    const size_t ub = (size_t)unit * B;
#pragma unroll
    for (int i = 0; i < NR; ++i) {
        const int s = tid + NT * i;
        if (s < B) cv.pos[ub + s] = (vmask >> i & 1u) ? pos[i] : -1;
    }
    if (tid == 0) cv.ustate[unit] = make_int2(n0, T_);
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
    const int G = p.G > 1 ? p.G : 1;
    rowstats_kernel<T, D><<<grid, 256, smem, st>>>(reinterpret_cast<const T*>(p.Q),
                                                 reinterpret_cast<const T*>(p.K), p.T, G, c.qscale, p.m2, p.l);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    colsum_kernel<T, D><<<grid, 256, smem, st>>>(reinterpret_cast<const T*>(p.Q),
                                               reinterpret_cast<const T*>(p.K), p.T, G, c.qscale, p.m2, p.l,
                                               p.c, p.bandB, p.bandr, p.wB, p.wr);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t gather_t(const CacheView& c, const PromptArgs& p, bool with_codes, cudaStream_t st)
{
    const long long warps = ((long long)c.U * c.B + kGatherSlots - 1) / kGatherSlots;
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
cudaError_t lsh_t(const CacheView& c, const PromptArgs& p, const float* W_host, cudaStream_t st)
{
    const long long ntok = (long long)c.U * p.T;
    int sms = 0, dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    long long blocks = (2 * ntok + kCodeThreads - 1) / kCodeThreads;
    if (blocks > 8LL * sms) blocks = 8LL * sms;
    WParam<D> wp;
    memcpy(wp.w, W_host, sizeof(wp.w));
    lsh_codes_kernel<T, D><<<(unsigned)blocks, kCodeThreads, 0, st>>>(
        reinterpret_cast<const T*>(p.Q), reinterpret_cast<const T*>(p.K), wp, ntok, p.cq, p.ck);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (c.r >= 2 && c.B > 96 && c.B <= 128 * 4) {
        // four warps per unit, one CTA each (measured against two and eight
        // warps: 538 / 599 / 598 us for the OPT-6.7B-shaped layer's prompt phase)
        const int nr = (c.B + 127) / 128;
        if (nr <= 1) lsh_replay_wide_kernel<1, 4><<<(unsigned)c.U, 128, 0, st>>>(c, p);
        else if (nr <= 2) lsh_replay_wide_kernel<2, 4><<<(unsigned)c.U, 128, 0, st>>>(c, p);
        else if (nr <= 3) lsh_replay_wide_kernel<3, 4><<<(unsigned)c.U, 128, 0, st>>>(c, p);
        else lsh_replay_wide_kernel<4, 4><<<(unsigned)c.U, 128, 0, st>>>(c, p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        return gather_t<T, D>(c, p, true, st);
    }
    if (c.r >= 2 && c.B <= 32 * 16) {
        const unsigned blocks = (unsigned)((c.U + 1) / 2);
        const int nr = (c.B + 31) / 32;
        if (nr <= 1) lsh_replay_pipe_kernel<1><<<blocks, 64, 0, st>>>(c, p);
        else if (nr <= 2) lsh_replay_pipe_kernel<2><<<blocks, 64, 0, st>>>(c, p);
        else if (nr <= 4) lsh_replay_pipe_kernel<4><<<blocks, 64, 0, st>>>(c, p);
        else if (nr <= 8) lsh_replay_pipe_kernel<8><<<blocks, 64, 0, st>>>(c, p);
        else if (nr <= 13) lsh_replay_pipe_kernel<13><<<blocks, 64, 0, st>>>(c, p);
        else lsh_replay_pipe_kernel<16><<<blocks, 64, 0, st>>>(c, p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        return gather_t<T, D>(c, p, true, st);
    }
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

namespace {

// Pivotal histories of the prompt (persistence of importance): the last
// WR = min(T, 32) query rows are steps; key j is pivotal for row i (j <= i)
// when its probability exceeds the uniform share, P_ij (i + 1) > 1.  Lane r
// of every warp holds row i0 + r (its scaled query in registers); each warp
// takes every NW-th key of a shared-memory tile and dots it with all rows at
// once (the key is broadcast to the lanes).  Pass 1: each lane's online
// (max, sum) over its warp's keys, merged across warps; pass 2 recomputes
// the logits, and the ballot of a key's flags, bit-reversed, is its history
// (bit T-1-i = row i).  Writes ck[j] = history and c[j] = set bits * T + j,
// a key that orders kept tokens by importance and then by newer position.
// Key tiles are fetched with 16-byte loads into registers one tile ahead
// (the next pass's first tile after a pass's last), so their latency
// overlaps the current tile's dot products.
constexpr int kShWarps = 4, kShTile = 32;

template <typename T, int D>
__global__ void __launch_bounds__(kShWarps * 32) sh_masks_kernel(const T* __restrict__ Q, const T* __restrict__ K,
                                                                int T_, float qscale, uint32_t* __restrict__ ck,
                                                                double* __restrict__ cout)
{
    __shared__ __align__(16) float ks[kShTile][D];
    __shared__ float wm[kShWarps][32], wl[kShWarps][32];
    const int unit = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int i0 = T_ > 32 ? T_ - 32 : 0, WR = T_ - i0;
    const int i = i0 + lane;                    // this lane's query row
    const bool row_ok = lane < WR;
    const T* Qu = Q + (size_t)unit * T_ * D;
    const T* Ku = K + (size_t)unit * T_ * D;
    float2 q2[D / 2];
#pragma unroll
    for (int e = 0; e < D / 2; ++e) {
        const float a = row_ok ? Elem<T>::to_f(Qu[(size_t)i * D + 2 * e]) : 0.f;
        const float b = row_ok ? Elem<T>::to_f(Qu[(size_t)i * D + 2 * e + 1]) : 0.f;
        q2[e] = make_float2(a * qscale, b * qscale);
    }
    constexpr int NT = kShWarps * 32;
    constexpr int VE = 16 / (int)sizeof(T);          // elements per 16-byte vector
    constexpr int RV = D / VE;                       // vectors per key row
    constexpr int VPT = kShTile * RV / NT;           // vectors per thread per tile
    static_assert(kShTile * RV % NT == 0, "a tile splits evenly over the threads");
    uint4 nxt[VPT];
    auto fetch = [&](int j0) {
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int x = tid + v * NT, jj = x / RV, cv = x - jj * RV;
            nxt[v] = (j0 + jj < T_) ? reinterpret_cast<const uint4*>(Ku + (size_t)(j0 + jj) * D)[cv]
                                    : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    // the fetched tile into shared memory, then the next fetch goes out
    auto stage = [&](int j0) {
        __syncthreads();                             // the previous tile is consumed
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int x = tid + v * NT, jj = x / RV, cv = x - jj * RV;
            float f[VE];
            chunk_to_f32<T>(nxt[v], f);
#pragma unroll
            for (int e = 0; e < VE; e += 4)
                *reinterpret_cast<float4*>(&ks[jj][cv * VE + e]) = make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
        }
        __syncthreads();
        fetch(j0 + kShTile < T_ ? j0 + kShTile : 0);
    };
    fetch(0);
    // logits of this lane's row against KG consecutive keys of the tile
    // (KG independent multiply-add chains)
    constexpr int KG = 4, KPW = kShTile / kShWarps;  // keys per group, keys per warp
    static_assert(KPW % KG == 0, "a warp's keys split into groups");
    auto logits = [&](int jj, float (&z)[KG]) {
        float2 acc[KG];
#pragma unroll
        for (int g = 0; g < KG; ++g) acc[g] = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < D / 4; ++e) {
#pragma unroll
            for (int g = 0; g < KG; ++g) {
                const float4 kv = reinterpret_cast<const float4*>(ks[jj + g])[e];
                acc[g] = __ffma2_rn(q2[2 * e], make_float2(kv.x, kv.y), acc[g]);
                acc[g] = __ffma2_rn(q2[2 * e + 1], make_float2(kv.z, kv.w), acc[g]);
            }
        }
#pragma unroll
        for (int g = 0; g < KG; ++g) z[g] = acc[g].x + acc[g].y;
    };
    // pass 1: row max and normaliser (base 2) over the keys j <= i
    float m = -INFINITY, l = 0.f;
    for (int j0 = 0; j0 < T_; j0 += kShTile) {
        stage(j0);
        for (int jg = warp * KPW; jg < warp * KPW + KPW; jg += KG) {
            float z[KG];
            logits(jg, z);
#pragma unroll
            for (int g = 0; g < KG; ++g) {
                const int j = j0 + jg + g;
                if (row_ok && j <= i) {
                    if (z[g] > m) { l = l * exp2f(m - z[g]) + 1.f; m = z[g]; }
                    else l += exp2f(z[g] - m);
                }
            }
        }
    }
    wm[warp][lane] = m;
    wl[warp][lane] = l;
    __syncthreads();
    float M = -INFINITY, L = 0.f;
#pragma unroll
    for (int w = 0; w < kShWarps; ++w) M = fmaxf(M, wm[w][lane]);
#pragma unroll
    for (int w = 0; w < kShWarps; ++w) L += (wm[w][lane] == -INFINITY) ? 0.f : wl[w][lane] * exp2f(wm[w][lane] - M);
    const float share = row_ok ? (float)(i + 1) / L : 0.f;   // P (i + 1) = exp2(z - M) * share
    // pass 2: flags
    for (int j0 = 0; j0 < T_; j0 += kShTile) {
        stage(j0);
        for (int jg = warp * KPW; jg < warp * KPW + KPW; jg += KG) {
            float z[KG];
            logits(jg, z);
#pragma unroll
            for (int g = 0; g < KG; ++g) {
                const int j = j0 + jg + g;
                const bool f = row_ok && j <= i && exp2f(z[g] - M) * share > 1.f;
                const unsigned bits = __ballot_sync(0xffffffffu, f);
                if (lane == g && j < T_) {
                    const uint32_t h = __brev(bits) >> (32 - WR);
                    ck[(size_t)unit * T_ + j] = h;
                    cout[(size_t)unit * T_ + j] = (double)__popc(h) * (double)T_ + (double)j;
                }
            }
        }
    }
}

template <typename T, int D>
cudaError_t sh_masks_t(const CacheView& c, const PromptArgs& p, cudaStream_t st)
{
    sh_masks_kernel<T, D><<<(unsigned)c.U, kShWarps * 32, 0, st>>>(
        reinterpret_cast<const T*>(p.Q), reinterpret_cast<const T*>(p.K), p.T, c.qscale, p.ck, p.c);
    return cudaGetLastError();
}

// A cache unit's column sums: its heads' sums added in head order.
__global__ void group_sum_kernel(const double* __restrict__ c, double* __restrict__ ckv, int U, int G, int T_)
{
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)U * T_) return;
    const long long u = i / T_, j = i - u * T_;
    const double* cu = c + (size_t)u * G * T_ + j;
    double s = 0.0;
    for (int g = 0; g < G; ++g) s += cu[(size_t)g * T_];
    ckv[i] = s;
}

}  // namespace

cudaError_t launch_sh_prompt(const CacheView& c, const PromptArgs& p, cudaStream_t st)
{
    const bool bf = c.dtype == 1;
    cudaError_t e;
    if (prompt_tc_supported(c) && p.m2 && p.l && !getenv_flag("H2O_PROMPT_CUDA_CORES")) e = launch_sh_flags_tc(c, p, st);
    else if (c.D == 128) e = bf ? sh_masks_t<__nv_bfloat16, 128>(c, p, st) : sh_masks_t<float, 128>(c, p, st);
    else if (c.D == 64) e = bf ? sh_masks_t<__nv_bfloat16, 64>(c, p, st) : sh_masks_t<float, 64>(c, p, st);
    else return cudaErrorInvalidValue;
    if (e == cudaSuccess) e = launch_select(c, p, st);
    if (e == cudaSuccess) e = launch_gather(c, p, true, st);
    return e;
}

cudaError_t launch_group_sum(const double* c, double* ckv, int U, int G, int T, cudaStream_t st)
{
    const long long n = (long long)U * T;
    group_sum_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(c, ckv, U, G, T);
    return cudaGetLastError();
}

cudaError_t launch_select(const CacheView& c, const PromptArgs& p, cudaStream_t st)
{
    // a block of 256 threads for prompts up to 4096 tokens (more units per
    // SM), 1024 above
    // keys in registers up to 4096 candidates (16 a thread); longer prompts
    // read them from L2 each round
    if (p.T <= 4096) select_kernel<256, 16><<<(unsigned)c.U, 256, 0, st>>>(c, p);
    else select_kernel<1024, 1><<<(unsigned)c.U, 1024, 0, st>>>(c, p);
    return cudaGetLastError();
}

// The selection with the kept rows' copy in the same kernel, for prompts up
// to 4096 tokens (one CTA of 256 threads per unit: enough units to cover the
// SMs) and rows kept as they are; longer prompts (few units would leave
// most SMs out of the copy) and quantised rows (their copy is arithmetic:
// measured 50 us slower per OPT-30B-shaped layer inside the selection's
// CTAs) select, then gather in a kernel of their own.
cudaError_t launch_select_gather(const CacheView& c, const PromptArgs& p, cudaStream_t st)
{
    if (p.T > 4096 || c.qbits) {
        cudaError_t e = launch_select(c, p, st);
        return e != cudaSuccess ? e : launch_gather(c, p, false, st);
    }
    const bool bf = c.dtype == 1;
    const unsigned grid = (unsigned)c.U;
    if (c.D == 128) {
        if (bf) select_kernel<256, 16, __nv_bfloat16, 128><<<grid, 256, 0, st>>>(c, p);
        else select_kernel<256, 16, float, 128><<<grid, 256, 0, st>>>(c, p);
    } else if (c.D == 64) {
        if (bf) select_kernel<256, 16, __nv_bfloat16, 64><<<grid, 256, 0, st>>>(c, p);
        else select_kernel<256, 16, float, 64><<<grid, 256, 0, st>>>(c, p);
    } else {
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_fg_policy(const CacheView& c, const PromptArgs& p, const FgArgs& f, cudaStream_t st)
{
    fg_policy_kernel<<<(unsigned)c.U, 256, 0, st>>>(c, p, f);
    return cudaGetLastError();
}

// The per-head policies' decode lists ["Model Tells You What to Discard"
// review page, method section: each head keeps its own policy's cache]:
// one CTA writes the units of the compressed policies (0, 1) and of the
// full cache (2), each list in unit order (a ballot and a running offset
// per 1024 units), so that each decode step can launch over each budget
// class with a split of its own.
__global__ void __launch_bounds__(1024) fg_lists_kernel(const int4* __restrict__ upol, int U, int* __restrict__ lists,
                                                        int* __restrict__ counts)
{
    __shared__ int wsum[2][32];
    __shared__ int base[2];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) { base[0] = 0; base[1] = 0; }
    __syncthreads();
    for (int u0 = 0; u0 < U; u0 += 1024) {
        const int u = u0 + tid;
        const bool live = u < U;
        const bool full = live && upol[u].w == 2;
        const unsigned mf = __ballot_sync(0xffffffffu, full), ms = __ballot_sync(0xffffffffu, live && !full);
        if (lane == 0) { wsum[0][warp] = __popc(ms); wsum[1][warp] = __popc(mf); }
        __syncthreads();
        int off0 = base[0], off1 = base[1];
        for (int w = 0; w < warp; ++w) { off0 += wsum[0][w]; off1 += wsum[1][w]; }
        const unsigned below = (1u << lane) - 1u;
        if (live && !full) lists[off0 + __popc(ms & below)] = u;
        if (full) lists[U + off1 + __popc(mf & below)] = u;
        __syncthreads();
        if (tid == 0) {
            for (int w = 0; w < 32; ++w) { base[0] += wsum[0][w]; base[1] += wsum[1][w]; }
        }
        __syncthreads();
    }
    if (tid == 0) { counts[0] = base[0]; counts[1] = base[1]; }
}

cudaError_t launch_fg_lists(const int4* upol, int U, int* lists, int* counts, cudaStream_t st)
{
    fg_lists_kernel<<<1, 1024, 0, st>>>(upol, U, lists, counts);
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

cudaError_t launch_lsh_prompt(const CacheView& c, const PromptArgs& p, const float* W, const float* W_host,
                              cudaStream_t st)
{
    (void)W;
    if (!W_host) return cudaErrorInvalidValue;
    const bool bf = c.dtype == 1;
    if (c.D == 128) return bf ? lsh_t<__nv_bfloat16, 128>(c, p, W_host, st) : lsh_t<float, 128>(c, p, W_host, st);
    if (c.D == 64) return bf ? lsh_t<__nv_bfloat16, 64>(c, p, W_host, st) : lsh_t<float, 64>(c, p, W_host, st);
    return cudaErrorInvalidValue;
}

}  // namespace h2o
