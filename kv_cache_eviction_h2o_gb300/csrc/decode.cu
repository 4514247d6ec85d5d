// decode.cu -- one decode step over every (batch, head) unit's budgeted cache.
//
// H2O step [H2O review page, 提案手法: accumulated attention ranks tokens,
// a greedy per-step eviction from local attention statistics; Scissorhands
// abstract: fixed budget]:
//   attend over the live slots and the new token, add each slot's
//   probability to its score, evict the lowest-score slot outside the recent
//   window (lowest slot on ties), write the new token there.
// HashEvict step [HashEvict abstract]: pick the victim before attention by
//   the largest Hamming distance between the query code and the key codes
//   (outside the recent window, lowest slot on ties), write the new token
//   there, then attend over the cache.
//
// Layout and parallel plan (GB300): a unit's slots are split into `split`
// contiguous chunks, one CTA each, the CTAs of a unit forming one
// thread-block cluster.  Inside a CTA every warp streams its own 8-slot
// groups of K and V rows with 1-D bulk copies (TMA) into a private ring of
// shared-memory buffers completed on mbarriers, and keeps its own online
// softmax (base-2 logits).  Warps merge through shared memory, CTAs merge
// through distributed shared memory into cluster rank 0.  H2O needs the
// global normaliser before any score update, so the cluster exchanges
// (max, sum) once, every CTA updates its own slots' scores from the logits
// it kept in shared memory (P never goes to HBM), and a second exchange
// reduces the arg-min.  Every wait is bounded; a wait that runs out sets the
// handle's error word.
#include <cfloat>
#include <climits>
#include <cstdlib>

#include "common.cuh"
#include "kernels.h"

namespace h2o {

namespace {

constexpr int kMaxSplit = 16;              // CTAs per cluster (non-portable above 8)
constexpr int kMaxChunk = 1024;            // slots per CTA
constexpr unsigned kFull = 0xffffffffu;

// Tile shape of the decode kernels: NW warps per CTA, each streaming groups of
// G slots through a private ring of NBUF shared-memory buffers.
template <int NW_, int G_, int NBUF_>
struct Tile {
    static constexpr int NW = NW_, NT = 32 * NW_, G = G_, NBUF = NBUF_;
    static constexpr int SPT = kMaxChunk / NT;            // slots per thread in the score pass
    static constexpr int LOG2G = G_ == 8 ? 3 : (G_ == 4 ? 2 : 1);
    static_assert(G_ == 2 || G_ == 4 || G_ == 8, "group size");
};

template <int D>
struct Exchange {                 // every CTA has one; rank 0's is the meeting point
    float m[kMaxSplit];           // per-CTA running max (base 2)
    float l[kMaxSplit];           // per-CTA normaliser at that max
    double cand_score[kMaxSplit]; // per-CTA arg-min over eviction candidates
    double all_score[kMaxSplit];  // per-CTA arg-min over every live slot
    int cand_slot[kMaxSplit];
    int all_slot[kMaxSplit];
    float o[kMaxSplit][D];        // per-CTA unnormalised output
};

template <typename T, int D, class TL>
struct DecodeSmem {
    T buf[TL::NW][TL::NBUF][2][TL::G * D];   // per-warp ring: [K rows | V rows]
    uint64_t bar[TL::NW][TL::NBUF];
    Exchange<D> x;
    float z[kMaxChunk];                   // base-2 logits of this CTA's slots
    float wo[TL::NW][D];
    alignas(16) float e[TL::NW][TL::G < 4 ? 4 : TL::G];
    float wm[TL::NW];
    float wl[TL::NW];
    float qf[D];
    float kf[D];
    double rd[2][TL::NW];
    int ri[2][TL::NW];
    unsigned long long ru[2][TL::NW];
    float M, invL, z_new, P_new;
    int victim;
    unsigned code_q, code_k;
};

// Sum G per-lane partials over the warp: each exchange level keeps half of
// the live partials and sends the other half, so lane l ends up with the
// total of partial j, j read from lane bits 4, 3, ... (most significant
// first); log2(G) + (5 - log2(G)) = 5 shuffle levels, G - 1 + 5 - log2(G)
// shuffles instead of 5 G.
template <int G>
__device__ __forceinline__ float reduce_transposed(float (&v)[G], int lane)
{
#pragma unroll
    for (int k = 0; (G >> k) > 1; ++k) {
        const int half = (G >> k) / 2;
        const bool up = (lane >> (4 - k)) & 1;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float keep = up ? v[i + half] : v[i];
            const float send = up ? v[i] : v[i + half];
            v[i] = keep + __shfl_xor_sync(kFull, send, 16 >> k);
        }
    }
    float c = v[0];
    constexpr int lg = G == 8 ? 3 : (G == 4 ? 2 : 1);
#pragma unroll
    for (int o = 16 >> lg; o > 0; o >>= 1) c += __shfl_xor_sync(kFull, c, o);
    return c;
}

// slot (within a group of G) whose total lane `lane` holds after the reduction
template <int G>
__device__ __forceinline__ int owned_slot(int lane)
{
    constexpr int lg = G == 8 ? 3 : (G == 4 ? 2 : 1);
    return (lane >> (5 - lg)) & (G - 1);
}

__device__ __forceinline__ float safe_exp2_diff(float a, float m)
{
    return (a == -INFINITY) ? 0.f : exp2f(a - m);
}

// Per-warp streaming online softmax over this CTA's chunk [c0, c1) of live
// slots.  `skip` (absolute slot) is left out of the softmax.  When keep_z,
// logits are stored in S.z[slot - c0].  Returns through (m_run, l_run, o).
template <typename T, int D, class TL>
__device__ __forceinline__ void attend_chunk(DecodeSmem<T, D, TL>& S, const T* Kc, const T* Vc,
                                             int c0, int c1, int skip, bool keep_z,
                                             const float (&qr)[D / 32], float& m_run,
                                             float& l_run, float (&o)[D / 32], int* err)
{
    constexpr int EPL = D / 32;
    constexpr int G = TL::G, NW = TL::NW, NBUF = TL::NBUF;
    constexpr int OWN = (1 << (5 - TL::LOG2G)) - 1;     // lanes sharing one slot's total
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int len = c1 - c0;
    const int ngroups = (len + G - 1) / G;
    bool timed_out = false;
    int it = 0;
    for (int g = warp; g < ngroups; g += NW, ++it) {
        const int b = it % NBUF;
        const uint32_t parity = (uint32_t)(it / NBUF) & 1u;
        if (!mbar_wait(&S.bar[warp][b], parity)) {
            if (!timed_out && lane == 0) atomicOr(err, kErrWaitTimeout);
            timed_out = true;
        }
        const T* kb = S.buf[warp][b][0];
        const T* vb = S.buf[warp][b][1];
        const int s0 = g * G;                     // chunk-relative first slot
        const int gl = min(G, len - s0);

        float part[G];
#pragma unroll
        for (int j = 0; j < G; ++j) {
            float kr[EPL];
            load_vec<T, EPL>(kb + j * D + lane * EPL, kr);
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc = fmaf(qr[e], kr[e], acc);
            part[j] = acc;
        }
        float zj = reduce_transposed<G>(part, lane);
        const int jl = owned_slot<G>(lane);
        if (jl >= gl || c0 + s0 + jl == skip) zj = -INFINITY;
        float gm = zj;
#pragma unroll
        for (int sh = 16; sh > OWN; sh >>= 1) gm = fmaxf(gm, __shfl_xor_sync(kFull, gm, sh));
        const float m_new = fmaxf(m_run, gm);
        const float alpha = safe_exp2_diff(m_run, m_new);
        const float ej = safe_exp2_diff(zj, m_new);
        if ((lane & OWN) == 0) {
            S.e[warp][jl] = ej;
            if (keep_z && jl < gl) S.z[s0 + jl] = zj;
        }
        __syncwarp();
        float ev[G];
#pragma unroll
        for (int j = 0; j < G; j += 4) {
            if (j + 4 <= G) {
                const float4 e4 = *reinterpret_cast<const float4*>(&S.e[warp][j]);
                ev[j] = e4.x; ev[j + 1] = e4.y; ev[j + 2] = e4.z; ev[j + 3] = e4.w;
            }
        }
        if (G < 4) {
#pragma unroll
            for (int j = 0; j < G; ++j) ev[j] = S.e[warp][j];
        }
        float esum = 0.f;
#pragma unroll
        for (int j = 0; j < G; ++j) esum += ev[j];
        if (m_new != -INFINITY) {
            l_run = l_run * alpha + esum;
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[e] *= alpha;
            m_run = m_new;
        }
#pragma unroll
        for (int j = 0; j < G; ++j) {
            if (j < gl) {
                float vr[EPL];
                load_vec<T, EPL>(vb + j * D + lane * EPL, vr);
#pragma unroll
                for (int e = 0; e < EPL; ++e) o[e] = fmaf(ev[j], vr[e], o[e]);
            }
        }
        __syncwarp();
        // refill this buffer with the warp's group NBUF rounds ahead
        if (lane == 0) {
            const int gn = g + NW * NBUF;
            if (gn < ngroups) {
                const int s = c0 + gn * G;
                const uint32_t bytes = (uint32_t)(min(G, c1 - s) * D * sizeof(T));
                mbar_arrive_expect_tx(&S.bar[warp][b], 2 * bytes);
                bulk_g2s(S.buf[warp][b][0], Kc + (size_t)s * D, bytes, &S.bar[warp][b]);
                bulk_g2s(S.buf[warp][b][1], Vc + (size_t)s * D, bytes, &S.bar[warp][b]);
            }
        }
    }
}

// Kick off the first NBUF groups of each warp (called by lane 0 of every warp
// after its barriers are initialised).
template <typename T, int D, class TL>
__device__ __forceinline__ void prime_ring(DecodeSmem<T, D, TL>& S, const T* Kc, const T* Vc,
                                           int c0, int c1)
{
    const int warp = threadIdx.x >> 5;
    const int ngroups = (c1 - c0 + TL::G - 1) / TL::G;
#pragma unroll
    for (int b = 0; b < TL::NBUF; ++b) {
        const int g = warp + TL::NW * b;
        if (g < ngroups) {
            const int s = c0 + g * TL::G;
            const uint32_t bytes = (uint32_t)(min(TL::G, c1 - s) * D * sizeof(T));
            mbar_arrive_expect_tx(&S.bar[warp][b], 2 * bytes);
            bulk_g2s(S.buf[warp][b][0], Kc + (size_t)s * D, bytes, &S.bar[warp][b]);
            bulk_g2s(S.buf[warp][b][1], Vc + (size_t)s * D, bytes, &S.bar[warp][b]);
        }
    }
}

// Merge the warps' softmax states; threads < D get their output column.
template <typename T, int D, class TL>
__device__ __forceinline__ void merge_warps(DecodeSmem<T, D, TL>& S, float m_run, float l_run,
                                            const float (&o)[D / 32], float& Mc, float& Lc,
                                            float& Oc)
{
    constexpr int EPL = D / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (lane == 0) { S.wm[warp] = m_run; S.wl[warp] = l_run; }
#pragma unroll
    for (int e = 0; e < EPL; ++e) S.wo[warp][lane * EPL + e] = o[e];
    __syncthreads();
    Mc = -INFINITY;
#pragma unroll
    for (int w = 0; w < TL::NW; ++w) Mc = fmaxf(Mc, S.wm[w]);
    Lc = 0.f;
    Oc = 0.f;
#pragma unroll
    for (int w = 0; w < TL::NW; ++w) {
        const float f = safe_exp2_diff(S.wm[w], Mc);
        Lc += S.wl[w] * f;
        if (tid < D) Oc += S.wo[w][tid] * f;
    }
}

template <typename T, int D>
__device__ __forceinline__ void copy_row(T* dst, const T* src, int t)
{
    constexpr int NV = D * (int)sizeof(T) / 16;
    if (t < NV) reinterpret_cast<uint4*>(dst)[t] = reinterpret_cast<const uint4*>(src)[t];
}

// ------------------------------------------------------------------ H2O

template <typename T, int D, class TL>
__global__ void __launch_bounds__(TL::NT) h2o_decode_kernel(const DecodeArgs a)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    auto& S = *reinterpret_cast<DecodeSmem<T, D, TL>*>(smem_raw);
    constexpr int EPL = D / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const CacheView& c = a.c;
    const int C = (int)cluster_nctarank();
    const int rank = (int)cluster_ctarank();
    const int unit = blockIdx.x / C;
    cluster_arrive_relaxed();     // paired with the wait before the first remote store

    const int B = c.B;
    const int2 us = c.ustate[unit];
    const int n = us.x, p = us.y;
    const bool full = (n >= B);
    int cs = (n + C - 1) / C;
    cs = (cs + TL::G - 1) / TL::G * TL::G;
    const int c0 = min(n, rank * cs), c1 = min(n, c0 + cs);
    const size_t ub = (size_t)unit * B;
    T* Kc = reinterpret_cast<T*>(c.K) + ub * D;
    T* Vc = reinterpret_cast<T*>(c.V) + ub * D;

    if (lane == 0) {
#pragma unroll
        for (int b = 0; b < TL::NBUF; ++b) mbar_init(&S.bar[warp][b], 1);
        fence_mbar_init();
        prime_ring<T, D, TL>(S, Kc, Vc, c0, c1);
    }

    // scores and positions of this thread's slots, consumed after the merge
    double sc_old[TL::SPT];
    int ps[TL::SPT];
#pragma unroll
    for (int i = 0; i < TL::SPT; ++i) {
        const int s = c0 + tid + i * TL::NT;
        sc_old[i] = 0.0;
        ps[i] = 0;
        if (s < c1) { sc_old[i] = c.score[ub + s]; ps[i] = c.pos[ub + s]; }
    }

    float qr[EPL];
    load_vec<T, EPL>(reinterpret_cast<const T*>(a.q) + (size_t)unit * D + lane * EPL, qr);
#pragma unroll
    for (int e = 0; e < EPL; ++e) qr[e] *= c.qscale;

    float m_run = -INFINITY, l_run = 0.f, o[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] = 0.f;
    if (rank == 0 && warp == 0) {          // the new token attends to itself
        float kr[EPL], vr[EPL];
        load_vec<T, EPL>(reinterpret_cast<const T*>(a.k) + (size_t)unit * D + lane * EPL, kr);
        load_vec<T, EPL>(reinterpret_cast<const T*>(a.v) + (size_t)unit * D + lane * EPL, vr);
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc = fmaf(qr[e], kr[e], acc);
        const float zn = warp_sum(acc);
        m_run = zn;
        l_run = 1.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] = vr[e];
        if (lane == 0) S.z_new = zn;
    }
    __syncwarp();

    attend_chunk<T, D, TL>(S, Kc, Vc, c0, c1, -1, true, qr, m_run, l_run, o, c.err);

    float Mc, Lc, Oc;
    merge_warps<T, D, TL>(S, m_run, l_run, o, Mc, Lc, Oc);

    // exchange 1: (max, normaliser, output) of every CTA into rank 0
    cluster_wait();
    const uint32_t x0 = map_to_rank(&S.x, 0);
    const uint32_t off_m = (uint32_t)offsetof(Exchange<D>, m), off_l = (uint32_t)offsetof(Exchange<D>, l);
    const uint32_t off_o = (uint32_t)offsetof(Exchange<D>, o);
    if (tid < D) st_cluster_f32(x0 + off_o + (uint32_t)((rank * D + tid) * 4), Oc);
    if (tid == 0) {
        st_cluster_f32(x0 + off_m + rank * 4, Mc);
        st_cluster_f32(x0 + off_l + rank * 4, Lc);
    }
    cluster_arrive();
    cluster_wait();

    if (warp == 0) {
        const float mj = lane < C ? ld_cluster_f32(x0 + off_m + lane * 4) : -INFINITY;
        const float lj = lane < C ? ld_cluster_f32(x0 + off_l + lane * 4) : 0.f;
        const float M = warp_max(mj);
        const float L = warp_sum(lane < C ? lj * safe_exp2_diff(mj, M) : 0.f);
        if (lane == 0) { S.M = M; S.invL = 1.f / L; }
    }
    __syncthreads();
    const float M = S.M, invL = S.invL;

    // accumulate this step's probabilities; arg-min over candidates
    double best = DBL_MAX, best_all = DBL_MAX;
    int bslot = INT_MAX, bslot_all = INT_MAX;
#pragma unroll
    for (int i = 0; i < TL::SPT; ++i) {
        const int s = c0 + tid + i * TL::NT;
        if (s < c1) {
            const float P = exp2f(S.z[s - c0] - M) * invL;
            const double ns = sc_old[i] + (double)P;
            c.score[ub + s] = ns;
            if (full) {
                if (ps[i] <= p - c.r && (ns < best || (ns == best && s < bslot))) { best = ns; bslot = s; }
                if (ns < best_all || (ns == best_all && s < bslot_all)) { best_all = ns; bslot_all = s; }
            }
        }
    }
    if (full) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const double ob = __shfl_xor_sync(kFull, best, off);
            const int os = __shfl_xor_sync(kFull, bslot, off);
            if (ob < best || (ob == best && os < bslot)) { best = ob; bslot = os; }
            const double oa = __shfl_xor_sync(kFull, best_all, off);
            const int osa = __shfl_xor_sync(kFull, bslot_all, off);
            if (oa < best_all || (oa == best_all && osa < bslot_all)) { best_all = oa; bslot_all = osa; }
        }
        if (lane == 0) {
            S.rd[0][warp] = best; S.ri[0][warp] = bslot;
            S.rd[1][warp] = best_all; S.ri[1][warp] = bslot_all;
        }
    }
    if (rank == 0 && tid < D) {
        float acc = 0.f;
        for (int j = 0; j < C; ++j) acc += S.x.o[j][tid] * safe_exp2_diff(S.x.m[j], M);
        a.out[(size_t)unit * D + tid] = acc * invL;
    }
    if (rank == 0 && tid == 0) S.P_new = exp2f(S.z_new - M) * invL;
    __syncthreads();
    if (full && tid == 0) {
        for (int w = 1; w < TL::NW; ++w) {
            if (S.rd[0][w] < best || (S.rd[0][w] == best && S.ri[0][w] < bslot)) { best = S.rd[0][w]; bslot = S.ri[0][w]; }
            if (S.rd[1][w] < best_all || (S.rd[1][w] == best_all && S.ri[1][w] < bslot_all)) {
                best_all = S.rd[1][w]; bslot_all = S.ri[1][w];
            }
        }
        const uint32_t base = x0;
        st_cluster_f64(base + (uint32_t)offsetof(Exchange<D>, cand_score) + rank * 8, best);
        st_cluster_s32(base + (uint32_t)offsetof(Exchange<D>, cand_slot) + rank * 4, bslot);
        st_cluster_f64(base + (uint32_t)offsetof(Exchange<D>, all_score) + rank * 8, best_all);
        st_cluster_s32(base + (uint32_t)offsetof(Exchange<D>, all_slot) + rank * 4, bslot_all);
    }
    // exchange 2: arg-min of every CTA into rank 0
    cluster_arrive();
    cluster_wait();
    if (rank != 0) return;

    if (tid == 0) {
        int victim = n;
        if (full) {
            double vb = DBL_MAX, va = DBL_MAX;
            int vs = INT_MAX, vsa = INT_MAX;
            for (int j = 0; j < C; ++j) {
                const double sj = S.x.cand_score[j];
                const int ij = S.x.cand_slot[j];
                if (ij != INT_MAX && (sj < vb || (sj == vb && ij < vs))) { vb = sj; vs = ij; }
                const double sa = S.x.all_score[j];
                const int ia = S.x.all_slot[j];
                if (ia != INT_MAX && (sa < va || (sa == va && ia < vsa))) { va = sa; vsa = ia; }
            }
            victim = (vs != INT_MAX) ? vs : vsa;
        }
        if (victim < 0 || victim >= B) victim = 0;   // n == 0 with B == 0 cannot happen
        S.victim = victim;
        c.score[ub + victim] = (double)S.P_new;
        c.pos[ub + victim] = p;
        c.ustate[unit] = make_int2(min(n + 1, B), p + 1);
        if (a.victim_out) a.victim_out[unit] = full ? victim : -1;
    }
    __syncthreads();
    const int victim = S.victim;
    constexpr int NV = D * (int)sizeof(T) / 16;
    if (tid < NV)
        copy_row<T, D>(Kc + (size_t)victim * D, reinterpret_cast<const T*>(a.k) + (size_t)unit * D, tid);
    else if (tid < 2 * NV)
        copy_row<T, D>(Vc + (size_t)victim * D, reinterpret_cast<const T*>(a.v) + (size_t)unit * D, tid - NV);
}

// ------------------------------------------------------------------ LSH

template <typename T, int D, class TL>
__global__ void __launch_bounds__(TL::NT) lsh_decode_kernel(const DecodeArgs a)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    auto& S = *reinterpret_cast<DecodeSmem<T, D, TL>*>(smem_raw);
    constexpr int EPL = D / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const CacheView& c = a.c;
    const int C = (int)cluster_nctarank();
    const int rank = (int)cluster_ctarank();
    const int unit = blockIdx.x / C;
    cluster_arrive_relaxed();

    const int B = c.B;
    const int2 us = c.ustate[unit];
    const int n = us.x, p = us.y;
    const bool full = (n >= B);
    int cs = (n + C - 1) / C;
    cs = (cs + TL::G - 1) / TL::G * TL::G;
    const int c0 = min(n, rank * cs), c1 = min(n, c0 + cs);
    const size_t ub = (size_t)unit * B;
    T* Kc = reinterpret_cast<T*>(c.K) + ub * D;
    T* Vc = reinterpret_cast<T*>(c.V) + ub * D;

    if (lane == 0) {
#pragma unroll
        for (int b = 0; b < TL::NBUF; ++b) mbar_init(&S.bar[warp][b], 1);
        fence_mbar_init();
        prime_ring<T, D, TL>(S, Kc, Vc, c0, c1);
    }

    const T* qg = reinterpret_cast<const T*>(a.q) + (size_t)unit * D;
    const T* kg = reinterpret_cast<const T*>(a.k) + (size_t)unit * D;
    if (tid < D) {
        S.qf[tid] = Elem<T>::to_f(qg[tid]);
        S.kf[tid] = Elem<T>::to_f(kg[tid]);
    }
    __syncthreads();
    // sign codes: lane j of warp 0 (query) / warp 1 (key) owns bit j; the
    // projection is an fp32 fused multiply-add chain in index order
    if (warp < 2) {
        const float* x = warp == 0 ? S.qf : S.kf;
        float acc = 0.f;
        for (int i = 0; i < D; ++i) acc = __fmaf_rn(x[i], __ldg(a.W + i * 32 + lane), acc);
        const unsigned code = __ballot_sync(kFull, acc > 0.f);
        if (lane == 0) {
            if (warp == 0) S.code_q = code; else S.code_k = code;
        }
    }
    __syncthreads();

    // victim: every CTA of the cluster decides it redundantly from the codes
    if (full) {
        const unsigned cq = S.code_q;
        unsigned long long bk = 0ull, bka = 0ull;    // (distance << 32) | ~slot, max wins
        for (int s = tid; s < n; s += TL::NT) {
            const unsigned long long key =
                ((unsigned long long)__popc(cq ^ c.code[ub + s]) << 32) | (unsigned)(0xffffffffu - (unsigned)s);
            if (c.pos[ub + s] <= p - c.r && key > bk) bk = key;
            if (key > bka) bka = key;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const unsigned long long o1 = __shfl_xor_sync(kFull, bk, off);
            const unsigned long long o2 = __shfl_xor_sync(kFull, bka, off);
            bk = o1 > bk ? o1 : bk;
            bka = o2 > bka ? o2 : bka;
        }
        if (lane == 0) { S.ru[0][warp] = bk; S.ru[1][warp] = bka; }
        __syncthreads();
        if (tid == 0) {
            for (int w = 1; w < TL::NW; ++w) {
                bk = S.ru[0][w] > bk ? S.ru[0][w] : bk;
                bka = S.ru[1][w] > bka ? S.ru[1][w] : bka;
            }
            const unsigned long long pick = bk ? bk : bka;
            S.victim = (int)(0xffffffffu - (unsigned)(pick & 0xffffffffull));
        }
    } else if (tid == 0) {
        S.victim = n;
    }
    __syncthreads();
    const int victim = S.victim;

    float qr[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) qr[e] = S.qf[lane * EPL + e] * c.qscale;
    float m_run = -INFINITY, l_run = 0.f, o[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] = 0.f;
    if (rank == 0 && warp == 0) {          // the new token, now in the victim slot
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc = fmaf(qr[e], S.kf[lane * EPL + e], acc);
        const float zn = warp_sum(acc);
        float vr[EPL];
        load_vec<T, EPL>(reinterpret_cast<const T*>(a.v) + (size_t)unit * D + lane * EPL, vr);
        m_run = zn;
        l_run = 1.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] = vr[e];
    }
    __syncwarp();

    attend_chunk<T, D, TL>(S, Kc, Vc, c0, c1, full ? victim : -1, false, qr, m_run, l_run, o,
                             c.err);

    float Mc, Lc, Oc;
    merge_warps<T, D, TL>(S, m_run, l_run, o, Mc, Lc, Oc);

    cluster_wait();
    const uint32_t x0 = map_to_rank(&S.x, 0);
    const uint32_t off_m = (uint32_t)offsetof(Exchange<D>, m), off_l = (uint32_t)offsetof(Exchange<D>, l);
    const uint32_t off_o = (uint32_t)offsetof(Exchange<D>, o);
    if (tid < D) st_cluster_f32(x0 + off_o + (uint32_t)((rank * D + tid) * 4), Oc);
    if (tid == 0) {
        st_cluster_f32(x0 + off_m + rank * 4, Mc);
        st_cluster_f32(x0 + off_l + rank * 4, Lc);
    }
    cluster_arrive();
    cluster_wait();
    if (rank != 0) return;

    if (tid < D) {
        float M = -INFINITY;
        for (int j = 0; j < C; ++j) M = fmaxf(M, S.x.m[j]);
        float L = 0.f, acc = 0.f;
        for (int j = 0; j < C; ++j) {
            const float f = safe_exp2_diff(S.x.m[j], M);
            L += S.x.l[j] * f;
            acc += S.x.o[j][tid] * f;
        }
        a.out[(size_t)unit * D + tid] = acc / L;
    }
    if (tid == 0) {
        c.code[ub + victim] = S.code_k;
        c.pos[ub + victim] = p;
        c.ustate[unit] = make_int2(min(n + 1, B), p + 1);
        if (a.victim_out) a.victim_out[unit] = full ? victim : -1;
    }
    constexpr int NV = D * (int)sizeof(T) / 16;
    if (tid < NV)
        copy_row<T, D>(Kc + (size_t)victim * D, kg, tid);
    else if (tid < 2 * NV)
        copy_row<T, D>(Vc + (size_t)victim * D, reinterpret_cast<const T*>(a.v) + (size_t)unit * D, tid - NV);
}

// ------------------------------------------------------------- launching

using TileDefault = Tile<8, 8, 2>;

template <typename T, int D, bool LSH, class TL>
cudaError_t launch_decode_t(const DecodeArgs& a, int split, cudaStream_t st)
{
    auto kern = LSH ? lsh_decode_kernel<T, D, TL> : h2o_decode_kernel<T, D, TL>;
    const size_t smem = sizeof(DecodeSmem<T, D, TL>);
    static bool configured[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.c.U * split), 1, 1);
    cfg.blockDim = dim3(TL::NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

// Tile variants for bf16 / head_dim 128, selectable with H2O_DECODE_TILE for
// tuning; every variant computes the same result.
int tile_variant()
{
    static int v = -1;
    if (v < 0) {
        const char* e = getenv("H2O_DECODE_TILE");
        v = e ? atoi(e) : 0;
    }
    return v;
}

template <bool LSH>
cudaError_t dispatch(const DecodeArgs& a, int split, cudaStream_t st)
{
    const bool bf = a.c.dtype == 1;
    if (a.c.D == 128 && bf) {
        switch (tile_variant()) {
        case 1: return launch_decode_t<__nv_bfloat16, 128, LSH, Tile<16, 8, 1>>(a, split, st);
        case 2: return launch_decode_t<__nv_bfloat16, 128, LSH, Tile<16, 4, 2>>(a, split, st);
        case 3: return launch_decode_t<__nv_bfloat16, 128, LSH, Tile<8, 4, 4>>(a, split, st);
        case 4: return launch_decode_t<__nv_bfloat16, 128, LSH, Tile<16, 8, 2>>(a, split, st);
        case 5: return launch_decode_t<__nv_bfloat16, 128, LSH, Tile<8, 8, 3>>(a, split, st);
        case 6: return launch_decode_t<__nv_bfloat16, 128, LSH, Tile<4, 8, 4>>(a, split, st);
        default: return launch_decode_t<__nv_bfloat16, 128, LSH, TileDefault>(a, split, st);
        }
    }
    if (a.c.D == 128) return launch_decode_t<float, 128, LSH, TileDefault>(a, split, st);
    if (a.c.D == 64)
        return bf ? launch_decode_t<__nv_bfloat16, 64, LSH, TileDefault>(a, split, st)
                  : launch_decode_t<float, 64, LSH, TileDefault>(a, split, st);
    return cudaErrorInvalidValue;
}

}  // namespace

int max_decode_split() { return kMaxSplit; }

// One CTA per unit whenever the units alone cover the SMs: the cluster
// exchange costs more than it saves.  Otherwise enough CTAs per unit to give
// every SM one, never more slots per CTA than the registers cover.
int auto_decode_split(int U, int B, int num_sms)
{
    int s = (num_sms + U - 1) / U;
    const int lo = (B + kMaxChunk - 1) / kMaxChunk;
    const int hi = (B + 63) / 64;
    if (s > hi) s = hi;
    if (s < lo) s = lo;
    if (s < 1) s = 1;
    if (s > kMaxSplit) s = kMaxSplit;
    return s;
}

cudaError_t launch_h2o_decode(const DecodeArgs& a, int split, cudaStream_t st)
{
    return dispatch<false>(a, split, st);
}

cudaError_t launch_lsh_decode(const DecodeArgs& a, int split, cudaStream_t st)
{
    return dispatch<true>(a, split, st);
}

}  // namespace h2o
