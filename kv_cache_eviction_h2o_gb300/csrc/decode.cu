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
// contiguous chunks, one CTA each, a unit's CTAs forming one cluster (a
// grouped-query cache: one CTA per query head).  In a CTA every warp streams
// its own 16-slot stages of K and V rows with 1-D bulk copies (TMA) into a
// private ring of shared-memory buffers completed on mbarriers, and keeps
// its own online softmax (base-2 logits).  Warps merge through shared
// memory, CTAs through distributed shared memory into cluster rank 0.  H2O
// needs the global normaliser before any score update, so the cluster
// exchanges (max, sum) once, every CTA updates its own slots' scores (or
// pivotal histories) from the logits it kept in shared memory (P never goes
// to HBM), and a second exchange reduces the arg-min.  Every wait is
// bounded; a wait that runs out sets the handle's error word.
#include <mutex>

#include "decode_common.cuh"

namespace h2o {

namespace {

// ------------------------------------------------------------------ H2O

// GQ: grouped-query cache.  The cluster's C CTAs are the C query heads that
// share cache unit `unit`; each CTA attends over every slot of the unit with
// its own query and softmax, and CTA g accumulates the heads' probabilities
// into the scores of its share [s0, s1) of the slots.  Otherwise the
// cluster's CTAs split one head's slots.
// SH: persistence of importance [Scissorhands abstract].  In place of a
// score every slot keeps a 32-step history of pivotal flags (`code`): this
// step shifts it and sets bit 0 when the slot's probability exceeds the
// uniform share, P (n + 1) > 1; the victim is the candidate with the fewest
// set bits, then the lowest position; the new token's history is its own
// flag.
template <typename T, int D, class TL, int QB, bool GQ, bool SH = false>
__global__ void __launch_bounds__(TL::NT, TL::MINB) h2o_decode_kernel(const DecodeArgs a)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    auto& S = *reinterpret_cast<DecodeSmem<T, D, TL, QB>*>(smem_raw);
    constexpr int EPL = D / 32;
    constexpr int NV = D * (int)sizeof(T) / 16;          // 16-byte vectors per row
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const CacheView& c = a.c;
    const int C = (int)cluster_nctarank();
    const int rank = (int)cluster_ctarank();
    int unit = blockIdx.x / C;
    if (a.ulist) {
        // a unit list (per-head policies): written by the handle's earlier
        // kernels, so read after the dependency wait unless the previous
        // kernel cannot have written it; a whole cluster exits together, and
        // only after the wait, so that this grid's end still implies the
        // previous kernel's (the next launch waits on this one alone)
        if (!a.early) grid_dependency_wait();
        if (unit >= *a.ucount) {
            if (a.early) grid_dependency_wait();
            return;
        }
        unit = a.ulist[unit];
    }
    const size_t qrow = GQ ? (size_t)blockIdx.x : (size_t)unit;   // query / output row

    const int B = c.B;
    const size_t ub = (size_t)unit * B;
    using CE = CacheElem<T, QB>;
    CE* Kc = reinterpret_cast<CE*>(c.K) + ub * RowElems<D, QB>;
    CE* Vc = reinterpret_cast<CE*>(c.V) + ub * RowElems<D, QB>;
    float2* Sc = QB ? c.kvs + (size_t)unit * c.Bp : nullptr;   // slot scale pairs
    // this unit's budget and recent window: the cache's own, or the unit's
    // policy (per-head policies; then the unit uses Bu of its B slots)
    int Bu = B, ru = c.r;
    int f0, f1, s0, s1;                      // fetched slots; slots whose scores this CTA updates
    auto unit_ranges = [&]() {
        if (c.upol) {
            const int4 pp = c.upol[unit];
            Bu = pp.x;
            ru = pp.z;
        }
        if constexpr (GQ) {
            f0 = 0;
            f1 = Bu;
            fetch_range(Bu, C, rank, s0, s1);
        } else {
            fetch_range(Bu, C, rank, f0, f1);
            s0 = f0;
            s1 = f1;
        }
    };
    // the policy is written by this handle's prompt phase only, so it is
    // read before the dependency wait under the same rule as the cache
    if (a.early || !c.upol) unit_ranges();
    if (lane == 0) {
#pragma unroll
        for (int b = 0; b < TL::NBUF; ++b) mbar_init(&S.bar[warp][b], 1);
        if (C > 1) fence_mbar_init(); else fence_proxy_async_smem();
    }
    // paired with the wait before the first exchange: by then every CTA of
    // the cluster runs, so its shared memory may be written
    if (C > 1) cluster_arrive_relaxed();
    const T* qg = reinterpret_cast<const T*>(a.q) + qrow * D;
    const T* kg = reinterpret_cast<const T*>(a.k) + (size_t)unit * D;
    const T* vg = reinterpret_cast<const T*>(a.v) + (size_t)unit * D;
    // the input rows are read only after the wait, but their lines can be
    // on their way to L2 meanwhile, ahead of the cache traffic below
    prefetch_rows_l2(qg, kg, vg, D * (int)sizeof(T), tid);
    // This unit's cache: the ring's first stages (the attention starts on
    // them, so their bulk copies go out first), the occupancy, and the scores
    // and positions of this thread's fetched slots (consumed after the merge).
    // When the previous kernel in the stream cannot have written the cache
    // this happens before the dependency wait, overlapping that kernel's end.
    int2 us = make_int2(0, 0);
    float2 sc_old[TL::SPT];
    int ps[TL::SPT];
    // (volatile loads: issued here, not sunk to their use after the stream)
    auto read_cache = [&]() {
        us = c.ustate[unit];
#pragma unroll
        for (int i = 0; i < TL::SPT; ++i) {
            const int s = s0 + tid + i * TL::NT;
            sc_old[i] = make_float2(0.f, 0.f);
            ps[i] = 0;
            if (s < s1) {
                if constexpr (SH) sc_old[i].x = __uint_as_float(ld_issue_u32(c.code + ub + s));
                else sc_old[i] = ld_issue_f2(c.score + ub + s);
                ps[i] = (int)ld_issue_u32(reinterpret_cast<const uint32_t*>(c.pos + ub + s));
            }
        }
    };
    // Early, only each warp's first buffer is filled before the wait: the
    // query row, requested right after the wait, then queues behind less
    // traffic, and the remaining buffers keep HBM busy while it is in flight.
    if (a.early) {
        if (lane == 0) prime_ring<T, D, TL, QB>(S, Kc, Vc, Sc, f0, f1, 0, 1);
        read_cache();
    }
    // everything below may read memory the previous kernel in the stream
    // has written (the inputs, and the cache unless read above)
    grid_dependency_wait();
    grid_launch_dependents();
    if (!a.early) {
        if (c.upol) unit_ranges();
        if (lane == 0) prime_ring<T, D, TL, QB>(S, Kc, Vc, Sc, f0, f1);
        read_cache();
    }
    // q, k, v in one round trip (requested before the rest of the ring)
    {
        const uint4 w = load_rows_16b<T, D>(qg, kg, vg, tid);
        if (a.early && lane == 0) prime_ring<T, D, TL, QB>(S, Kc, Vc, Sc, f0, f1, 1, TL::NBUF);
        store_rows_16b<T, D>(S.in, w, tid);
    }
    __syncthreads();
    const T* qs = reinterpret_cast<const T*>(S.in[0]);
    const T* ks = reinterpret_cast<const T*>(S.in[1]);
    const T* vs = reinterpret_cast<const T*>(S.in[2]);
    QVec<T, D, QB> qv;
    load_qvec<QB, T, D>(qs, c.qscale, lane, QB ? S.qpl[warp] : nullptr, qv);
    // the new token's row, written into the victim slot at the end
    uint4 newrow = make_uint4(0u, 0u, 0u, 0u);
    if (rank == 0 && tid < 2 * NV) newrow = reinterpret_cast<const uint4*>(S.in[1])[tid];

    const int n = us.x, p = us.y;
    const bool full = (n >= Bu);
    const int c0 = f0, c1 = min(n, f1);     // live slots of this CTA

    float m_run = -INFINITY, l_run = 0.f, o[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] = 0.f;
    if ((GQ || rank == 0) && warp == 0) {  // the new token attends to itself
        float vr[EPL];
        const float zn = new_logit<QB, T, D>(qs, ks, c.qscale, qv, lane);
        load_vec<T, EPL>(vs + lane * EPL, vr);
        m_run = zn;
        l_run = lane == 0 ? 1.f : 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] = vr[e];
        if (lane == 0) S.z_new = zn;
    }
    __syncwarp();

    attend_chunk<T, D, TL, QB>(S, Kc, Vc, Sc, f0, f1, n, -1, true, qv, m_run, l_run, o, c.err);

    float Mc, Lc, Oc;
    merge_warps<T, D, TL, QB>(S, m_run, l_run, o, Mc, Lc, Oc);
    if (C > 1) cluster_wait();               // every CTA of the cluster runs (arrive at the start)
    const uint32_t x0 = map_to_rank(&S.x, 0);

    // Write the new token into the victim slot (slot n while the cache is
    // not full) with score `snew`.  `write_row` runs in the threads holding
    // `newrow`.
    auto finish = [&](int victim, float2 snew) {
        if (victim < 0 || victim >= Bu) victim = 0;   // n == 0 with Bu == 0 cannot happen
        if (tid == 0) {
            if constexpr (SH) c.code[ub + victim] = S.P_new * (float)(n + 1) > 1.f ? 1u : 0u;
            else c.score[ub + victim] = snew;
            c.pos[ub + victim] = p;
            c.ustate[unit] = make_int2(min(n + 1, Bu), p + 1);
            if (a.victim_out) a.victim_out[unit] = full ? victim : -1;
        }
        if constexpr (QB != 0) {
            store_row_quant<QB, T, D>(newrow, tid, Kc, Vc, Sc, victim);
        } else {
            if (tid < NV)
                reinterpret_cast<uint4*>(Kc + (size_t)victim * D)[tid] = newrow;
            else if (tid < 2 * NV)
                reinterpret_cast<uint4*>(Vc + (size_t)victim * D)[tid - NV] = newrow;
        }
    };

    if constexpr (GQ) {
        // this head's output, then its probabilities in place of its logits
        const float invL = 1.f / Lc;
        if (tid < D) a.out[qrow * D + tid] = Oc * invL;
        for (int s = tid; s < n; s += TL::NT) S.z[s] = ex2_approx(S.z[s] - Mc) * invL;
        if (tid == 0) S.P_new = ex2_approx(S.z_new - Mc) * invL;
        cluster_arrive();                    // every head's probabilities are in place
        cluster_wait();
        // scores of this CTA's share: add the heads' probabilities in head
        // order; arg-min as in the split path
        const int sc1 = min(n, s1);
        ArgMin best = argmin_none(), best_all = argmin_none();
#pragma unroll
        for (int i = 0; i < TL::SPT; ++i) {
            const int s = s0 + tid + i * TL::NT;
            if (s < sc1) {
                float2 ns = sc_old[i];
                for (int j = 0; j < C; ++j) ns = pair_add(ns, ld_cluster_f32(map_to_rank(&S.z[s], j)));
                c.score[ub + s] = ns;
                if (full) {
                    const ArgMin k = ArgMin{ord_key(ns.x), ord_key(ns.y), (unsigned)s};
                    if (ps[i] <= p - ru) argmin_take(best, k);
                    argmin_take(best_all, k);
                }
            }
        }
        if (full) {
            best = warp_argmin(best);
            best_all = warp_argmin(best_all);
            if (lane == 0) {
                S.am[0][0][warp] = best.hi; S.am[0][1][warp] = best.lo; S.am[0][2][warp] = best.slot;
                S.am[1][0][warp] = best_all.hi; S.am[1][1][warp] = best_all.lo; S.am[1][2][warp] = best_all.slot;
            }
        }
        __syncthreads();
        if (warp == 0) {
            // this CTA's arg-mins and its head's new-token probability, pushed
            // into rank 0's exchange
            if (full) {
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    ArgMin w = lane < TL::NW ? ArgMin{S.am[k][0][lane], S.am[k][1][lane], S.am[k][2][lane]} : argmin_none();
                    w = warp_argmin(w);
                    if (lane == 0) {
                        const uint32_t base = x0 + (uint32_t)offsetof(Exchange<D>, am) + (uint32_t)(k * 3 * kMaxSplit * 4);
                        st_cluster_s32(base + rank * 4, (int)w.hi);
                        st_cluster_s32(base + (kMaxSplit + rank) * 4, (int)w.lo);
                        st_cluster_s32(base + (2 * kMaxSplit + rank) * 4, (int)w.slot);
                    }
                }
            }
            if (lane == 0) st_cluster_f32(x0 + (uint32_t)offsetof(Exchange<D>, m) + rank * 4, S.P_new);
        }
        cluster_arrive();                    // exchange complete; no CTA reads another's memory after this
        cluster_wait();
        if (rank != 0) return;
        if (tid == 0) {
            int victim = n;
            if (full) {
                ArgMin vc = argmin_none(), va = argmin_none();
                for (int j = 0; j < C; ++j) {
                    argmin_take(vc, ArgMin{S.x.am[0][0][j], S.x.am[0][1][j], S.x.am[0][2][j]});
                    argmin_take(va, ArgMin{S.x.am[1][0][j], S.x.am[1][1][j], S.x.am[1][2][j]});
                }
                victim = (int)(vc.slot != 0xffffffffu ? vc.slot : va.slot);
            }
            S.victim = victim;
        }
        __syncthreads();
        float2 snew = make_float2(0.f, 0.f);
        if (tid == 0)
            for (int j = 0; j < C; ++j) snew = pair_add(snew, S.x.m[j]);
        finish(S.victim, snew);
        return;
    }

    // exchange 1: (max, normaliser, output) of every CTA into rank 0; a
    // single-CTA unit already has them
    float M, invL;
    if (C > 1) {
        // every CTA's (max, normaliser) into every CTA, its output into rank 0
        const uint32_t off_m = (uint32_t)offsetof(Exchange<D>, m), off_l = (uint32_t)offsetof(Exchange<D>, l);
        const uint32_t off_o = (uint32_t)offsetof(Exchange<D>, o);
        if (tid < D) st_cluster_f32(x0 + off_o + (uint32_t)((rank * D + tid) * 4), Oc);
        if (tid < C) {
            const uint32_t xt = map_to_rank(&S.x, (uint32_t)tid);
            st_cluster_f32(xt + off_m + rank * 4, Mc);
            st_cluster_f32(xt + off_l + rank * 4, Lc);
        }
        cluster_arrive();
        cluster_wait();
        float Mx = -INFINITY, Lx = 0.f;
        for (int j = 0; j < C; ++j) Mx = fmaxf(Mx, S.x.m[j]);
        for (int j = 0; j < C; ++j) Lx += S.x.l[j] * safe_exp2_diff(S.x.m[j], Mx);
        M = Mx;
        invL = 1.f / Lx;
    } else {
        M = Mc;
        invL = 1.f / Lc;
    }

    // accumulate this step's probabilities; arg-min over candidates (slots
    // whose position is at most p - r)
    ArgMin best = argmin_none(), best_all = argmin_none();
#pragma unroll
    for (int i = 0; i < TL::SPT; ++i) {
        const int s = c0 + tid + i * TL::NT;
        if (s < c1) {
            const float P = ex2_approx(S.z[s - c0] - M) * invL;
            ArgMin k;
            if constexpr (SH) {
                const uint32_t h = (__float_as_uint(sc_old[i].x) << 1) | (P * (float)(n + 1) > 1.f ? 1u : 0u);
                c.code[ub + s] = h;
                k = ArgMin{(unsigned)__popc(h), (unsigned)ps[i], (unsigned)s};
            } else {
                const float2 ns = pair_add(sc_old[i], P);
                c.score[ub + s] = ns;
                k = ArgMin{ord_key(ns.x), ord_key(ns.y), (unsigned)s};
            }
            if (full) {
                if (ps[i] <= p - ru) argmin_take(best, k);
                if (C > 1) argmin_take(best_all, k);
            }
        }
    }
    if (full) {
        best = warp_argmin(best);
        if (C > 1) best_all = warp_argmin(best_all);
        if (lane == 0) {
            S.am[0][0][warp] = best.hi; S.am[0][1][warp] = best.lo; S.am[0][2][warp] = best.slot;
            S.am[1][0][warp] = best_all.hi; S.am[1][1][warp] = best_all.lo; S.am[1][2][warp] = best_all.slot;
        }
    }
    if (rank == 0 && tid < D) {
        float acc = Oc;
        if (C > 1) {
            acc = 0.f;
            for (int j = 0; j < C; ++j) acc += S.x.o[j][tid] * safe_exp2_diff(S.x.m[j], M);
        }
        a.out[qrow * D + tid] = acc * invL;
    }
    if (rank == 0 && tid == 0) S.P_new = ex2_approx(S.z_new - M) * invL;
    __syncthreads();

    if (C == 1) {
        // one CTA holds the unit: warp 0 reduces the warps' candidates; with
        // no candidate at all (possible only for loaded states) every live
        // slot competes, its new score re-read from global memory (written
        // above by this CTA)
        int victim = n;
        if (warp == 0 && full) {
            ArgMin w = lane < TL::NW ? ArgMin{S.am[0][0][lane], S.am[0][1][lane], S.am[0][2][lane]} : argmin_none();
            w = warp_argmin(w);
            if (w.slot == 0xffffffffu) {
                ArgMin al = argmin_none();
                for (int s = lane; s < n; s += 32) {
                    if constexpr (SH) {
                        argmin_take(al, ArgMin{(unsigned)__popc(c.code[ub + s]), (unsigned)c.pos[ub + s], (unsigned)s});
                    } else {
                        const float2 sc = c.score[ub + s];
                        argmin_take(al, ArgMin{ord_key(sc.x), ord_key(sc.y), (unsigned)s});
                    }
                }
                w = warp_argmin(al);
            }
            victim = (int)w.slot;
        }
        if constexpr (2 * NV <= 32) {
            if (warp == 0) finish(victim, make_float2(S.P_new, 0.f));
        } else {
            if (tid == 0) S.victim = victim;
            __syncthreads();
            finish(S.victim, make_float2(S.P_new, 0.f));
        }
        return;
    }

    if (full && warp == 0) {
        // this CTA's arg-min over its warps, pushed into rank 0's exchange
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            ArgMin w = lane < TL::NW ? ArgMin{S.am[k][0][lane], S.am[k][1][lane], S.am[k][2][lane]} : argmin_none();
            w = warp_argmin(w);
            if (lane == 0) {
                const uint32_t base = x0 + (uint32_t)offsetof(Exchange<D>, am) + (uint32_t)(k * 3 * kMaxSplit * 4);
                st_cluster_s32(base + rank * 4, (int)w.hi);
                st_cluster_s32(base + (kMaxSplit + rank) * 4, (int)w.lo);
                st_cluster_s32(base + (2 * kMaxSplit + rank) * 4, (int)w.slot);
            }
        }
    }
    // exchange 2: arg-min of every CTA into rank 0
    cta_group_sync(C);
    if (rank != 0) return;

    if (tid == 0) {
        int victim = n;
        if (full) {
            ArgMin vc = argmin_none(), va = argmin_none();
            for (int j = 0; j < C; ++j) {
                argmin_take(vc, ArgMin{S.x.am[0][0][j], S.x.am[0][1][j], S.x.am[0][2][j]});
                argmin_take(va, ArgMin{S.x.am[1][0][j], S.x.am[1][1][j], S.x.am[1][2][j]});
            }
            victim = (int)(vc.slot != 0xffffffffu ? vc.slot : va.slot);
        }
        S.victim = victim;
    }
    __syncthreads();
    finish(S.victim, make_float2(S.P_new, 0.f));
}

// ------------------------------------------------------------ grouped query
//
// Grouped-query H2O step in one pass over each cache unit's rows for all of
// its G query heads [H2O review page, 提案手法; the grouped form is this
// library's reading: a slot's score grows by the sum of its G heads'
// probabilities, added in head order].  A CTA -- or a cluster of C CTAs
// splitting the unit's slots -- has NW = G * NG warps: stage group sg takes
// the 16-slot stages sg, sg + NG, ... of the CTA's slots, and its G warps,
// one per head, read each stage from a ring the group shares (filled by the
// group's head-0 warp with 1-D bulk copies; a full and an empty mbarrier per
// buffer, G arrivals on the empty one).  Every K and V row therefore crosses
// from L2 once per unit, not once per head.  Each warp keeps its head's
// online softmax and logits; after the stream the heads' states are merged
// per head (and across the cluster), one score pass adds the G
// probabilities to each slot, and one arg-min and insert follow.

template <int G>
struct GqaShape {
    static constexpr int NW = 8;                          // warps
    static constexpr int NG = NW / G;                     // stage groups
    static constexpr int NT = 32 * NW;
    // about 128 KB of stages in flight per CTA (one CTA per SM: registers)
    static constexpr int NBUF = 16 / NG;
    static constexpr int CMAX = 32 / G;                   // the exchange holds C * G <= 32 head states
    static constexpr int SPT = (kMaxChunk + NT - 1) / NT;
    static_assert(NW % G == 0, "heads divide the warps");
};

// cluster exchange of the grouped-query kernel: every CTA's per-head max
// and normaliser (index rank * G + head), outputs gathered in rank 0, and
// the CTAs' arg-min keys
template <int D>
struct GqaExchange {
    float m[32];
    float l[32];
    unsigned am[2][3][kMaxSplit];
    float o[32][D];
};

template <typename T, int D, int G>
struct GqaSmem {
    using SH = GqaShape<G>;
    union {
        struct {
            T kbuf[SH::NG][SH::NBUF][kStage * D];
            T vbuf[SH::NG][SH::NBUF][kStage * D];
        } ring;
        float wo[SH::NW][D];                  // per-warp outputs at the merge
    } u;
    GqaExchange<D> x;
    alignas(16) unsigned char in[G + 2][D * sizeof(T)];   // the G heads' q, then k, v
    uint64_t full[SH::NG][SH::NBUF];
    uint64_t empty[SH::NG][SH::NBUF];
    float z[G][kMaxChunk];                    // base-2 logits of this CTA's slots, per head
    alignas(16) float e[SH::NW][kStage];
    float wm[SH::NW], wl[SH::NW];
    float hm[G], hl[G];                       // this CTA's per-head max and normaliser
    float M[G], invL[G];                      // per-head max and 1 / normaliser over the unit
    float zn[G];                              // the new token's logit per head
    unsigned am[2][3][SH::NW];
    float2 P_new;                             // the new token's score: its G probabilities
    int victim;
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(GqaShape<G>::NT, 1) gqa_decode_kernel(const DecodeArgs a)
{
    using SH = GqaShape<G>;
    constexpr int EPL = D / 32, NV = D * (int)sizeof(T) / 16, NW = SH::NW, NG = SH::NG, NBUF = SH::NBUF;
    constexpr int NT = SH::NT, SPT = SH::SPT;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    auto& S = *reinterpret_cast<GqaSmem<T, D, G>*>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int head = warp % G, sg = warp / G;
    const bool leader = (head == 0);          // refills its group's ring
    const int r = lane & 15, hh = lane >> 4;
    const CacheView& c = a.c;
    const int C = (int)cluster_nctarank(), rank = (int)cluster_ctarank();
    const int unit = blockIdx.x / C;
    const int B = c.B;
    const size_t ub = (size_t)unit * B;
    T* Kc = reinterpret_cast<T*>(c.K) + ub * D;
    T* Vc = reinterpret_cast<T*>(c.V) + ub * D;
    int f0, f1;
    fetch_range(B, C, rank, f0, f1);
    const int nst = (f1 - f0 + kStage - 1) / kStage;
    if (leader && lane == 0) {
#pragma unroll
        for (int b = 0; b < NBUF; ++b) {
            mbar_init(&S.full[sg][b], 1);
            mbar_init(&S.empty[sg][b], G);
        }
        if (C > 1) fence_mbar_init(); else fence_proxy_async_smem();
    }
    if (C > 1) cluster_arrive_relaxed();      // paired with the wait before the exchange
    const T* qg = reinterpret_cast<const T*>(a.q) + (size_t)unit * G * D;
    const T* kg = reinterpret_cast<const T*>(a.k) + (size_t)unit * D;
    const T* vg = reinterpret_cast<const T*>(a.v) + (size_t)unit * D;
    {
        // the input rows' lines on their way to L2 before the wait
        constexpr int lines = (D * (int)sizeof(T) + 127) / 128;
        if (tid < (G + 2) * lines) {
            const int row = tid / lines, l = tid - row * lines;
            const T* base = row < G ? qg + (size_t)row * D : (row == G ? kg : vg);
            prefetch_l2(reinterpret_cast<const char*>(base) + 128 * l);
        }
    }
    __syncthreads();                          // the group barriers are initialised
    // stage j (CTA-relative) of group sg into buffer b
    auto issue = [&](int j, int b) {
        const int s = f0 + j * kStage;
        const int rows = min(kStage, f1 - s);
        const uint32_t bytes = (uint32_t)(rows * D * sizeof(T));
        mbar_arrive_expect_tx(&S.full[sg][b], 2 * bytes);
        bulk_g2s(S.u.ring.kbuf[sg][b], Kc + (size_t)s * D, bytes, &S.full[sg][b]);
        bulk_g2s(S.u.ring.vbuf[sg][b], Vc + (size_t)s * D, bytes, &S.full[sg][b]);
    };
    auto prime = [&](int b_lo, int b_hi) {
        for (int b = b_lo; b < b_hi; ++b) {
            const int j = sg + NG * b;
            if (j < nst) issue(j, b);
        }
    };
    int2 us = make_int2(0, 0);
    float2 sc_old[SPT];
    int ps[SPT];
    auto read_cache = [&]() {
        us = c.ustate[unit];
#pragma unroll
        for (int i = 0; i < SPT; ++i) {
            const int s = f0 + tid + i * NT;
            sc_old[i] = make_float2(0.f, 0.f);
            ps[i] = 0;
            if (s < f1) {
                sc_old[i] = ld_issue_f2(c.score + ub + s);
                ps[i] = (int)ld_issue_u32(reinterpret_cast<const uint32_t*>(c.pos + ub + s));
            }
        }
    };
    if (a.early) {
        if (leader && lane == 0) prime(0, 1);
        read_cache();
    }
    grid_dependency_wait();
    grid_launch_dependents();
    if (!a.early) {
        if (leader && lane == 0) prime(0, NBUF);
        read_cache();
    }
    {
        // the G heads' q, k and v in one round trip
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (tid < (G + 2) * NV) {
            const int row = tid / NV;
            const T* base = row < G ? qg + (size_t)row * D : (row == G ? kg : vg);
            w = reinterpret_cast<const uint4*>(base)[tid - row * NV];
        }
        if (a.early && leader && lane == 0) prime(1, NBUF);
        if (tid < (G + 2) * NV) reinterpret_cast<uint4*>(S.in[tid / NV])[tid % NV] = w;
    }
    __syncthreads();
    const T* qs = reinterpret_cast<const T*>(S.in[head]);
    const T* ks = reinterpret_cast<const T*>(S.in[G]);
    const T* vs = reinterpret_cast<const T*>(S.in[G + 1]);
    float qp[D / 2];
    {
        QRaw<T, D> qraw;
        load_q_raw<T, D>(qs, lane, qraw);
        widen_q<T, D>(qraw, c.qscale, qp);
    }
    uint4 newrow = make_uint4(0u, 0u, 0u, 0u);       // k then v (adjacent rows of S.in)
    if (rank == 0 && tid < 2 * NV) newrow = reinterpret_cast<const uint4*>(S.in[G])[tid];
    const int n = us.x, p = us.y;
    const bool full = (n >= B);
    const int c1 = min(n, f1);

    float m_ref = -INFINITY, l_lane = 0.f, o[EPL], o2[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) { o[e] = 0.f; o2[e] = 0.f; }
    if (rank == 0 && sg == 0) {              // each head's new token attends to itself
        const float zn = row_dot<T, D, T>(ks, qp, lane);
        float vr[EPL];
        load_vec<T, EPL>(vs + lane * EPL, vr);
        m_ref = zn;
        l_lane = lane == 0 ? 1.f : 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] = vr[e];
        if (lane == 0) S.zn[head] = zn;
    }
    __syncwarp();
    auto vfma = [&](float pw, const float* vr, bool odd) {
        const float2 pj = make_float2(pw, pw);
#pragma unroll
        for (int e = 0; e < EPL; e += 2) {
            float* acc = odd ? o2 : o;
            const float2 rr = fma2(pj, make_float2(vr[e], vr[e + 1]), make_float2(acc[e], acc[e + 1]));
            acc[e] = rr.x;
            acc[e + 1] = rr.y;
        }
    };
    bool timed_out = false;
    int it = 0;
    for (int j = sg; j < nst; j += NG, ++it) {
        const int b = it % NBUF;
        const uint32_t par = (uint32_t)(it / NBUF) & 1u;
        if (!mbar_wait(&S.full[sg][b], par)) {
            if (!timed_out && lane == 0) atomicOr(c.err, kErrWaitTimeout);
            timed_out = true;
        }
        const int s0 = j * kStage;                         // CTA-relative first slot
        const int gl = max(0, min(kStage, n - (f0 + s0)));  // live rows of this stage
        if (gl > 0) {
            const T* kst = S.u.ring.kbuf[sg][b];
            const T* vst = S.u.ring.vbuf[sg][b];
            float z = row_dot<T, D, T>(kst + r * D, qp, lane);
            if (r >= gl) z = -INFINITY;
            if (__any_sync(kFull, z > m_ref + 8.f)) {
                float zm = z;
#pragma unroll
                for (int sh = 1; sh < 16; sh <<= 1) zm = fmaxf(zm, __shfl_xor_sync(kFull, zm, sh));
                const float alpha = safe_exp2_diff(m_ref, zm);
                l_lane *= alpha;
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    o[e] *= alpha;
                    o2[e] *= alpha;
                }
                m_ref = zm;
            }
            const float er = safe_exp2_diff(z, m_ref);
            if (hh == 0) {
                l_lane += er;
                S.e[warp][r] = er;
                if (r < gl) S.z[head][s0 + r] = z;
            }
            __syncwarp();
            float ev[kStage];
#pragma unroll
            for (int q4 = 0; q4 < kStage; q4 += 4) {
                const float4 e4 = *reinterpret_cast<const float4*>(&S.e[warp][q4]);
                ev[q4] = e4.x; ev[q4 + 1] = e4.y; ev[q4 + 2] = e4.z; ev[q4 + 3] = e4.w;
            }
            using RV = typename RawT<EPL * sizeof(T)>::type;
            if (gl == kStage) {
#pragma unroll
                for (int j0 = 0; j0 < kStage; j0 += kStage / 2) {
                    RV vraw[kStage / 2];
#pragma unroll
                    for (int jj = 0; jj < kStage / 2; ++jj)
                        vraw[jj] = *reinterpret_cast<const RV*>(vst + (j0 + jj) * D + lane * EPL);
#pragma unroll
                    for (int jj = 0; jj < kStage / 2; ++jj) {
                        float vr[EPL];
                        widen_raw<T, EPL>(vraw[jj], vr);
                        vfma(ev[j0 + jj], vr, jj & 1);
                    }
                }
            } else {
#pragma unroll
                for (int jj = 0; jj < kStage; ++jj) {
                    if (jj < gl) {
                        float vr[EPL];
                        load_vec<T, EPL>(vst + jj * D + lane * EPL, vr);
                        vfma(ev[jj], vr, jj & 1);
                    }
                }
            }
            __syncwarp();
        }
        // this head is done with the buffer; the group's head-0 warp refills
        // it once every head has released it
        if (lane == 0) mbar_arrive_one(&S.empty[sg][b]);
        if (leader && lane == 0) {
            const int jn = j + NG * NBUF;
            if (jn < nst) {
                if (!mbar_wait(&S.empty[sg][b], par)) {
                    if (!timed_out) atomicOr(c.err, kErrWaitTimeout);
                    timed_out = true;
                }
                issue(jn, b);
            }
        }
        __syncwarp();
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] += o2[e];

    // merge: per head over the stage groups (and then the cluster)
    const float l_warp = warp_sum(l_lane);
    __syncthreads();                          // every warp is past the ring the outputs overlay
    if (lane == 0) { S.wm[warp] = m_ref; S.wl[warp] = l_warp; }
#pragma unroll
    for (int e = 0; e < EPL; ++e) S.u.wo[warp][lane * EPL + e] = o[e];
    __syncthreads();
    if (tid < G) {
        float mx = -INFINITY, lx = 0.f;
        for (int q = 0; q < NG; ++q) mx = fmaxf(mx, S.wm[q * G + tid]);
        for (int q = 0; q < NG; ++q) lx += S.wl[q * G + tid] * safe_exp2_diff(S.wm[q * G + tid], mx);
        S.hm[tid] = mx;
        S.hl[tid] = lx;
    }
    __syncthreads();
    const uint32_t x0 = map_to_rank(&S.x, 0);
    if (C > 1) {
        cluster_wait();                      // every CTA of the cluster runs (arrive at the start)
        const uint32_t off_m = (uint32_t)offsetof(GqaExchange<D>, m), off_l = (uint32_t)offsetof(GqaExchange<D>, l);
        const uint32_t off_o = (uint32_t)offsetof(GqaExchange<D>, o);
        for (int idx = tid; idx < G * D; idx += NT) {
            const int g = idx / D, e = idx - g * D;
            float oc = 0.f;
            for (int q = 0; q < NG; ++q) oc += S.u.wo[q * G + g][e] * safe_exp2_diff(S.wm[q * G + g], S.hm[g]);
            st_cluster_f32(x0 + off_o + (uint32_t)(((rank * G + g) * D + e) * 4), oc);
        }
        if (tid < C * G) {
            const int t = tid / G, g = tid - t * G;
            const uint32_t xt = map_to_rank(&S.x, (uint32_t)t);
            st_cluster_f32(xt + off_m + (uint32_t)((rank * G + g) * 4), S.hm[g]);
            st_cluster_f32(xt + off_l + (uint32_t)((rank * G + g) * 4), S.hl[g]);
        }
        cluster_arrive();
        cluster_wait();
        if (tid < G) {
            float mx = -INFINITY, lx = 0.f;
            for (int t = 0; t < C; ++t) mx = fmaxf(mx, S.x.m[t * G + tid]);
            for (int t = 0; t < C; ++t) lx += S.x.l[t * G + tid] * safe_exp2_diff(S.x.m[t * G + tid], mx);
            S.M[tid] = mx;
            S.invL[tid] = 1.f / lx;
        }
        __syncthreads();
        if (rank == 0) {
            for (int idx = tid; idx < G * D; idx += NT) {
                const int g = idx / D, e = idx - g * D;
                float acc = 0.f;
                for (int t = 0; t < C; ++t) acc += S.x.o[t * G + g][e] * safe_exp2_diff(S.x.m[t * G + g], S.M[g]);
                a.out[((size_t)unit * G + g) * D + e] = acc * S.invL[g];
            }
        }
    } else {
        if (tid < G) {
            S.M[tid] = S.hm[tid];
            S.invL[tid] = 1.f / S.hl[tid];
        }
        __syncthreads();
        for (int idx = tid; idx < G * D; idx += NT) {
            const int g = idx / D, e = idx - g * D;
            float oc = 0.f;
            for (int q = 0; q < NG; ++q) oc += S.u.wo[q * G + g][e] * safe_exp2_diff(S.wm[q * G + g], S.M[g]);
            a.out[((size_t)unit * G + g) * D + e] = oc * S.invL[g];
        }
    }

    // accumulate: every live slot gains its G heads' probabilities (head
    // order); arg-min over candidates (position <= p - r)
    ArgMin best = argmin_none(), best_all = argmin_none();
#pragma unroll
    for (int i = 0; i < SPT; ++i) {
        const int s = f0 + tid + i * NT;
        if (s < c1) {
            float2 ns = sc_old[i];
#pragma unroll
            for (int g = 0; g < G; ++g) ns = pair_add(ns, ex2_approx(S.z[g][s - f0] - S.M[g]) * S.invL[g]);
            c.score[ub + s] = ns;
            const ArgMin k = ArgMin{ord_key(ns.x), ord_key(ns.y), (unsigned)s};
            if (full) {
                if (ps[i] <= p - c.r) argmin_take(best, k);
                argmin_take(best_all, k);
            }
        }
    }
    if (full) {
        best = warp_argmin(best);
        best_all = warp_argmin(best_all);
        if (lane == 0) {
            S.am[0][0][warp] = best.hi; S.am[0][1][warp] = best.lo; S.am[0][2][warp] = best.slot;
            S.am[1][0][warp] = best_all.hi; S.am[1][1][warp] = best_all.lo; S.am[1][2][warp] = best_all.slot;
        }
    }
    if (rank == 0 && tid == 0) {
        float2 pn = make_float2(0.f, 0.f);
#pragma unroll
        for (int g = 0; g < G; ++g) pn = pair_add(pn, ex2_approx(S.zn[g] - S.M[g]) * S.invL[g]);
        S.P_new = pn;
    }
    __syncthreads();
    if (full && warp == 0) {
        // this CTA's arg-mins; with C > 1 into rank 0's exchange
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            ArgMin w = lane < NW ? ArgMin{S.am[k][0][lane], S.am[k][1][lane], S.am[k][2][lane]} : argmin_none();
            w = warp_argmin(w);
            if (lane == 0) {
                const uint32_t base = x0 + (uint32_t)offsetof(GqaExchange<D>, am) + (uint32_t)(k * 3 * kMaxSplit * 4);
                st_cluster_s32(base + rank * 4, (int)w.hi);
                st_cluster_s32(base + (kMaxSplit + rank) * 4, (int)w.lo);
                st_cluster_s32(base + (2 * kMaxSplit + rank) * 4, (int)w.slot);
            }
        }
    }
    cta_group_sync(C);
    if (rank != 0) return;
    if (tid == 0) {
        int victim = n;
        if (full) {
            ArgMin vc = argmin_none(), va = argmin_none();
            for (int t = 0; t < C; ++t) {
                argmin_take(vc, ArgMin{S.x.am[0][0][t], S.x.am[0][1][t], S.x.am[0][2][t]});
                argmin_take(va, ArgMin{S.x.am[1][0][t], S.x.am[1][1][t], S.x.am[1][2][t]});
            }
            victim = (int)(vc.slot != 0xffffffffu ? vc.slot : va.slot);
        }
        if (victim < 0 || victim >= B) victim = 0;
        S.victim = victim;
        c.score[ub + victim] = S.P_new;
        c.pos[ub + victim] = p;
        c.ustate[unit] = make_int2(min(n + 1, B), p + 1);
        if (a.victim_out) a.victim_out[unit] = full ? victim : -1;
    }
    __syncthreads();
    const int victim = S.victim;
    if (tid < NV)
        reinterpret_cast<uint4*>(Kc + (size_t)victim * D)[tid] = newrow;
    else if (tid < 2 * NV)
        reinterpret_cast<uint4*>(Vc + (size_t)victim * D)[tid - NV] = newrow;
}

// ------------------------------------------------------------------ LSH

template <typename T, int D, class TL, int QB>
__global__ void __launch_bounds__(TL::NT, TL::MINB) lsh_decode_kernel(const DecodeArgs a)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    auto& S = *reinterpret_cast<DecodeSmem<T, D, TL, QB>*>(smem_raw);
    constexpr int EPL = D / 32;
    constexpr int NV = D * (int)sizeof(T) / 16;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const CacheView& c = a.c;
    const int C = (int)cluster_nctarank();
    const int rank = (int)cluster_ctarank();
    const int unit = blockIdx.x / C;

    const int B = c.B;
    const size_t ub = (size_t)unit * B;
    using CE = CacheElem<T, QB>;
    CE* Kc = reinterpret_cast<CE*>(c.K) + ub * RowElems<D, QB>;
    CE* Vc = reinterpret_cast<CE*>(c.V) + ub * RowElems<D, QB>;
    float2* Sc = QB ? c.kvs + (size_t)unit * c.Bp : nullptr;   // slot scale pairs
    int f0, f1;
    fetch_range(B, C, rank, f0, f1);
    if (lane == 0) {
#pragma unroll
        for (int b = 0; b < TL::NBUF; ++b) mbar_init(&S.bar[warp][b], 1);
        if (C > 1) fence_mbar_init(); else fence_proxy_async_smem();
    }
    if (C > 1) cluster_arrive_relaxed();     // paired with the wait before the exchange
    const T* qg = reinterpret_cast<const T*>(a.q) + (size_t)unit * D;
    const T* kg = reinterpret_cast<const T*>(a.k) + (size_t)unit * D;
    const T* vg = reinterpret_cast<const T*>(a.v) + (size_t)unit * D;
    // the input rows are read only after the wait, but their lines can be
    // on their way to L2 meanwhile, ahead of the cache traffic below
    prefetch_rows_l2(qg, kg, vg, D * (int)sizeof(T), tid);
    // The projection matrix is written once when the cache is created, never
    // by a previous kernel in the stream, so it is read before the wait:
    // warp w holds rows [w*RPW, w*RPW + RPW) of W, lane j the column of bit j.
    // Rows past D hold zeros (in x as well), which leave the sign of every
    // partial sum above zero unchanged.
    constexpr int RPW = (D + TL::NW - 1) / TL::NW;
    static_assert(TL::NW <= 16, "one named barrier (1..15) per hand-off");
    float wreg[RPW];
#pragma unroll
    for (int t = 0; t < RPW; ++t) {
        const int row = warp * RPW + t;
        wreg[t] = row < D ? __ldg(a.W + row * 32 + lane) : 0.f;
    }
    // This unit's occupancy, and the codes and positions of the slots this
    // thread scans (fetched for all B slots before the occupancy is known).
    // When the previous kernel in the stream cannot have written the cache,
    // these (and the first ring buffers, below) are read before the wait.
    constexpr int PF = 4;
    int2 us = make_int2(0, 0);
    unsigned pcode[PF];
    int ppos[PF];
    auto read_state = [&]() {
        us = c.ustate[unit];
#pragma unroll
        for (int i = 0; i < PF; ++i) {
            const int s = tid + i * TL::NT;
            pcode[i] = 0u;
            ppos[i] = 0;
            if (s < B) { pcode[i] = c.code[ub + s]; ppos[i] = c.pos[ub + s]; }
        }
    };
    // Early, each warp's first ring buffer is filled before the wait too;
    // the rest follow the small loads after it (priming the whole ring early
    // measured slower: its data landed while the victim was still being
    // decided, and HBM then idled until the attention started).
    if (a.early) {
        read_state();
        if (lane == 0) prime_ring<T, D, TL, QB>(S, Kc, Vc, Sc, f0, f1, 0, 1);
    }
    // everything below may read memory the previous kernel in the stream
    // has written (the inputs, and the cache unless read above)
    grid_dependency_wait();
    grid_launch_dependents();
    // the victim (which gates the attention) depends only on small loads:
    // q, k, v in one round trip, before the bulk copies, which would
    // otherwise delay them
    {
        const uint4 w = load_rows_16b<T, D>(qg, kg, vg, tid);
        if (!a.early) read_state();
        if (lane == 0) prime_ring<T, D, TL, QB>(S, Kc, Vc, Sc, f0, f1, a.early ? 1 : 0, TL::NBUF);
        store_rows_16b<T, D>(S.in, w, tid);
    }
    __syncthreads();
    const T* qs = reinterpret_cast<const T*>(S.in[0]);
    const T* ks = reinterpret_cast<const T*>(S.in[1]);
    const T* vs = reinterpret_cast<const T*>(S.in[2]);
    uint4 newrow = make_uint4(0u, 0u, 0u, 0u);
    if (rank == 0 && tid < 2 * NV) newrow = reinterpret_cast<const uint4*>(S.in[1])[tid];
    QRaw<T, D> qraw;
    load_q_raw<T, D>(qs, lane, qraw);
    const int n = us.x, p = us.y;
    const bool full = (n >= B);

    if (tid < D) {
        S.qf[tid] = Elem<T>::to_f(qs[tid]);
        S.kf[tid] = Elem<T>::to_f(ks[tid]);
    }
    __syncthreads();
    // sign codes: bit j is the sign of an fp32 fused multiply-add chain over
    // x[i] * W[i][j] in index order; the chain runs through the warps in turn
    // (lane j carries bit j's partial sums for query and key in S.hacc).
    // Every warp first pulls its rows of q and k into registers, so a turn
    // is a chain of register FMAs only.
    float xqr[RPW], xkr[RPW];
#pragma unroll
    for (int t = 0; t < RPW; ++t) {
        const int row = warp * RPW + t;
        xqr[t] = row < D ? S.qf[row] : 0.f;
        xkr[t] = row < D ? S.kf[row] : 0.f;
    }
    // Warp w takes the partial sums from warp w-1 through named barrier w
    // (64 threads: w-1 arrives, w waits), so a hand-off involves two warps.
    {
        float aq = 0.f, ak = 0.f;
        if (warp > 0) {
            named_barrier_sync(warp, 64);
            aq = S.hacc[0][lane];
            ak = S.hacc[1][lane];
        }
#pragma unroll
        for (int t = 0; t < RPW; ++t) {
            aq = __fmaf_rn(xqr[t], wreg[t], aq);
            ak = __fmaf_rn(xkr[t], wreg[t], ak);
        }
        if (warp + 1 < TL::NW) {
            S.hacc[0][lane] = aq;
            S.hacc[1][lane] = ak;
            named_barrier_arrive(warp + 1, 64);
        } else {
            const unsigned cq = __ballot_sync(kFull, aq > 0.f);
            const unsigned ck = __ballot_sync(kFull, ak > 0.f);
            if (lane == 0) { S.code_q = cq; S.code_k = ck; }
        }
    }
    __syncthreads();

    // victim: the largest Hamming distance, lowest slot on ties, packed as
    // (distance << 20) | (2^20 - 1 - slot) so one unsigned max decides;
    // every CTA of the cluster decides it redundantly
    if (full) {
        const unsigned cq = S.code_q;
        unsigned bk = 0u, bka = 0u;
#pragma unroll
        for (int i = 0; i < PF; ++i) {
            const int s = tid + i * TL::NT;
            if (s < n) {
                const unsigned key = ((unsigned)__popc(cq ^ pcode[i]) << 20) | (0xFFFFFu - (unsigned)s);
                if (ppos[i] <= p - c.r) bk = max(bk, key);
                bka = max(bka, key);
            }
        }
        for (int s = tid + PF * TL::NT; s < n; s += TL::NT) {
            const unsigned key = ((unsigned)__popc(cq ^ c.code[ub + s]) << 20) | (0xFFFFFu - (unsigned)s);
            if (c.pos[ub + s] <= p - c.r) bk = max(bk, key);
            bka = max(bka, key);
        }
        bk = __reduce_max_sync(kFull, bk);
        bka = __reduce_max_sync(kFull, bka);
        if (lane == 0) { S.ru[0][warp] = bk; S.ru[1][warp] = bka; }
        __syncthreads();
        if (warp == 0) {
            unsigned k0 = lane < TL::NW ? S.ru[0][lane] : 0u;
            unsigned k1 = lane < TL::NW ? S.ru[1][lane] : 0u;
            k0 = __reduce_max_sync(kFull, k0);
            k1 = __reduce_max_sync(kFull, k1);
            if (lane == 0) S.victim = (int)(0xFFFFFu - ((k0 ? k0 : k1) & 0xFFFFFu));
        }
    } else if (tid == 0) {
        S.victim = n;
    }
    __syncthreads();
    const int victim = S.victim;
    QVec<T, D, QB> qv;
    if constexpr (QB != 0) load_q_fix<QB, T, D>(qs, c.qscale, lane, S.qpl[warp], qv);
    else widen_q<T, D>(qraw, c.qscale, qv.v);

    float m_run = -INFINITY, l_run = 0.f, o[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] = 0.f;
    if (rank == 0 && warp == 0) {          // the new token, now in the victim slot
        const float zn = new_logit<QB, T, D>(qs, ks, c.qscale, qv, lane);
        float vr[EPL];
        load_vec<T, EPL>(vs + lane * EPL, vr);
        m_run = zn;
        l_run = lane == 0 ? 1.f : 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] = vr[e];
    }
    __syncwarp();

    attend_chunk<T, D, TL, QB>(S, Kc, Vc, Sc, f0, f1, n, full ? victim : -1, false, qv, m_run, l_run, o,
                               c.err);

    float Mc, Lc, Oc;
    merge_warps<T, D, TL, QB>(S, m_run, l_run, o, Mc, Lc, Oc);

    if (C > 1) {
        cluster_wait();                      // every CTA of the cluster runs (arrive at the start)
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
            float Mx = -INFINITY;
            for (int j = 0; j < C; ++j) Mx = fmaxf(Mx, S.x.m[j]);
            float L = 0.f, acc = 0.f;
            for (int j = 0; j < C; ++j) {
                const float f = safe_exp2_diff(S.x.m[j], Mx);
                L += S.x.l[j] * f;
                acc += S.x.o[j][tid] * f;
            }
            a.out[(size_t)unit * D + tid] = acc / L;
        }
    } else if (tid < D) {
        a.out[(size_t)unit * D + tid] = Oc / Lc;
    }
    if (tid == 0) {
        c.code[ub + victim] = S.code_k;
        c.pos[ub + victim] = p;
        c.ustate[unit] = make_int2(min(n + 1, B), p + 1);
        if (a.victim_out) a.victim_out[unit] = full ? victim : -1;
    }
    if constexpr (QB != 0) {
        store_row_quant<QB, T, D>(newrow, tid, Kc, Vc, Sc, victim);
    } else {
        if (tid < NV)
            reinterpret_cast<uint4*>(Kc + (size_t)victim * D)[tid] = newrow;
        else if (tid < 2 * NV)
            reinterpret_cast<uint4*>(Vc + (size_t)victim * D)[tid - NV] = newrow;
    }
}

// ------------------------------------------------------------- launching

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

template <typename T, int D, bool LSH, class TL, int QB = 0, bool GQ = false, bool SH = false>
cudaError_t launch_decode_t(const DecodeArgs& a, int split, cudaStream_t st)
{
    void (*kern)(const DecodeArgs);
    if constexpr (LSH) kern = lsh_decode_kernel<T, D, TL, QB>;
    else kern = h2o_decode_kernel<T, D, TL, QB, GQ, SH>;
    if constexpr (GQ) split = a.G;             // one CTA per query head of a cache unit
    const size_t smem = sizeof(DecodeSmem<T, D, TL, QB>);
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
    // programmatic dependent launch: this grid may be scheduled while the
    // previous one drains; the kernel waits for it before reading memory
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    int na = 1;
    if (split > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)split;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        na = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename T, int D, int G>
cudaError_t launch_gqa_t(const DecodeArgs& a, cudaStream_t st)
{
    void (*kern)(const DecodeArgs) = gqa_decode_kernel<T, D, G>;
    const size_t smem = sizeof(GqaSmem<T, D, G>);
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
    // CTAs per unit: enough to give every SM one while the exchange holds
    // their head states, never fewer than one per kMaxChunk slots
    int split = a.num_sms > 0 ? a.num_sms / max(1, a.c.U) : 1;
    if (const char* ev = getenv("H2O_GQA_SPLIT")) split = atoi(ev);   // tuning override
    split = max(split, (a.c.B + kMaxChunk - 1) / kMaxChunk);
    split = max(1, min(split, GqaShape<G>::CMAX));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.c.U * split), 1, 1);
    cfg.blockDim = dim3(GqaShape<G>::NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    int na = 1;
    if (split > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)split;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        na = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

// the one-pass grouped-query kernel unless H2O_GQA_PATH=cluster (one CTA per
// query head, kept for comparison); H2O_GQA_PATH=one takes it for every
// shape it serves (for comparisons)
int gqa_path()
{
    static int v = -1;
    if (v < 0) {
        const char* e = getenv("H2O_GQA_PATH");
        v = (e && strcmp(e, "cluster") == 0) ? 0 : (e && strcmp(e, "one") == 0) ? 2 : 1;
    }
    return v;
}
bool gqa_one_pass() { return gqa_path() != 0; }

// One row form QB over the dtypes and head sizes: tile TL, or TLF for bf16
// rows of 128 with fewer units than SMs (one-head caches).
template <bool LSH, int QB, class TL, class TLF, bool GQ = false>
cudaError_t dispatch_form(const DecodeArgs& a, int split, cudaStream_t st)
{
    const bool bf = a.c.dtype == 1;
    if (a.c.D == 128) {
        if (!GQ && bf && a.num_sms > 0 && a.c.U < a.num_sms)
            return launch_decode_t<__nv_bfloat16, 128, LSH, TLF, QB, GQ>(a, split, st);
        return bf ? launch_decode_t<__nv_bfloat16, 128, LSH, TL, QB, GQ>(a, split, st)
                  : launch_decode_t<float, 128, LSH, TL, QB, GQ>(a, split, st);
    }
    if (a.c.D == 64)
        return bf ? launch_decode_t<__nv_bfloat16, 64, LSH, TL, QB, GQ>(a, split, st)
                  : launch_decode_t<float, 64, LSH, TL, QB, GQ>(a, split, st);
    return cudaErrorInvalidValue;
}

template <bool LSH>
cudaError_t dispatch(const DecodeArgs& a, int split, cudaStream_t st)
{
    const bool bf = a.c.dtype == 1;
    if constexpr (!LSH) {
        if (a.G <= 1 && split == 1) {
            // one CTA per unit would do and the units are many: one warp per
            // unit instead (decode_warp.cu)
            bool used = false;
            const cudaError_t e = launch_h2o_decode_warps(a, st, &used);
            if (used || e != cudaSuccess) return e;
        }
        if (a.G > 1) {
            // one pass over each unit's rows for all heads (bf16 rows of 128,
            // 2, 4 or 8 heads per unit)
            // (4 heads on fewer units than half the SMs: the cluster path below
            // measured faster -- each of its CTAs walks fewer stages)
            const bool small4 = a.G == 4 && a.num_sms > 0 && 2 * a.c.U < a.num_sms && gqa_path() != 2;
            if (a.c.D == 128 && bf && a.c.qbits == 0 && gqa_one_pass() && !small4) {
                if (a.G == 2) return launch_gqa_t<__nv_bfloat16, 128, 2>(a, st);
                if (a.G == 4) return launch_gqa_t<__nv_bfloat16, 128, 4>(a, st);
                if (a.G == 8) return launch_gqa_t<__nv_bfloat16, 128, 8>(a, st);
            }
            // grouped-query cache (default tile), one CTA per query head: every dtype and row form
            if (a.c.qbits == 8) return dispatch_form<false, 8, TileDefault, TileDefault, true>(a, split, st);
            if (a.c.qbits == 4) return dispatch_form<false, 4, TileDefault, TileDefault, true>(a, split, st);
            return dispatch_form<false, 0, TileDefault, TileDefault, true>(a, split, st);
        }
    }
    // quantised rows: one CTA per SM with 8 warps when the units do not fill
    // the SMs (bf16 rows of 128), else 5 (int8) or 6 (4-bit) warps x 4 stages
    if (a.c.qbits == 8) return dispatch_form<LSH, 8, TileQ8, TileQ8Few>(a, split, st);
    if (a.c.qbits == 4) return dispatch_form<LSH, 4, TileQ4, TileQ4Few>(a, split, st);
    if (a.c.D == 128 && bf) {
        switch (tile_variant() ? tile_variant() : auto_tile(a.c.U, a.num_sms)) {
        case 1: return launch_decode_t<__nv_bfloat16, 128, LSH, Tile<4, 2>>(a, split, st);
        case 3: return launch_decode_t<__nv_bfloat16, 128, LSH, TileMany>(a, split, st);
        case 6: return launch_decode_t<__nv_bfloat16, 128, LSH, TileFew>(a, split, st);
        case 9: return launch_decode_t<__nv_bfloat16, 128, LSH, Tile<8, 3>>(a, split, st);
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

namespace {

// The bounded wait on a barrier that expects one arrival which never comes.
__global__ void wait_selftest_kernel(int* err)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_proxy_async_smem();
        if (!mbar_wait(&bar, 0)) atomicOr(err, kErrWaitTimeout);
    }
}

}  // namespace

cudaError_t launch_wait_selftest(int* err, cudaStream_t st)
{
    wait_selftest_kernel<<<1, 32, 0, st>>>(err);
    return cudaGetLastError();
}

int max_decode_split() { return kMaxSplit; }

namespace {

// Largest number of clusters of `split` CTAs of the few-units H2O or
// HashEvict kernel (bf16, head_dim 128; TileFew, or TileQ8Few / TileQ4Few
// for int8 / 4-bit rows) that the device runs at once; 0 on error.
template <class TL, int QB>
int clusters_that_fit_t(int split, bool lsh)
{
    void (*kern)(const DecodeArgs);
    if (lsh) kern = lsh_decode_kernel<__nv_bfloat16, 128, TL, QB>;
    else kern = h2o_decode_kernel<__nv_bfloat16, 128, TL, QB, false>;
    const size_t smem = sizeof(DecodeSmem<__nv_bfloat16, 128, TL, QB>);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)split, 1, 1);
    cfg.blockDim = dim3(TL::NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (const void*)kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

int clusters_that_fit(int split, bool lsh, int qbits)
{
    if (qbits == 8) return clusters_that_fit_t<TileQ8Few, 8>(split, lsh);
    if (qbits == 4) return clusters_that_fit_t<TileQ4Few, 4>(split, lsh);
    return clusters_that_fit_t<TileFew, 0>(split, lsh);
}

}  // namespace

// Decode split for a bf16, head_dim 128 one-head H2O or HashEvict cache with
// fewer units than SMs (the TileFew kernel, one CTA per SM): the most CTAs
// per unit with all U clusters resident at once (clusters are placed within
// a GPC, so U * split <= num_sms alone does not ensure it), at least one
// CTA per 1024 slots.  Results are cached per (device, U, B, kernel).
int few_units_split(int U, int B, int num_sms, bool lsh, int qbits)
{
    struct Entry { int dev, U, B, lsh, split; };
    const int key = (lsh ? 1 : 0) | (qbits << 1);
    static std::mutex mu;
    static Entry cache[64];
    static int n_cache = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < n_cache; ++i)
            if (cache[i].dev == dev && cache[i].U == U && cache[i].B == B && cache[i].lsh == key)
                return cache[i].split;
    }
    const int lo = max(1, (B + kMaxChunk - 1) / kMaxChunk);
    const int hi = max(1, (B + 63) / 64);
    int s = min(kMaxSplit, min(hi, max(lo, num_sms / max(U, 1))));
    while (s > lo && clusters_that_fit(s, lsh, qbits) < U) --s;
    std::lock_guard<std::mutex> lock(mu);
    if (n_cache < 64) cache[n_cache++] = Entry{dev, U, B, key, s};
    return s;
}

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

cudaError_t launch_sh_decode(const DecodeArgs& a, int split, cudaStream_t st)
{
    const bool bf = a.c.dtype == 1;
    if (a.c.qbits || a.G > 1) return cudaErrorInvalidValue;
    if (a.c.D == 128)
        return bf ? launch_decode_t<__nv_bfloat16, 128, false, TileDefault, 0, false, true>(a, split, st)
                  : launch_decode_t<float, 128, false, TileDefault, 0, false, true>(a, split, st);
    if (a.c.D == 64)
        return bf ? launch_decode_t<__nv_bfloat16, 64, false, TileDefault, 0, false, true>(a, split, st)
                  : launch_decode_t<float, 64, false, TileDefault, 0, false, true>(a, split, st);
    return cudaErrorInvalidValue;
}

}  // namespace h2o
