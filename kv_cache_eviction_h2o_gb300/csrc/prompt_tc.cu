// prompt_tc.cu -- the H2O prompt scorer on the 5th-generation tensor cores.
//
// [H2O review page, 提案手法: the accumulated attention of prompt token j,
//  c_j = sum_{i >= j} exp(z_ij - m_i) / l_i, ranks the heavy hitters.]
//
// Two passes over the causal 128 x 128 score tiles of each (batch, head)
// unit, bf16 inputs, head_dim 128:
//   pass 1  S = Q_blk K_blk^T        -> per row i: m2_i (base-2 max), l_i
//   pass 2  S^T = K_blk Q_blk^T      -> per key j: c_j = sum_i 2^(s_ij - m2_i) / l_i
// Pass 2 computes the transposed tile so that TMEM lane = key: each epilogue
// thread owns one key and sums its 128 query columns in registers; no
// cross-thread reduction is needed for the column sums.
//
// Per CTA (320 threads, two CTAs per SM): warp 0 issues TMA loads (128-byte
// swizzled boxes of 128 rows x 64 columns) into a ring of stages; lane 0 of
// warp 1 issues tcgen05.mma (M = N = 128, K = 16 per instruction, fp32
// accumulate) into one of two TMEM accumulators and commits to mbarriers;
// warps 2..5 drain accumulator 0 and warps 6..9 accumulator 1 with
// tcgen05.ld (thread = TMEM lane = tile row), so the exponentials of two
// tiles run at once and each scheduler has four epilogue warps to switch
// between.  Every wait is
// bounded: a wait that runs out sets the handle's error word (when there is
// one) and the CTA abandons its loop, writes NaN into the statistics it owns
// (so pass 2 and every reader of the column sums see the failure), waits
// (bounded) for its copies in flight, frees its TMEM and returns.
#include <cuda.h>
#include <algorithm>
#include <cfloat>
#include <cstddef>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace h2o {

namespace {

constexpr int kT = 128;                          // tile rows / columns
constexpr int kD = 128;                          // head dim handled here
constexpr uint32_t kBox = kT * 64 * 2;           // one 128 x 64 bf16 box: 16 KB
constexpr uint32_t kTile = 2 * kBox;             // 128 x 128 bf16: 32 KB
constexpr int kThreads = 192;                   // one epilogue group (persistence-of-importance flags)
constexpr int kThreadsW = 320;                  // two epilogue groups (the score passes)
constexpr int kScoreCtasPerSM = 2;
constexpr int kPersistBlocks = 32;               // prompts of up to 32 blocks run on a persistent grid

// instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bits
// 4-5 = 1), bf16 A and B (bits 7-9, 10-12 = 1), both K-major (bits 15, 16 =
// 0), N >> 3 at bits 17-22, M >> 4 at bits 24-28
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kT >> 3) << 17) |
                            ((uint32_t)(kT >> 4) << 24);

// ----------------------------------------------------------------- PTX

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* holder, uint32_t cols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(holder)),
                 "r"(cols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

// arrive on `bar` once every tcgen05 operation issued so far has completed
__device__ __forceinline__ void tc_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Issue the load of 32 consecutive fp32 columns of this thread's TMEM lane;
// the registers are valid only after tc_ld32_wait on the same array.
__device__ __forceinline__ void tc_ld32_issue(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// Wait for every TMEM load issued so far; taking r as in/out operands keeps
// the compiler from reading them before the wait.
__device__ __forceinline__ void tc_ld32_wait(uint32_t (&r)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]) :: "memory");
}

// The same for 16 columns.
__device__ __forceinline__ void tc_ld16_issue(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tc_ld16_wait(uint32_t (&r)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]) :: "memory");
}
__device__ __forceinline__ void tc_ld_issue(uint32_t taddr, uint32_t (&r)[16]) { tc_ld16_issue(taddr, r); }
__device__ __forceinline__ void tc_ld_wait(uint32_t (&r)[16]) { tc_ld16_wait(r); }

// max(a, b, c) in one instruction
__device__ __forceinline__ float max3f(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// 2^x by the MUFU instruction (2 ulp; results below 2^-126 flush to 0)
__device__ __forceinline__ float ex2_fast(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzled layout TMA writes: start address >> 4 (bits 0-13), leading
// offset 1 (unused for this layout), stride between 8-row groups 1024 B
// (bits 32-45, >> 4), descriptor version 1 (bits 46-47), swizzle mode
// 128 B (value 2 at bits 61-63).
__device__ __forceinline__ uint64_t sw128_desc(const void* p)
{
    const uint32_t a = smem_u32(p);
    return (uint64_t)((a & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Issue the 8 MMAs of one 128 x 128 x 128 tile: K slice k (16 elements,
// 32 bytes) sits in box k / 4 at byte offset 32 (k % 4) of each 128-byte
// swizzled row.
__device__ __forceinline__ void tile_mma(uint32_t d_tmem, const uint8_t* a, const uint8_t* b)
{
#pragma unroll
    for (int k = 0; k < kD / 16; ++k) {
        const uint32_t off = (uint32_t)(k / 4) * kBox + (uint32_t)(k % 4) * 32u;
        tc_mma(d_tmem, sw128_desc(a + off), sw128_desc(b + off), k > 0 ? 1u : 0u);
    }
}

// The same from the descriptors of the two tiles' starts: K slice k adds
// the slice's byte offset >> 4 to the start-address field (bits 0-13; the
// tiles lie below 256 KB, so the sum stays in the field).
__device__ __forceinline__ void tile_mma_desc(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc)
{
#pragma unroll
    for (int k = 0; k < kD / 16; ++k) {
        const uint64_t off = (uint64_t)(((uint32_t)(k / 4) * kBox + (uint32_t)(k % 4) * 32u) >> 4);
        tc_mma(d_tmem, adesc + off, bdesc + off, k > 0 ? 1u : 0u);
    }
}

// Shared memory of a scorer CTA: NA buffers of the A tile (the item's own
// block), a ring of NS B stages (the swept blocks), NACC fp32 accumulators
// of 128 TMEM columns, NGRP epilogue groups of four warps (group e drains
// accumulator e).
template <int NA, int NS, int NACC, int NGRP>
struct alignas(1024) TcSmemT {
    static constexpr int kA = NA, kS = NS, kAcc = NACC, kGrp = NGRP;
    static constexpr uint32_t kCols = (uint32_t)NACC * kT;   // TMEM columns (a power of 2)
    uint8_t a[NA][kTile];             // the item's own block (Q in pass 1, K in pass 2)
    uint8_t b[NS][kTile];             // ring of the swept blocks
    // pass 2: per warp of each group, its tile's 128 query biases -(m2 + log2(l)) (read as float4);
    // the flags kernel: two buffers of the 128 queries' thresholds ([0][0], [0][1])
    alignas(16) float colstat[NGRP][4][kT];
    double xch[2][NGRP > 1 ? NGRP - 1 : 1][3][kT];   // groups 1.. hand their per-item results to group 0, two items deep
    uint64_t a_full[NA];
    uint64_t a_empty[NA];             // the MMAs have read the A buffer
    uint64_t b_full[NS];
    uint64_t b_empty[NS];
    uint64_t acc_full[NACC];
    uint64_t acc_empty[NACC];
    uint32_t tmem_base;
    int abort;
};
// persistence-of-importance flags: one item per CTA, two CTAs per SM
using TcSmem = TcSmemT<1, 2, 2, 1>;
// the score passes: two CTAs per SM, each with two accumulators drained by
// two epilogue groups.  (One CTA per SM holding all of TMEM, with four
// groups, a double-buffered A tile and four B stages, measured 20-30 %
// slower: its groups meet at every item's merge and share one in-order
// MMA issuer.)
using TcSmemW = TcSmemT<1, 2, 2, 2>;
static_assert(TcSmemW::kAcc == TcSmemW::kGrp, "group e drains accumulator e");
static_assert(TcSmemW::kGrp * 128 + 64 == kThreadsW, "a producer warp, an MMA warp and the epilogue groups");
static_assert(offsetof(TcSmem, colstat) % 16 == 0, "colstat is read as float4");
static_assert(offsetof(TcSmem, b) % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(offsetof(TcSmemW, colstat) % 16 == 0, "colstat is read as float4");
static_assert(offsetof(TcSmemW, b) % 1024 == 0, "swizzled tiles need 1024-byte alignment");
// the dynamic size (the struct and its alignment slack) and the SM's 1 KB
// per CTA, for the CTAs that share an SM, within its 228 KB
static_assert(kScoreCtasPerSM * (sizeof(TcSmemW) + 1024 + 1024) <= 228 * 1024, "the score-pass CTAs must fit one SM");
static_assert(2 * (sizeof(TcSmem) + 1024 + 1024) <= 228 * 1024, "two flag CTAs must fit one SM");

template <class SM>
__device__ __forceinline__ SM& tc_smem(unsigned char* raw)
{
    const uintptr_t p = (reinterpret_cast<uintptr_t>(raw) + 1023) & ~(uintptr_t)1023;
    return *reinterpret_cast<SM*>(p);
}

// bounded wait that also watches the CTA's abort flag
template <class SM>
__device__ __forceinline__ bool tc_wait(SM& S, uint64_t* bar, uint32_t parity, int* err)
{
    if (mbar_wait(bar, parity)) return true;
    if (err) atomicOr(err, kErrWaitTimeout);
    *(volatile int*)&S.abort = 1;
    return false;
}

template <class SM>
__device__ __forceinline__ bool aborted(SM& S) { return *(volatile int*)&S.abort != 0; }

// OR of `pred` over the 128 epilogue threads of the flags kernel (named
// barrier ID); also orders their earlier shared-memory writes before the
// later reads
template <int ID = 1>
__device__ __forceinline__ bool epilogue_any(bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "barrier.red.or.pred q, %2, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "n"(ID)
        : "memory");
    return r != 0;
}

// All epilogue groups (named barrier 5): groups 1.. have put their per-item
// results in `xch` for group 0
template <int NG>
__device__ __forceinline__ void groups_sync()
{
    asm volatile("bar.sync 5, %0;" ::"n"(NG * 128) : "memory");
}

template <class SM>
__device__ __forceinline__ void tc_setup(SM& S, int warp)
{
    if (threadIdx.x == 0) {
        for (int k = 0; k < SM::kA; ++k) {
            mbar_init(&S.a_full[k], 1);
            mbar_init(&S.a_empty[k], 1);
        }
        for (int s = 0; s < SM::kS; ++s) {
            mbar_init(&S.b_full[s], 1);
            mbar_init(&S.b_empty[s], 1);
        }
        for (int b = 0; b < SM::kAcc; ++b) {
            mbar_init(&S.acc_full[b], 1);
            mbar_init(&S.acc_empty[b], 4);        // one arrival per warp of the group draining it
        }
        S.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&S.tmem_base, SM::kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// End of a one-item CTA (the flags kernel).
__device__ __forceinline__ void tc_teardown(TcSmem& S, int warp, int n_b_loads)
{
    constexpr int NS = TcSmem::kS;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (aborted(S) && threadIdx.x == 0) {
        // copies may still be in flight: wait (bounded) for every stage's
        // last load before the CTA's shared memory is released
        for (int t = (n_b_loads > NS ? n_b_loads - NS : 0); t < n_b_loads; ++t)
            mbar_wait(&S.b_full[t % NS], (uint32_t)(t / NS) & 1u);
        mbar_wait(&S.a_full[0], 0);
    }
    if (warp == 1) tmem_dealloc(S.tmem_base, TcSmem::kCols);
}

// Producer of a one-item CTA: its own block once, then the swept blocks
// `first..last` (inclusive) through the ring.
__device__ __forceinline__ void tc_producer(TcSmem& S, const CUtensorMap* map_a, const CUtensorMap* map_b,
                                            int row_a, int row0_b, int first, int last, int* err)
{
    constexpr int NS = TcSmem::kS;
    mbar_arrive_expect_tx(&S.a_full[0], kTile);
    tma_load_2d(S.a[0], map_a, 0, row_a, &S.a_full[0]);
    tma_load_2d(S.a[0] + kBox, map_a, 64, row_a, &S.a_full[0]);
    for (int t = 0; first + t <= last; ++t) {
        const int s = t % NS;
        if (t >= NS && !tc_wait(S, &S.b_empty[s], ((uint32_t)(t / NS) & 1u) ^ 1u, err)) return;
        if (aborted(S)) return;
        mbar_arrive_expect_tx(&S.b_full[s], kTile);
        tma_load_2d(S.b[s], map_b, 0, row0_b + (first + t) * kT, &S.b_full[s]);
        tma_load_2d(S.b[s] + kBox, map_b, 64, row0_b + (first + t) * kT, &S.b_full[s]);
    }
}

// MMA issuer of a one-item CTA (one thread): tile t of the sweep into
// accumulator t & 1.
__device__ __forceinline__ void tc_mma_loop(TcSmem& S, uint32_t tbase, int ntiles, int* err)
{
    constexpr int NS = TcSmem::kS;
    if (!tc_wait(S, &S.a_full[0], 0, err)) return;
    for (int t = 0; t < ntiles; ++t) {
        const int s = t % NS, b = t & 1;
        if (!tc_wait(S, &S.b_full[s], (uint32_t)(t / NS) & 1u, err)) return;
        if (t >= 2 && !tc_wait(S, &S.acc_empty[b], ((uint32_t)(t >> 1) & 1u) ^ 1u, err)) return;
        if (aborted(S)) return;
        tc_fence_after();
        tile_mma(tbase + (uint32_t)b * kT, S.a[0], S.b[s]);
        tc_commit(&S.b_empty[s]);       // the stage is free once these MMAs have read it
        tc_commit(&S.acc_full[b]);      // and the accumulator is ready for the epilogue
    }
}

// ------------------------------------------------ persistent item loops
//
// The score passes run on a persistent grid: CTA c takes one work item per
// round of P = gridDim.x items (walk_item), an item being one (unit, block)
// of group_order below; with P = the item count every CTA takes one item.
// TMEM, the barriers and the ring stay live across items, and every role
// counts ring stages, accumulators and A tiles over the whole walk, so the
// next item's tiles are loaded and multiplied while the epilogue still
// drains this item's accumulators.  Item k's A tile goes to buffer k % NA;
// the MMA issuer commits that buffer's `a_empty` after the item's last MMA
// and the producer waits for it before loading item k + NA there.

struct ItemWalk {
    int n_b;                          // B tiles the producer issued
    int n_a;                          // A tiles the producer issued
};

// Item of this CTA in round i of the walk (nitems if none): round i covers
// items i P .. i P + P - 1, taken in CTA order on even rounds and in reverse
// on odd ones, so a CTA that drew a heavy block (many tiles) in one round
// draws a light one in the next.
__device__ __forceinline__ int walk_item(int i, int nitems)
{
    const int P = (int)gridDim.x, c = (int)blockIdx.x;
    const int x = i * P + ((i & 1) ? P - 1 - c : c);
    return x < nitems ? x : nitems;
}

// Producer over the items: `item(x, row_a, row0_b, first, last)` gives the
// A row, the first B row and the swept block range of item x.
template <class SM, class ItemFn>
__device__ __forceinline__ ItemWalk tc_producer_items(SM& S, const CUtensorMap* map_a, const CUtensorMap* map_b,
                                                      int nitems, ItemFn item, int* err)
{
    constexpr int NA = SM::kA, NS = SM::kS;
    ItemWalk w{0, 0};
    for (int i = 0; i * (int)gridDim.x < nitems; ++i) {
        const int x = walk_item(i, nitems);
        if (x >= nitems) continue;
        int row_a, row0_b, first, last;
        item(x, row_a, row0_b, first, last);
        const int ka = w.n_a % NA;
        // the buffer's previous item (w.n_a - NA) has been multiplied
        if (w.n_a >= NA && !tc_wait(S, &S.a_empty[ka], (uint32_t)((w.n_a / NA - 1) & 1), err)) return w;
        if (aborted(S)) return w;
        mbar_arrive_expect_tx(&S.a_full[ka], kTile);
        tma_load_2d(S.a[ka], map_a, 0, row_a, &S.a_full[ka]);
        tma_load_2d(S.a[ka] + kBox, map_a, 64, row_a, &S.a_full[ka]);
        ++w.n_a;
        for (int bk = first; bk <= last; ++bk) {
            const int s = w.n_b % NS;
            if (w.n_b >= NS && !tc_wait(S, &S.b_empty[s], ((uint32_t)(w.n_b / NS) & 1u) ^ 1u, err))
                return w;
            if (aborted(S)) return w;
            mbar_arrive_expect_tx(&S.b_full[s], kTile);
            tma_load_2d(S.b[s], map_b, 0, row0_b + bk * kT, &S.b_full[s]);
            tma_load_2d(S.b[s] + kBox, map_b, 64, row0_b + bk * kT, &S.b_full[s]);
            ++w.n_b;
        }
    }
    return w;
}

// MMA issuer over the items: `tiles(x)` is item x's tile count.  Tile g of
// the walk goes to accumulator g % NACC.
template <class SM, class TilesFn>
__device__ __forceinline__ void tc_mma_items(SM& S, uint32_t tbase, int nitems, TilesFn tiles, int* err)
{
    constexpr int NA = SM::kA, NS = SM::kS, NACC = SM::kAcc;
    int g = 0, ia = 0;
    for (int i = 0; i * (int)gridDim.x < nitems; ++i) {
        const int x = walk_item(i, nitems);
        if (x >= nitems) continue;
        const int ntiles = tiles(x);
        const int ka = ia % NA;
        const uint64_t adesc = sw128_desc(S.a[ka]);
        if (!tc_wait(S, &S.a_full[ka], (uint32_t)((ia / NA) & 1), err)) return;
        for (int t = 0; t < ntiles; ++t, ++g) {
            const int s = g % NS, b = g % NACC;
            if (!tc_wait(S, &S.b_full[s], (uint32_t)(g / NS) & 1u, err)) return;
            if (g >= NACC && !tc_wait(S, &S.acc_empty[b], ((uint32_t)(g / NACC) & 1u) ^ 1u, err)) return;
            if (aborted(S)) return;
            tc_fence_after();
            tile_mma_desc(tbase + (uint32_t)b * kT, adesc, sw128_desc(S.b[s]));
            tc_commit(&S.b_empty[s]);     // the stage is free once these MMAs have read it
            tc_commit(&S.acc_full[b]);    // and the accumulator is ready for the epilogue
        }
        tc_commit(&S.a_empty[ka]);        // this item's A tile has been read
        ++ia;
    }
    // the last releases land before the CTA can leave
    for (int k = (ia > NA ? ia - NA : 0); k < ia; ++k) tc_wait(S, &S.a_empty[k % NA], (uint32_t)((k / NA) & 1), err);
}

// End of a walk: every role is past its loop.  An aborted CTA waits
// (bounded) for the copies it may still have in flight -- the last stages of
// the ring and the last A tiles -- before its shared memory is released.
template <class SM>
__device__ __forceinline__ void tc_teardown_items(SM& S, int warp, const ItemWalk& w)
{
    constexpr int NA = SM::kA, NS = SM::kS;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (aborted(S) && threadIdx.x == 0) {
        for (int t = (w.n_b > NS ? w.n_b - NS : 0); t < w.n_b; ++t)
            mbar_wait(&S.b_full[t % NS], (uint32_t)(t / NS) & 1u);
        for (int k = (w.n_a > NA ? w.n_a - NA : 0); k < w.n_a; ++k)
            mbar_wait(&S.a_full[k % NA], (uint32_t)((k / NA) & 1));
    }
    if (warp == 1) tmem_dealloc(S.tmem_base, SM::kCols);
}

// ------------------------------------------------------- CTA schedule

// CTA x -> (unit u, block rank k): units go in groups of g, and within a
// group the k-th heaviest block of every unit comes before the (k+1)-th.  A
// group's blocks all sweep the same K (pass 1) or Q (pass 2) tiles of its g
// units, so with g about the number of resident CTAs over the blocks per
// unit those tiles are read from HBM about once and then served by L2,
// while the heaviest blocks still start first.
__device__ __forceinline__ void group_order(int x, int U, int nb, int g, int& u, int& k)
{
    const int grp = x / (g * nb);
    const int u0 = grp * g;
    const int gs = min(g, U - u0);
    const int r = x - grp * g * nb;
    k = r / gs;
    u = u0 + r % gs;
}

// ------------------------------------------------------------- pass 1

// Items x < nitems (U * nb, or U * nq for the last nq blocks with g = U):
// item x is row block ib = nb - 1 - k of unit u (group_order); it sweeps key
// blocks 0..ib.  Persistent grid (see the item loops above).
__global__ void __launch_bounds__(kThreadsW, kScoreCtasPerSM)
    rowstats_tc_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK, int U,
                       int G, int T, int nb, int g, int nitems, float c2, float* __restrict__ m2,
                       float* __restrict__ lout, float* __restrict__ nbias, int* err)
{
    extern __shared__ unsigned char smem_raw[];
    TcSmemW& S = tc_smem<TcSmemW>(smem_raw);
    constexpr int NG = TcSmemW::kGrp;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto unit_block = [&](int x, int& u, int& ib) {
        int k;
        group_order(x, U, nb, g, u, k);
        ib = nb - 1 - k;
    };
    tc_setup(S, warp);
    const uint32_t tbase = S.tmem_base;
    ItemWalk w{0, 0};

    if (warp == 0) {
        if (lane == 0)
            w = tc_producer_items(S, &mapQ, &mapK, nitems,
                                  [&](int x, int& row_a, int& row0_b, int& first, int& last) {
                                      int u, ib;
                                      unit_block(x, u, ib);
                                      row_a = u * T + ib * kT;
                                      row0_b = (u / G) * T;
                                      first = 0;
                                      last = ib;
                                  },
                                  err);
    } else if (warp == 1) {
        if (lane == 0)
            tc_mma_items(S, tbase, nitems,
                         [&](int x) {
                             int u, ib;
                             unit_block(x, u, ib);
                             return ib + 1;
                         },
                         err);
        __syncwarp();
    } else {
        // Four epilogue groups of four warps: group e drains accumulator e,
        // that is tiles g of the walk with g % 4 == e, so four tiles are in
        // the exponentials at once and each scheduler holds four epilogue
        // warps.  Each group keeps the running statistics of its own tiles;
        // at the end of an item groups 1..3 hand their (m, l) to group 0,
        // which merges and writes.
        const int q = warp & 3;                   // TMEM lane quarter of this warp
        const int grp = (warp - 2) >> 2;
        const int kk = 32 * q + lane;             // row of the block (TMEM lane)
        int gt = 0;                               // tiles of the walk so far (both groups)
        int ia = 0;                               // items so far
        bool dead = false;                        // a wait ran out: the rest is NaN
        const float qnan = __int_as_float(0x7fffffff);
        for (int r = 0; r * (int)gridDim.x < nitems; ++r) {
            const int x = walk_item(r, nitems);
            if (x >= nitems) continue;
            int u, ib;
            unit_block(x, u, ib);
            const int i = ib * kT + kk;               // query row within the unit
            const int ntiles = ib + 1;
            float m = -INFINITY, l = 0.f, lc = 0.f;   // running base-2 max, Kahan-summed normaliser
            for (int t = (grp - (gt & (NG - 1))) & (NG - 1); t < ntiles && !dead; t += NG) {
                const int gg = gt + t;                // this tile of the walk: accumulator grp
                const bool ok = tc_wait(S, &S.acc_full[grp], (uint32_t)(gg / NG) & 1u, err);
                if (__any_sync(0xffffffffu, !ok || aborted(S))) {
                    dead = true;
                    break;
                }
                tc_fence_after();
                const bool diag = (t == ib);
                // the four 32-column chunks, each load issued while the
                // previous chunk is processed
                const uint32_t tcol = tbase + ((uint32_t)(32 * q) << 16) + (uint32_t)(grp * kT);
                uint32_t ra[32], rb[32];
                tc_ld32_issue(tcol, ra);
                tc_ld32_wait(ra);
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t (&cur)[32] = (ch & 1) ? rb : ra;
                    uint32_t (&nxt)[32] = (ch & 1) ? ra : rb;
                    if (ch + 1 < 4) tc_ld32_issue(tcol + (uint32_t)((ch + 1) * 32), nxt);
                    float v[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(cur[e]);
                    const int j0 = t * kT + ch * 32;
                    if (diag) {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (j0 + e > i) v[e] = -INFINITY;
                    }
                    // the chunk's max as a tree of three-input max
                    // instructions: 17 of them, four deep (a chain of 16
                    // would put all of them on the critical path)
                    float t1[11];
#pragma unroll
                    for (int k = 0; k < 10; ++k) t1[k] = max3f(v[3 * k], v[3 * k + 1], v[3 * k + 2]);
                    t1[10] = fmaxf(v[30], v[31]);
                    const float t20 = max3f(t1[0], t1[1], t1[2]), t21 = max3f(t1[3], t1[4], t1[5]);
                    const float t22 = max3f(t1[6], t1[7], t1[8]), t23 = fmaxf(t1[9], t1[10]);
                    const float cm = fmaxf(max3f(t20, t21, t22), t23);
                    {
                        // branch-free rescale: alpha is exactly 1 when the max
                        // stays, 0 before the first finite column; a chunk of
                        // masked columns (-inf) leaves m, and adds nothing
                        const float mn = fmaxf(m, cm * c2);
                        const float alpha = (mn == m) ? 1.f : ex2_fast(m - mn);   // ex2(-inf) = 0
                        l *= alpha;
                        lc *= alpha;
                        m = mn;
                        // exponent arguments and running sums two columns at a time
                        const float2 c22 = make_float2(c2, c2), nm2 = make_float2(-m, -m);
                        float2 sa = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f);
#pragma unroll
                        for (int e = 0; e < 32; e += 4) {
                            const float2 ta = __ffma2_rn(make_float2(v[e], v[e + 1]), c22, nm2);
                            const float2 tb = __ffma2_rn(make_float2(v[e + 2], v[e + 3]), c22, nm2);
                            sa = __fadd2_rn(sa, make_float2(ex2_fast(ta.x), ex2_fast(ta.y)));
                            sb = __fadd2_rn(sb, make_float2(ex2_fast(tb.x), ex2_fast(tb.y)));
                        }
                        // Kahan step
                        const float y = ((sa.x + sa.y) + (sb.x + sb.y)) - lc;
                        const float tsum = l + y;
                        lc = (tsum - l) - y;
                        l = tsum;
                    }
                    if (ch + 1 < 4) tc_ld32_wait(nxt);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.acc_empty[grp]);
            }
            gt += ntiles;
            // merge the groups' statistics of the block's rows:
            // m = max_e m_e, l = sum_e l_e 2^(m_e - m)
            if (grp > 0) {
                float* xm = reinterpret_cast<float*>(S.xch[ia & 1][grp - 1][0]);
                xm[kk] = dead ? qnan : m;
                xm[kT + kk] = dead ? qnan : l - lc;
            }
            groups_sync<NG>();
            if (grp == 0 && i < T) {
                float me[NG], le[NG];
                me[0] = m;
                le[0] = dead ? qnan : l - lc;
#pragma unroll
                for (int e = 1; e < NG; ++e) {
                    const float* xm = reinterpret_cast<const float*>(S.xch[ia & 1][e - 1][0]);
                    me[e] = xm[kk];
                    le[e] = xm[kT + kk];
                }
                float mo = -INFINITY, lo = 0.f;
                bool bad = false;
#pragma unroll
                for (int e = 0; e < NG; ++e) {
                    bad |= isnan(le[e]);
                    mo = fmaxf(mo, me[e]);
                }
#pragma unroll
                for (int e = 0; e < NG; ++e) lo += (me[e] == -INFINITY) ? 0.f : le[e] * exp2f(me[e] - mo);
                // an abandoned walk leaves NaN, which the column sums carry on
                m2[(size_t)u * T + i] = bad ? qnan : mo;
                lout[(size_t)u * T + i] = bad ? qnan : lo;
                // the row's bias in the second pass: a weight is 2^(s c2 + bias)
                if (nbias) nbias[(size_t)u * T + i] = bad ? qnan : -(mo + log2f(lo));
            }
            ++ia;
        }
    }
    tc_teardown_items(S, warp, w);
}

// ------------------------------------------------------------- pass 2

// Items x < U * nb: item x is key block jb = k of unit u (group_order:
// heaviest blocks, small jb, first within a group of units); it sweeps query
// blocks jb..nb-1.  Persistent grid (see the item loops above).
// BAND: also the band sums of the per-head policy profile (a separate
// instantiation, so the plain pass carries none of their instructions).
template <bool BAND>
__global__ void __launch_bounds__(kThreadsW, kScoreCtasPerSM)
    colsum_tc_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK, int U,
                     int G, int T, int nb, int g, int nitems, float c2, const float* __restrict__ nbias,
                     double* __restrict__ cout, double* __restrict__ bandB, double* __restrict__ bandr, int wB,
                     int wr, int* err)
{
    extern __shared__ unsigned char smem_raw[];
    TcSmemW& S = tc_smem<TcSmemW>(smem_raw);
    constexpr int NG = TcSmemW::kGrp;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    tc_setup(S, warp);
    const uint32_t tbase = S.tmem_base;
    ItemWalk w{0, 0};

    if (warp == 0) {
        if (lane == 0)
            w = tc_producer_items(S, &mapK, &mapQ, nitems,
                                  [&](int x, int& row_a, int& row0_b, int& first, int& last) {
                                      int u, jb;
                                      group_order(x, U, nb, g, u, jb);
                                      row_a = (u / G) * T + jb * kT;
                                      row0_b = u * T;
                                      first = jb;
                                      last = nb - 1;
                                  },
                                  err);
    } else if (warp == 1) {
        if (lane == 0)
            tc_mma_items(S, tbase, nitems,
                         [&](int x) {
                             int u, jb;
                             group_order(x, U, nb, g, u, jb);
                             return nb - jb;
                         },
                         err);
        __syncwarp();
    } else {
        // Four epilogue groups as in pass 1: group e drains the tiles g of
        // the walk with g % 4 == e; each keeps its own sums of the block's
        // keys, and groups 1..3 hand theirs to group 0 at the end of an item.
        const int q = warp & 3;
        const int grp = (warp - 2) >> 2;
        const int kk = 32 * q + lane;             // key of the block (TMEM lane)
        const int wmax = max(wB, wr);
        const double nan = __longlong_as_double(0x7ff8000000000000LL);
        const int P = (int)gridDim.x;
        int gt = 0;                               // tiles of the walk so far (both groups)
        int ia = 0;                               // items so far
        bool dead = false;                        // a wait ran out: the rest is NaN
        // unit and query block of tile `target` of the walk, searching from
        // round r, whose item starts at tile g0; false past the walk's end
        auto locate = [&](int r, int g0, int target, int& uo, int& ibo) {
            for (; r * P < nitems; ++r) {
                const int x = walk_item(r, nitems);
                if (x >= nitems) continue;
                int u, jb;
                group_order(x, U, nb, g, u, jb);
                const int nt = nb - jb;
                if (target < g0 + nt) {
                    uo = u;
                    ibo = jb + (target - g0);
                    return true;
                }
                g0 += nt;
            }
            return false;
        };
        // Each warp stages its own copy of a tile's 128 query biases
        // (written by pass 1: a weight is 2^(s c2 + bias); -inf past T,
        // weight 0), four per lane, so no barrier joins the group's warps:
        // the next tile's four are loaded at the start of a tile and stored
        // after it.
        float* wbias = S.colstat[grp][q];
        auto load_bias = [&](int uq, int ibq, float (&bq)[4]) {
            const int iq0 = ibq * kT + 4 * lane;
            const float* src = nbias + (size_t)uq * T + iq0;
            if (iq0 + 3 < T && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
                // the four in one 16-byte load where the address allows
                const float4 b4 = __ldg(reinterpret_cast<const float4*>(src));
                bq[0] = b4.x; bq[1] = b4.y; bq[2] = b4.z; bq[3] = b4.w;
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) bq[k] = iq0 + k < T ? src[k] : -INFINITY;
            }
        };
        auto store_bias = [&](const float (&bq)[4]) {
            __syncwarp();                         // every lane is past its reads of the last tile's biases
            *reinterpret_cast<float4*>(wbias + 4 * lane) = make_float4(bq[0], bq[1], bq[2], bq[3]);
            __syncwarp();
        };
        {
            // the group's first tile: walk tile grp
            int u0, ib0;
            if (locate(0, 0, grp, u0, ib0)) {
                float b0[4];
                load_bias(u0, ib0, b0);
                store_bias(b0);
            }
        }
        for (int r = 0; r * P < nitems; ++r) {
            const int x = walk_item(r, nitems);
            if (x >= nitems) continue;
            int u, jb;
            group_order(x, U, nb, g, u, jb);
            const int ntiles = nb - jb;
            const int j = jb * kT + kk;               // key within the unit
            float cs = 0.f, cc = 0.f;                 // Kahan-summed column sum
            double bsB = 0.0, bsr = 0.0;              // band sums (rows j .. j+w-1)
            for (int t = (grp - (gt & (NG - 1))) & (NG - 1); t < ntiles && !dead; t += NG) {
                const int gg = gt + t;                // this tile of the walk: accumulator grp
                const int ib = jb + t;
                // some key of the block has rows of this tile in its band
                const bool band = BAND && ib * kT < (jb + 1) * kT + wmax;
                // the group's next tile (gg + NG): its biases are loaded now
                // and staged after this tile
                int un = u, ibn = ib + NG;
                const bool more = t + NG < ntiles || locate(r, gt, gg + NG, un, ibn);
                float bnext[4];
                if (more) load_bias(un, ibn, bnext);
                const bool ok = tc_wait(S, &S.acc_full[grp], (uint32_t)(gg / NG) & 1u, err);
                if (__any_sync(0xffffffffu, !ok || aborted(S))) {
                    dead = true;
                    break;
                }
                tc_fence_after();
                const bool edge = (t == 0) || ((ib + 1) * kT > T);
                const float* bs = wbias;
                const int dj = ib * kT - j;               // i - j of the tile's first row
                float part = 0.f, partB = 0.f, partr = 0.f;
                const uint32_t tcol = tbase + ((uint32_t)(32 * q) << 16) + (uint32_t)(grp * kT);
                // chunks of CW columns, each load issued while the previous
                // chunk is processed (16: measured 2 % faster than 32 here,
                // and the band sums' registers leave no room for two
                // 32-column buffers)
                constexpr int CW = 16, NCH = kT / CW;
                uint32_t ra[CW], rb[CW];
                tc_ld_issue(tcol, ra);
                tc_ld_wait(ra);
                // the causal and past-T masks are compiled only into the edge
                // tiles' copy of the chunk loop
                auto chunks = [&](auto edge_tag) {
                    constexpr bool EDGE = decltype(edge_tag)::value;
#pragma unroll
                    for (int ch = 0; ch < NCH; ++ch) {
                        uint32_t (&cur)[CW] = (ch & 1) ? rb : ra;
                        uint32_t (&nxt)[CW] = (ch & 1) ? ra : rb;
                        if (ch + 1 < NCH) tc_ld_issue(tcol + (uint32_t)((ch + 1) * CW), nxt);
                        const int i0 = ib * kT + ch * CW;
                        const float2 c22 = make_float2(c2, c2);
                        float2 pa = make_float2(0.f, 0.f), pb = make_float2(0.f, 0.f);
#pragma unroll
                        for (int e = 0; e < CW; e += 4) {
                            const float4 b4 = *reinterpret_cast<const float4*>(bs + ch * CW + e);
                            const float2 ta = __ffma2_rn(make_float2(__uint_as_float(cur[e]), __uint_as_float(cur[e + 1])),
                                                         c22, make_float2(b4.x, b4.y));
                            const float2 tb = __ffma2_rn(make_float2(__uint_as_float(cur[e + 2]), __uint_as_float(cur[e + 3])),
                                                         c22, make_float2(b4.z, b4.w));
                            float w0 = ex2_fast(ta.x), w1 = ex2_fast(ta.y), w2 = ex2_fast(tb.x), w3 = ex2_fast(tb.y);
                            if constexpr (EDGE) {
                                if (i0 + e < j) w0 = 0.f;
                                if (i0 + e + 1 < j) w1 = 0.f;
                                if (i0 + e + 2 < j) w2 = 0.f;
                                if (i0 + e + 3 < j) w3 = 0.f;
                            }
                            pa = __fadd2_rn(pa, make_float2(w0, w1));
                            pb = __fadd2_rn(pb, make_float2(w2, w3));
                            if (band) {
                                const int d0 = dj + ch * CW + e;
                                partB += (d0 < wB ? w0 : 0.f) + (d0 + 1 < wB ? w1 : 0.f) + (d0 + 2 < wB ? w2 : 0.f) +
                                         (d0 + 3 < wB ? w3 : 0.f);
                                partr += (d0 < wr ? w0 : 0.f) + (d0 + 1 < wr ? w1 : 0.f) + (d0 + 2 < wr ? w2 : 0.f) +
                                         (d0 + 3 < wr ? w3 : 0.f);
                            }
                        }
                        part += (pa.x + pa.y) + (pb.x + pb.y);
                        if (ch + 1 < NCH) tc_ld_wait(nxt);
                    }
                };
                if (edge) chunks(std::true_type{});
                else chunks(std::false_type{});
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.acc_empty[grp]);
                const float y = part - cc;
                const float tsum = cs + y;
                cc = (tsum - cs) - y;
                cs = tsum;
                if (band) {
                    bsB += (double)partB;
                    bsr += (double)partr;
                }
                if (more) store_bias(bnext);
            }
            gt += ntiles;
            // groups 1..3 hand their sums to group 0, which adds and writes
            if (grp > 0) {
                S.xch[ia & 1][grp - 1][0][kk] = dead ? nan : (double)cs - (double)cc;
                if constexpr (BAND) {
                    S.xch[ia & 1][grp - 1][1][kk] = bsB;
                    S.xch[ia & 1][grp - 1][2][kk] = bsr;
                }
            }
            groups_sync<NG>();
            if (grp == 0 && j < T) {
                double ct = dead ? nan : (double)cs - (double)cc, bt = bsB, rt = bsr;
#pragma unroll
                for (int e = 1; e < NG; ++e) {
                    ct += S.xch[ia & 1][e - 1][0][kk];
                    if constexpr (BAND) {
                        bt += S.xch[ia & 1][e - 1][1][kk];
                        rt += S.xch[ia & 1][e - 1][2][kk];
                    }
                }
                // an abandoned walk leaves NaN in its columns (NaN propagates through the sum)
                cout[(size_t)u * T + j] = ct;
                if constexpr (BAND) {
                    bandB[(size_t)u * T + j] = isnan(ct) ? nan : bt;
                    bandr[(size_t)u * T + j] = isnan(ct) ? nan : rt;
                }
            }
            ++ia;
        }
    }
    tc_teardown_items(S, warp, w);
}

// ------------------------------------------------- persistence of importance

// Prompt pivotal histories [Scissorhands abstract; the rule is this
// library's reading]: the rows i of the window [max(0, T-32), T) are steps;
// key j <= i is pivotal for row i when P_ij (i + 1) > 1, that is when
// s_ij c2 > m2_i + log2(l_i / (i + 1)) -- a comparison, no exponential.
// grid: U * nb CTAs; CTA x takes key block jb = x / U of unit x % U and
// sweeps only the query blocks that hold window rows, from max(jb, qb0) to
// nb - 1 (one or two).  Each epilogue thread owns one key, sets bit T-1-i
// of its history for every pivotal window row i, and writes the history
// and the selection key (set bits * T + j).
__global__ void __launch_bounds__(kThreads, 2)
    sh_flags_tc_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK, int U,
                       int T, int nb, int qb0, float c2, const float* __restrict__ m2, const float* __restrict__ lin,
                       uint32_t* __restrict__ ck, double* __restrict__ cout, int* err)
{
    extern __shared__ unsigned char smem_raw[];
    static_assert(TcSmem::kGrp == 1, "the flags kernel drains with one group of four warps");
    TcSmem& S = tc_smem<TcSmem>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int u = blockIdx.x % U;
    const int jb = (int)(blockIdx.x / U);
    const int row0 = u * T;
    const int first = jb > qb0 ? jb : qb0;
    const int ntiles = nb - first;
    const int w0 = T > 32 ? T - 32 : 0;
    const float* m2u = m2 + (size_t)u * T;
    const float* lu = lin + (size_t)u * T;
    tc_setup(S, warp);
    const uint32_t tbase = S.tmem_base;

    // threshold of query row i in base-2 logit units; +inf outside the window
    auto thr = [&](int i) { return (i >= w0 && i < T) ? m2u[i] + log2f(lu[i] / (float)(i + 1)) : INFINITY; };

    if (warp == 0) {
        if (lane == 0) tc_producer(S, &mapK, &mapQ, row0 + jb * kT, row0, first, nb - 1, err);
    } else if (warp == 1) {
        if (lane == 0) tc_mma_loop(S, tbase, ntiles, err);
        __syncwarp();
    } else {
        const int et = threadIdx.x - 64;          // epilogue thread 0..127
        const int q = warp & 3;
        const int j = jb * kT + 32 * q + lane;    // key within the unit
        S.colstat[0][0][et] = thr(first * kT + et);
        uint32_t hist = 0u;
        for (int t = 0; t < ntiles; ++t) {
            const int b = t & 1;
            const int ib = first + t;
            const float nthr = (t + 1 < ntiles) ? thr((ib + 1) * kT + et) : INFINITY;
            const bool ok = tc_wait(S, &S.acc_full[b], (uint32_t)(t >> 1) & 1u, err);
            // agreed by all epilogue threads; also publishes last iteration's thresholds
            if (epilogue_any(!ok || aborted(S))) break;
            tc_fence_after();
            const float* th = S.colstat[0][b];
            const uint32_t tcol = tbase + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * kT);
            uint32_t ra[32], rb[32];
            tc_ld32_issue(tcol, ra);
            tc_ld32_wait(ra);
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t (&cur)[32] = (ch & 1) ? rb : ra;
                uint32_t (&nxt)[32] = (ch & 1) ? ra : rb;
                if (ch + 1 < 4) tc_ld32_issue(tcol + (uint32_t)((ch + 1) * 32), nxt);
                const int i0 = ib * kT + ch * 32;
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int i = i0 + e;
                    if (i >= j && __uint_as_float(cur[e]) * c2 > th[ch * 32 + e]) hist |= 1u << ((T - 1 - i) & 31);
                }
                if (ch + 1 < 4) tc_ld32_wait(nxt);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.acc_empty[b]);
            if (t + 1 < ntiles) S.colstat[0][b ^ 1][et] = nthr;
        }
        if (j < T && !aborted(S)) {
            ck[(size_t)u * T + j] = hist;
            cout[(size_t)u * T + j] = (double)__popc(hist) * (double)T + (double)j;
        }
    }
    tc_teardown(S, warp, ntiles);
}

// ------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// [rows][128] bf16 row-major, boxes of 128 rows x 64 columns, 128-byte swizzle
bool make_map(CUtensorMap* m, const void* base, long long rows)
{
    EncodeTiledFn enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    const cuuint32_t box[2] = {64u, (cuuint32_t)kT};
    const cuuint32_t estr[2] = {1u, 1u};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool prompt_tc_supported(const CacheView& c) { return c.dtype == 1 && c.D == kD; }

namespace {

// SM count of the current device (cached per device)
int sm_count()
{
    static int n[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!n[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        n[dev] = v;
    }
    return n[dev];
}

}  // namespace

cudaError_t launch_prompt_stats_tc(const CacheView& c, const PromptArgs& p, cudaStream_t st)
{
    CUtensorMap mq, mk;
    const int G = p.G > 1 ? p.G : 1;
    const long long rows = (long long)c.U * p.T;
    if (!p.nb) return cudaErrorInvalidValue;      // pass 2 reads the row biases pass 1 writes there
    if (!make_map(&mq, p.Q, rows) || !make_map(&mk, p.K, rows / G)) return cudaErrorInvalidValue;
    const size_t smem = sizeof(TcSmemW) + 1024;
    static bool configured[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(rowstats_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(colsum_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(colsum_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const int nb = (p.T + kT - 1) / kT;
    const int nitems = c.U * nb;
    // Persistent grid of the resident CTAs for prompts of up to
    // 32 blocks (4096 tokens), where an item's 1..32 tiles leave the per-CTA
    // set-up a large share; longer prompts take one item per CTA, whose
    // hardware scheduling (heaviest first) balances items of up to nb tiles
    // better than the fixed walk.
    const int resident = kScoreCtasPerSM * sm_count();
    const unsigned grid = nb <= kPersistBlocks ? (unsigned)std::min(nitems, resident) : (unsigned)nitems;
    // units per schedule group: the resident CTAs over the blocks per unit
    const int g = std::max(1, std::min(c.U, resident / nb));
    rowstats_tc_kernel<<<grid, kThreadsW, smem, st>>>(mq, mk, c.U, G, p.T, nb, g, nitems, c.qscale, p.m2, p.l,
                                                     p.nb, c.err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (p.bandB)
        colsum_tc_kernel<true><<<grid, kThreadsW, smem, st>>>(mq, mk, c.U, G, p.T, nb, g, nitems, c.qscale, p.nb,
                                                             p.c, p.bandB, p.bandr, p.wB, p.wr, c.err);
    else
        colsum_tc_kernel<false><<<grid, kThreadsW, smem, st>>>(mq, mk, c.U, G, p.T, nb, g, nitems, c.qscale, p.nb,
                                                              p.c, nullptr, nullptr, 0, 0, c.err);
    return cudaGetLastError();
}

// Prompt histories of the persistence-of-importance cache on the tensor
// cores: row statistics of the query blocks holding the last 32 rows only
// (the row-statistics kernel takes its blocks from the last one down, so a
// grid of U * nq CTAs covers exactly the last nq blocks), then the flags.
cudaError_t launch_sh_flags_tc(const CacheView& c, const PromptArgs& p, cudaStream_t st)
{
    CUtensorMap mq, mk;
    const long long rows = (long long)c.U * p.T;
    if (!make_map(&mq, p.Q, rows) || !make_map(&mk, p.K, rows)) return cudaErrorInvalidValue;
    const size_t smem = sizeof(TcSmem) + 1024, smemW = sizeof(TcSmemW) + 1024;
    static bool configured[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(rowstats_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smemW);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(sh_flags_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const int nb = (p.T + kT - 1) / kT;
    const int w0 = p.T > 32 ? p.T - 32 : 0;
    const int qb0 = w0 / kT, nq = nb - qb0;
    const int nitems = c.U * nq;
    rowstats_tc_kernel<<<(unsigned)std::min(nitems, kScoreCtasPerSM * sm_count()), kThreadsW, smemW, st>>>(
        mq, mk, c.U, 1, p.T, nb, c.U, nitems, c.qscale, p.m2, p.l, nullptr, c.err);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    sh_flags_tc_kernel<<<(unsigned)(c.U * nb), kThreads, smem, st>>>(mq, mk, c.U, p.T, nb, qb0, c.qscale, p.m2, p.l,
                                                                     p.ck, p.c, c.err);
    return cudaGetLastError();
}

}  // namespace h2o
