// common.cuh -- device helpers shared by the library's kernels: element
// loads, mbarrier / bulk-copy (TMA) wrappers with bounded waits, cluster
// barriers, and the launch-side structures.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace h2o {

constexpr float kLog2e = 1.4426950408889634f;

// bit flags OR-ed into a handle's device error word
enum DeviceError : int {
    kErrNone = 0,
    kErrWaitTimeout = 1,   // an mbarrier wait ran out of its bound
};

// ----------------------------------------------------------------- elements

template <typename T> struct Elem;

template <> struct Elem<float> {
    __device__ __forceinline__ static float to_f(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
    __device__ __forceinline__ static float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
};

// Load E consecutive elements starting at p (E * sizeof(T) bytes, naturally
// aligned) and widen them to fp32.
template <typename T, int E>
__device__ __forceinline__ void load_vec(const T* p, float* out)
{
    if constexpr (sizeof(T) == 2) {
        static_assert(E == 2 || E == 4 || E == 8, "bf16 vector width");
        if constexpr (E == 2) {
            uint32_t w = *reinterpret_cast<const uint32_t*>(p);
            out[0] = __uint_as_float(w << 16);
            out[1] = __uint_as_float(w & 0xffff0000u);
        } else if constexpr (E == 4) {
            uint2 w = *reinterpret_cast<const uint2*>(p);
            out[0] = __uint_as_float(w.x << 16); out[1] = __uint_as_float(w.x & 0xffff0000u);
            out[2] = __uint_as_float(w.y << 16); out[3] = __uint_as_float(w.y & 0xffff0000u);
        } else {
            uint4 w = *reinterpret_cast<const uint4*>(p);
            out[0] = __uint_as_float(w.x << 16); out[1] = __uint_as_float(w.x & 0xffff0000u);
            out[2] = __uint_as_float(w.y << 16); out[3] = __uint_as_float(w.y & 0xffff0000u);
            out[4] = __uint_as_float(w.z << 16); out[5] = __uint_as_float(w.z & 0xffff0000u);
            out[6] = __uint_as_float(w.w << 16); out[7] = __uint_as_float(w.w & 0xffff0000u);
        }
    } else {
        static_assert(E == 2 || E == 4, "fp32 vector width");
        if constexpr (E == 2) {
            float2 w = *reinterpret_cast<const float2*>(p);
            out[0] = w.x; out[1] = w.y;
        } else {
            float4 w = *reinterpret_cast<const float4*>(p);
            out[0] = w.x; out[1] = w.y; out[2] = w.z; out[3] = w.w;
        }
    }
}

// ------------------------------------------------------- shared-memory PTX

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// make mbarrier initialisation visible to the async (bulk-copy) proxy and
// to the rest of the cluster
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// one arrival (no transaction bytes) on `bar`
__device__ __forceinline__ void mbar_arrive_one(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase: gives up after ~2^31 SM clocks (about
// a second) or 2^24 polls, whichever comes first, and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (int it = 0; it < (1 << 24); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > (1LL << 31)) break;
    }
    return false;
}

// --------------------------------------------------------- cluster barrier

__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
// arrival with no memory ordering: marks this CTA as started for the
// matching cluster_wait
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
// address of the same shared-memory variable in CTA `rank` of this cluster
__device__ __forceinline__ uint32_t map_to_rank(const void* p, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v)
{
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_s32(uint32_t addr, int v)
{
    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// ------------------------------------------------------- fp32 pair scores
//
// Accumulated scores are held as an unevaluated pair hi + lo of fp32 values
// with |lo| <= ulp(hi) / 2 (about 48 significant bits), so the per-step
// accumulate and the eviction comparisons stay on the fp32 and integer
// pipes; GB300's fp64 pipe is far too narrow for the decode epilogue.

// (hi, lo) + x, exactly up to the final rounding of lo (TwoSum, then a
// renormalising Fast2Sum).
__device__ __forceinline__ float2 pair_add(float2 a, float x)
{
    const float s = a.x + x;
    const float bp = s - a.x;
    const float err = (a.x - (s - bp)) + (x - bp);
    const float t = a.y + err;
    const float hi = s + t;
    const float lo = t - (hi - s);
    return make_float2(hi, lo);
}

// Order-preserving map of an fp32 value to an unsigned key.
__device__ __forceinline__ unsigned ord_key(float x)
{
    const unsigned b = __float_as_uint(x);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Loads whose issue point is fixed (volatile): a value needed only much
// later is requested where the load is written, so its latency hides under
// the work in between instead of being paid at the use.
__device__ __forceinline__ uint32_t ld_issue_u32(const uint32_t* p)
{
    uint32_t v;
    asm volatile("ld.global.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ float2 ld_issue_f2(const float2* p)
{
    float2 v;
    asm volatile("ld.global.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
    return v;
}

// ---------------------------------------------- programmatic dependent launch

// Block until the grid this one depends on (the previous kernel in the
// stream) has completed and its memory is visible; a no-op when the grid was
// launched without a programmatic dependency.
// Ask L2 for the 128-byte line holding p (no register is written; L2 is the
// device's coherence point, so a later load still sees any write that lands
// in between).
__device__ __forceinline__ void prefetch_l2(const void* p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Prefetch the lines of three input rows of `bytes` each (q, k, v of a
// unit), one line per calling thread tid < 3 * lines.
__device__ __forceinline__ void prefetch_rows_l2(const void* q, const void* k, const void* v, int bytes, int tid)
{
    const int lines = (bytes + 127) / 128;
    if (tid < 3 * lines) {
        const int r = tid / lines, l = tid - r * lines;
        const char* base = static_cast<const char*>(r == 0 ? q : r == 1 ? k : v);
        prefetch_l2(base + 128 * l);
    }
}

// 2^x by the MUFU instruction (about 2 ulp; results below 2^-126 flush to
// 0, ex2(-inf) = 0)
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Let the next grid in the stream be scheduled; it still waits for this
// grid's completion in grid_dependency_wait before touching memory.
__device__ __forceinline__ void grid_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------ int8 rows
// A cache row x is stored as int8 codes with one fp32 scale: amax = max|x|,
// inv = 127 / amax (0 when amax = 0), code = rint(x * inv) within +-127
// (fp32 product, half to even), scale = amax / 127.  IEEE division and a
// separate product keep the codes identical on every correct fp32 path.
__device__ __forceinline__ float q8_inv(float amax) { return amax > 0.f ? __fdiv_rn(127.f, amax) : 0.f; }
__device__ __forceinline__ float q8_scale(float amax) { return __fdiv_rn(amax, 127.f); }

__device__ __forceinline__ uint32_t q8_code(float x, float inv)
{
    int c = __float2int_rn(__fmul_rn(x, inv));
    c = max(-127, min(127, c));
    return (uint32_t)c & 0xffu;
}

// Four fp32 values -> four int8 codes packed little-endian.
__device__ __forceinline__ uint32_t q8_pack4(const float* x, float inv)
{
    return q8_code(x[0], inv) | (q8_code(x[1], inv) << 8) | (q8_code(x[2], inv) << 16) | (q8_code(x[3], inv) << 24);
}

// Four int8 codes (little-endian in w) -> fp32, exactly: each biased byte
// becomes the low mantissa byte of 2^23, and the bias (2^23 + 128) is
// subtracted two values at a time.
__device__ __forceinline__ void q8_unpack4(uint32_t w, float* f)
{
    const uint32_t x = w ^ 0x80808080u;
    const float2 nb = make_float2(-8388736.f, -8388736.f);
    const float2 lo = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7540)),
                                             __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7541))), nb);
    const float2 hi = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7542)),
                                             __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7543))), nb);
    f[0] = lo.x; f[1] = lo.y; f[2] = hi.x; f[3] = hi.y;
}

// ------------------------------------------------------------ 4-bit rows
// A cache row x is stored as 4-bit codes with one fp32 scale: amax = max|x|,
// inv = 7 / amax (0 when amax = 0), code = rint(inv * x) within +-7 (fp32
// product, half to even), scale = amax / 7.  Two codes share a byte, element
// 2i in the low nibble, each nibble in offset binary (code + 8), so widening
// needs no sign handling.
__device__ __forceinline__ float q4_inv(float amax) { return amax > 0.f ? __fdiv_rn(7.f, amax) : 0.f; }
__device__ __forceinline__ float q4_scale(float amax) { return __fdiv_rn(amax, 7.f); }

__device__ __forceinline__ uint32_t q4_nibble(float x, float inv)
{
    int c = __float2int_rn(__fmul_rn(inv, x));
    c = max(-7, min(7, c));
    return (uint32_t)(c + 8);
}

// 2K fp32 values -> K bytes of packed codes, little-endian (K = 2 or 4).
template <int K>
__device__ __forceinline__ uint32_t q4_pack(const float* x, float inv)
{
    uint32_t w = 0u;
#pragma unroll
    for (int i = 0; i < 2 * K; ++i) w |= q4_nibble(x[i], inv) << (4 * i);
    return w;
}

// One 32-bit word of eight codes (elements 0..7) -> fp32, exactly, in the
// order 0, 2, 4, 6, 1, 3, 5, 7: the even elements' nibbles are masked into
// bytes, the odd ones' shifted down first; each byte becomes the low
// mantissa byte of 2^23 and the bias (2^23 + 8) is subtracted two values at
// a time.
__device__ __forceinline__ void q4_unpack8(uint32_t w, float* f)
{
    const uint32_t lo = w & 0x0F0F0F0Fu;
    const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;
    const float2 nb = make_float2(-8388616.f, -8388616.f);
    const float2 a = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7540)),
                                            __uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7541))), nb);
    const float2 b = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7542)),
                                            __uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7543))), nb);
    const float2 c = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7540)),
                                            __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7541))), nb);
    const float2 d = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7542)),
                                            __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7543))), nb);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

// The low 16 bits of w hold four codes (elements 0..3) -> fp32 in element
// order: (w | w << 12) & 0x0F0F0F0F puts elements 0, 2, 1, 3 in bytes 0..3.
__device__ __forceinline__ void q4_unpack4(uint32_t w, float* f)
{
    const uint32_t x = (w | (w << 12)) & 0x0F0F0F0Fu;
    const float2 nb = make_float2(-8388616.f, -8388616.f);
    const float2 a = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7540)),
                                            __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7542))), nb);
    const float2 b = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7541)),
                                            __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7543))), nb);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}

// The low 8 bits of w hold two codes (elements 0, 1) -> fp32.
__device__ __forceinline__ void q4_unpack2(uint32_t w, float* f)
{
    const uint32_t x = (w | (w << 12)) & 0x000F000Fu;
    const float2 a = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7540)),
                                            __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7542))),
                                make_float2(-8388616.f, -8388616.f));
    f[0] = a.x; f[1] = a.y;
}

// Named CTA barriers (ids 1..15; id 0 is __syncthreads).  Memory
// accesses made before the arrive are visible to the threads that pass the
// sync.  The id is an immediate in the instruction (a register id makes the
// compiler reserve all sixteen barriers).
template <int ID>
__device__ __forceinline__ void bar_sync_imm(int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"n"(ID), "r"(nthreads) : "memory");
}

template <int ID>
__device__ __forceinline__ void bar_arrive_imm(int nthreads)
{
    asm volatile("bar.arrive %0, %1;" ::"n"(ID), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void named_barrier_sync(int id, int nthreads)
{
    switch (id) {
    case 1: bar_sync_imm<1>(nthreads); break;
    case 2: bar_sync_imm<2>(nthreads); break;
    case 3: bar_sync_imm<3>(nthreads); break;
    case 4: bar_sync_imm<4>(nthreads); break;
    case 5: bar_sync_imm<5>(nthreads); break;
    case 6: bar_sync_imm<6>(nthreads); break;
    case 7: bar_sync_imm<7>(nthreads); break;
    case 8: bar_sync_imm<8>(nthreads); break;
    case 9: bar_sync_imm<9>(nthreads); break;
    case 10: bar_sync_imm<10>(nthreads); break;
    case 11: bar_sync_imm<11>(nthreads); break;
    case 12: bar_sync_imm<12>(nthreads); break;
    case 13: bar_sync_imm<13>(nthreads); break;
    case 14: bar_sync_imm<14>(nthreads); break;
    case 15: bar_sync_imm<15>(nthreads); break;
    default: break;
    }
}

__device__ __forceinline__ void named_barrier_arrive(int id, int nthreads)
{
    switch (id) {
    case 1: bar_arrive_imm<1>(nthreads); break;
    case 2: bar_arrive_imm<2>(nthreads); break;
    case 3: bar_arrive_imm<3>(nthreads); break;
    case 4: bar_arrive_imm<4>(nthreads); break;
    case 5: bar_arrive_imm<5>(nthreads); break;
    case 6: bar_arrive_imm<6>(nthreads); break;
    case 7: bar_arrive_imm<7>(nthreads); break;
    case 8: bar_arrive_imm<8>(nthreads); break;
    case 9: bar_arrive_imm<9>(nthreads); break;
    case 10: bar_arrive_imm<10>(nthreads); break;
    case 11: bar_arrive_imm<11>(nthreads); break;
    case 12: bar_arrive_imm<12>(nthreads); break;
    case 13: bar_arrive_imm<13>(nthreads); break;
    case 14: bar_arrive_imm<14>(nthreads); break;
    case 15: bar_arrive_imm<15>(nthreads); break;
    default: break;
    }
}

// Cheapest proxy fence that makes mbarrier initialisation visible to the
// bulk-copy engine of this CTA.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------- reductions

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace h2o
