// decode_common.cuh -- pieces shared by the decode kernels: tiles, row
// geometry, the shared-memory layout of a CTA, the row dot products (input
// type, int8 and 4-bit rows), the per-warp stage ring fed by 1-D bulk
// copies, the per-stage online softmax, and the warps' merge.  Everything
// sits in an unnamed namespace: each decode translation unit instantiates
// its own kernels.
#pragma once

#include <cfloat>
#include <climits>
#include <cstdlib>
#include <cstring>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace h2o {

namespace {

constexpr int kMaxSplit = 16;              // CTAs per cluster (non-portable above 8)
constexpr int kMaxChunk = 1024;            // slots per CTA
constexpr int kStage = 16;                 // slots per warp stage
constexpr unsigned kFull = 0xffffffffu;

// NW warps per CTA, each streaming 16-slot stages through a private ring of
// NBUF shared-memory buffers.
template <int NW_, int NBUF_>
struct Tile {
    static constexpr int NW = NW_, NT = 32 * NW_, NBUF = NBUF_;
    static constexpr int SPT = (kMaxChunk + NT - 1) / NT; // slots per thread in the score pass (SPT * NT >= kMaxChunk)
    static_assert(SPT * NT >= kMaxChunk, "the score pass covers every slot of a chunk");
    static constexpr int MINB = NT <= 192 ? 2 : 1;        // CTAs per SM the registers must allow
};

// Row geometry.  For the logits a stage's 16 rows are split between the two
// half-warps: lane (r = lane & 15, h = lane >> 4) computes the dot of row r's
// half h with the matching half of q.  Rows are read as 16-byte chunks in
// the order c ^ (r & XM): eight consecutive lanes then touch eight distinct
// chunk positions, so the row-major stage is read without bank conflicts;
// each lane holds its half of q already permuted into that order.
template <typename T, int D>
struct Rows {
    static constexpr int VE = 16 / (int)sizeof(T);        // elements per 16-byte chunk
    static constexpr int HALF = D / 2;                    // elements per half row
    static constexpr int HCH = HALF / VE;                 // chunks per half row
    static constexpr int XM = HCH >= 8 ? 7 : HCH - 1;     // chunk rotation mask
    static constexpr int EPL = D / 32;                    // value elements per lane
};

template <int D>
struct Exchange {                 // every CTA has one; rank 0's is the meeting point
    float m[kMaxSplit];           // per-CTA running max (base 2)
    float l[kMaxSplit];           // per-CTA normaliser at that max
    unsigned am[2][3][kMaxSplit]; // per-CTA arg-min keys (hi, lo, slot): [0] candidates, [1] every live slot
    float o[kMaxSplit][D];        // per-CTA unnormalised output
};

// Form of a cache row, QB: 0 = the input type, 8 = int8 codes, 4 = 4-bit
// codes (two per byte, offset binary).  CacheElem is the element a row is
// addressed in and RowElems<D, QB> the elements of one row.
template <typename T, int QB>
using CacheElem = typename std::conditional<QB == 8, int8_t,
                  typename std::conditional<QB == 4, uint8_t, T>::type>::type;

template <int D, int QB>
constexpr int RowElems = QB == 4 ? D / 2 : D;

template <typename T, int D, class TL, int QB>
struct Ring {
    CacheElem<T, QB> kbuf[TL::NW][TL::NBUF][kStage * RowElems<D, QB>];   // per-warp ring of K rows
    CacheElem<T, QB> vbuf[TL::NW][TL::NBUF][kStage * RowElems<D, QB>];   // per-warp ring of V rows
};

template <int D, class TL>
struct Epilogue {
    float wo[TL::NW][D];
};

template <typename T, int D, class TL, int QB>
struct DecodeSmem {
    // the epilogue buffers reuse the ring once every copy has landed and
    // been consumed (after the barrier that opens merge_warps)
    union {
        Ring<T, D, TL, QB> ring;
        Epilogue<D, TL> epi;
    } u;
    // the cluster exchange lies outside the ring, so other CTAs may write
    // into it while this one still streams
    Exchange<D> x;
    // this step's q, k, v rows, fetched in one round trip after the wait
    alignas(16) unsigned char in[3][D * sizeof(T)];
    // quantised rows: {K scale, V scale} of every slot of a ring stage
    alignas(16) float2 sbuf[QB ? TL::NW : 1][TL::NBUF][kStage];
    // quantised rows: each warp's byte planes of q (built per warp)
    alignas(16) unsigned char qpl[QB ? TL::NW : 1][QB ? 3 * D : 16];
    uint64_t bar[TL::NW][TL::NBUF];
    float z[kMaxChunk];                     // base-2 logits of this CTA's slots
    alignas(16) float e[TL::NW][kStage];
    float wm[TL::NW];
    float wl[TL::NW];
    float qf[D];
    float kf[D];
    unsigned am[2][3][TL::NW];              // per-warp arg-min keys
    unsigned ru[2][TL::NW];                  // per-warp HashEvict arg-max keys
    float M, invL, z_new, P_new;
    int victim;
    unsigned code_q, code_k;
    float hacc[2][32];                      // HashEvict projection partial sums
};

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c)
{
    return __ffma2_rn(a, b, c);
}

__device__ __forceinline__ float safe_exp2_diff(float a, float m)
{
    return (a == -INFINITY) ? 0.f : ex2_approx(a - m);
}

// Lexicographic arg-min over (score hi, score lo, slot), each an unsigned
// key; all-ones means "no slot".
struct ArgMin {
    unsigned hi, lo, slot;
};

__device__ __forceinline__ ArgMin argmin_none() { return ArgMin{0xffffffffu, 0xffffffffu, 0xffffffffu}; }

__device__ __forceinline__ void argmin_take(ArgMin& a, const ArgMin& b)
{
    if (b.hi < a.hi || (b.hi == a.hi && (b.lo < a.lo || (b.lo == a.lo && b.slot < a.slot)))) a = b;
}

__device__ __forceinline__ ArgMin warp_argmin(const ArgMin& a)
{
    const unsigned mh = __reduce_min_sync(kFull, a.hi);
    const unsigned ml = __reduce_min_sync(kFull, a.hi == mh ? a.lo : 0xffffffffu);
    const unsigned ms = __reduce_min_sync(kFull, (a.hi == mh && a.lo == ml) ? a.slot : 0xffffffffu);
    return ArgMin{mh, ml, ms};
}

// This lane's half of q as raw 16-byte chunks in its rotated chunk order.
// Loading and widening are separate so that nothing consumes the load
// before the ring's bulk copies are issued.
template <typename T, int D>
struct QRaw {
    uint4 w[Rows<T, D>::HCH];
};

template <typename T, int D>
__device__ __forceinline__ void load_q_raw(const T* q, int lane, QRaw<T, D>& raw)
{
    using R = Rows<T, D>;
    const int r = lane & 15, h = lane >> 4;
#pragma unroll
    for (int c = 0; c < R::HCH; ++c)
        raw.w[c] = *reinterpret_cast<const uint4*>(q + h * R::HALF + (c ^ (r & R::XM)) * R::VE);
}

// This step's q, k and v rows as 16-byte vectors: thread tid < 3 * NV loads
// vector tid % NV of row tid / NV (q, k, v); the others return zeros.
template <typename T, int D>
__device__ __forceinline__ uint4 load_rows_16b(const T* q, const T* k, const T* v, int tid)
{
    constexpr int NV = D * (int)sizeof(T) / 16;
    if (tid >= 3 * NV) return make_uint4(0u, 0u, 0u, 0u);
    const int r = tid / NV;
    const T* row = r == 0 ? q : r == 1 ? k : v;
    return reinterpret_cast<const uint4*>(row)[tid - r * NV];
}

template <typename T, int D>
__device__ __forceinline__ void store_rows_16b(unsigned char (*in)[D * sizeof(T)], uint4 w, int tid)
{
    constexpr int NV = D * (int)sizeof(T) / 16;
    if (tid < 3 * NV) reinterpret_cast<uint4*>(in[tid / NV])[tid % NV] = w;
}

// Widen the raw chunks to fp32 and scale them to base-2 logits.
template <typename T, int D>
__device__ __forceinline__ void widen_q(const QRaw<T, D>& raw, float scale, float (&qp)[D / 2])
{
    using R = Rows<T, D>;
#pragma unroll
    for (int c = 0; c < R::HCH; ++c) {
        const uint32_t u[4] = {raw.w[c].x, raw.w[c].y, raw.w[c].z, raw.w[c].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if constexpr (sizeof(T) == 2) {
                qp[c * R::VE + 2 * k] = __uint_as_float(u[k] << 16) * scale;
                qp[c * R::VE + 2 * k + 1] = __uint_as_float(u[k] & 0xffff0000u) * scale;
            } else {
                qp[c * R::VE + k] = __uint_as_float(u[k]) * scale;
            }
        }
    }
}

// Half-row dot product of row `row` (global or shared, elements of type T)
// with the rotated q half; every lane returns the full dot of its
// row after one exchange between the half-warps.
// Raw 32-bit words of a vector of E elements of T, and their fp32 values.
template <int BYTES> struct RawT;
template <> struct RawT<4> { using type = uint32_t; };
template <> struct RawT<8> { using type = uint2; };
template <> struct RawT<16> { using type = uint4; };

__device__ __forceinline__ void raw_words(uint32_t w, uint32_t* u) { u[0] = w; }
__device__ __forceinline__ void raw_words(uint2 w, uint32_t* u) { u[0] = w.x; u[1] = w.y; }
__device__ __forceinline__ void raw_words(uint4 w, uint32_t* u) { u[0] = w.x; u[1] = w.y; u[2] = w.z; u[3] = w.w; }

template <typename T, int E>
__device__ __forceinline__ void widen_raw(const typename RawT<E * sizeof(T)>::type& w, float* out)
{
    constexpr int NWD = E * (int)sizeof(T) / 4;
    uint32_t u[NWD];
    raw_words(w, u);
#pragma unroll
    for (int k = 0; k < NWD; ++k) {
        if constexpr (sizeof(T) == 2) {
            out[2 * k] = __uint_as_float(u[k] << 16);
            out[2 * k + 1] = __uint_as_float(u[k] & 0xffff0000u);
        } else {
            out[k] = __uint_as_float(u[k]);
        }
    }
}

// Pairwise sum of the per-chunk partial sums s[0..N) over the chunk index:
// level w adds s[c + w] into s[c] for c a multiple of 2w.  A lane that read
// its chunks in the order c ^ m (m < N) holds, at every node of this tree,
// the sum of the same data chunks as a lane with any other m (the XOR maps
// aligned blocks onto aligned blocks), and fp32 addition is commutative, so
// every lane -- every slot of a stage -- gets the same bits for the same
// row: equal keys give equal logits wherever they sit.
template <int N>
__device__ __forceinline__ float chunk_tree(float (&s)[N])
{
    static_assert((N & (N - 1)) == 0, "power-of-two chunk count");
#pragma unroll
    for (int w = 1; w < N; w <<= 1) {
#pragma unroll
        for (int c = 0; c < N; c += 2 * w) s[c] = s[c] + s[c + w];
    }
    return s[0];
}

// Half-row dot product of row `row` (global or shared, elements of type T)
// with the rotated q half; every lane returns the full dot of its row after
// one exchange between the half-warps.  All chunks are loaded before the
// first multiply; each chunk's products are summed in element order, and
// the chunks by chunk_tree, so the result does not depend on the slot's
// place in its stage.
template <typename T, int D, typename E>
__device__ __forceinline__ float row_dot(const E* row, const float (&qp)[D / 2], int lane)
{
    using R = Rows<T, D>;
    const int r = lane & 15, h = lane >> 4;
    const E* half = row + h * R::HALF;
    static_assert(sizeof(E) == sizeof(T), "rows hold the input type");
    float part[R::HCH];
    {
        uint4 raw[R::HCH];
#pragma unroll
        for (int c = 0; c < R::HCH; ++c)
            raw[c] = *reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(half) + (c ^ (r & R::XM)) * R::VE);
#pragma unroll
        for (int c = 0; c < R::HCH; ++c) {
            float kf[R::VE];
            widen_raw<T, R::VE>(raw[c], kf);
            float2 t = fma2(make_float2(qp[c * R::VE], qp[c * R::VE + 1]), make_float2(kf[0], kf[1]),
                            make_float2(0.f, 0.f));
#pragma unroll
            for (int e = 2; e < R::VE; e += 2)
                t = fma2(make_float2(qp[c * R::VE + e], qp[c * R::VE + e + 1]), make_float2(kf[e], kf[e + 1]), t);
            part[c] = t.x + t.y;
        }
    }
    const float zh = chunk_tree<R::HCH>(part);
    return zh + __shfl_xor_sync(kFull, zh, 16);
}

// int8 rows (QB): a row of D codes is D / 16 chunks of 16.  Lane (r, h)
// takes half hh = h ^ ((r / HCH) & 1) of row r -- the halves swap every HCH
// rows -- and at step c reads chunk HCH * hh + (c ^ (r % HCH)), so the 8
// lanes of one 16-byte shared-memory phase hit 8 different bank groups
// although every 128-byte row starts in the same one.  q is held in the
// same order, scaled to base-2 logits.
template <int D>
__device__ __forceinline__ int q8_chunk(int lane, int c)
{
    constexpr int HCH = D / 32;
    const int r = lane & 15, h = lane >> 4;
    const int hh = h ^ ((r / HCH) & 1);
    return HCH * hh + (c ^ (r % HCH));
}

// The new token's row, held as 16 bytes of T by threads tid < 2 * NV (K rows
// first, then V), stored quantised into slot `victim`: the NV threads of a
// row form an aligned lane group, which reduces the row's max magnitude.
// Every lane of the calling warps must take part (shuffles).
template <typename T, int D>
__device__ __forceinline__ void store_row_q8(uint4 newrow, int tid, int8_t* Kc8, int8_t* Vc8, float2* slot_scales,
                                             int victim)
{
    constexpr int NV = D * (int)sizeof(T) / 16, VE = 16 / (int)sizeof(T);
    static_assert(NV <= 32, "a row's threads must fit one warp");
    float x[VE];
    const uint32_t u[4] = {newrow.x, newrow.y, newrow.z, newrow.w};
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
    const float inv = q8_inv(amax);
    if (tid < 2 * NV) {
        const bool isv = tid >= NV;
        const int v = isv ? tid - NV : tid;
        int8_t* dst = (isv ? Vc8 : Kc8) + (size_t)victim * D + v * VE;
        if constexpr (VE == 8)
            *reinterpret_cast<uint2*>(dst) = make_uint2(q8_pack4(&x[0], inv), q8_pack4(&x[4], inv));
        else
            *reinterpret_cast<uint32_t*>(dst) = q8_pack4(&x[0], inv);
        if (v == 0) reinterpret_cast<float*>(slot_scales + victim)[isv ? 1 : 0] = q8_scale(amax);
    }
}

// 4-bit rows (QB 4): a row of D codes is D / 2 bytes, D / 32 chunks of 16
// bytes (32 codes each), HC = D / 64 per half.  Lane (r, h) takes half
// hh = h ^ ((r >> S) & 1) of row r and at step c reads chunk
// HC * hh + (c ^ ((r >> (S + 1)) & (HC - 1))), S = log2(4 / HC): the rows'
// own offsets separate r mod 4 / HC, the half and chunk swaps the rest, so
// the 8 lanes of one 16-byte shared-memory phase hit 8 different bank
// groups.  q is held per 32-bit code word in the order q4_unpack8 widens
// (elements 0, 2, 4, 6, 1, 3, 5, 7), scaled to base-2 logits.
template <int D>
__device__ __forceinline__ int q4_chunk(int lane, int c)
{
    constexpr int HC = D / 64, SH = HC == 2 ? 1 : 2;
    static_assert(HC == 1 || HC == 2, "head_dim 64 or 128");
    const int r = lane & 15, h = lane >> 4;
    const int hh = h ^ ((r >> SH) & 1);
    return HC * hh + (c ^ ((r >> (SH + 1)) & (HC - 1)));
}

// As store_row_q8, for 4-bit rows: each thread's 16 bytes of T become
// VE / 2 bytes of codes.
template <typename T, int D>
__device__ __forceinline__ void store_row_q4(uint4 newrow, int tid, uint8_t* Kc4, uint8_t* Vc4, float2* slot_scales,
                                             int victim)
{
    constexpr int NV = D * (int)sizeof(T) / 16, VE = 16 / (int)sizeof(T);
    static_assert(NV <= 32, "a row's threads must fit one warp");
    float x[VE];
    const uint32_t u[4] = {newrow.x, newrow.y, newrow.z, newrow.w};
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
    const float inv = q4_inv(amax);
    if (tid < 2 * NV) {
        const bool isv = tid >= NV;
        const int v = isv ? tid - NV : tid;
        uint8_t* dst = (isv ? Vc4 : Kc4) + (size_t)victim * (D / 2) + v * (VE / 2);
        if constexpr (VE == 8) *reinterpret_cast<uint32_t*>(dst) = q4_pack<4>(x, inv);
        else *reinterpret_cast<uint16_t*>(dst) = (uint16_t)q4_pack<2>(x, inv);
        if (v == 0) reinterpret_cast<float*>(slot_scales + victim)[isv ? 1 : 0] = q4_scale(amax);
    }
}

// ------------------------------------------------ q against quantised rows
//
// The logit of a quantised row is an integer dot product: the codes against
// q held as fixed point.  x = q * scale (base-2 logit units, fp32) is
// rounded to xi = rint(x * 2^F), F chosen per row so that |xi| < 2^23, and
// xi is split into three byte planes, xi = 2^16 b2 + 2^8 b1 + b0 (b2 signed,
// b1 and b0 unsigned).  dp4a sums four code x byte products exactly in
// 32-bit integers, so a row's dot is (2^16 A2 + 2^8 A1 + A0) * 2^-F with
// A_k = sum_e code_e * b_k,e exact whatever order the lanes take: equal
// rows give equal bits in every slot.  The rounding of x to the 2^-F grid
// is at most 2^-23 of the row's largest |x|, the size of an fp32 rounding.
// Lane (r, h) holds its half row in the order of its chunk reads.
template <typename T, int D, int QB>
struct QVec {                     // q for rows of the input type
    float v[D / 2];
};

template <typename T, int D>
struct QFix {
    uint32_t p[3][D / 8];         // byte planes b0, b1, b2 of the lane's D / 2 elements, 4 per word
    int s[3];                     // 4-bit rows: the lane's sum of every plane (for the code offset)
    float unscale;                // 2^-F
};
template <typename T, int D> struct QVec<T, D, 8> : QFix<T, D> {};
template <typename T, int D> struct QVec<T, D, 4> : QFix<T, D> {};

__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Building the planes: the warp's lanes take EPL = D / 32 consecutive
// elements each, round them (one multiply-add onto 1.5 * 2^23 rounds to the
// nearest integer, ties to even, for |x 2^F| < 2^22), and write their plane
// bytes to a 3 x D shared buffer -- int8 rows in element order, 4-bit rows
// with every group of 8 elements stored even elements first -- from which
// every lane reads the words of its chunks.  A plane's sum over each half
// row (for the offset of 4-bit codes) is reduced over the 16 lanes holding
// that half.  pl: this warp's 3 * D bytes, 16-byte aligned.
template <int QB, int D>
__device__ __forceinline__ int qfix_pos(int e)
{
    if constexpr (QB == 8) return e;
    else return (e & ~7) + (e & 1) * 4 + ((e & 7) >> 1);
}

template <int QB, typename T, int D>
__device__ __forceinline__ void load_q_fix(const T* q, float scale, int lane, unsigned char* pl, QFix<T, D>& qf)
{
    constexpr int EPL = D / 32, NWD = D / 8;
    float x[EPL];
    load_vec<T, EPL>(q + lane * EPL, x);
    float m = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        x[e] *= scale;
        m = fmaxf(m, fabsf(x[e]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    // m < 2^E, read from the exponent field (frexpf for the rare subnormal m)
    int E = 0;
    if (m >= FLT_MIN) E = (int)((__float_as_uint(m) >> 23) & 0xffu) - 126;
    else if (m > 0.f) frexpf(m, &E);
    const int F = 22 - E;                            // |x| 2^F < 2^22
    // 2^F and 2^-F, built from their exponent fields while they are normal
    const float up = (F >= -126 && F <= 127) ? __uint_as_float((uint32_t)(F + 127) << 23) : ldexpf(1.f, F);
    qf.unscale = m > 0.f ? ((F >= -127 && F <= 126) ? __uint_as_float((uint32_t)(127 - F) << 23) : ldexpf(1.f, -F))
                         : 1.f;
    int ps[3] = {0, 0, 0};
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        const int xi = m > 0.f ? __float_as_int(__fmaf_rn(x[e], up, 12582912.f)) - 0x4B400000 : 0;
        const int pos = qfix_pos<QB, D>(lane * EPL + e);
        pl[pos] = (unsigned char)(xi & 0xff);
        pl[D + pos] = (unsigned char)((xi >> 8) & 0xff);
        pl[2 * D + pos] = (unsigned char)((xi >> 16) & 0xff);
        ps[0] += xi & 0xff;
        ps[1] += (xi >> 8) & 0xff;
        ps[2] += xi >> 16;
    }
    __syncwarp();
    // the half of the row this lane reads: the half its first chunk lies in
    int hh;
    if constexpr (QB == 8) hh = q8_chunk<D>(lane, 0) >= D / 32;
    else hh = q4_chunk<D>(lane, 0) >= D / 64;
    if constexpr (QB == 4) {
        // lanes 0..15 hold elements of the first half, 16..31 of the second
#pragma unroll
        for (int k = 0; k < 3; ++k) {
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) ps[k] += __shfl_xor_sync(kFull, ps[k], o);
            const int s0 = __shfl_sync(kFull, ps[k], 0), s1 = __shfl_sync(kFull, ps[k], 16);
            qf.s[k] = hh ? s1 : s0;
        }
    } else {
        qf.s[0] = qf.s[1] = qf.s[2] = 0;
    }
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const unsigned char* plane = pl + k * D;
        if constexpr (QB == 8) {
#pragma unroll
            for (int c = 0; c < NWD / 4; ++c) {
                const uint4 w = *reinterpret_cast<const uint4*>(plane + q8_chunk<D>(lane, c) * 16);
                qf.p[k][4 * c] = w.x; qf.p[k][4 * c + 1] = w.y; qf.p[k][4 * c + 2] = w.z; qf.p[k][4 * c + 3] = w.w;
            }
        } else {
            // chunk c: 32 elements = 4 groups of 8 = 32 plane bytes
#pragma unroll
            for (int c = 0; c < NWD / 8; ++c) {
                const unsigned char* src = plane + q4_chunk<D>(lane, c) * 32;
                const uint4 w0 = *reinterpret_cast<const uint4*>(src);
                const uint4 w1 = *reinterpret_cast<const uint4*>(src + 16);
                uint32_t* dst = &qf.p[k][8 * c];
                dst[0] = w0.x; dst[1] = w0.y; dst[2] = w0.z; dst[3] = w0.w;
                dst[4] = w1.x; dst[5] = w1.y; dst[6] = w1.z; dst[7] = w1.w;
            }
        }
    }
    __syncwarp();                                    // pl may be written again
}

template <int QB, typename T, int D>
__device__ __forceinline__ void load_qvec(const T* q, float scale, int lane, unsigned char* pl, QVec<T, D, QB>& qv)
{
    if constexpr (QB == 0) {
        QRaw<T, D> raw;
        load_q_raw<T, D>(q, lane, raw);
        widen_q<T, D>(raw, scale, qv.v);
    } else {
        load_q_fix<QB, T, D>(q, scale, lane, pl, qv);
    }
}

// Dot (unscaled by the row's scale) of a quantised row with q; every lane
// returns the full dot of its row.
template <int QB, int D, typename T>
__device__ __forceinline__ float row_dot_fix(const CacheElem<T, QB>* row, const QFix<T, D>& qf, int lane)
{
    int a0 = 0, a1 = 0, a2 = 0;
    if constexpr (QB == 8) {
        constexpr int HCH = D / 32;
        uint4 raw[HCH];
#pragma unroll
        for (int c = 0; c < HCH; ++c)
            raw[c] = *reinterpret_cast<const uint4*>(reinterpret_cast<const int8_t*>(row) + q8_chunk<D>(lane, c) * 16);
#pragma unroll
        for (int c = 0; c < HCH; ++c) {
            const uint32_t u[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = 4 * c + i;
                a0 = dp4a_su(u[i], qf.p[0][j], a0);
                a1 = dp4a_su(u[i], qf.p[1][j], a1);
                a2 = dp4a_ss(u[i], qf.p[2][j], a2);
            }
        }
    } else {
        // offset-binary nibbles: sum (code + 8) b, then take 8 sum b off
        constexpr int HC = D / 64;
        uint4 raw[HC];
#pragma unroll
        for (int c = 0; c < HC; ++c)
            raw[c] = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(row) + q4_chunk<D>(lane, c) * 16);
#pragma unroll
        for (int c = 0; c < HC; ++c) {
            const uint32_t u[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = 2 * (4 * c + i);
                const uint32_t lo = u[i] & 0x0F0F0F0Fu, hi = (u[i] >> 4) & 0x0F0F0F0Fu;
                a0 = dp4a_uu(lo, qf.p[0][j], a0);
                a0 = dp4a_uu(hi, qf.p[0][j + 1], a0);
                a1 = dp4a_uu(lo, qf.p[1][j], a1);
                a1 = dp4a_uu(hi, qf.p[1][j + 1], a1);
                a2 = dp4a_us(lo, qf.p[2][j], a2);
                a2 = dp4a_us(hi, qf.p[2][j + 1], a2);
            }
        }
        a0 -= 8 * qf.s[0];
        a1 -= 8 * qf.s[1];
        a2 -= 8 * qf.s[2];
    }
    a0 += __shfl_xor_sync(kFull, a0, 16);
    a1 += __shfl_xor_sync(kFull, a1, 16);
    a2 += __shfl_xor_sync(kFull, a2, 16);
    return __fmaf_rn((float)a2, 65536.f, __fmaf_rn((float)a1, 256.f, (float)a0)) * qf.unscale;
}

// Dot of q and k (rows of T in shared memory) times scale, in fp32: the new
// token's logit on the quantised paths (any lane order; every lane gets it).
template <typename T, int D>
__device__ __forceinline__ float new_token_dot(const T* q, const T* k, float scale, int lane)
{
    constexpr int EPL = D / 32;
    float qv[EPL], kv[EPL];
    load_vec<T, EPL>(q + lane * EPL, qv);
    load_vec<T, EPL>(k + lane * EPL, kv);
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc = __fmaf_rn(qv[e], kv[e], acc);
    return warp_sum(acc) * scale;
}

// Logit (before the row's scale) of row `row` against q: the float path for
// rows of the input type, the integer path for codes.
template <int QB, typename T, int D>
__device__ __forceinline__ float row_logit(const CacheElem<T, QB>* row, const QVec<T, D, QB>& qv, int lane)
{
    if constexpr (QB == 0) return row_dot<T, D, T>(row, qv.v, lane);
    else return row_dot_fix<QB, D, T>(row, qv, lane);
}

// The new token's logit: row_dot for rows of the input type (the same
// arithmetic as a cached row), new_token_dot otherwise.
template <int QB, typename T, int D>
__device__ __forceinline__ float new_logit(const T* q, const T* k, float scale, const QVec<T, D, QB>& qv, int lane)
{
    if constexpr (QB == 0) return row_dot<T, D, T>(k, qv.v, lane);
    else return new_token_dot<T, D>(q, k, scale, lane);
}

template <int QB, typename T, int D, typename E>
__device__ __forceinline__ void store_row_quant(uint4 newrow, int tid, E* Kc, E* Vc, float2* slot_scales, int victim)
{
    if constexpr (QB == 8) store_row_q8<T, D>(newrow, tid, Kc, Vc, slot_scales, victim);
    else store_row_q4<T, D>(newrow, tid, Kc, Vc, slot_scales, victim);
}

// Bulk copies of one stage (slots s .. min(s + 16, f1) - 1) into this warp's
// ring buffer b: K and V rows and, for int8 rows, the slots' scale pairs
// (an even count, so the copy stays a multiple of 16 bytes; the scale rows
// are padded to an even length).
template <typename T, int D, class TL, int QB>
__device__ __forceinline__ void issue_stage(DecodeSmem<T, D, TL, QB>& S, const CacheElem<T, QB>* Kc,
                                            const CacheElem<T, QB>* Vc, const float2* Sc, int s, int f1, int b)
{
    const int warp = threadIdx.x >> 5;
    const int rows = min(kStage, f1 - s);
    constexpr int RE = RowElems<D, QB>;
    const uint32_t bytes = (uint32_t)(rows * RE * sizeof(CacheElem<T, QB>));
    const uint32_t sbytes = QB ? (uint32_t)(((rows + 1) & ~1) * sizeof(float2)) : 0u;
    mbar_arrive_expect_tx(&S.bar[warp][b], 2 * bytes + sbytes);
    bulk_g2s(S.u.ring.kbuf[warp][b], Kc + (size_t)s * RE, bytes, &S.bar[warp][b]);
    bulk_g2s(S.u.ring.vbuf[warp][b], Vc + (size_t)s * RE, bytes, &S.bar[warp][b]);
    if constexpr (QB != 0) bulk_g2s(S.sbuf[warp][b], Sc + s, sbytes, &S.bar[warp][b]);
}

// One 16-slot stage held in shared memory at kst / vst (with its slots'
// scale pairs at sc for quantised rows): logits of its gl live rows (row
// skip_r left out), the online softmax update and the weighted V rows;
// e_buf is the warp's 16-float weight buffer.  When zdst is given, row r's
// logit goes to zdst[r].  The warp keeps one reference max m_ref
// and rescales only when a logit exceeds it by more than 8 (weights stay
// below 2^8), so most stages need no cross-lane max.  l_lane is this lane's
// share of the normaliser (lanes 0..15 count their slot once); o holds the
// lane's EPL output columns lane*EPL.. of the unnormalised sum (even rows of
// every stage), o2 the odd rows' share (which halves the dependent
// multiply-add chain of a stage), both relative to m_ref.
template <typename T, int D, int QB>
__device__ __forceinline__ void attend_rows(const CacheElem<T, QB>* kst, const CacheElem<T, QB>* vst,
                                            const float2* sc, float* e_buf, float* zdst, int gl, int skip_r,
                                            const QVec<T, D, QB>& qv, float& m_ref, float& l_lane,
                                            float (&o)[D / 32], float (&o2)[D / 32])
{
    using R = Rows<T, D>;
    constexpr int EPL = R::EPL;
    const int lane = threadIdx.x & 31;
    const int r = lane & 15, h = lane >> 4;
    auto vfma = [&](float p, const float* vr, bool odd) {
        const float2 pj = make_float2(p, p);
#pragma unroll
        for (int e = 0; e < EPL; e += 2) {
            float* acc = odd ? o2 : o;
            const float2 rr = fma2(pj, make_float2(vr[e], vr[e + 1]), make_float2(acc[e], acc[e + 1]));
            acc[e] = rr.x;
            acc[e + 1] = rr.y;
        }
    };
    float z;
    if constexpr (QB != 0) z = row_logit<QB, T, D>(kst + r * RowElems<D, QB>, qv, lane) * sc[r].x;
    else z = row_logit<QB, T, D>(kst + r * D, qv, lane);
    if (r >= gl || r == skip_r) z = -INFINITY;
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
    if (h == 0) {
        l_lane += er;
        // quantised values: the slot's V scale is folded into its weight
        if constexpr (QB != 0) e_buf[r] = er * sc[r].y;
        else e_buf[r] = er;
        if (zdst && r < gl) zdst[r] = z;
    }
    __syncwarp();
    float ev[kStage];
#pragma unroll
    for (int j = 0; j < kStage; j += 4) {
        const float4 e4 = *reinterpret_cast<const float4*>(&e_buf[j]);
        ev[j] = e4.x; ev[j + 1] = e4.y; ev[j + 2] = e4.z; ev[j + 3] = e4.w;
    }
    if constexpr (QB != 0) {
        // quantised values (weights already carry the V scales); a full
        // stage loads each half's code words before the first widening, as
        // the bf16 path does
        constexpr int RE = RowElems<D, QB>;
        auto v_word = [&](int j) -> uint32_t {
            if constexpr (QB == 8 && EPL == 4) return *reinterpret_cast<const uint32_t*>(vst + j * RE + lane * EPL);
            else if constexpr (QB == 8) return (uint32_t)*reinterpret_cast<const uint16_t*>(vst + j * RE + lane * EPL);
            else if constexpr (EPL == 4) return (uint32_t)*reinterpret_cast<const uint16_t*>(vst + j * RE + lane * 2);
            else return (uint32_t)vst[j * RE + lane];
        };
        auto v_acc = [&](uint32_t w, float p, bool odd) {
            float vr[4];
            if constexpr (QB == 8) q8_unpack4(w, vr);
            else if constexpr (EPL == 4) q4_unpack4(w, vr);
            else q4_unpack2(w, vr);
            vfma(p, vr, odd);
        };
        if (gl == kStage) {
#pragma unroll
            for (int j0 = 0; j0 < kStage; j0 += kStage / 2) {
                uint32_t vw[kStage / 2];
#pragma unroll
                for (int j = 0; j < kStage / 2; ++j) vw[j] = v_word(j0 + j);
#pragma unroll
                for (int j = 0; j < kStage / 2; ++j) v_acc(vw[j], ev[j0 + j], j & 1);
            }
        } else {
#pragma unroll
            for (int j = 0; j < kStage; ++j)
                if (j < gl) v_acc(v_word(j), ev[j], j & 1);
        }
    } else {
        using RV = typename RawT<EPL * sizeof(T)>::type;
        if (gl == kStage) {
            // a full stage: each half's value fragments are loaded before the
            // first multiply (rows past gl of a partial stage may hold stale
            // data and are never read)
#pragma unroll
            for (int j0 = 0; j0 < kStage; j0 += kStage / 2) {
                RV vraw[kStage / 2];
#pragma unroll
                for (int j = 0; j < kStage / 2; ++j)
                    vraw[j] = *reinterpret_cast<const RV*>(vst + (j0 + j) * D + lane * EPL);
#pragma unroll
                for (int j = 0; j < kStage / 2; ++j) {
                    float vr[EPL];
                    widen_raw<T, EPL>(vraw[j], vr);
                    vfma(ev[j0 + j], vr, j & 1);
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < kStage; ++j) {
                if (j < gl) {
                    float vr[EPL];
                    load_vec<T, EPL>(vst + j * D + lane * EPL, vr);
                    vfma(ev[j], vr, j & 1);
                }
            }
        }
    }
    __syncwarp();
}

// attend_rows on stage buffer b of this warp's ring in S (slot offset s0
// within the fetched range starting at f0; `skip` is an absolute slot; when
// keep_z the logits go to S.z[s0 + r]).
template <typename T, int D, class TL, int QB>
__device__ __forceinline__ void attend_stage(DecodeSmem<T, D, TL, QB>& S, int b, int s0, int gl, int f0, int skip,
                                             bool keep_z, const QVec<T, D, QB>& qv, float& m_ref, float& l_lane,
                                             float (&o)[D / 32], float (&o2)[D / 32])
{
    const int warp = threadIdx.x >> 5;
    const int sr = skip - f0 - s0;
    attend_rows<T, D, QB>(S.u.ring.kbuf[warp][b], S.u.ring.vbuf[warp][b], QB ? S.sbuf[warp][b] : nullptr, S.e[warp],
                          keep_z ? &S.z[s0] : nullptr, gl, (sr >= 0 && sr < kStage) ? sr : -1, qv, m_ref, l_lane,
                          o, o2);
}

// Per-warp streaming softmax over the rows this CTA fetched, [f0, f1); only
// slots < n are live and `skip` (absolute slot) is left out.  When keep_z,
// logits go to S.z[slot - f0].  Stage g of the range goes to warp g % NW,
// buffer (g / NW) % NBUF; after a stage the warp refills its buffer with its
// stage NBUF rounds ahead.
template <typename T, int D, class TL, int QB>
__device__ __forceinline__ void attend_chunk(DecodeSmem<T, D, TL, QB>& S, const CacheElem<T, QB>* Kc,
                                             const CacheElem<T, QB>* Vc, const float2* Sc,
                                             int f0, int f1, int n, int skip, bool keep_z,
                                             const QVec<T, D, QB>& qv, float& m_ref,
                                             float& l_lane, float (&o)[D / 32], int* err)
{
    constexpr int EPL = D / 32, NW = TL::NW, NBUF = TL::NBUF;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nst = (f1 - f0 + kStage - 1) / kStage;
    bool timed_out = false;
    float o2[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) o2[e] = 0.f;
    int it = 0;
    for (int g = warp; g < nst; g += NW, ++it) {
        const int b = it % NBUF;
        const uint32_t parity = (uint32_t)(it / NBUF) & 1u;
        if (!mbar_wait(&S.bar[warp][b], parity)) {
            if (!timed_out && lane == 0) atomicOr(err, kErrWaitTimeout);
            timed_out = true;
        }
        const int s0 = g * kStage;                 // fetch-relative first slot
        const int gl = max(0, min(kStage, n - (f0 + s0)));   // live rows of this stage
        if (gl > 0) attend_stage<T, D, TL, QB>(S, b, s0, gl, f0, skip, keep_z, qv, m_ref, l_lane, o, o2);
        __syncwarp();                              // every lane is past the wait and the buffer
        // refill this buffer with the warp's stage NBUF rounds ahead
        if (lane == 0) {
            const int gn = g + NW * NBUF;
            if (gn < nst) issue_stage<T, D, TL, QB>(S, Kc, Vc, Sc, f0 + gn * kStage, f1, b);
        }
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] += o2[e];
}

// Kick off ring buffers [b_lo, b_hi) of each warp -- by default all NBUF --
// with their first stages (called by lane 0 of every warp after its barriers
// are initialised).
template <typename T, int D, class TL, int QB>
__device__ __forceinline__ void prime_ring(DecodeSmem<T, D, TL, QB>& S, const CacheElem<T, QB>* Kc,
                                           const CacheElem<T, QB>* Vc, const float2* Sc,
                                           int c0, int c1, int b_lo = 0, int b_hi = TL::NBUF)
{
    const int warp = threadIdx.x >> 5;
    const int nst = (c1 - c0 + kStage - 1) / kStage;
#pragma unroll
    for (int b = 0; b < TL::NBUF; ++b) {
        if (b < b_lo || b >= b_hi) continue;
        const int g = warp + TL::NW * b;
        if (g < nst) issue_stage<T, D, TL, QB>(S, Kc, Vc, Sc, c0 + g * kStage, c1, b);
    }
}

// Merge the warps' softmax states; threads < D get their output column.
// The warps' outputs meet in `wo` (by default the epilogue buffer that
// overlays the ring, free once every warp is past it).
template <typename T, int D, class TL, int QB>
__device__ __forceinline__ void merge_warps(DecodeSmem<T, D, TL, QB>& S, float m_run, float l_run,
                                            const float (&o)[D / 32], float& Mc, float& Lc,
                                            float& Oc, float (*wo)[D] = nullptr)
{
    constexpr int EPL = D / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (!wo) wo = S.u.epi.wo;
    const float l_warp = warp_sum(l_run);
    __syncthreads();                         // every warp is past the ring it overlays
    if (lane == 0) { S.wm[warp] = m_run; S.wl[warp] = l_warp; }
#pragma unroll
    for (int e = 0; e < EPL; ++e) wo[warp][lane * EPL + e] = o[e];
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
        if (tid < D) Oc += wo[w][tid] * f;
    }
}

// Cluster-wide barrier; a single-CTA cluster only needs the CTA barrier.
__device__ __forceinline__ void cta_group_sync(int C)
{
    if (C > 1) {
        cluster_arrive();
        cluster_wait();
    } else {
        __syncthreads();
    }
}

// Fetch range of this CTA: its share of all B slots, rounded to stages.  The
// range does not depend on the occupancy, so the bulk copies can start
// before the unit's state is read.
__device__ __forceinline__ void fetch_range(int B, int C, int rank, int& f0, int& f1)
{
    int cs = (B + C - 1) / C;
    cs = (cs + kStage - 1) / kStage * kStage;
    f0 = min(B, rank * cs);
    f1 = min(B, f0 + cs);
}

// ----------------------------------------------------------------- tiles

using TileDefault = Tile<6, 2>;
// bf16 rows of 128: fewer units than SMs (one CTA per SM, often a cluster
// per unit) stream with 8 warps; very many units with 4 warps x 3 stages
using TileFew = Tile<8, 2>;
using TileMany = Tile<4, 3>;
// int8 rows: a stage holds the same 16 slots in half the bytes, so twice the
// stages keep as many bytes in flight as the bf16 tiles
using TileQ8 = Tile<5, 4>;
using TileQ8Few = Tile<8, 4>;
// 4-bit rows: a quarter of the bf16 bytes per stage; six warps measured
// faster than five or eight
using TileQ4 = Tile<6, 4>;
using TileQ4Few = Tile<8, 4>;

// Tile for bf16 rows of 128 (numbers as H2O_DECODE_TILE): TileFew when the
// units do not fill the SMs, TileMany from four units per SM on, else the
// default.
int auto_tile(int U, int num_sms)
{
    if (num_sms > 0 && U < num_sms) return 6;
    if (num_sms > 0 && U >= 4 * num_sms) return 3;
    return 2;
}

// Programmatic dependent launch is on unless H2O_PDL=0 (for comparisons).
bool pdl_enabled()
{
    static int v = -1;
    if (v < 0) {
        const char* e = getenv("H2O_PDL");
        v = (e && e[0] == '0') ? 0 : 1;
    }
    return v == 1;
}

}  // namespace

}  // namespace h2o
