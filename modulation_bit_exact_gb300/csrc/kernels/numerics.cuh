// numerics.cuh -- arithmetic building blocks of the sm_103a kernels.
//
// Every binary32 operation of a lossless path is an explicitly rounded PTX
// instruction (add/sub/mul/fma/div/sqrt .rn), so no multiply-add is ever
// contracted and no approximate instruction is used.  Two packed forms carry
// most of the work:
//   * f32x2 -- add/sub/mul/fma.rn.f32x2 operate on two independent binary32
//     values in a 64-bit register pair (two Welford lanes, or two adjacent
//     elements), each half rounded exactly like the scalar instruction.  A
//     packed product is never fed to a packed sum: ptxas fuses that pair into
//     one multiply-add even with explicit .rn and -fmad=false, so wherever a
//     rounded product feeds a sum the scalar __fmul_rn / __fadd_rn intrinsics
//     (documented never to be merged) are used instead;
//   * bf16x2 -- mul/add.rn.bf16x2 compute bf16(a*b) and bf16(a+b) from the
//     exact result.  For bfloat16 operands these equal rounding the binary32
//     result to bfloat16 (the product of two 8-bit significands and the sum of
//     two bfloat16 values are exact in binary32 except far below the smallest
//     normal, where the intermediate grid is 2^16 times finer than bfloat16's
//     and cannot create a new halfway case); mbx_selftest(1|2) checks this on
//     every pair of operands.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <type_traits>

namespace mbx {

typedef unsigned long long u64;

// ---------------------------------------------------------------- bfloat16

// A 32-bit word holds two bfloat16 values: element 2i in the low half and
// element 2i+1 in the high half (little-endian memory order).
__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// bf16 of two binary32 values, nearest-even; `lo` goes to the low half.
__device__ __forceinline__ uint32_t pack_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t bmul(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t badd(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// The same two operations written as binary32 arithmetic plus one rounding:
// the definition the packed instructions are checked against.
__device__ __forceinline__ uint32_t bmul_ref(uint32_t a, uint32_t b) {
    return pack_rn(__fmul_rn(lo_f(a), lo_f(b)), __fmul_rn(hi_f(a), hi_f(b)));
}
__device__ __forceinline__ uint32_t badd_ref(uint32_t a, uint32_t b) {
    return pack_rn(__fadd_rn(lo_f(a), lo_f(b)), __fadd_rn(hi_f(a), hi_f(b)));
}

__device__ __forceinline__ uint32_t bf16_bits(float v) {  // a bfloat16 splat (v exact in bf16)
    uint32_t h = __float_as_uint(v) >> 16;
    return h | (h << 16);
}

// ---------------------------------------------------------------- f32x2

__device__ __forceinline__ u64 f2(float lo, float hi) {
    u64 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float f2lo(u64 v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2hi(u64 v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ u64 add2(u64 a, u64 b) {
    u64 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ u64 sub2(u64 a, u64 b) {
    u64 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ u64 mul2(u64 a, u64 b) {
    u64 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ u64 fma2(u64 a, u64 b, u64 c) {
    u64 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

__device__ __forceinline__ uint32_t min_u16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("min.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Two adjacent bfloat16 elements of a word, widened to an f32x2.
__device__ __forceinline__ u64 widen2(uint32_t w) { return f2(lo_f(w), hi_f(w)); }
// Element e (0/1) of word a and the same element of word b as an f32x2.
__device__ __forceinline__ u64 pair_elem(uint32_t a, uint32_t b, int e) {
    return e ? f2(hi_f(a), hi_f(b)) : f2(lo_f(a), lo_f(b));
}
__device__ __forceinline__ uint32_t pack2_rn(u64 v) { return pack_rn(f2lo(v), f2hi(v)); }

// ---------------------------------------------------------------- division by k

// Correctly rounded d / K for a compile-time count K (1 <= K <= 64), by
// multiplication with the reciprocal split into two binary32 words
// (Brisebarre, Muller & Raina, "Accelerating correctly rounded floating-point
// division when the divisor is known in advance", IEEE Trans. Computers 53(8),
// 2004): with yh = RN(1/K) and yl = RN(1/K - yh), q = RN(d*yh + RN(d*yl)),
// one multiply and one fused multiply-add.  That paper shows the result is
// RN(d/K) for most but not all divisors, and gives a test per divisor;
// here the test is exhaustive on this GPU: the fast form equals div.rn.f32 for
// every K and every d with |d| >= 2^-100 and for d = +0 (mbx_selftest(3)),
// and the guarded form sends |d| < 2^-90 (zeros included) to div.rn and
// equals it for every finite d (mbx_selftest(0)).
// (A non-finite d only occurs in a row whose mean and M2 are already inf/NaN;
// every output of such a row is the canonical NaN whatever the quotient.)
template <int K>
struct Recip {
    static_assert(K >= 1 && K <= 64, "Welford counts are 1..64");
    static constexpr float yh = 1.0f / (float)K;
    static constexpr float yl = (float)(1.0 / (double)K - (double)yh);
};

constexpr float kDivTiny = 0x1p-90f;

// K a power of two: d/K and d*(1/K) are the same correctly rounded value
// (1/K is exact), for every d including subnormal results; K = 1 is d itself.
template <int K>
constexpr bool kPow2 = (K & (K - 1)) == 0;

template <int K>
__device__ __forceinline__ float div_k_fast(float d) {
    if constexpr (K == 1) return d;
    if constexpr (kPow2<K>) return __fmul_rn(d, Recip<K>::yh);
    return __fmaf_rn(d, Recip<K>::yh, __fmul_rn(d, Recip<K>::yl));
}

template <int K>
__device__ __forceinline__ float div_k(float d) {
    if constexpr (kPow2<K>) return div_k_fast<K>(d);
    if (fabsf(d) < kDivTiny) return __fdiv_rn(d, (float)K);
    return div_k_fast<K>(d);
}

template <int K>
__device__ __forceinline__ u64 div_k2_fast(u64 d) {
    if constexpr (K == 1) return d;
    if constexpr (kPow2<K>) return mul2(d, f2(Recip<K>::yh, Recip<K>::yh));
    return fma2(d, f2(Recip<K>::yh, Recip<K>::yh), mul2(d, f2(Recip<K>::yl, Recip<K>::yl)));
}

template <int K>
__device__ __forceinline__ u64 div_k2(u64 d) {
    if constexpr (kPow2<K>) return div_k2_fast<K>(d);
    const float dl = f2lo(d), dh = f2hi(d);
    if (fminf(fabsf(dl), fabsf(dh)) < kDivTiny) return f2(__fdiv_rn(dl, (float)K), __fdiv_rn(dh, (float)K));
    return div_k2_fast<K>(d);
}

// ---------------------------------------------------------------- compile-time loops

template <int I, int N, typename F>
__device__ __forceinline__ void static_for(F&& f) {
    if constexpr (I < N) {
        f(std::integral_constant<int, I>{});
        static_for<I + 1, N>(f);
    }
}

// ---------------------------------------------------------------- Welford

// One Welford step of count K on two lanes at once (x, mean, m2 as f32x2):
//   d = x - mean; mean += d / K; m2 += d * (x - mean)
// GUARD = false is the fast division, valid for a lane whose nonzero
// elements all have |x| >= 2^-60 (see lane_is_plain in rowops.cuh).
// nz holds -0.0f in both halves, passed in at run time (see LnModParams):
// fma(d, t, -0) is the correctly rounded product d*t for every d and t (adding
// -0 changes neither a nonzero product nor the sign of a zero one), and as the
// compiler cannot see the constant it cannot fold the fma back into a multiply
// and contract that with the add that follows.
template <int K, bool GUARD>
__device__ __forceinline__ void welford_step2(u64 x, u64& mean, u64& m2, u64 nz) {
    u64 d = sub2(x, mean);
    if constexpr (GUARD) mean = add2(mean, div_k2<K>(d));
    else mean = add2(mean, div_k2_fast<K>(d));
    const u64 t = sub2(x, mean);
    m2 = add2(m2, fma2(d, t, nz));
}

template <int K, bool GUARD>
__device__ __forceinline__ void welford_step(float x, float& mean, float& m2) {
    float d = __fsub_rn(x, mean);
    if constexpr (GUARD) mean = __fadd_rn(mean, div_k<K>(d));
    else mean = __fadd_rn(mean, div_k_fast<K>(d));
    m2 = __fadd_rn(m2, __fmul_rn(d, __fsub_rn(x, mean)));
}

struct Wf {
    float mean, m2, n;
};

// Chan pairwise combine, a = lower lane:  n = na+nb; d = mb-ma; r = nb/n;
// mean = ma + d*r; m2 = (qa+qb) + (d*d)*(na*r).  An empty side is an identity.
__device__ __forceinline__ Wf wf_combine(Wf a, Wf b) {
    if (b.n == 0.0f) return a;
    if (a.n == 0.0f) return b;
    Wf c;
    c.n = __fadd_rn(a.n, b.n);
    float d = __fsub_rn(b.mean, a.mean);
    // nb/(na+nb) is exactly 0.5 when the counts are equal (the common case)
    float r = a.n == b.n ? 0.5f : __fdiv_rn(b.n, c.n);
    c.mean = __fadd_rn(a.mean, __fmul_rn(d, r));
    c.m2 = __fadd_rn(__fadd_rn(a.m2, b.m2), __fmul_rn(__fmul_rn(d, d), __fmul_rn(a.n, r)));
    return c;
}

// The same combine when both sides hold the same nonzero count (every lane
// full): r = nb/(na+nb) = 0.5 exactly, no empty side.  Same operations, same
// bits, no branches.
__device__ __forceinline__ Wf wf_combine_eq(Wf a, Wf b) {
    Wf c;
    c.n = __fadd_rn(a.n, b.n);
    float d = __fsub_rn(b.mean, a.mean);
    c.mean = __fadd_rn(a.mean, __fmul_rn(d, 0.5f));
    c.m2 = __fadd_rn(__fadd_rn(a.m2, b.m2), __fmul_rn(__fmul_rn(d, d), __fmul_rn(a.n, 0.5f)));
    return c;
}

__device__ __forceinline__ Wf wf_shfl_down(Wf v, int s, unsigned mask = 0xffffffffu) {
    Wf o;
    o.mean = __shfl_down_sync(mask, v.mean, s);
    o.m2 = __shfl_down_sync(mask, v.m2, s);
    o.n = __shfl_down_sync(mask, v.n, s);
    return o;
}

// ---------------------------------------------------------------- memory

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation may begin while the kernel before it in the stream is still
// running, so it touches no global memory that kernel may read or write until
// grid_dep_wait() has returned (the earlier grid has completed and its writes
// are visible).  grid_dep_launch() lets the next kernel in the stream begin
// launching; that kernel's own wait still covers this whole grid.  Both are
// no-ops in a kernel launched without the attribute.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Bring [p, p + n) into L2 (p 16-byte aligned, n a multiple of 16), or the
// line holding p.  L2 is the device's point of coherence: a write the earlier
// kernel makes after the prefetch lands in the L2 copy, so a prefetch may be
// issued before grid_dep_wait().
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t n) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(n) : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// 16-byte streaming load (read once: not kept in L1).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
// 16-byte streaming load of an operand the same kernel may overwrite (an
// exact in-place residual update): a weak, coherent load.  ld.global.nc is
// reserved for data that stays read-only while the kernel runs.
__device__ __forceinline__ uint4 ld_stream_rw(const void* p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
// 16-byte load of data shared by many rows (kept in L1).
__device__ __forceinline__ uint4 ld_shared_row(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ void st_v4(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}
// The hardware tanh (one MUFU operation; relative error about 2^-11, a small
// fraction of a bfloat16 ulp): used only by the single-pass "high" variants,
// whose contract is a bound on the error, not a rounding order.
__device__ __forceinline__ float tanh_hw(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two binary32 values to FP8 E4M3 (round to nearest even, finite overflow
// and infinities saturate to +-448, NaN to 0x7F): `lo` in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float hi, float lo) {
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}

// Four bf16 values (two packed words) times `inv`, each product rounded once,
// to four E4M3 bytes in element order.
__device__ __forceinline__ uint32_t e4m3x4_of_bf16(uint32_t w0, uint32_t w1, float inv) {
    const uint32_t a = e4m3x2(__fmul_rn(hi_f(w0), inv), __fmul_rn(lo_f(w0), inv));
    const uint32_t b = e4m3x2(__fmul_rn(hi_f(w1), inv), __fmul_rn(lo_f(w1), inv));
    return a | (b << 16);
}

// Eight binary32 values to eight FP4 E2M1 codes (nearest, ties to even,
// saturating; cvt.rn.satfinite.e2m1x2.f32), element 2i in the low nibble of
// byte i.
__device__ __forceinline__ uint32_t e2m1x8(const float (&v)[8]) {
    uint32_t d;
    asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
        "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
        : "=r"(d)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return d;
}

// The value of an E4M3 code (exact, through the hardware conversion to f16).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
    uint32_t h2;
    const uint16_t c = (uint16_t)(code & 0xffu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
}

// max with NaN propagation (max.NaN.f32)
__device__ __forceinline__ float max_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// Byte offset of the scale of (row r, block b) in the 128x4 tile layout of
// NVFP4 block scales: tiles of 128 rows x 4 blocks (512 bytes) in row-major
// order; inside a tile (r mod 32, (r mod 128) / 32, b mod 4) in that order.
__device__ __forceinline__ int64_t nvfp4_sf_offset(int64_t r, int b, int col_tiles) {
    return ((r >> 7) * col_tiles + (b >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (b & 3);
}
// The same split into its row part (once per row) and its block part.
__device__ __forceinline__ int64_t nvfp4_sf_row(int64_t r, int col_tiles) {
    return (r >> 7) * col_tiles * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
}
__device__ __forceinline__ int nvfp4_sf_block(int b) { return (b >> 2) * 512 + (b & 3); }

__device__ __forceinline__ void st_u32(void* p, uint32_t a) {
    asm volatile("st.global.u32 [%0], %1;" ::"l"(p), "r"(a) : "memory");
}

__device__ __forceinline__ void st_v2(void* p, uint32_t a, uint32_t b) {
    asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ uint16_t ld_u16(const void* p) {
    uint16_t v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}
// Coherent 2-byte load (see ld_stream_rw).
__device__ __forceinline__ uint16_t ld_u16_rw(const void* p) {
    uint16_t v;
    asm volatile("ld.global.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ void st_u16(void* p, uint16_t v) {
    asm volatile("st.global.u16 [%0], %1;" ::"l"(p), "h"(v) : "memory");
}

__device__ __forceinline__ uint32_t w_of(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}
__device__ __forceinline__ void w_set(uint4& v, int i, uint32_t w) {
    if (i == 0) v.x = w;
    else if (i == 1) v.y = w;
    else if (i == 2) v.z = w;
    else v.w = w;
}

// max.NaN of two bf16 pairs (a max selects an operand: exact)
__device__ __forceinline__ uint32_t bmax_nan(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// max.NaN.xorsign.abs of two bf16 pairs: per half, the larger magnitude (an
// exact selection), NaN propagating; the sign bit is the xor of the operands'
// signs, so callers clear it.
__device__ __forceinline__ uint32_t bmaxabs_nan(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// |largest| of the eight bf16 values of a chunk, NaN propagating: pairwise
// magnitude maxima, then the larger of the two halves with the sign cleared.
__device__ __forceinline__ float amax8_bf16(const uint4& o) {
    const uint32_t a = bmaxabs_nan(bmaxabs_nan(o.x, o.y), bmaxabs_nan(o.z, o.w));
    return max_nan(fabsf(lo_f(a)), fabsf(hi_f(a)));
}

// NVFP4 block step: from the block's amax and the global scale gs, the E4M3
// block scale s = e4m3(RN(RN(amax * gs) / 6)) and its value.  The division by
// 6 is the guarded two-word reciprocal form (equal to div.rn for every finite numerator,
// mbx_selftest(0)); an infinite or NaN numerator takes div.rn itself.
__device__ __forceinline__ float div6(float d) {
    return isfinite(d) ? div_k<6>(d) : __fdiv_rn(d, 6.0f);
}
__device__ __forceinline__ uint32_t nvfp4_block_scale(float amax16, float gs, float& sv) {
    const uint32_t s = e4m3x2(0.0f, div6(__fmul_rn(amax16, gs))) & 0xffu;
    sv = e4m3_value(s);
    return s;
}

// The E4M3 code of RN(d / 6), without a branch.  For |d| >= 2^-100 the
// unguarded two-word quotient is RN(d / 6) (mbx_selftest(3)).  Below that
// both it and RN(d / 6) have magnitude under 2^-102, far below half the
// smallest E4M3 subnormal (2^-10), and carry the sign of d, so both convert
// to the same signed zero.  An infinite or NaN d gives an infinite or NaN
// quotient either way, which converts to the same code (saturated 0x7E / 0xFE,
// or 0x7F for NaN).
__device__ __forceinline__ uint32_t e4m3_of_div6(float d) {
    const float q = div_k_fast<6>(d);
    return e4m3x2(0.0f, isfinite(d) ? q : d) & 0xffu;
}

// The same step with the element factor gs / value(s) looked up in a table of
// all 256 codes (built once per CTA by nvfp4_fill_table): returns s and sets
// esc.
__device__ __forceinline__ uint32_t nvfp4_block_scale_tab(float amax16, float gs, const float* tab, float& esc) {
    const uint32_t s = e4m3_of_div6(__fmul_rn(amax16, gs));
    esc = tab[s];
    return s;
}
__device__ __forceinline__ void nvfp4_fill_table(float* tab, float gs) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) {
        const float sv = e4m3_value((uint32_t)i);
        tab[i] = __fdiv_rn(gs, sv);  // the two zero codes' entries only feed discarded codes
    }
}

// The eight E2M1 codes of a chunk given the block scale code s and the
// element factor esc = gs / value(s); every code is 0 when value(s) is 0 (s is
// +0 or -0), whatever esc.  The products are packed (each one rounding; they
// feed conversions, not sums).
__device__ __forceinline__ uint32_t nvfp4_codes_esc(const uint4& o, uint32_t s, float esc) {
    const u64 e2 = f2(esc, esc);
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const u64 pr = mul2(widen2(w_of(o, i)), e2);
        v[2 * i] = f2lo(pr);
        v[2 * i + 1] = f2hi(pr);
    }
    const uint32_t q = e2m1x8(v);
    return (s & 0x7fu) != 0u ? q : 0u;  // selected, not branched
}

// The eight E2M1 codes of a chunk, e2m1(RN(y * RN(gs / sv))); 0 when sv is 0.
__device__ __forceinline__ uint32_t nvfp4_codes(const uint4& o, float gs, float sv) {
    if (sv == 0.0f) return 0u;
    const float esc = __fdiv_rn(gs, sv);
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __fmul_rn(lo_f(w_of(o, i)), esc);
        v[2 * i + 1] = __fmul_rn(hi_f(w_of(o, i)), esc);
    }
    return e2m1x8(v);
}

}  // namespace mbx
