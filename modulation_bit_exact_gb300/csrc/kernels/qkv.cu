// qkv.cu -- fused post-GEMM QKV epilogue.
//
// "Agent-assisted SGLang diffusion kernel optimisation: Qwen-Image, FLUX.2 and
// video models" (tahou.com), section 合并QKV投影时的数值问题: after the merged
// QKV GEMM one kernel performs (1) Q/K RMSNorm, (2) interleaved RoPE, (3) the
// V copy and (4) writes text and image tokens into the joint QKV buffer,
// reading the GEMM output through strided row views, so no intermediate
// tensor is materialised.
//
// Work decomposition: a CTA owns one (token, head-pass) unit at a time
// (persistent loop; a head pass is `slots` heads, all H heads when they fit in
// 512 threads).  Its threads form `slots` head units of hd/8 threads; thread l
// of a unit holds the 8-element chunk l of the head, which is also logical
// lane l of the 128-lane order (a head has at most 32 chunks, so the levels
// s >= 32 of the fixed tree only add empty lanes and the remaining levels are
// warp shuffles within the unit).  The Q, K and V chunks of the next unit and
// its table entries are loaded while the current unit is computed (a register
// double buffer); a thread's Q and K sums travel together in one f32x2.
//
// Lossless Q/K head: the BF16-native RMSNorm chain without the scale
// (sq = bf16(x*x), S over the lanes, ms = bf16(S/hd),
// rstd = bf16(1/sqrt(bf16(ms+eps))), n = bf16(bf16(x*rstd)*w)), then for each
// pair (2i, 2i+1): o0 = bf16(n0*c - n1*s), o1 = bf16(n0*s + n1*c) in binary32
// with c, s the token's table entries for pair i.  V is a bit copy.
#include <type_traits>

#include "launch.h"
#include "rowops.cuh"
#include "rstd_bf16_table.inc"

namespace mbx {

__device__ __forceinline__ float4 ld_f4(const float* p) {
    float4 v;
    asm volatile("ld.global.nc.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ unsigned fast_div(unsigned n, const FastDiv& f) {
    return (unsigned)(((unsigned long long)n * f.m) >> f.shift);
}

// bf16(1 / sqrt(inner)) for a bfloat16 `inner` (binary32 sqrt and division,
// each correctly rounded): a lookup in a table generated from exactly that
// definition and compared with div.rn(1, sqrt.rn(v)) on this GPU for every
// bfloat16 v (mbx_selftest(4)).  NaN gives the canonical NaN.
__device__ __forceinline__ float rstd_bf16(float inner) {
    const uint32_t ib = __float_as_uint(inner) >> 16;
    const uint32_t r = ib <= 0x7f80u ? (uint32_t)kRstdBf16[ib] : 0x7fffu;
    return __uint_as_float(r << 16);
}

// One unit of work: the heads [hp*slots, hp*slots + slots) of one token.
// Index arithmetic in I: 32-bit unsigned when every element offset of the
// call fits (the launcher checks), else 64-bit.
template <class I>
struct QkvUnit {
    I b, s, sb;
    bool txt;
    const uint16_t* src;
    const float* cos_row;
    const float* sin_row;
};

template <int HD, class I>
__device__ __forceinline__ QkvUnit<I> qkv_unit(const QkvParams& p, I tok) {
    QkvUnit<I> u;
    const I s_txt = (I)p.s_txt, s_tot = (I)(p.s_txt + p.s_img);
    u.b = (I)fast_div((unsigned)tok, p.by_stot);
    u.s = tok - u.b * s_tot;  // position in the joint sequence
    u.txt = u.s < s_txt;
    u.sb = u.txt ? u.s : u.s - s_txt;  // position within the branch
    u.src = u.txt ? p.txt + (u.b * s_txt + u.sb) * (I)p.txt_stride
                  : p.img + (u.b * (I)p.s_img + u.sb) * (I)p.img_stride;
    u.cos_row = (u.txt ? p.cos_txt : p.cos_img) + u.sb * (I)(HD / 2);
    u.sin_row = (u.txt ? p.sin_txt : p.sin_img) + u.sb * (I)(HD / 2);
    return u;
}

template <int TPH, bool HIGH, bool I32>
__global__ void __launch_bounds__(512) qkv_epilogue_kernel(QkvParams p) {
    using I = typename std::conditional<I32, uint32_t, int64_t>::type;
    grid_dep_wait();  // launched programmatically: the previous kernel has finished
    grid_dep_launch();
    constexpr int HD = TPH * kChunk;
    const int l = threadIdx.x % TPH;     // chunk / lane within the head
    const int slot = threadIdx.x / TPH;  // head unit within the CTA
    const int slots = blockDim.x / TPH;
    const int H = p.heads;
    const I s_tot = (I)(p.s_txt + p.s_img);
    const int hpasses = p.hpasses;
    const int64_t units = p.batch * (p.s_txt + p.s_img) * hpasses;
    const I part_stride = (I)H * HD;  // columns between Q, K and V

    // software pipeline: the next unit's chunks and table entries are in
    // flight while the current one is computed
    uint4 nx[3];
    float4 nc, ns;
    auto fetch = [&](int64_t unit) {
        const I tok = hpasses == 1 ? (I)unit : (I)fast_div((unsigned)unit, p.by_hpass);
        const int hp = (int)((I)unit - tok * (I)hpasses);
        const QkvUnit<I> u = qkv_unit<HD, I>(p, tok);
        const int h = hp * slots + slot;
#pragma unroll
        for (int part = 0; part < 3; ++part)
            nx[part] = h < H ? ld_stream(u.src + ((I)part * part_stride + (I)h * HD + (I)(l * kChunk)))
                             : make_uint4(0, 0, 0, 0);
        nc = ld_f4(u.cos_row + 4 * l);
        ns = ld_f4(u.sin_row + 4 * l);
    };
    int64_t unit = blockIdx.x;
    if (unit < units) fetch(unit);
    for (; unit < units; unit += gridDim.x) {
        const uint4 xq = nx[0], xk = nx[1], xv = nx[2];
        const float4 c4 = nc, s4 = ns;
        if (unit + gridDim.x < units) fetch(unit + gridDim.x);

        const I tok = hpasses == 1 ? (I)unit : (I)fast_div((unsigned)unit, p.by_hpass);
        const int hp = (int)((I)unit - tok * (I)hpasses);
        const QkvUnit<I> u = qkv_unit<HD, I>(p, tok);
        const int h = hp * slots + slot;
        const bool active = h < H;
        uint16_t* const dst_q = p.joint + (((((u.b * 3) * (I)H + (I)h) * s_tot + u.s) * (I)HD) + (I)(l * kChunk));
        const I part_out = (I)H * s_tot * (I)HD;  // between the Q, K and V planes
        if (active) st_v4(dst_q + 2 * part_out, xv);  // V: bit copy

        const uint4 wq = ld_shared_row((u.txt ? p.wq_txt : p.wq_img) + l * kChunk);
        const uint4 wk = ld_shared_row((u.txt ? p.wk_txt : p.wk_img) + l * kChunk);
        // lane sums of squares of the Q and K heads side by side (f32x2:
        // Q in the low half, K in the high half), element order
        u64 acc = f2(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t a = w_of(xq, i), b = w_of(xk, i);
            if constexpr (!HIGH) {
                const uint32_t sa = bmul(a, a), sb = bmul(b, b);
                acc = add2(acc, pair_elem(sa, sb, 0));
                acc = add2(acc, pair_elem(sa, sb, 1));
            } else {
                acc = fma2(pair_elem(a, b, 0), pair_elem(a, b, 0), acc);
                acc = fma2(pair_elem(a, b, 1), pair_elem(a, b, 1), acc);
            }
        }
#pragma unroll
        for (int sh = TPH / 2; sh >= 1; sh /= 2)
            acc = add2(acc, f2(__shfl_down_sync(0xffffffffu, f2lo(acc), sh, TPH),
                               __shfl_down_sync(0xffffffffu, f2hi(acc), sh, TPH)));
        const float Sq = __shfl_sync(0xffffffffu, f2lo(acc), 0, TPH);
        const float Sk = __shfl_sync(0xffffffffu, f2hi(acc), 0, TPH);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            const uint4 x = part == 0 ? xq : xk, w = part == 0 ? wq : wk;
            const float S = part == 0 ? Sq : Sk;
            uint4 o;
            if constexpr (!HIGH) {
                // S / HD: HD is a power of two, so the product is the correctly
                // rounded quotient
                const float ms = lo_f(pack_rn(__fmul_rn(S, 1.0f / HD), 0.0f));
                const float inner = lo_f(pack_rn(__fadd_rn(ms, p.eps), 0.0f));
                const uint32_t r2 = bf16_bits(rstd_bf16(inner));
                // pairs i and i+1 side by side in f32x2: each product is one
                // correctly rounded fma(a, b, -0) (nz, a run-time -0), each
                // sum or difference one rounded add
                const u64 nz = f2(p.neg_zero, p.neg_zero);
#pragma unroll
                for (int i = 0; i < 4; i += 2) {
                    const uint32_t na = bmul(bmul(w_of(x, i), r2), w_of(w, i));
                    const uint32_t nb = bmul(bmul(w_of(x, i + 1), r2), w_of(w, i + 1));
                    const u64 n0 = f2(lo_f(na), lo_f(nb)), n1 = f2(hi_f(na), hi_f(nb));
                    const u64 c = i == 0 ? f2(c4.x, c4.y) : f2(c4.z, c4.w);
                    const u64 sn = i == 0 ? f2(s4.x, s4.y) : f2(s4.z, s4.w);
                    const u64 o0 = sub2(fma2(n0, c, nz), fma2(n1, sn, nz));
                    const u64 o1 = add2(fma2(n0, sn, nz), fma2(n1, c, nz));
                    w_set(o, i, pack_rn(f2lo(o0), f2lo(o1)));
                    w_set(o, i + 1, pack_rn(f2hi(o0), f2hi(o1)));
                }
            } else {
                const float rstd = rsqrtf(S / (float)HD + p.eps);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t xw = w_of(x, i), ww = w_of(w, i);
                    const float n0 = lo_f(xw) * rstd * lo_f(ww), n1 = hi_f(xw) * rstd * hi_f(ww);
                    const float c = i == 0 ? c4.x : i == 1 ? c4.y : i == 2 ? c4.z : c4.w;
                    const float sn = i == 0 ? s4.x : i == 1 ? s4.y : i == 2 ? s4.z : s4.w;
                    w_set(o, i, pack_rn(fmaf(n0, c, -n1 * sn), fmaf(n0, sn, n1 * c)));
                }
            }
            if (active) st_v4(dst_q + part * part_out, o);
        }
    }
}

// Whether every element offset the kernel forms fits in 32 bits: the joint
// buffer, and each branch's rows (last row start plus the Q, K, V columns).
static bool qkv_fits_32(const QkvParams& p) {
    const int64_t lim = (int64_t)1 << 32;
    const int64_t s_tot = p.s_txt + p.s_img, cols = 3 * (int64_t)p.heads * p.head_dim;
    if (p.batch * 3 * p.heads * s_tot * p.head_dim >= lim) return false;
    for (int t = 0; t < 2; ++t) {
        const int64_t rows = p.batch * (t == 0 ? p.s_txt : p.s_img), stride = t == 0 ? p.txt_stride : p.img_stride;
        if (rows > 0 && (rows - 1) * stride + cols >= lim) return false;
        if (rows * stride >= lim) return false;  // the row-start product itself
    }
    return true;
}

template <int TPH, bool HIGH, bool I32>
static cudaError_t launch_one(const QkvParams& p0, cudaStream_t s) {
    auto k = qkv_epilogue_kernel<TPH, HIGH, I32>;
    int slots = p0.heads < 512 / TPH ? (int)p0.heads : 512 / TPH;
    int block = slots * TPH;
    if (block % 32) block += 32 - block % 32;  // whole warps (extra units idle)
    slots = block / TPH;
    QkvParams p = p0;
    p.hpasses = (p.heads + slots - 1) / slots;
    const int64_t tokens = p.batch * (p.s_txt + p.s_img);
    if (tokens * p.hpasses >= (1ll << 31)) return cudaErrorInvalidValue;
    p.by_stot = make_fastdiv((unsigned)(p.s_txt + p.s_img));
    p.by_hpass = make_fastdiv((unsigned)p.hpasses);
    int grid = grid_for_rows(reinterpret_cast<const void*>(k), tokens * p.hpasses, 1, block);
    if (grid < 0) return cudaErrorUnknown;
    return launch_pdl(k, grid, block, 0, s, p);
}

template <int TPH>
static cudaError_t launch_hd(const QkvParams& p, bool high, cudaStream_t s) {
    if (qkv_fits_32(p)) return high ? launch_one<TPH, true, true>(p, s) : launch_one<TPH, false, true>(p, s);
    return high ? launch_one<TPH, true, false>(p, s) : launch_one<TPH, false, false>(p, s);
}

cudaError_t launch_qkv_epilogue(const QkvParams& p, bool high, cudaStream_t s) {
    switch (p.head_dim) {
        case 64: return launch_hd<8>(p, high, s);
        case 128: return launch_hd<16>(p, high, s);
        case 256: return launch_hd<32>(p, high, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mbx
