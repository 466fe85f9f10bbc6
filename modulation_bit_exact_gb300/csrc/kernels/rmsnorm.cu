// rmsnorm.cu -- BF16-native RMSNorm kernels: rmsnorm_scale and
// rmsnorm_tanh_residual.
//
// "#34085 [diffusion] Clean up kernels and shared fast paths" (prhub.com.cn),
// section 关键源码片段 (rmsnorm_scale): every product and the reduction result
// are rounded back to bfloat16 at the points of the eager bf16 chain:
//   sq = bf16(x*x); S = sum of sq in binary32 (here over the fixed 128-lane
//   order and tree of rowops.cuh); ms = bf16(S / D);
//   rstd = bf16(1 / sqrt(bf16(ms + eps)))   (sqrt and divide correctly rounded)
//   rmsnorm_scale:         out = bf16(bf16(bf16(x*rstd) * w) * scale)
//   rmsnorm_tanh_residual: n = bf16(bf16(x*rstd) * w); tg = bf16 nearest to
//                          tanh(g); out = bf16(r + bf16(tg * n))
// (same digest, 实现拆解 item 2; "AI Agent 驱动的 SGLang Kernel 一等公民",
// 163.com, 3.2: rmsnorm + tanh(gate)·x + residual).
// High path: binary32 throughout (unrounded squares, rsqrt, tanhf, fused
// multiply-add) with one rounding at the output.
#include "launch.h"
#include "rowops.cuh"
#include "tanh_bf16_table.inc"

namespace mbx {

// tanh of one bfloat16 (bits in the low 16 of h), from the shared-memory
// table for MBX_TANH_LO <= |g| < MBX_TANH_HI.
__device__ __forceinline__ uint32_t tanh_half(uint32_t h, const unsigned short* tab) {
    uint32_t a = h & 0x7fffu, s = h & 0x8000u;
    uint32_t idx = a - MBX_TANH_LO;
    uint32_t t = (a >= MBX_TANH_LO && a < MBX_TANH_HI) ? (s | tab[idx]) : h;
    t = a >= MBX_TANH_HI ? (s | 0x3f80u) : t;
    return a > 0x7f80u ? 0x7fffu : t;
}
__device__ __forceinline__ uint32_t tanh2(uint32_t w, const unsigned short* tab) {
    return tanh_half(w & 0xffffu, tab) | (tanh_half(w >> 16, tab) << 16);
}

// Sum of bf16(x*x) per lane (lanes paired in f32x2 when M >= 2).  Elements
// past D were loaded as zero and add exactly nothing.
template <class C>
__device__ __forceinline__ void sumsq_lanes(const uint4 (&v)[C::M][C::J], float (&L)[C::M]) {
    if constexpr (C::M >= 2) {
        constexpr int P = C::M / 2;
        u64 acc[P];
#pragma unroll
        for (int p = 0; p < P; ++p) acc[p] = f2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < C::J; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    uint32_t a = w_of(v[p][j], i), b = w_of(v[p + P][j], i);
                    uint32_t sa = bmul(a, a), sb = bmul(b, b);
                    acc[p] = add2(acc[p], pair_elem(sa, sb, 0));
                    acc[p] = add2(acc[p], pair_elem(sa, sb, 1));
                }
#pragma unroll
        for (int p = 0; p < P; ++p) {
            L[p] = f2lo(acc[p]);
            L[p + P] = f2hi(acc[p]);
        }
    } else {
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < C::J; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t a = w_of(v[0][j], i), sa = bmul(a, a);
                acc = __fadd_rn(acc, lo_f(sa));
                acc = __fadd_rn(acc, hi_f(sa));
            }
        L[0] = acc;
    }
}

// High path: unrounded binary32 sum of squares, any order.
template <class C>
__device__ __forceinline__ void sumsq_lanes_f32(const uint4 (&v)[C::M][C::J], float (&L)[C::M]) {
#pragma unroll
    for (int m = 0; m < C::M; ++m) {
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < C::J; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t w = w_of(v[m][j], i);
                acc = fmaf(lo_f(w), lo_f(w), acc);
                acc = fmaf(hi_f(w), hi_f(w), acc);
            }
        L[m] = acc;
    }
}

// rstd of the row, valid in every thread of the group.
template <class C, bool HIGH>
__device__ __forceinline__ float row_rstd(const uint4 (&v)[C::M][C::J], const RowLoop& rl,
                                          TreeSmem& sm, int D, float eps) {
    float L[C::M];
    if constexpr (!HIGH) sumsq_lanes<C>(v, L);
    else sumsq_lanes_f32<C>(v, L);
    float S = tree_reduce<C>(L, rl.t, sm, rl.bar_id, sum_combine);
    float rstd = 0.0f, unused = 0.0f;
    if (rl.t == 0) {
        if constexpr (!HIGH) {
            float ms = lo_f(pack_rn(__fdiv_rn(S, (float)D), 0.0f));
            float inner = lo_f(pack_rn(__fadd_rn(ms, eps), 0.0f));
            rstd = lo_f(pack_rn(__fdiv_rn(1.0f, __fsqrt_rn(inner)), 0.0f));
        } else {
            rstd = rsqrtf(S / (float)D + eps);
        }
    }
    group_bcast<C>(rstd, unused, rl.t, sm, rl.bar_id);
    return rstd;
}

template <int TPR, int J, bool VEC, bool HIGH>
__global__ void __launch_bounds__(kBlock) rmsnorm_scale_kernel(RmsScaleParams p) {
    using C = RowCfg<TPR, J, VEC>;
    __shared__ TreeSmem smem[C::RPC];
    const RowLoop rl = row_loop<C>();
    TreeSmem& sm = smem[rl.group];
    const int D = p.D;
    const int nch = (D + kChunk - 1) / kChunk;
    const bool per_token = p.seq == 1;

    for (int64_t row = rl.first; row < p.rows; row += rl.step) {
        uint4 v[C::M][C::J];
        load_row<C>(v, p.x + row * p.x_stride, rl.t, D, true);
        const float rstd = row_rstd<C, HIGH>(v, rl, sm, D, p.eps);
        const uint32_t r2 = bf16_bits(rstd);
        const int64_t mrow = per_token ? row : row / p.seq;
        const uint16_t* sc_row = p.scale + mrow * p.scale_stride;
        uint16_t* out_row = p.out + row * p.out_stride;
#pragma unroll
        for (int j = 0; j < C::J; ++j)
#pragma unroll
            for (int m = 0; m < C::M; ++m) {
                int c = rl.t + C::TPR * m + kLanes * j;
                if (c >= nch) continue;
                uint4 w = load_chunk<VEC>(p.weight, c, D, false);
                uint4 sc = load_chunk<VEC>(sc_row, c, D, per_token);
                uint4 o;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t xw = w_of(v[m][j], i);
                    uint32_t ow;
                    if constexpr (!HIGH) {
                        ow = bmul(bmul(bmul(xw, r2), w_of(w, i)), w_of(sc, i));
                    } else {
                        uint32_t ww = w_of(w, i), sw = w_of(sc, i);
                        ow = pack_rn(lo_f(xw) * rstd * lo_f(ww) * lo_f(sw),
                                     hi_f(xw) * rstd * hi_f(ww) * hi_f(sw));
                    }
                    w_set(o, i, ow);
                }
                store_chunk<VEC>(out_row, c, D, o);
            }
    }
}

template <int TPR, int J, bool VEC, bool HIGH>
__global__ void __launch_bounds__(kBlock) rmsnorm_tanh_residual_kernel(RmsTanhParams p) {
    using C = RowCfg<TPR, J, VEC>;
    __shared__ TreeSmem smem[C::RPC];
    __shared__ unsigned short tab[MBX_TANH_HI - MBX_TANH_LO];
    if constexpr (!HIGH) {
        for (int i = threadIdx.x; i < (int)(MBX_TANH_HI - MBX_TANH_LO); i += blockDim.x)
            tab[i] = kTanhBf16[i];
        __syncthreads();
    }
    const RowLoop rl = row_loop<C>();
    TreeSmem& sm = smem[rl.group];
    const int D = p.D;
    const int nch = (D + kChunk - 1) / kChunk;
    const bool per_token = p.seq == 1;

    for (int64_t row = rl.first; row < p.rows; row += rl.step) {
        uint4 v[C::M][C::J];
        load_row<C>(v, p.x + row * p.x_stride, rl.t, D, true);
        const float rstd = row_rstd<C, HIGH>(v, rl, sm, D, p.eps);
        const uint32_t r2 = bf16_bits(rstd);
        const int64_t grow = per_token ? row : row / p.seq;
        const uint16_t* g_row = p.gate + grow * p.gate_stride;
        const uint16_t* r_row = p.residual + row * p.res_stride;
        uint16_t* out_row = p.out + row * p.out_stride;
#pragma unroll
        for (int j = 0; j < C::J; ++j)
#pragma unroll
            for (int m = 0; m < C::M; ++m) {
                int c = rl.t + C::TPR * m + kLanes * j;
                if (c >= nch) continue;
                uint4 w = load_chunk<VEC>(p.weight, c, D, false);
                uint4 g = load_chunk<VEC>(g_row, c, D, per_token);
                uint4 r = load_chunk<VEC>(r_row, c, D, true);
                uint4 o;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t xw = w_of(v[m][j], i), ww = w_of(w, i), gw = w_of(g, i), rw = w_of(r, i);
                    uint32_t ow;
                    if constexpr (!HIGH) {
                        uint32_t n = bmul(bmul(xw, r2), ww);
                        ow = badd(rw, bmul(tanh2(gw, tab), n));
                    } else {
                        float y0 = fmaf(tanhf(lo_f(gw)), lo_f(xw) * rstd * lo_f(ww), lo_f(rw));
                        float y1 = fmaf(tanhf(hi_f(gw)), hi_f(xw) * rstd * hi_f(ww), hi_f(rw));
                        ow = pack_rn(y0, y1);
                    }
                    w_set(o, i, ow);
                }
                store_chunk<VEC>(out_row, c, D, o);
            }
    }
}

// ------------------------------------------------------------------ host

template <class P, int TPR, int J, bool VEC, bool HIGH>
static cudaError_t launch_one(const P& p, cudaStream_t s) {
    void (*k)(P);
    if constexpr (std::is_same<P, RmsScaleParams>::value) k = rmsnorm_scale_kernel<TPR, J, VEC, HIGH>;
    else k = rmsnorm_tanh_residual_kernel<TPR, J, VEC, HIGH>;
    int grid = grid_for_rows(reinterpret_cast<const void*>(k), p.rows, kBlock / TPR, kBlock);
    if (grid < 0) return cudaErrorUnknown;
    k<<<grid, kBlock, 0, s>>>(p);
    return cudaGetLastError();
}

template <class P, int TPR, int J>
static cudaError_t launch_j(const P& p, bool vec, bool high, cudaStream_t s) {
    if (vec)
        return high ? launch_one<P, TPR, J, true, true>(p, s) : launch_one<P, TPR, J, true, false>(p, s);
    return high ? launch_one<P, TPR, J, false, true>(p, s) : launch_one<P, TPR, J, false, false>(p, s);
}

template <class P>
static cudaError_t launch_rms(const P& p, bool vec, bool high, cudaStream_t s) {
    switch (chunks_per_lane(p.D)) {
        case 1: return launch_j<P, 32, 1>(p, vec, high, s);
        case 2: return launch_j<P, 32, 2>(p, vec, high, s);
        case 3: return launch_j<P, 64, 3>(p, vec, high, s);
        case 4: return launch_j<P, 64, 4>(p, vec, high, s);
        case 5: return launch_j<P, 64, 5>(p, vec, high, s);
        case 6: return launch_j<P, 128, 6>(p, vec, high, s);
        case 7: return launch_j<P, 128, 7>(p, vec, high, s);
        case 8: return launch_j<P, 128, 8>(p, vec, high, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_rmsnorm_scale(const RmsScaleParams& p, bool vec, bool high, cudaStream_t s) {
    return launch_rms(p, vec, high, s);
}
cudaError_t launch_rmsnorm_tanh_residual(const RmsTanhParams& p, bool vec, bool high, cudaStream_t s) {
    return launch_rms(p, vec, high, s);
}

}  // namespace mbx
