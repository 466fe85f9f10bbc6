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
// High path: binary32 throughout (unrounded squares, rsqrt, the hardware tanh, fused
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
    grid_dep_wait();  // launched programmatically: the previous kernel has finished
    grid_dep_launch();
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
    grid_dep_wait();  // launched programmatically: the previous kernel has finished
    grid_dep_launch();
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
                uint4 r = load_chunk<VEC, true>(r_row, c, D, true);  // out may be the residual
                uint4 o;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t xw = w_of(v[m][j], i), ww = w_of(w, i), gw = w_of(g, i), rw = w_of(r, i);
                    uint32_t ow;
                    if constexpr (!HIGH) {
                        uint32_t n = bmul(bmul(xw, r2), ww);
                        ow = badd(rw, bmul(tanh2(gw, tab), n));
                    } else {
                        float y0 = fmaf(tanh_hw(lo_f(gw)), lo_f(xw) * rstd * lo_f(ww), lo_f(rw));
                        float y1 = fmaf(tanh_hw(hi_f(gw)), hi_f(xw) * rstd * hi_f(ww), hi_f(rw));
                        ow = pack_rn(y0, y1);
                    }
                    w_set(o, i, ow);
                }
                store_chunk<VEC>(out_row, c, D, o);
            }
    }
}

// ------------------------------------------------------------------ pipelined path
//
// 16-byte-aligned rows: the same lanes, order and roundings as above, with x
// streamed through a per-row-group ring of shared-memory stages by cp.async,
// the weight row (plus per-sample modulation rows, when a CTA's block of rows
// spans at most two samples) staged once per CTA (for the tanh op, tanh of a
// per-sample gate is staged instead of the gate), and per-row modulation and
// the tanh op's residual loaded into registers.  OP 0: rmsnorm_scale
// (mod = scale); OP 1: rmsnorm_tanh_residual (mod = gate, plus the residual).
enum { kRmsScale = 0, kRmsTanh = 1 };
enum { kRmsModRing = 0, kRmsModStaged = 1 };

template <int OP>
struct RmsPipeArgs;
template <>
struct RmsPipeArgs<kRmsScale> {
    using P = RmsScaleParams;
    static __device__ const uint16_t* mod(const P& p) { return p.scale; }
    static __device__ int64_t mod_stride(const P& p) { return p.scale_stride; }
    static __device__ const uint16_t* residual(const P&) { return nullptr; }
    static __device__ int64_t res_stride(const P&) { return 0; }
};
template <>
struct RmsPipeArgs<kRmsTanh> {
    using P = RmsTanhParams;
    static __device__ const uint16_t* mod(const P& p) { return p.gate; }
    static __device__ int64_t mod_stride(const P& p) { return p.gate_stride; }
    static __device__ const uint16_t* residual(const P& p) { return p.residual; }
    static __device__ int64_t res_stride(const P& p) { return p.res_stride; }
};

// Sum of bf16(x*x) per lane, chunks read from ring stage s (absent chunks
// add nothing).
template <class C, class RingT>
__device__ __forceinline__ void sumsq_stage(const RingT& ring, int s, int t, int nch, float (&L)[C::M]) {
    if constexpr (C::M >= 2) {
        constexpr int P = C::M / 2;
        u64 acc[P];
#pragma unroll
        for (int p = 0; p < P; ++p) acc[p] = f2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < C::J; ++j)
#pragma unroll
            for (int p = 0; p < P; ++p) {
                const int ca = t + C::TPR * p + kLanes * j, cb = ca + C::TPR * P;
                const uint4 A = ca < nch ? lds16(ring.at(s, 0, ca)) : make_uint4(0, 0, 0, 0);
                const uint4 B = cb < nch ? lds16(ring.at(s, 0, cb)) : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t a = w_of(A, i), b = w_of(B, i), sa = bmul(a, a), sb = bmul(b, b);
                    acc[p] = add2(acc[p], pair_elem(sa, sb, 0));
                    acc[p] = add2(acc[p], pair_elem(sa, sb, 1));
                }
            }
#pragma unroll
        for (int p = 0; p < P; ++p) {
            L[p] = f2lo(acc[p]);
            L[p + P] = f2hi(acc[p]);
        }
    } else {
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < C::J; ++j) {
            const int c = t + kLanes * j;
            if (c >= nch) continue;
            const uint4 A = lds16(ring.at(s, 0, c));
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t a = w_of(A, i), sa = bmul(a, a);
                acc = __fadd_rn(acc, lo_f(sa));
                acc = __fadd_rn(acc, hi_f(sa));
            }
        }
        L[0] = acc;
    }
}

template <class C, class RingT>
__device__ __forceinline__ void sumsq_stage_f32(const RingT& ring, int s, int t, int nch, float (&L)[C::M]) {
#pragma unroll
    for (int m = 0; m < C::M; ++m) {
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < C::J; ++j) {
            const int c = t + C::TPR * m + kLanes * j;
            if (c >= nch) continue;
            const uint4 A = lds16(ring.at(s, 0, c));
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t w = w_of(A, i);
                acc = fmaf(lo_f(w), lo_f(w), acc);
                acc = fmaf(hi_f(w), hi_f(w), acc);
            }
        }
        L[m] = acc;
    }
}

// rows per group brought into L2 before the wait on the previous kernel
constexpr int kRmsPrefetchRows = 2;

template <int TPR, int J, int NS, bool HIGH, int OP, int MODE>
__global__ void __launch_bounds__(512, 1) rmsnorm_pipe_kernel(typename RmsPipeArgs<OP>::P p, int64_t rows_per_cta) {
    using A = RmsPipeArgs<OP>;
    using C = RowCfg<TPR, J, true>;
    // the ring holds x alone: it is read twice (sum of squares, output), while a
    // per-row modulation row and the tanh op's residual are read once, by the
    // output pass, and go straight from global memory into registers
    constexpr bool DMOD = MODE == kRmsModRing;
    constexpr bool DRES = OP == kRmsTanh;
    using R = Ring<C, NS, 1>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int groups = blockDim.x / TPR;
    const int g = threadIdx.x / TPR, t = threadIdx.x % TPR;
    const int D = p.D;
    const int nch = D / kChunk;
    TreeAll<TPR>& sm = reinterpret_cast<TreeAll<TPR>*>(smem_raw)[g];
    uint4* wsm = reinterpret_cast<uint4*>(smem_raw + groups * sizeof(TreeAll<TPR>));  // weight [nch]
    uint4* msm = wsm + nch;                                                       // mod [2][nch]
    unsigned short* tab = reinterpret_cast<unsigned short*>(msm + (MODE == kRmsModStaged ? 2 * nch : 0));
    constexpr int kTab = OP == kRmsTanh && MODE == kRmsModRing ? (MBX_TANH_HI - MBX_TANH_LO) : 0;
    const R ring{reinterpret_cast<uint4*>(tab + ((kTab + 7) / 8) * 8) + (size_t)g * (R::kBytes / 16)};
    const int bar_id = 1 + g;
    const int64_t r0 = (int64_t)blockIdx.x * rows_per_cta;
    const int64_t r1 = r0 + rows_per_cta < p.rows ? r0 + rows_per_cta : p.rows;
    const int64_t m0 = r0 / p.seq;
    const int64_t split = (m0 + 1) * p.seq;  // staged: rows from here use slot 1
    const uint16_t* modp = A::mod(p);
    const int64_t mod_stride = A::mod_stride(p);
    // rows go to the groups in reverse order, so a block's extra rows (its row
    // count mod the groups) fall to the highest-numbered groups, whose warps
    // the schedulers serve first (measured: they finish a round earliest)
    const int64_t first = r0 + (groups - 1 - g);
    RowDiv here(first, groups, p.seq);  // modulation row of the row being processed
    // while the previous kernel in the stream drains, bring the weight and the
    // per-sample modulation of this block's rows (first: every row group needs
    // them before its first row) and this group's first rows into L2, and copy
    // the tanh table (constant) into shared memory; then wait for it before
    // reading anything it may write
    if (t == 0 && g == 0 && r1 > r0) {
        prefetch_l2_bulk(p.weight, (uint32_t)D * 2);
        if constexpr (MODE == kRmsModStaged) {
            const int64_t m_last = (r1 - 1) / p.seq;
            for (int64_t m = m0; m <= m_last && m <= m0 + 1; ++m) prefetch_l2_bulk(modp + m * mod_stride, (uint32_t)D * 2);
        }
    }
    if (t == 0)
#pragma unroll
        for (int s = 0; s < kRmsPrefetchRows; ++s) {
            const int64_t r = first + s * groups;
            if (r >= r1) break;
            prefetch_l2_bulk(p.x + r * p.x_stride, (uint32_t)D * 2);
            if constexpr (DRES) prefetch_l2_bulk(A::residual(p) + r * A::res_stride(p), (uint32_t)D * 2);
        }
    if constexpr (OP == kRmsTanh && !HIGH && MODE == kRmsModRing)
        for (int i = threadIdx.x; i < kTab; i += blockDim.x) tab[i] = kTanhBf16[i];
    grid_dep_wait();
    grid_dep_launch();

    auto issue = [&](int s, int64_t row) { ring.issue(s, 0, p.x + row * p.x_stride, t, nch); };
#pragma unroll
    for (int s = 0; s < NS - 1; ++s) {
        const int64_t r = first + s * groups;
        if (r < r1) issue(s, r);
        cp_async_commit();
    }
    // the first rows are on their way; stage the per-CTA data meanwhile
    for (int c = threadIdx.x; c < nch; c += blockDim.x) wsm[c] = ld_shared_row(p.weight + (int64_t)c * kChunk);
    if constexpr (MODE == kRmsModStaged) {
        const int slots = (int)((r1 - 1) / p.seq - m0 + 1);
        for (int i = threadIdx.x; i < slots * nch; i += blockDim.x) {
            const int slot = i / nch, c = i - slot * nch;
            uint4 v = ld_shared_row(modp + (m0 + slot) * mod_stride + (int64_t)c * kChunk);
            if constexpr (OP == kRmsTanh && !HIGH) {
                // a per-sample gate is shared by all its rows: stage tanh(gate)
                v.x = tanh2(v.x, kTanhBf16);
                v.y = tanh2(v.y, kTanhBf16);
                v.z = tanh2(v.z, kTanhBf16);
                v.w = tanh2(v.w, kTanhBf16);
            }
            msm[slot * nch + c] = v;
        }
    }
    __syncthreads();

    int cur = 0, par = 0;
    for (int64_t row = first; row < r1; row += groups) {
        const int64_t rn = row + (NS - 1) * groups;
        const int sn = cur == 0 ? NS - 1 : cur - 1;
        if (rn < r1) issue(sn, rn);
        cp_async_commit();
        cp_async_wait<NS - 1>();

        // this row's modulation and residual chunks, in flight during the reduction
        uint4 dMD[DMOD ? C::J : 1][DMOD ? C::M : 1], dRS[DRES ? C::J : 1][DRES ? C::M : 1];
        {
            const uint16_t* md_row = modp + here.q * mod_stride;
            const uint16_t* rs_row = nullptr;
            if constexpr (DRES) rs_row = A::residual(p) + row * A::res_stride(p);
#pragma unroll
            for (int j = 0; j < C::J; ++j)
#pragma unroll
                for (int m = 0; m < C::M; ++m) {
                    const int c = t + C::TPR * m + kLanes * j;
                    if (c >= nch) continue;
                    if constexpr (DMOD) dMD[DMOD ? j : 0][DMOD ? m : 0] = ld_stream(md_row + (int64_t)c * kChunk);
                    if constexpr (DRES) dRS[DRES ? j : 0][DRES ? m : 0] = ld_stream_rw(rs_row + (int64_t)c * kChunk);
                }
        }

        float L[C::M];
        if constexpr (!HIGH) sumsq_stage<C>(ring, cur, t, nch, L);
        else sumsq_stage_f32<C>(ring, cur, t, nch, L);
        const float rstd = tree_w0_sum<C>(L, t, sm, bar_id, par, [&](float S) {
            float r;
            if constexpr (!HIGH) {
                const float ms = lo_f(pack_rn(__fdiv_rn(S, (float)D), 0.0f));
                const float inner = lo_f(pack_rn(__fadd_rn(ms, p.eps), 0.0f));
                r = lo_f(pack_rn(__fdiv_rn(1.0f, __fsqrt_rn(inner)), 0.0f));
            } else {
                r = rsqrtf(S / (float)D + p.eps);
            }
            return make_float2(r, 0.0f);
        }).x;
        const uint32_t r2 = bf16_bits(rstd);
        const uint4* mrow = MODE == kRmsModStaged ? msm + (row >= split ? nch : 0) : nullptr;
        uint16_t* out_row = p.out + row * p.out_stride;
#pragma unroll
        for (int j = 0; j < C::J; ++j)
#pragma unroll
            for (int m = 0; m < C::M; ++m) {
                const int c = t + C::TPR * m + kLanes * j;
                if (c >= nch) continue;
                const uint4 X = lds16(ring.at(cur, 0, c));
                const uint4 W = lds16(wsm + c);
                uint4 MD;
                if constexpr (MODE == kRmsModStaged) MD = lds16(mrow + c);
                else MD = dMD[DMOD ? j : 0][DMOD ? m : 0];
                uint4 RS = make_uint4(0, 0, 0, 0);
                if constexpr (DRES) RS = dRS[DRES ? j : 0][DRES ? m : 0];
                uint4 o;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t xw = w_of(X, i), ww = w_of(W, i), mw = w_of(MD, i);
                    uint32_t ow;
                    if constexpr (OP == kRmsScale) {
                        if constexpr (!HIGH) {
                            ow = bmul(bmul(bmul(xw, r2), ww), mw);
                        } else {
                            ow = pack_rn(lo_f(xw) * rstd * lo_f(ww) * lo_f(mw), hi_f(xw) * rstd * hi_f(ww) * hi_f(mw));
                        }
                    } else {
                        const uint32_t rw = w_of(RS, i);
                        if constexpr (!HIGH) {
                            const uint32_t n = bmul(bmul(xw, r2), ww);
                            const uint32_t tg = MODE == kRmsModStaged ? mw : tanh2(mw, tab);
                            ow = badd(rw, bmul(tg, n));
                        } else {
                            ow = pack_rn(fmaf(tanh_hw(lo_f(mw)), lo_f(xw) * rstd * lo_f(ww), lo_f(rw)),
                                         fmaf(tanh_hw(hi_f(mw)), hi_f(xw) * rstd * hi_f(ww), hi_f(rw)));
                        }
                    }
                    w_set(o, i, ow);
                }
                st_v4(out_row + (int64_t)c * kChunk, o);
            }
        cur = cur + 1 == NS ? 0 : cur + 1;
        par ^= 1;
        if constexpr (DMOD) here.advance();
    }
    cp_async_wait<0>();
}

template <int TPR, int J, int NS, bool HIGH, int OP, int MODE>
static cudaError_t launch_rms_pipe(const typename RmsPipeArgs<OP>::P& p, cudaStream_t s) {
    auto k = rmsnorm_pipe_kernel<TPR, J, NS, HIGH, OP, MODE>;
    using C = RowCfg<TPR, J, true>;
    using R = Ring<C, NS, 1>;
    const int nch = p.D / kChunk;
    const int tab_bytes = OP == kRmsTanh && MODE == kRmsModRing ? (((MBX_TANH_HI - MBX_TANH_LO) + 7) / 8) * 16 : 0;
    const int fixed = nch * 16 + (MODE == kRmsModStaged ? 2 * nch * 16 : 0) + tab_bytes;
    PipeShape sh;
    if (!pipe_shape(reinterpret_cast<const void*>(k), TPR, (int)sizeof(TreeAll<TPR>) + R::kBytes, fixed, p.rows, &sh))
        return cudaErrorInvalidConfiguration;
    return launch_pdl(k, sh.grid, sh.groups * TPR, sh.smem, s, p, sh.rows_per_cta);
}

template <int OP, int TPR, int J, int NS>
static cudaError_t launch_rms_pipe_v(const typename RmsPipeArgs<OP>::P& p, bool high, cudaStream_t s) {
    const bool staged = pipe_rows_per_cta(p.rows) <= p.seq;
    if (high)
        return staged ? launch_rms_pipe<TPR, J, NS, true, OP, kRmsModStaged>(p, s)
                      : launch_rms_pipe<TPR, J, NS, true, OP, kRmsModRing>(p, s);
    return staged ? launch_rms_pipe<TPR, J, NS, false, OP, kRmsModStaged>(p, s)
                  : launch_rms_pipe<TPR, J, NS, false, OP, kRmsModRing>(p, s);
}

// Threads per row and ring stages, measured per row width, operation and
// row count: three stages at 2048 and 3072 (and for the tanh op at 8192),
// two elsewhere; one warp per row
// up to 2048 elements (two for the tanh op at 2048), two at 3072 and 4096,
// four above; four warps at 3072 for rmsnorm_scale from 32768 rows and at
// 4096 from 16384 rows (faster there, slower on fewer rows); two warps for
// lossless rmsnorm_scale with per-sample modulation at 5120, 6144 and 8192
// (+2..4%; the high variant is slower with two).
template <int OP>
static cudaError_t launch_rms_pipe_d(const typename RmsPipeArgs<OP>::P& p, bool high, cudaStream_t s) {
    const bool staged_lossless = !high && pipe_rows_per_cta(p.rows) <= p.seq;
    switch (chunks_per_lane(p.D)) {
        case 1: return launch_rms_pipe_v<OP, 32, 1, 2>(p, high, s);
        case 2:
            if constexpr (OP == kRmsTanh) return launch_rms_pipe_v<OP, 64, 2, 3>(p, high, s);
            else return launch_rms_pipe_v<OP, 32, 2, 3>(p, high, s);
        case 3:
            if constexpr (OP == kRmsScale) {
                if (p.rows >= 32768) return launch_rms_pipe_v<OP, 128, 3, 3>(p, high, s);
            }
            return launch_rms_pipe_v<OP, 64, 3, 3>(p, high, s);
        case 4:
            if (p.rows >= 16384) return launch_rms_pipe_v<OP, 128, 4, 2>(p, high, s);
            return launch_rms_pipe_v<OP, 64, 4, 2>(p, high, s);
        case 5:
            if constexpr (OP == kRmsScale) {
                if (staged_lossless) return launch_rms_pipe<64, 5, 2, false, OP, kRmsModStaged>(p, s);
            }
            return launch_rms_pipe_v<OP, 128, 5, 2>(p, high, s);
        case 6:
            if constexpr (OP == kRmsScale) {
                if (staged_lossless) return launch_rms_pipe<64, 6, 2, false, OP, kRmsModStaged>(p, s);
            }
            return launch_rms_pipe_v<OP, 128, 6, 2>(p, high, s);
        case 7: return launch_rms_pipe_v<OP, 128, 7, 2>(p, high, s);
        case 8:
            if constexpr (OP == kRmsTanh) {
                return launch_rms_pipe_v<OP, 128, 8, 3>(p, high, s);
            } else {
                if (staged_lossless) return launch_rms_pipe<64, 8, 2, false, OP, kRmsModStaged>(p, s);
                return launch_rms_pipe_v<OP, 128, 8, 2>(p, high, s);
            }
        default: return cudaErrorInvalidValue;
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
    return launch_pdl(k, grid, kBlock, 0, s, p);
}

template <class P, int TPR, int J>
static cudaError_t launch_j(const P& p, bool, bool high, cudaStream_t s) {
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
    if (vec) return launch_rms_pipe_d<kRmsScale>(p, high, s);
    return launch_rms(p, vec, high, s);
}
cudaError_t launch_rmsnorm_tanh_residual(const RmsTanhParams& p, bool vec, bool high, cudaStream_t s) {
    if (vec) return launch_rms_pipe_d<kRmsTanh>(p, high, s);
    return launch_rms(p, vec, high, s);
}

}  // namespace mbx
