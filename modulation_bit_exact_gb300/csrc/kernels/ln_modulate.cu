// ln_modulate.cu -- LayerNorm (no affine) fused with AdaLN modulate.
//
// "Agent-assisted SGLang diffusion kernel optimisation: Qwen-Image, FLUX.2 and
// video models" (tahou.com), section 扩散Kernel对数值精度的敏感性:
//   y = LN(x); y = y * (1 + scale) + shift
// Lossless path (bit-exact to the eager BF16 chain, in the fixed order of
// rowops.cuh):
//   per lane, Welford over its elements: n += 1; d = x - mean;
//     mean += d / n (correctly rounded: a two-word reciprocal of the
//     compile-time count); m2 += d * (x - mean)
//   fixed tree of Chan combines; var = m2 / D; rstd = 1 / sqrt(var + eps)
//   nrm = bf16((x - mean) * rstd)          (the BF16 store between LN and modulate)
//   out = bf16(bf16(nrm * bf16(1 + scale)) + shift)
// High path: the same formula in one binary32 pass (two-pass mean/variance
// over registers, fused multiply-add allowed) with one rounding at the output.
#include "ln_pipe.cuh"

namespace mbx {

// Welford statistics of every lane this thread owns (GUARD: division safe for
// any d; otherwise the fast division, for lanes that pass lanes_plain).
template <class C, bool GUARD>
__device__ __forceinline__ void welford_lanes(const uint4 (&v)[C::M][C::J], int t, int D,
                                              Wf (&L)[C::M], u64 nz) {
    // elements left in the last chunk of each lane (<= 0: no last chunk)
    int lim[C::M];
#pragma unroll
    for (int m = 0; m < C::M; ++m) lim[m] = D - kChunk * (t + C::TPR * m + kLanes * (C::J - 1));

    if constexpr (C::M >= 2) {
        constexpr int P = C::M / 2;  // lane pairs (m, m + P) share an f32x2
        u64 mean[P], m2[P];
#pragma unroll
        for (int p = 0; p < P; ++p) mean[p] = m2[p] = f2(0.0f, 0.0f);
        static_for<0, C::J>([&](auto jc) {
            constexpr int j = decltype(jc)::value;
            static_for<0, kChunk>([&](auto ec) {
                constexpr int e = decltype(ec)::value;
                constexpr int K = kChunk * j + e + 1;
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    u64 x = pair_elem(w_of(v[p][j], e / 2), w_of(v[p + P][j], e / 2), e & 1);
                    if constexpr (j < C::J - 1) {
                        welford_step2<K, GUARD>(x, mean[p], m2[p], nz);
                    } else {
                        u64 mn = mean[p], q = m2[p];
                        welford_step2<K, GUARD>(x, mn, q, nz);
                        bool va = e < lim[p], vb = e < lim[p + P];
                        mean[p] = sel2(va, vb, mn, mean[p]);
                        m2[p] = sel2(va, vb, q, m2[p]);
                    }
                }
            });
        });
#pragma unroll
        for (int p = 0; p < P; ++p) {
            L[p].mean = f2lo(mean[p]);
            L[p].m2 = f2lo(m2[p]);
            L[p + P].mean = f2hi(mean[p]);
            L[p + P].m2 = f2hi(m2[p]);
        }
    } else {
        float mean = 0.0f, m2 = 0.0f;
        static_for<0, C::J>([&](auto jc) {
            constexpr int j = decltype(jc)::value;
            static_for<0, kChunk>([&](auto ec) {
                constexpr int e = decltype(ec)::value;
                constexpr int K = kChunk * j + e + 1;
                uint32_t w = w_of(v[0][j], e / 2);
                float x = (e & 1) ? hi_f(w) : lo_f(w);
                if constexpr (j < C::J - 1) {
                    welford_step<K, GUARD>(x, mean, m2);
                } else {
                    float mn = mean, q = m2;
                    welford_step<K, GUARD>(x, mn, q);
                    if (e < lim[0]) {
                        mean = mn;
                        m2 = q;
                    }
                }
            });
        });
        L[0].mean = mean;
        L[0].m2 = m2;
    }
#pragma unroll
    for (int m = 0; m < C::M; ++m) {
        int last = lim[m] <= 0 ? 0 : (lim[m] >= kChunk ? kChunk : lim[m]);
        L[m].n = (float)(kChunk * (C::J - 1) + last);
    }
}

template <int TPR, int J, bool VEC, bool HIGH>
__global__ void __launch_bounds__(kBlock) ln_modulate_kernel(LnModParams p) {
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

        float mean, rstd;
        if constexpr (!HIGH) {
            Wf L[C::M];
            const u64 nz = f2(p.neg_zero, p.neg_zero);
            if (lanes_plain<C>(v, rl.t, nch)) welford_lanes<C, false>(v, rl.t, D, L, nz);
            else welford_lanes<C, true>(v, rl.t, D, L, nz);
            Wf s = tree_reduce<C>(L, rl.t, sm, rl.bar_id, wf_combine);
            mean = s.mean;
            if (rl.t == 0) {
                float var = __fdiv_rn(s.m2, (float)D);
                rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(var, p.eps)));
            }
        } else {
            float acc[C::M];
#pragma unroll
            for (int m = 0; m < C::M; ++m) {
                acc[m] = 0.0f;
#pragma unroll
                for (int j = 0; j < C::J; ++j)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t w = w_of(v[m][j], i);
                        acc[m] += lo_f(w) + hi_f(w);
                    }
            }
            float s = tree_reduce<C>(acc, rl.t, sm, rl.bar_id, sum_combine);
            float dummy = 0.0f;
            mean = s / (float)D;
            group_bcast<C>(mean, dummy, rl.t, sm, rl.bar_id);
#pragma unroll
            for (int m = 0; m < C::M; ++m) {
                acc[m] = 0.0f;
                int lim = D - kChunk * (rl.t + C::TPR * m + kLanes * (C::J - 1));
#pragma unroll
                for (int j = 0; j < C::J; ++j)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t w = w_of(v[m][j], i);
                        float d0 = lo_f(w) - mean, d1 = hi_f(w) - mean;
                        if (j == C::J - 1) {
                            d0 = 2 * i < lim ? d0 : 0.0f;
                            d1 = 2 * i + 1 < lim ? d1 : 0.0f;
                        }
                        acc[m] += d0 * d0 + d1 * d1;
                    }
            }
            float q = tree_reduce<C>(acc, rl.t, sm, rl.bar_id, sum_combine);
            if (rl.t == 0) rstd = rsqrtf(q / (float)D + p.eps);
        }
        group_bcast<C>(mean, rstd, rl.t, sm, rl.bar_id);

        const int64_t mrow = per_token ? row : row / p.seq;
        const uint16_t* sc_row = p.scale + mrow * p.scale_stride;
        const uint16_t* sh_row = p.shift + mrow * p.shift_stride;
        uint16_t* out_row = p.out + row * p.out_stride;
        const u64 mean2 = f2(mean, mean), rstd2 = f2(rstd, rstd);
        const uint32_t one2 = 0x3f803f80u;
#pragma unroll
        for (int j = 0; j < C::J; ++j)
#pragma unroll
            for (int m = 0; m < C::M; ++m) {
                int c = rl.t + C::TPR * m + kLanes * j;
                if (c >= nch) continue;
                uint4 sc = load_chunk<VEC>(sc_row, c, D, per_token);
                uint4 sh = load_chunk<VEC>(sh_row, c, D, per_token);
                uint4 o;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t xw = w_of(v[m][j], i), sw = w_of(sc, i), hw = w_of(sh, i);
                    uint32_t ow;
                    if constexpr (!HIGH) {
                        uint32_t nrm = pack2_rn(mul2(sub2(widen2(xw), mean2), rstd2));
                        ow = badd(bmul(nrm, badd(one2, sw)), hw);
                    } else {
                        float y0 = fmaf((lo_f(xw) - mean) * rstd, 1.0f + lo_f(sw), lo_f(hw));
                        float y1 = fmaf((hi_f(xw) - mean) * rstd, 1.0f + hi_f(sw), hi_f(hw));
                        ow = pack_rn(y0, y1);
                    }
                    w_set(o, i, ow);
                }
                store_chunk<VEC>(out_row, c, D, o);
            }
    }
}

// ------------------------------------------------------------------ host

template <int TPR, int J, bool VEC, bool HIGH>
static cudaError_t launch_one(const LnModParams& p, cudaStream_t s) {
    auto k = ln_modulate_kernel<TPR, J, VEC, HIGH>;
    int grid = grid_for_rows(reinterpret_cast<const void*>(k), p.rows, kBlock / TPR, kBlock);
    if (grid < 0) return cudaErrorUnknown;
    return launch_pdl(k, grid, kBlock, 0, s, p);
}

template <int TPR, int J>
static cudaError_t launch_j(const LnModParams& p, bool, bool high, cudaStream_t s) {
    return high ? launch_one<TPR, J, false, true>(p, s) : launch_one<TPR, J, false, false>(p, s);
}

// First half of the composed gated op: r' = bf16(x + bf16(gate * a)) into
// res_out; returns the parameters of the LN pass over r'.
cudaError_t launch_gated_add_part(const LnModParams& p, bool vec, cudaStream_t s, LnModParams* ln) {
    GateAddParams g;
    g.out = p.res_out;
    g.out_stride = p.res_out_stride;
    g.x = p.x;
    g.x_stride = p.x_stride;
    g.gate = p.gate;
    g.gate_stride = p.gate_stride;
    g.y = p.update;
    g.y_stride = p.update_stride;
    g.rows = p.rows;
    g.D = p.D;
    g.seq = p.seq;
    g.bias = p.bias;
    *ln = p;
    ln->x = p.res_out;
    ln->x_stride = p.res_out_stride;
    ln->update = nullptr;
    ln->gate = nullptr;
    ln->bias = nullptr;
    ln->res_out = nullptr;
    return launch_residual_gate_add(g, vec, false, s);
}

cudaError_t launch_gated_residual_ln_modulate(const LnModParams& p, bool vec, bool high, cudaStream_t s) {
    if (vec && fused_fits(p, high, false)) return launch_pipe_d<true, false>(p, high, s);
    // unaligned or ragged rows, or rows too wide for the fused ring: the same
    // definition as two steps, the gated residual into res_out, then
    // LayerNorm + modulate of res_out
    return launch_all_or_none([&]() {
        LnModParams q;
        const cudaError_t e = launch_gated_add_part(p, vec, s, &q);
        if (e != cudaSuccess) return e;
        return vec ? launch_pipe_d<false, false>(q, high, s) : launch_ln_modulate(q, false, high, s);
    });
}

// The FP8 copy outside the pipelined kernel: quantise the bf16 output after it
// is written (the same definition: the copy is of the bf16 value).
static cudaError_t quantise_out(const LnModParams& p, cudaStream_t s) {
    QuantParams q;
    q.out = p.out_fp8;
    q.out_stride = p.out_fp8_stride;
    q.y = p.out;
    q.y_stride = p.out_stride;
    q.rows = p.rows;
    q.D = p.D;
    q.scale = p.fp8_scale;
    return launch_quant_e4m3(q, s);
}

cudaError_t launch_ln_modulate_fp8(const LnModParams& p, bool vec, bool high, cudaStream_t s) {
    if (vec) return launch_pipe_d<false, false>(p, high, s);
    return launch_all_or_none([&]() {
        LnModParams q = p;
        q.out_fp8 = nullptr;
        const cudaError_t e = launch_ln_modulate(q, false, high, s);
        return e != cudaSuccess ? e : quantise_out(p, s);
    });
}

cudaError_t launch_gated_residual_ln_modulate_fp8(const LnModParams& p, bool vec, bool high, cudaStream_t s) {
    if (vec && fused_fits(p, high, false)) return launch_pipe_d<true, false>(p, high, s);
    if (vec) return launch_gated_residual_ln_modulate(p, true, high, s);  // composed; the LN pass writes the FP8 copy
    return launch_all_or_none([&]() {
        LnModParams q = p;
        q.out_fp8 = nullptr;
        const cudaError_t e = launch_gated_residual_ln_modulate(q, false, high, s);
        return e != cudaSuccess ? e : quantise_out(p, s);
    });
}

cudaError_t launch_ln_modulate(const LnModParams& p, bool vec, bool high, cudaStream_t s) {
    const int J = chunks_per_lane(p.D);
    if (vec) return launch_pipe_d<false, false>(p, high, s);
    switch (J) {
        // threads per row: enough that a thread holds at most ~5 chunks of x
        case 1: return launch_j<32, 1>(p, vec, high, s);
        case 2: return launch_j<32, 2>(p, vec, high, s);
        case 3: return launch_j<64, 3>(p, vec, high, s);
        case 4: return launch_j<64, 4>(p, vec, high, s);
        case 5: return launch_j<64, 5>(p, vec, high, s);
        case 6: return launch_j<128, 6>(p, vec, high, s);
        case 7: return launch_j<128, 7>(p, vec, high, s);
        case 8: return launch_j<128, 8>(p, vec, high, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mbx
