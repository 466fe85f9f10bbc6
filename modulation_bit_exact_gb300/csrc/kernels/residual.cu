// residual.cu -- gated residual add, out = bf16(x + bf16(gate * y)).
//
// "#34085 [diffusion] Clean up kernels and shared fast paths" (prhub.com.cn),
// section 实现拆解 item 3 (the unified residual_gate_add entry); "AI Agent
// 驱动的 SGLang Kernel 一等公民" (163.com), 3.2 (residual + gate·update).
// Lossless: the product and the sum are each rounded to bfloat16, as the
// eager chain x + gate * y does.  High: one fused multiply-add in binary32,
// rounded once.
#include "launch.h"
#include "rowops.cuh"

namespace mbx {

template <int J, bool VEC, bool HIGH>
__global__ void __launch_bounds__(kBlock) residual_gate_add_kernel(GateAddParams p) {
    grid_dep_wait();  // launched programmatically: the previous kernel has finished
    grid_dep_launch();
    using C = RowCfg<128, J, VEC>;  // one 128-thread group per row, no reduction
    const RowLoop rl = row_loop<C>();
    const int D = p.D;
    const int nch = (D + kChunk - 1) / kChunk;
    const bool per_token = p.seq == 1;

    for (int64_t row = rl.first; row < p.rows; row += rl.step) {
        const uint16_t* x_row = p.x + row * p.x_stride;
        const uint16_t* y_row = p.y + row * p.y_stride;
        const uint16_t* g_row = p.gate + (per_token ? row : row / p.seq) * p.gate_stride;
        uint16_t* out_row = p.out + row * p.out_stride;
        uint4 xv[J], yv[J], gv[J];
#pragma unroll
        for (int j = 0; j < J; ++j) {
            int c = rl.t + kLanes * j;
            if (c < nch) {
                xv[j] = load_chunk<VEC, true>(x_row, c, D, true);  // out may be x
                yv[j] = load_chunk<VEC>(y_row, c, D, true);
                gv[j] = load_chunk<VEC>(g_row, c, D, per_token);
                if (p.bias) {  // internal use: the fused entry point's fallback
                    const uint4 b = load_chunk<VEC>(p.bias, c, D, false);
                    yv[j].x = badd(yv[j].x, b.x);
                    yv[j].y = badd(yv[j].y, b.y);
                    yv[j].z = badd(yv[j].z, b.z);
                    yv[j].w = badd(yv[j].w, b.w);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < J; ++j) {
            int c = rl.t + kLanes * j;
            if (c >= nch) continue;
            uint4 o;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t xw = w_of(xv[j], i), yw = w_of(yv[j], i), gw = w_of(gv[j], i);
                uint32_t ow;
                if constexpr (!HIGH) {
                    ow = badd(xw, bmul(gw, yw));
                } else {
                    ow = pack_rn(fmaf(lo_f(gw), lo_f(yw), lo_f(xw)), fmaf(hi_f(gw), hi_f(yw), hi_f(xw)));
                }
                w_set(o, i, ow);
            }
            store_chunk<VEC>(out_row, c, D, o);
        }
    }
}

// Aligned rows (D % 8 == 0): the tensor as one list of 16-byte chunks, rows
// back to back, so every thread gets within one chunk of the same share
// (rows would leave the last round of row slots partly idle).  Each thread
// issues the loads of kFlatU chunks before it computes and stores them; the
// row and modulation row of a chunk come from multiply-shift divisions.
constexpr int kFlatU = 4;

__device__ __forceinline__ unsigned fdiv_u(unsigned n, const FastDiv& f) {
    return (unsigned)(((unsigned long long)n * f.m) >> f.shift);
}

// BIAS (internal: the composed gated LN): y is replaced by bf16(y + bias).
template <bool HIGH, bool BIAS>
__global__ void __launch_bounds__(kBlock) residual_gate_add_flat_kernel(GateAddParams p, FastDiv by_nch,
                                                                        FastDiv by_seq, unsigned total) {
    const unsigned nch = (unsigned)p.D / kChunk;
    const unsigned stride = gridDim.x * kBlock * kFlatU;
    // while the previous kernel in the stream drains, bring this thread's
    // first chunks of x and y into L2; then wait for it
#pragma unroll
    for (int u = 0; u < kFlatU; ++u) {
        const unsigned q = blockIdx.x * kBlock * kFlatU + threadIdx.x + u * kBlock;
        if (q >= total) break;
        const unsigned row = fdiv_u(q, by_nch), col = q - row * nch;
        prefetch_l2(p.x + (int64_t)row * p.x_stride + col * kChunk);
        prefetch_l2(p.y + (int64_t)row * p.y_stride + col * kChunk);
    }
    grid_dep_wait();
    grid_dep_launch();
    for (unsigned base = blockIdx.x * kBlock * kFlatU + threadIdx.x; base < total; base += stride) {
        uint4 xv[kFlatU], yv[kFlatU], gv[kFlatU];
        unsigned row[kFlatU], col[kFlatU];
#pragma unroll
        for (int u = 0; u < kFlatU; ++u) {
            const unsigned q = base + u * kBlock;
            if (q >= total) continue;
            row[u] = fdiv_u(q, by_nch);
            col[u] = q - row[u] * nch;
            const unsigned mrow = fdiv_u(row[u], by_seq);
            xv[u] = ld_stream_rw(p.x + (int64_t)row[u] * p.x_stride + col[u] * kChunk);  // out may be x
            yv[u] = ld_stream(p.y + (int64_t)row[u] * p.y_stride + col[u] * kChunk);
            gv[u] = ld_shared_row(p.gate + (int64_t)mrow * p.gate_stride + col[u] * kChunk);
            if constexpr (BIAS) {
                const uint4 b = ld_shared_row(p.bias + col[u] * kChunk);
                yv[u] = make_uint4(badd(yv[u].x, b.x), badd(yv[u].y, b.y), badd(yv[u].z, b.z), badd(yv[u].w, b.w));
            }
        }
#pragma unroll
        for (int u = 0; u < kFlatU; ++u) {
            const unsigned q = base + u * kBlock;
            if (q >= total) continue;
            uint4 o;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t xw = w_of(xv[u], i), yw = w_of(yv[u], i), gw = w_of(gv[u], i);
                uint32_t ow;
                if constexpr (!HIGH) ow = badd(xw, bmul(gw, yw));
                else ow = pack_rn(fmaf(lo_f(gw), lo_f(yw), lo_f(xw)), fmaf(hi_f(gw), hi_f(yw), hi_f(xw)));
                w_set(o, i, ow);
            }
            st_v4(p.out + (int64_t)row[u] * p.out_stride + col[u] * kChunk, o);
        }
    }
}

template <int J, bool VEC, bool HIGH>
static cudaError_t launch_one(const GateAddParams& p, cudaStream_t s) {
    auto k = residual_gate_add_kernel<J, VEC, HIGH>;
    int grid = grid_for_rows(reinterpret_cast<const void*>(k), p.rows, kBlock / 128, kBlock);
    if (grid < 0) return cudaErrorUnknown;
    return launch_pdl(k, grid, kBlock, 0, s, p);
}

template <int J>
static cudaError_t launch_j(const GateAddParams& p, bool vec, bool high, cudaStream_t s) {
    if (vec) return high ? launch_one<J, true, true>(p, s) : launch_one<J, true, false>(p, s);
    return high ? launch_one<J, false, true>(p, s) : launch_one<J, false, false>(p, s);
}

template <bool HIGH, bool BIAS>
static cudaError_t launch_flat(const GateAddParams& p, cudaStream_t s) {
    auto k = residual_gate_add_flat_kernel<HIGH, BIAS>;
    const unsigned total = (unsigned)(p.rows * (p.D / kChunk));
    const int grid = grid_for_rows(reinterpret_cast<const void*>(k), (total + kBlock * kFlatU - 1) / (kBlock * kFlatU), 1, kBlock);
    if (grid < 0) return cudaErrorUnknown;
    return launch_pdl(k, grid, kBlock, 0, s, p, make_fastdiv((unsigned)(p.D / kChunk)), make_fastdiv((unsigned)p.seq),
                      total);
}

cudaError_t launch_residual_gate_add(const GateAddParams& p, bool vec, bool high, cudaStream_t s) {
    // the flat form when its 32-bit chunk index fits
    if (vec && p.rows * (p.D / kChunk) < (1ll << 31)) {
        if (p.bias != nullptr) return high ? launch_flat<true, true>(p, s) : launch_flat<false, true>(p, s);
        return high ? launch_flat<true, false>(p, s) : launch_flat<false, false>(p, s);
    }
    switch (chunks_per_lane(p.D)) {
        case 1: return launch_j<1>(p, vec, high, s);
        case 2: return launch_j<2>(p, vec, high, s);
        case 3: return launch_j<3>(p, vec, high, s);
        case 4: return launch_j<4>(p, vec, high, s);
        case 5: return launch_j<5>(p, vec, high, s);
        case 6: return launch_j<6>(p, vec, high, s);
        case 7: return launch_j<7>(p, vec, high, s);
        case 8: return launch_j<8>(p, vec, high, s);
        default: return cudaErrorInvalidValue;
    }
}

// Static E4M3 copy of a bf16 matrix (the FP8 producers' fallback for rows
// the pipelined kernel does not take): one element per step, any alignment.
__global__ void __launch_bounds__(kBlock) quant_e4m3_kernel(QuantParams p) {
    grid_dep_wait();  // launched programmatically: the previous kernel has finished
    grid_dep_launch();
    const float inv = __fdiv_rn(1.0f, __ldg(p.scale));
    for (int64_t r = blockIdx.x; r < p.rows; r += gridDim.x) {
        const uint16_t* y = p.y + r * p.y_stride;
        uint8_t* o = p.out + r * p.out_stride;
        for (int e = threadIdx.x; e < p.D; e += blockDim.x) {
            const float v = __uint_as_float((uint32_t)ld_u16(y + e) << 16);
            o[e] = (uint8_t)(e4m3x2(0.0f, __fmul_rn(v, inv)) & 0xffu);
        }
    }
}

cudaError_t launch_quant_e4m3(const QuantParams& p, cudaStream_t s) {
    const int grid = grid_for_rows(reinterpret_cast<const void*>(quant_e4m3_kernel), p.rows, 1, kBlock);
    if (grid < 0) return cudaErrorUnknown;
    return launch_pdl(quant_e4m3_kernel, grid, kBlock, 0, s, p);
}

// NVFP4 copy of a bf16 matrix, one 16-element block per thread, any
// alignment (the fallback of the NVFP4 producers).
__global__ void __launch_bounds__(kBlock) quant_nvfp4_kernel(QuantFp4Params p) {
    grid_dep_wait();  // launched programmatically: the previous kernel has finished
    grid_dep_launch();
    const float gs = __ldg(p.gs);
    const int blocks = p.D / 16;
    const int64_t total = p.rows * blocks;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / blocks;
        const int b = (int)(i - r * blocks);
        const uint16_t* y = p.y + r * p.y_stride + b * 16;
        uint4 lo, hi;
        uint32_t wv[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) wv[k] = (uint32_t)ld_u16(y + 2 * k) | ((uint32_t)ld_u16(y + 2 * k + 1) << 16);
        lo = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        hi = make_uint4(wv[4], wv[5], wv[6], wv[7]);
        float sv;
        const uint32_t sc = nvfp4_block_scale(max_nan(amax8_bf16(lo), amax8_bf16(hi)), gs, sv);
        const uint32_t q0 = nvfp4_codes(lo, gs, sv), q1 = nvfp4_codes(hi, gs, sv);
        uint8_t* o = p.out + r * p.out_stride + b * 8;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            o[k] = (uint8_t)(q0 >> (8 * k));
            o[4 + k] = (uint8_t)(q1 >> (8 * k));
        }
        p.sf[nvfp4_sf_offset(r, b, p.sf_col_tiles)] = (uint8_t)sc;
    }
}

cudaError_t launch_quant_nvfp4(const QuantFp4Params& p, cudaStream_t s) {
    const int64_t total = p.rows * (p.D / 16);
    const int grid = grid_for_rows(reinterpret_cast<const void*>(quant_nvfp4_kernel), (total + kBlock - 1) / kBlock, 1, kBlock);
    if (grid < 0) return cudaErrorUnknown;
    return launch_pdl(quant_nvfp4_kernel, grid, kBlock, 0, s, p);
}

}  // namespace mbx
