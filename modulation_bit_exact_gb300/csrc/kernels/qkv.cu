// qkv.cu -- fused post-GEMM QKV epilogue.
//
// "Agent-assisted SGLang diffusion kernel optimisation: Qwen-Image, FLUX.2 and
// video models" (tahou.com), section 合并QKV投影时的数值问题: after the merged
// QKV GEMM one kernel performs (1) Q/K RMSNorm, (2) interleaved RoPE, (3) the
// V copy and (4) writes text and image tokens into the joint QKV buffer,
// reading the GEMM output through strided row views, so no intermediate
// tensor is materialised.
//
// Work decomposition: a CTA owns one token at a time (persistent loop over
// tokens).  Its threads form `slots` head units of hd/8 threads; thread l of a
// unit holds the 8-element chunk l of the head, which is also logical lane l
// of the 128-lane order (a head has at most 32 chunks, so the levels s >= 32
// of the fixed tree only add empty lanes and the remaining levels are warp
// shuffles within the unit).  All three parts of the token are loaded before
// any is processed; every warp works on heads of a single part, so the
// shuffles of a Q/K head never meet a V unit.
//
// Lossless Q/K head: the BF16-native RMSNorm chain without the scale
// (sq = bf16(x*x), S over the lanes, ms = bf16(S/hd),
// rstd = bf16(1/sqrt(bf16(ms+eps))), n = bf16(bf16(x*rstd)*w)), then for each
// pair (2i, 2i+1): o0 = bf16(n0*c - n1*s), o1 = bf16(n0*s + n1*c) in binary32
// with c, s the token's table entries for pair i.  V is a bit copy.
#include "launch.h"
#include "rowops.cuh"

namespace mbx {

__device__ __forceinline__ float4 ld_f4(const float* p) {
    float4 v;
    asm volatile("ld.global.nc.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

template <int TPH, bool HIGH>
__global__ void __launch_bounds__(1024) qkv_epilogue_kernel(QkvParams p) {
    constexpr int HD = TPH * kChunk;
    const int l = threadIdx.x % TPH;     // chunk / lane within the head
    const int slot = threadIdx.x / TPH;  // head unit within the CTA
    const int slots = blockDim.x / TPH;
    const int H = p.heads;
    const int64_t s_tot = p.s_txt + p.s_img;
    const int64_t tokens = p.batch * s_tot;
    const int hpasses = (H + slots - 1) / slots;
    const int64_t part_stride = (int64_t)H * HD;  // columns between Q, K and V

    for (int64_t tok = blockIdx.x; tok < tokens; tok += gridDim.x) {
        const int64_t b = tok / s_tot;
        const int64_t s = tok - b * s_tot;  // position in the joint sequence
        const bool txt = s < p.s_txt;
        const int64_t sb = txt ? s : s - p.s_txt;  // position within the branch
        const uint16_t* src = txt ? p.txt + (b * p.s_txt + sb) * p.txt_stride
                                  : p.img + (b * p.s_img + sb) * p.img_stride;
        const float* cos_row = (txt ? p.cos_txt : p.cos_img) + sb * (HD / 2);
        const float* sin_row = (txt ? p.sin_txt : p.sin_img) + sb * (HD / 2);
        const uint16_t* wq = txt ? p.wq_txt : p.wq_img;
        const uint16_t* wk = txt ? p.wk_txt : p.wk_img;

        for (int hp = 0; hp < hpasses; ++hp) {
            const int h = hp * slots + slot;
            const bool active = h < H;
            // all three parts of this head first (more bytes in flight)
            uint4 xv[3];
#pragma unroll
            for (int part = 0; part < 3; ++part)
                xv[part] = active ? ld_stream(src + part * part_stride + (int64_t)h * HD + l * kChunk)
                                  : make_uint4(0, 0, 0, 0);
            const float4 c4 = ld_f4(cos_row + 4 * l);
            const float4 s4 = ld_f4(sin_row + 4 * l);
#pragma unroll
            for (int part = 0; part < 3; ++part) {
                uint16_t* dst = p.joint + ((((b * 3 + part) * H + h) * s_tot + s) * HD) + l * kChunk;
                if (part == 2) {
                    if (active) st_v4(dst, xv[2]);
                    continue;
                }
                const uint4 x = xv[part];
                const uint4 w = ld_shared_row((part == 0 ? wq : wk) + l * kChunk);
                // lane sum of squares, element order
                float acc = 0.0f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t xw = w_of(x, i);
                    if constexpr (!HIGH) {
                        uint32_t sq = bmul(xw, xw);
                        acc = __fadd_rn(acc, lo_f(sq));
                        acc = __fadd_rn(acc, hi_f(sq));
                    } else {
                        acc = fmaf(lo_f(xw), lo_f(xw), acc);
                        acc = fmaf(hi_f(xw), hi_f(xw), acc);
                    }
                }
#pragma unroll
                for (int sh = TPH / 2; sh >= 1; sh /= 2)
                    acc = __fadd_rn(acc, __shfl_down_sync(0xffffffffu, acc, sh, TPH));
                const float S = __shfl_sync(0xffffffffu, acc, 0, TPH);
                uint4 o;
                if constexpr (!HIGH) {
                    float ms = lo_f(pack_rn(__fdiv_rn(S, (float)HD), 0.0f));
                    float inner = lo_f(pack_rn(__fadd_rn(ms, p.eps), 0.0f));
                    float rstd = lo_f(pack_rn(__fdiv_rn(1.0f, __fsqrt_rn(inner)), 0.0f));
                    const uint32_t r2 = bf16_bits(rstd);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t n = bmul(bmul(w_of(x, i), r2), w_of(w, i));
                        float c = i == 0 ? c4.x : i == 1 ? c4.y : i == 2 ? c4.z : c4.w;
                        float sn = i == 0 ? s4.x : i == 1 ? s4.y : i == 2 ? s4.z : s4.w;
                        // two roundings per product, one per sum: scalar
                        // intrinsics, never merged into a fused multiply-add
                        const float n0 = lo_f(n), n1 = hi_f(n);
                        const float o0 = __fsub_rn(__fmul_rn(n0, c), __fmul_rn(n1, sn));
                        const float o1 = __fadd_rn(__fmul_rn(n0, sn), __fmul_rn(n1, c));
                        w_set(o, i, pack_rn(o0, o1));
                    }
                } else {
                    float rstd = rsqrtf(S / (float)HD + p.eps);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t xw = w_of(x, i), ww = w_of(w, i);
                        float n0 = lo_f(xw) * rstd * lo_f(ww), n1 = hi_f(xw) * rstd * hi_f(ww);
                        float c = i == 0 ? c4.x : i == 1 ? c4.y : i == 2 ? c4.z : c4.w;
                        float sn = i == 0 ? s4.x : i == 1 ? s4.y : i == 2 ? s4.z : s4.w;
                        w_set(o, i, pack_rn(fmaf(n0, c, -n1 * sn), fmaf(n0, sn, n1 * c)));
                    }
                }
                if (active) st_v4(dst, o);
            }
        }
    }
}

template <int TPH, bool HIGH>
static cudaError_t launch_one(const QkvParams& p, cudaStream_t s) {
    auto k = qkv_epilogue_kernel<TPH, HIGH>;
    int slots = p.heads < 1024 / TPH ? (int)p.heads : 1024 / TPH;
    int block = slots * TPH;
    if (block % 32) block += 32 - block % 32;  // whole warps (extra units idle)
    int grid = grid_for_rows(reinterpret_cast<const void*>(k), p.batch * (p.s_txt + p.s_img), 1, block);
    if (grid < 0) return cudaErrorUnknown;
    k<<<grid, block, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_qkv_epilogue(const QkvParams& p, bool high, cudaStream_t s) {
    switch (p.head_dim) {
        case 64: return high ? launch_one<8, true>(p, s) : launch_one<8, false>(p, s);
        case 128: return high ? launch_one<16, true>(p, s) : launch_one<16, false>(p, s);
        case 256: return high ? launch_one<32, true>(p, s) : launch_one<32, false>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mbx
