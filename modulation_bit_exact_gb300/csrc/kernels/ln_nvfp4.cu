// ln_nvfp4.cu -- the NVFP4 producers: LayerNorm + AdaLN (and the gated
// residual form) writing the bf16 result and its NVFP4 copy in the ring
// kernel's store pass (instantiated here with FP4 = true, apart from the
// plain kernels), or, for rows the ring kernel does not take, from the written
// bf16 output by the separate quantiser.
//
// "Agent-assisted SGLang diffusion kernel optimisation: Qwen-Image, FLUX.2 and
// video models" (tahou.com), section 将FP8量化融合到前序算子, NVFP4 part: the
// residual update, layer_norm and (1 + scale)/shift chain ending in
// fp4_quantize, one kernel writing E2M1 packed values and 128x4-swizzled E4M3
// block scales.  The block rule and the tile order are stated with
// mbx_ln_modulate_nvfp4 in the public header.
#include "ln_pipe.cuh"

namespace mbx {

static cudaError_t quantise_out_fp4(const LnModParams& p, cudaStream_t s) {
    QuantFp4Params q;
    q.out = p.out_fp4;
    q.out_stride = p.out_fp4_stride;
    q.sf = p.out_sf;
    q.sf_col_tiles = p.sf_col_tiles;
    q.y = p.out;
    q.y_stride = p.out_stride;
    q.rows = p.rows;
    q.D = p.D;
    q.gs = p.fp4_scale;
    return launch_quant_nvfp4(q, s);
}

cudaError_t launch_ln_modulate_nvfp4(const LnModParams& p, bool vec, bool high, cudaStream_t s) {
    if (vec) return launch_pipe_d<false, true>(p, high, s);
    return launch_all_or_none([&]() {
        LnModParams q = p;
        q.out_fp4 = nullptr;
        const cudaError_t e = launch_ln_modulate(q, false, high, s);
        return e != cudaSuccess ? e : quantise_out_fp4(p, s);
    });
}

cudaError_t launch_gated_residual_ln_modulate_nvfp4(const LnModParams& p, bool vec, bool high, cudaStream_t s) {
    if (vec && fused_fits(p, high, true)) return launch_pipe_d<true, true>(p, high, s);
    if (vec) {  // rows too wide for the fused ring: gated add, then the NVFP4 LN pass
        return launch_all_or_none([&]() {
            LnModParams q;
            const cudaError_t e = launch_gated_add_part(p, true, s, &q);
            return e != cudaSuccess ? e : launch_pipe_d<false, true>(q, high, s);
        });
    }
    return launch_all_or_none([&]() {
        LnModParams q = p;
        q.out_fp4 = nullptr;
        const cudaError_t e = launch_gated_residual_ln_modulate(q, false, high, s);
        return e != cudaSuccess ? e : quantise_out_fp4(p, s);
    });
}

}  // namespace mbx
