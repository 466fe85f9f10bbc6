// launch.h -- internal interface between the C ABI (mbx_api.cu) and the
// kernel translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mbx {

struct LnModParams {
    uint16_t* out;
    int64_t out_stride;
    const uint16_t* x;
    int64_t x_stride;
    const uint16_t* scale;
    int64_t scale_stride;
    const uint16_t* shift;
    int64_t shift_stride;
    int64_t rows;
    int D;
    int64_t seq;  // rows / mod_rows: row r uses modulation row r / seq
    float eps;
    // gated residual front pass (fused entry point only; x is the residual):
    // r' = bf16(x + bf16(gate * a)), a = update or bf16(update + bias)
    const uint16_t* update = nullptr;
    int64_t update_stride = 0;
    const uint16_t* gate = nullptr;
    int64_t gate_stride = 0;
    const uint16_t* bias = nullptr;  // [D] or null
    uint16_t* res_out = nullptr;
    int64_t res_out_stride = 0;
    // -0.0f as a kernel argument: the packed Welford update takes its product
    // as fma(d, t, neg_zero), which the compiler cannot turn into a multiply
    float neg_zero = -0.0f;
    // static E4M3 copy of out (the FP8 producers): q = e4m3(out * (1/scale))
    uint8_t* out_fp8 = nullptr;
    int64_t out_fp8_stride = 0;
    const float* fp8_scale = nullptr;  // device, one per-tensor scale
    // NVFP4 copy of out (16-element blocks): packed E2M1 [rows, D/2] bytes and
    // E4M3 block scales in the 128x4 tile layout (sf_col_tiles tiles per row band)
    uint8_t* out_fp4 = nullptr;
    int64_t out_fp4_stride = 0;
    uint8_t* out_sf = nullptr;
    int sf_col_tiles = 0;
    const float* fp4_scale = nullptr;  // device, the per-tensor global scale
};

// NVFP4 copy of a bf16 matrix (the same definition as the LN kernel's store).
struct QuantFp4Params {
    uint8_t* out;
    int64_t out_stride;
    uint8_t* sf;
    int sf_col_tiles;
    const uint16_t* y;
    int64_t y_stride;
    int64_t rows;
    int D;
    const float* gs;
};
cudaError_t launch_quant_nvfp4(const QuantFp4Params& p, cudaStream_t s);

// Static E4M3 copy of a bf16 matrix: out[r][e] = e4m3(y[r][e] * (1/scale)).
struct QuantParams {
    uint8_t* out;
    int64_t out_stride;
    const uint16_t* y;
    int64_t y_stride;
    int64_t rows;
    int D;
    const float* scale;
};
cudaError_t launch_quant_e4m3(const QuantParams& p, cudaStream_t s);

struct RmsScaleParams {
    uint16_t* out;
    int64_t out_stride;
    const uint16_t* x;
    int64_t x_stride;
    const uint16_t* weight;
    const uint16_t* scale;
    int64_t scale_stride;
    int64_t rows;
    int D;
    int64_t seq;
    float eps;
};

struct RmsTanhParams {
    uint16_t* out;
    int64_t out_stride;
    const uint16_t* x;
    int64_t x_stride;
    const uint16_t* gate;
    int64_t gate_stride;
    const uint16_t* residual;
    int64_t res_stride;
    const uint16_t* weight;
    int64_t rows;
    int D;
    int64_t seq;
    float eps;
};

struct GateAddParams {
    uint16_t* out;
    int64_t out_stride;
    const uint16_t* x;
    int64_t x_stride;
    const uint16_t* gate;
    int64_t gate_stride;
    const uint16_t* y;
    int64_t y_stride;
    int64_t rows;
    int D;
    int64_t seq;
    const uint16_t* bias = nullptr;  // internal: y is replaced by bf16(y + bias) when set
};

// Exact unsigned division by a runtime constant for numerators below 2^31
// (Granlund & Montgomery, PLDI 1994): q = (n * m) >> shift with
// shift = 31 + ceil(log2 d) and m = ceil(2^shift / d).
struct FastDiv {
    unsigned long long m;
    unsigned shift;
};
inline FastDiv make_fastdiv(unsigned d) {
    unsigned l = 0;
    while ((1ull << l) < d) ++l;
    FastDiv f;
    f.shift = 31 + l;
    f.m = ((1ull << f.shift) + d - 1) / d;
    return f;
}

struct QkvParams {
    uint16_t* joint;
    const uint16_t* txt;
    int64_t txt_stride;
    const uint16_t* img;
    int64_t img_stride;
    int64_t s_txt, s_img, batch;
    int heads, head_dim;
    const uint16_t *wq_txt, *wk_txt, *wq_img, *wk_img;
    const float *cos_txt, *sin_txt, *cos_img, *sin_img;
    float eps;
    // -0.0f passed at run time: RoPE products are taken as fma(a, b, neg_zero),
    // the correctly rounded product, which the compiler cannot contract with
    // the sum that follows
    float neg_zero = -0.0f;
    // filled by the launcher
    int hpasses;       // head passes per token
    FastDiv by_stot;   // token -> batch index
    FastDiv by_hpass;  // unit -> token
};

// Set while a composed call (several launches for one entry point) runs its
// dispatch once without enqueueing anything: every launch is configured
// (occupancy, shape, shared-memory opt-in) and launch_pdl returns before
// cudaLaunchKernelEx.  One flag per host thread.
inline thread_local bool t_dry_run = false;

struct DryRun {
    bool prev;
    DryRun() : prev(t_dry_run) { t_dry_run = true; }
    ~DryRun() { t_dry_run = prev; }
};

// Run a composed dispatch f() so that a configuration error is reported
// before its first launch is enqueued: f() first runs dry, then for real.
template <class F>
inline cudaError_t launch_all_or_none(F&& f) {
    {
        DryRun dry;
        const cudaError_t e = f();
        if (e != cudaSuccess) return e;
    }
    return f();
}

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel in the stream drains, and calls grid_dep_wait() before
// it touches global memory that kernel may use.
template <class... KArgs, class... Args>
inline cudaError_t launch_pdl(void (*k)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t s,
                              Args... args) {
    if (t_dry_run) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k, args...);
    const cudaError_t last = cudaGetLastError();
    return e != cudaSuccess ? e : last;
}

// ceil(ceil(D / 8) / 128): chunks per lane of a row of D elements.
inline int chunks_per_lane(int D) { return ((D + 7) / 8 + 127) / 128; }

// Persistent grid size: min(ceil(units / units_per_block), SMs x resident
// blocks of `kernel` at `block` threads); -1 if the runtime cannot tell.
int grid_for_rows(const void* kernel, int64_t units, int units_per_block, int block);

// Launch shape of a pipelined row kernel: one CTA per SM, each owning a
// contiguous block of rows_per_cta rows, with as many row groups of `tpr`
// threads as shared memory allows (smem_fixed bytes per CTA plus
// smem_per_group per group), at most 512 threads (and at most 15 groups when
// a group spans several warps: one named barrier each).
struct PipeShape {
    int grid, groups, smem;
    int64_t rows_per_cta;
};
int64_t pipe_rows_per_cta(int64_t rows);
bool pipe_shape(const void* kernel, int tpr, int smem_per_group, int smem_fixed, int64_t rows, PipeShape* out);


// Per-token modulation table: out[k*rows + r][d] = table[k][d] + temb[r][k*D + d].
struct ModTableParams {
    float* out;
    int64_t out_stride;
    const void* table;
    int64_t table_stride;
    bool table_f32;
    const void* temb;
    int64_t temb_stride;
    bool temb_f32;
    int64_t rows;
    int D;
    FastDiv by_nch;  // chunk index within a token row -> plane k (vector path)
};
cudaError_t launch_modulation_table_add(const ModTableParams& p, bool vec, cudaStream_t s);

cudaError_t launch_ln_modulate(const LnModParams& p, bool vec, bool high, cudaStream_t s);
cudaError_t launch_rmsnorm_scale(const RmsScaleParams& p, bool vec, bool high, cudaStream_t s);
cudaError_t launch_rmsnorm_tanh_residual(const RmsTanhParams& p, bool vec, bool high, cudaStream_t s);
cudaError_t launch_residual_gate_add(const GateAddParams& p, bool vec, bool high, cudaStream_t s);
cudaError_t launch_gated_residual_ln_modulate(const LnModParams& p, bool vec, bool high, cudaStream_t s);
cudaError_t launch_ln_modulate_fp8(const LnModParams& p, bool vec, bool high, cudaStream_t s);
cudaError_t launch_gated_residual_ln_modulate_fp8(const LnModParams& p, bool vec, bool high, cudaStream_t s);
cudaError_t launch_gated_add_part(const LnModParams& p, bool vec, cudaStream_t s, LnModParams* ln);
cudaError_t launch_ln_modulate_nvfp4(const LnModParams& p, bool vec, bool high, cudaStream_t s);
cudaError_t launch_gated_residual_ln_modulate_nvfp4(const LnModParams& p, bool vec, bool high, cudaStream_t s);
cudaError_t launch_qkv_epilogue(const QkvParams& p, bool high, cudaStream_t s);
cudaError_t launch_selftest(int which, unsigned long long* counts, cudaStream_t s);

}  // namespace mbx
