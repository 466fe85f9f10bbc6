/*
 * mbx.h -- C ABI of libmbx.so, bit-exact DiT norm/modulation kernels for GB300
 * (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Tensors are described by views: a 2-D [rows, cols] array of bfloat16 whose
 * last dimension is contiguous and whose rows start `row_stride` elements
 * apart (row_stride >= cols; padding between rows is never read or written).
 * `data` is a device pointer on the CUDA device that is current on the calling
 * thread.  The caller owns every buffer: the library allocates nothing, frees
 * nothing and never synchronises; work is enqueued on `stream` (a
 * cudaStream_t; NULL is the legacy default stream) and the call returns once
 * it is enqueued.
 *
 * Every argument is validated on the host before anything is launched; on
 * any error the call returns a negative MBX_E_* status and launches nothing
 * (mbx_status_string() names it).  The checks are the guard set of the
 * BF16-native RMSNorm wrapper in "#34085 [diffusion] Clean up kernels and
 * shared fast paths" (prhub.com.cn), sections 实现拆解 item 2 and 关键源码片段:
 * one device, all bfloat16, hidden size <= 8192, non-empty, weight of shape
 * [D] and contiguous, flat row stride, rows of x a multiple of the modulation
 * rows.  In addition every view must lie inside one device allocation
 * (MBX_E_BOUNDS), and an output may not overlap an input except where an
 * entry point allows in-place use (MBX_E_ALIAS).
 *
 * Modulation broadcast: a modulation view (scale, shift, gate) has `mod_rows`
 * rows with rows(x) % mod_rows == 0, and row r of x uses modulation row
 * r / (rows(x) / mod_rows): per-sample modulation is mod_rows = batch,
 * per-token modulation is mod_rows = rows(x) (same digest, 关键源码片段:
 * batch = row // seq_len).
 *
 * Variants: MBX_LOSSLESS reproduces, bit for bit, the rounding order of the
 * eager BF16 chain ("Agent-assisted SGLang diffusion kernel optimisation:
 * Qwen-Image, FLUX.2 and video models", tahou.com, section
 * 扩散Kernel对数值精度的敏感性); MBX_HIGH evaluates the same formula in one
 * binary32 pass with a single rounding to bfloat16 at the output (same
 * section: the "plain fusion" the lossless path replaces; same article,
 * section 质量分级机制: the non-lossless quality tiers).
 *
 * Aligned fast path: rows whose start addresses are 16-byte aligned, with
 * cols a multiple of 8, use 128-bit accesses; any other view takes a scalar
 * path with the same arithmetic and order, so results are identical.
 */
#ifndef MBX_H
#define MBX_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MBX_API __attribute__((visibility("default")))
#else
#define MBX_API
#endif

#define MBX_ABI_VERSION 1

/* dtype codes.  Every operation takes bfloat16 operands, except that the
 * modulation-table add also accepts binary32 inputs and writes binary32, and
 * the FP8 producers write an extra FP8 E4M3 (one byte per element) output and
 * the NVFP4 producers packed FP4 E2M1 pairs (MBX_E2M1X2, one byte per two
 * elements) with E4M3 block scales. */
enum { MBX_BF16 = 1, MBX_F32 = 2, MBX_E4M3 = 3, MBX_E2M1X2 = 4 };

/* variant codes */
enum { MBX_LOSSLESS = 0, MBX_HIGH = 1 };

/* status codes */
enum {
    MBX_OK = 0,
    MBX_E_NULL = -1,          /* a required pointer is NULL                       */
    MBX_E_DTYPE = -2,         /* an operand has a dtype the operation does not take */
    MBX_E_EMPTY = -3,         /* rows or cols is zero (or negative)               */
    MBX_E_DIM_TOO_LARGE = -4, /* cols (hidden size) above 8192                    */
    MBX_E_SHAPE = -5,         /* shapes disagree, or rows % mod_rows != 0         */
    MBX_E_STRIDE = -6,        /* row_stride < cols                                */
    MBX_E_ALIGN = -7,         /* a pointer is not aligned to its element type     */
    MBX_E_ALIAS = -8,         /* an output overlaps an input                      */
    MBX_E_DEVICE = -9,        /* a pointer is not device memory of this device    */
    MBX_E_BOUNDS = -10,       /* a view runs past the end of its allocation       */
    MBX_E_VARIANT = -11,      /* variant is not MBX_LOSSLESS or MBX_HIGH          */
    MBX_E_ARG = -12,          /* another argument is out of range (eps, heads...) */
    MBX_E_CUDA = -13          /* the CUDA runtime reported an error               */
};

/* Read-only view of a [rows, cols] array of `dtype` elements (row_stride in
 * elements). */
typedef struct {
    const void* data;
    int64_t rows;
    int64_t cols;
    int64_t row_stride;
    int32_t dtype;
} mbx_cview;

/* Writable view, same layout rules. */
typedef struct {
    void* data;
    int64_t rows;
    int64_t cols;
    int64_t row_stride;
    int32_t dtype;
} mbx_view;

/*
 * LayerNorm (no affine) fused with AdaLN modulate.
 * Defined in: tahou.com SGLang diffusion article, section
 * 扩散Kernel对数值精度的敏感性 -- y = LN(x); y = y*(1+scale)+shift.
 *   lossless: mean and M2 by Welford over 128 lanes (8-element chunks, chunk c
 *     on lane c mod 128) combined by a fixed halving tree; var = M2/D;
 *     rstd = 1/sqrt(var+eps) (correctly rounded); n = bf16((x-mean)*rstd);
 *     out = bf16(bf16(n * bf16(1+scale)) + shift).
 *   high: the same formula in one binary32 pass, rounded once.
 * out [rows, D]; x [rows, D]; scale, shift [mod_rows, D].  eps >= 0, finite.
 * out must not overlap x, scale or shift.
 */
MBX_API int mbx_ln_modulate(const mbx_view* out, const mbx_cview* x, const mbx_cview* scale,
                            const mbx_cview* shift, float eps, int variant, void* stream);

/*
 * BF16-native RMSNorm times weight times scale.
 * Defined in: prhub.com.cn digest of SGLang PR #34085, section 关键源码片段
 * (rmsnorm_scale): squares rounded to bf16, row sum in binary32 (here over the
 * same 128 lanes and tree as LayerNorm), ms = bf16(sum/D),
 * rstd = bf16(1/sqrt(bf16(ms+eps))), out = bf16(bf16(bf16(x*rstd)*w)*scale).
 * out [rows, D]; x [rows, D]; weight [1, D] contiguous; scale [mod_rows, D].
 */
MBX_API int mbx_rmsnorm_scale(const mbx_view* out, const mbx_cview* x, const mbx_cview* weight,
                              const mbx_cview* scale, float eps, int variant, void* stream);

/*
 * out = residual + tanh(gate) * RMSNorm(x) * weight, BF16-native.
 * Defined in: PR #34085 digest, 实现拆解 item 2 (rmsnorm_tanh_residual);
 * "AI Agent 驱动的 SGLang Kernel 一等公民" (163.com), 3.2 (rmsnorm +
 * tanh(gate)·x + residual).  n = bf16(bf16(x*rstd)*w) with rstd as in
 * mbx_rmsnorm_scale; tg = the bfloat16 nearest to tanh(gate);
 * out = bf16(residual + bf16(tg*n)).
 * out, x, residual [rows, D]; gate [mod_rows, D]; weight [1, D].
 * out may be exactly residual (same pointer and stride) for an in-place
 * residual update; any other overlap is MBX_E_ALIAS.
 */
MBX_API int mbx_rmsnorm_tanh_residual(const mbx_view* out, const mbx_cview* x,
                                      const mbx_cview* gate, const mbx_cview* residual,
                                      const mbx_cview* weight, float eps, int variant,
                                      void* stream);

/*
 * Gated residual add: out = bf16(x + bf16(gate * y)).
 * Defined in: PR #34085 digest, 实现拆解 item 3 (residual_gate_add); 163.com
 * article, 3.2 (residual + gate·update).
 * out, x, y [rows, D]; gate [mod_rows, D].  out may be exactly x (in-place
 * residual update); any other overlap is MBX_E_ALIAS.
 */
MBX_API int mbx_residual_gate_add(const mbx_view* out, const mbx_cview* x, const mbx_cview* gate,
                                  const mbx_cview* y, int variant, void* stream);

/*
 * Gated residual update fused into LayerNorm + AdaLN modulate.
 * Defined in: tahou.com SGLang diffusion article, section
 * Qwen-Image FP8和NVFP4优化 -- residual = residual + gate * (attention + bias);
 * hidden = layer_norm(residual); hidden = hidden * (1 + scale) + shift -- the
 * chain the pages fuse into one producer (here without the FP4 quantisation).
 *   r'  = bf16(residual + bf16(gate * a)), a = update, or bf16(update + bias)
 *   out = the mbx_ln_modulate chain of r' (lossless or high)
 * r' is written to residual_out in both variants with the eager rounding
 * (it is the residual stream the next layer reads); `variant` applies to the
 * norm.  One pass reads residual and update and writes r' and out (8 bytes per
 * element, against 10 for mbx_residual_gate_add then mbx_ln_modulate).
 * residual_out, out, residual, update [rows, D]; gate, scale, shift
 * [mod_rows, D] with the same mod_rows; bias [1, D] or NULL.
 * residual_out may be exactly residual (in-place update of the stream); out
 * overlaps nothing; any other overlap is MBX_E_ALIAS.
 */
MBX_API int mbx_gated_residual_ln_modulate(const mbx_view* residual_out, const mbx_view* out,
                                           const mbx_cview* residual, const mbx_cview* gate,
                                           const mbx_cview* update, const mbx_cview* bias,
                                           const mbx_cview* scale, const mbx_cview* shift,
                                           float eps, int variant, void* stream);

/*
 * FP8 producers: the two LayerNorm + AdaLN entry points above with a second,
 * static E4M3 output.
 * Defined in: tahou.com SGLang diffusion article, section 将FP8量化融合到前序算子
 * -- LayerNorm/AdaLN and gated residual + LayerNorm/AdaLN write the BF16
 * result (kept for the residual branch) and its static-scale E4M3 copy (fed
 * to the next GEMM) in the same pass, instead of a separate quantisation
 * kernel re-reading the BF16 tensor:
 *   out_fp8 = e4m3(float(out) * inv),  inv = 1 / *fp8_scale
 * inv is the correctly rounded binary32 reciprocal (the pages' quantiser
 * takes it with div.full.f32, an approximation; see the design notes), the
 * product is rounded once, and the conversion rounds to nearest even,
 * saturates finite overflow and infinities to +-448 and maps NaN to 0x7F
 * (cvt.rn.satfinite; mbx_selftest(5) checks it against the definition).
 * out_fp8: MBX_E4M3 [rows, D] (row_stride in bytes-as-elements), overlapping
 * nothing.  fp8_scale: device pointer to one binary32 per-tensor scale
 * (caller-owned, read on the stream, so it may change between calls without
 * a sync).  Everything else as in mbx_ln_modulate /
 * mbx_gated_residual_ln_modulate.
 */
MBX_API int mbx_ln_modulate_fp8(const mbx_view* out, const mbx_view* out_fp8, const mbx_cview* x,
                                const mbx_cview* scale, const mbx_cview* shift,
                                const float* fp8_scale, float eps, int variant, void* stream);
MBX_API int mbx_gated_residual_ln_modulate_fp8(const mbx_view* residual_out, const mbx_view* out,
                                               const mbx_view* out_fp8, const mbx_cview* residual,
                                               const mbx_cview* gate, const mbx_cview* update,
                                               const mbx_cview* bias, const mbx_cview* scale,
                                               const mbx_cview* shift, const float* fp8_scale,
                                               float eps, int variant, void* stream);

/*
 * NVFP4 producers: the two LayerNorm + AdaLN entry points with an NVFP4 copy of
 * the bf16 output -- packed E2M1 values and E4M3 block scales.
 * Defined in: tahou.com SGLang diffusion article, section 将FP8量化融合到前序算子,
 * NVFP4 part -- the gated residual + layer_norm + (1 + scale)/shift chain
 * ending in fp4_quantize, writing E2M1 packed values and 128x4-swizzled E4M3
 * scales in one kernel.  The pages name the output, not the rule; this
 * library's rule (every operation a correctly rounded binary32 operation):
 *   blocks  16 consecutive elements of a row of out; amax = max |out| (NaN
 *           propagates)
 *   scale   s = e4m3(RN(RN(amax * gs) / 6)), gs = *fp4_scale, the per-tensor
 *           global scale (e.g. 448*6 / tensor amax), read on the stream
 *   values  q = e2m1(RN(out * RN(gs / value(s)))), nearest, ties to the code
 *           with mantissa 0, saturating to +-6 (cvt.rn.satfinite; checked by
 *           mbx_selftest(6)); every q of a block whose s is 0 is 0
 *   out_fp4 MBX_E2M1X2 [rows, D/2]: byte i of a row = q[2i] | q[2i+1] << 4
 *   out_sf  MBX_E4M3 [pad128(rows), pad4(D/16)], contiguous: the block scale of
 *           (row r, block b) at byte ((r/128)*(cols/4) + b/4)*512 + (r%32)*16 +
 *           ((r%128)/32)*4 + b%4 (tiles of 128 rows x 4 blocks); padding bytes
 *           are not written
 * D must be a multiple of 16.  No output overlaps another output or an input.
 */
MBX_API int mbx_ln_modulate_nvfp4(const mbx_view* out, const mbx_view* out_fp4, const mbx_view* out_sf,
                                  const mbx_cview* x, const mbx_cview* scale, const mbx_cview* shift,
                                  const float* fp4_scale, float eps, int variant, void* stream);
MBX_API int mbx_gated_residual_ln_modulate_nvfp4(
    const mbx_view* residual_out, const mbx_view* out, const mbx_view* out_fp4, const mbx_view* out_sf,
    const mbx_cview* residual, const mbx_cview* gate, const mbx_cview* update, const mbx_cview* bias,
    const mbx_cview* scale, const mbx_cview* shift, const float* fp4_scale, float eps, int variant,
    void* stream);

/*
 * Per-token modulation table, written in the (6, rows, D) layout.
 * Defined in: tahou.com SGLang diffusion article, section
 * Wan视频模型的数据搬运优化 -- the eager (table.unsqueeze(0) + temb.float())
 * .chunk(6, dim=2) of a Wan block builds a binary32 [B, S, 6, D] temporary and
 * hands out six strided views; here the six chunks are written as contiguous
 * planes with the same binary32 additions:
 *   out[k*rows + r][d] = float(table[k][d]) + float(temb[r][k*D + d]),  k = 0..5
 * table [6, D] and temb [rows, 6*D] (rows = B*S tokens) are MBX_BF16 or
 * MBX_F32 (each widened exactly); out [6*rows, D] is MBX_F32, plane k being
 * rows k*rows .. k*rows + rows - 1 (a contiguous (6, B, S, D) tensor).
 * One addition per element: bit-exact to the eager expression on the GPU.
 * out may not overlap table or temb (MBX_E_ALIAS); 6*D must be below 2^31.
 */
MBX_API int mbx_modulation_table_add(const mbx_view* out, const mbx_cview* table,
                                     const mbx_cview* temb, void* stream);

/*
 * Fused post-GEMM QKV epilogue.
 * Defined in: tahou.com SGLang diffusion article, section 合并QKV投影时的数值问题:
 * after the merged QKV GEMM one kernel does Q/K RMSNorm, interleaved RoPE,
 * the V copy, and writes text and image tokens into one joint QKV buffer,
 * reading the GEMM output through strided views.
 *   txt_qkv [batch*S_txt, 3*H*hd], img_qkv [batch*S_img, 3*H*hd]: columns
 *     [0,H*hd) are Q, [H*hd,2H*hd) K, [2H*hd,3H*hd) V; head h of a part is
 *     its columns [h*hd, (h+1)*hd).  Either branch may have 0 rows (NULL data).
 *   joint [batch*3*H*(S_txt+S_img), hd], contiguous: element
 *     (b, part, h, s, e) at row ((b*3+part)*H+h)*(S_txt+S_img)+s; text tokens
 *     occupy s in [0,S_txt), image tokens [S_txt, S_txt+S_img).
 *   wq_*, wk_* [1, hd]: per-branch Q and K RMSNorm weights.
 *   cos_*, sin_* : binary32 [S, hd/2] per-token tables (device pointers,
 *     16-byte aligned); pair i = (2i, 2i+1) of a head of token s rotates by
 *     (cos[s][i], sin[s][i]): o0 = n0*c - n1*s, o1 = n0*s + n1*c.
 *   lossless: Q/K heads use the mbx_rmsnorm_scale chain without the scale
 *     (n = bf16(bf16(x*rstd)*w)), then o = bf16 of the binary32 rotation.
 *   hd must be 64, 128 or 256; branch rows must be 16-byte aligned;
 *   batch * (S_txt + S_img) * heads must stay below 2^31 (MBX_E_ARG).
 */
MBX_API int mbx_qk_norm_rope_qkv_epilogue(const mbx_view* joint, const mbx_cview* txt_qkv,
                                          const mbx_cview* img_qkv, int64_t batch, int64_t heads,
                                          const mbx_cview* wq_txt, const mbx_cview* wk_txt,
                                          const mbx_cview* wq_img, const mbx_cview* wk_img,
                                          const float* cos_txt, const float* sin_txt,
                                          const float* cos_img, const float* sin_img, float eps,
                                          int variant, void* stream);

/*
 * Validation only: the same checks as the matching entry point, nothing is
 * launched and no stream is touched.  Returns MBX_OK or the status the entry
 * point would return (the "can_use" query of the tahou.com article, section
 * SGLang扩散Kernel的验证流程).
 */
MBX_API int mbx_check_ln_modulate(const mbx_view* out, const mbx_cview* x, const mbx_cview* scale,
                                  const mbx_cview* shift, float eps, int variant);
MBX_API int mbx_check_rmsnorm_scale(const mbx_view* out, const mbx_cview* x,
                                    const mbx_cview* weight, const mbx_cview* scale, float eps,
                                    int variant);
MBX_API int mbx_check_rmsnorm_tanh_residual(const mbx_view* out, const mbx_cview* x,
                                            const mbx_cview* gate, const mbx_cview* residual,
                                            const mbx_cview* weight, float eps, int variant);
MBX_API int mbx_check_residual_gate_add(const mbx_view* out, const mbx_cview* x,
                                        const mbx_cview* gate, const mbx_cview* y, int variant);
MBX_API int mbx_check_ln_modulate_fp8(const mbx_view* out, const mbx_view* out_fp8,
                                      const mbx_cview* x, const mbx_cview* scale,
                                      const mbx_cview* shift, const float* fp8_scale, float eps,
                                      int variant);
MBX_API int mbx_check_gated_residual_ln_modulate_fp8(
    const mbx_view* residual_out, const mbx_view* out, const mbx_view* out_fp8,
    const mbx_cview* residual, const mbx_cview* gate, const mbx_cview* update,
    const mbx_cview* bias, const mbx_cview* scale, const mbx_cview* shift,
    const float* fp8_scale, float eps, int variant);
MBX_API int mbx_check_ln_modulate_nvfp4(const mbx_view* out, const mbx_view* out_fp4,
                                        const mbx_view* out_sf, const mbx_cview* x,
                                        const mbx_cview* scale, const mbx_cview* shift,
                                        const float* fp4_scale, float eps, int variant);
MBX_API int mbx_check_gated_residual_ln_modulate_nvfp4(
    const mbx_view* residual_out, const mbx_view* out, const mbx_view* out_fp4, const mbx_view* out_sf,
    const mbx_cview* residual, const mbx_cview* gate, const mbx_cview* update, const mbx_cview* bias,
    const mbx_cview* scale, const mbx_cview* shift, const float* fp4_scale, float eps, int variant);
MBX_API int mbx_check_modulation_table_add(const mbx_view* out, const mbx_cview* table,
                                           const mbx_cview* temb);
MBX_API int mbx_check_gated_residual_ln_modulate(const mbx_view* residual_out,
                                                 const mbx_view* out, const mbx_cview* residual,
                                                 const mbx_cview* gate, const mbx_cview* update,
                                                 const mbx_cview* bias, const mbx_cview* scale,
                                                 const mbx_cview* shift, float eps, int variant);
MBX_API int mbx_check_qk_norm_rope_qkv_epilogue(
    const mbx_view* joint, const mbx_cview* txt_qkv, const mbx_cview* img_qkv, int64_t batch,
    int64_t heads, const mbx_cview* wq_txt, const mbx_cview* wk_txt, const mbx_cview* wq_img,
    const mbx_cview* wk_img, const float* cos_txt, const float* sin_txt, const float* cos_img,
    const float* sin_img, float eps, int variant);

/*
 * Exhaustive self-test of the kernels' arithmetic building blocks against the
 * GPU's own correctly rounded binary32 operations (no counterpart on the
 * pages; it backs the bit-exactness of the lossless paths):
 *   which = 0: division by each Welford count k = 1..64 (the kernels'
 *              multiply by a two-word reciprocal, one multiply and one
 *              fused multiply-add) vs div.rn, for every finite binary32
 *              numerator;
 *   which = 1: the bfloat16-pair multiply vs binary32 multiply + round, for
 *              every pair of bfloat16 operands;
 *   which = 2: the bfloat16-pair add vs binary32 add + round, every pair;
 *   which = 3: the unguarded division the kernels use for lanes whose
 *              elements all have |x| >= 2^-60, vs div.rn, for every count
 *              k = 1..64 and every binary32 numerator with |d| >= 2^-100,
 *              and +0;
 *   which = 4: the reciprocal-square-root table of the QKV epilogue vs
 *              bf16(div.rn(1, sqrt.rn(v))) for every non-negative bfloat16 v
 *              (finite and +inf);
 *   which = 5: the hardware binary32 -> FP8 E4M3 conversion used by the FP8
 *              producers vs the E4M3 definition (nearest even, saturation
 *              to +-448, NaN -> 0x7F) for every binary32 pattern; the second
 *              counter holds NaN inputs whose byte is not 0x7F;
 *   which = 6: the hardware binary32 -> FP4 E2M1 conversion used by the
 *              NVFP4 producers vs the E2M1 definition (nearest, ties to the
 *              code with mantissa 0, saturation to +-6) for every binary32
 *              pattern; the second counter holds NaN inputs whose code is
 *              not 0x7.
 * counts: device pointer to 2 uint64 counters (caller-owned), overwritten
 * with {mismatches between non-NaN results, mismatches where either is NaN}.
 * Enqueued on `stream`; the caller synchronises before reading counts.
 */
MBX_API int mbx_selftest(int which, unsigned long long* counts, void* stream);

/* Static name of a status code ("MBX_OK", "MBX_E_SHAPE: ..."). */
MBX_API const char* mbx_status_string(int status);

/* MBX_ABI_VERSION of the loaded library. */
MBX_API int mbx_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MBX_H */
