/*
 * mbx_oracle.c -- plain, slow CPU oracle for the DiT norm/modulation path.
 *
 * TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the CPU
 * baseline leg of the benchmark are the only callers.  The product path (the
 * CUDA library and its Python binding) never loads, links or calls this file,
 * and this file shares no code, header or table with it.
 *
 * What is computed, and where it is defined:
 *   [AdaLN]   "Agent-assisted SGLang diffusion kernel optimisation: Qwen-Image,
 *             FLUX.2 and video models" (tahou.com), section 扩散Kernel对数值精度
 *             的敏感性 ("numerical sensitivity of diffusion kernels"): y = LN(x);
 *             y = y*(1+scale)+shift, rounded to BF16 at the same points as the
 *             eager chain; the bit-exact LN uses a 128-thread Welford, a fixed
 *             shuffle tree, div.rn and a reciprocal-square-root step.
 *   [RMS]     "#34085 [diffusion] Clean up kernels and shared fast paths"
 *             (prhub.com.cn), section 关键源码片段 (key source excerpts): the
 *             BF16-native rmsnorm_scale rounding points; section 实现拆解 item 2:
 *             rmsnorm_tanh_residual and the guard set; item 3: residual_gate_add.
 *   [QKV]     tahou.com article, section 合并QKV投影时的数值问题 (merged QKV
 *             projection): Q/K RMSNorm, interleaved RoPE, V copy, text and image
 *             tokens written into one joint QKV buffer.
 *   [FP8]     tahou.com article, section 将FP8量化融合到前序算子 (fusing FP8
 *             quantisation into the producer): LayerNorm/AdaLN and gated
 *             residual + LayerNorm/AdaLN write a BF16 output and its static
 *             (per-tensor scale) E4M3 copy.
 *   [FP4]     tahou.com article, section 将FP8量化融合到前序算子, last part (the
 *             NVFP4 path): the gated residual + LN + modulate chain ending in
 *             fp4_quantize, writing packed E2M1 values and 128x4-swizzled E4M3
 *             block scales.  The block-scale rule and the swizzle are not on
 *             the pages; the readings are stated at orc_quant_nvfp4.
 *   [WAN]     tahou.com article, section Wan视频模型的数据搬运优化 (Wan data
 *             movement): the per-token modulation table
 *             (table.unsqueeze(0) + temb.float()).chunk(6, dim=2), written as six
 *             contiguous planes with the same binary32 additions.
 *
 * Readings taken where the pages are silent (each is a definition this oracle
 * owns; the CUDA path must reproduce it bit for bit):
 *   R1  bf16(v): IEEE binary32 -> bfloat16, round to nearest, ties to even, on
 *       the bit pattern; overflow goes to +-inf; subnormals are kept; every NaN
 *       becomes the canonical NaN 0x7FFF (the result of the GPU's own
 *       binary32->bf16 conversion, which is what an eager chain on the GPU
 *       stores).
 *   R2  The 128-lane ownership: chunk c = floor(e/8) belongs to lane c mod 128;
 *       a lane visits its chunks in ascending order and the elements of a
 *       chunk in ascending order.
 *   R3  The fixed tree: for s = 64,32,16,8,4,2,1 and every lane l < s,
 *       L[l] = combine(L[l], L[l+s]).
 *   R4  Welford step: n += 1; d = x - mean; mean += d / n; M2 += d*(x - mean).
 *       Chan combine with r = nB/n; an empty side is an exact identity.
 *   R5  var = M2 / D (biased); rstd = 1 / sqrt(var + eps), each correctly
 *       rounded (sqrt then divide, no approximate reciprocal square root).
 *   R6  RMSNorm sums bf16(x*x) in binary32 over the same lanes and tree.
 *   R7  tanh_bf16(g) is the bfloat16 nearest to the exact tanh(g).
 *
 * Every floating-point operation here is a single IEEE-754 binary32 (or, in the
 * *_f64 references, binary64) operation rounded to nearest-even.  This file
 * must be compiled with -ffp-contract=off and without fast-math: no multiply
 * and add may be fused.  orc_probe_mul_add() lets a test confirm that.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_LANES 128
#define ORC_CHUNK 8

/* ------------------------------------------------------------------------ */
/* bfloat16 <-> binary32                                                    */
/* ------------------------------------------------------------------------ */

/* Widen a bfloat16 bit pattern to binary32 (exact). */
static float f_of(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Reading R1: round a binary32 to bfloat16, nearest-even, on the bit pattern. */
static uint16_t bf16_of(float v) {
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fff; /* any NaN */
    uint32_t hi = u >> 16;     /* truncated result (sign, exponent, 7 bits) */
    uint32_t lo = u & 0xffffu; /* discarded bits                            */
    /* Magnitude rounding: up when above the halfway point, or exactly at it
     * with an odd kept part.  A carry out of the mantissa moves to the next
     * binade, and from the largest finite value to infinity. */
    if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u;
    return (uint16_t)hi;
}

/* bf16 -> binary32 -> bf16 helpers used in the eager chains. */
static float fb(float v) { return f_of(bf16_of(v)); }

void orc_f32_to_bf16(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_of(in[i]);
}

void orc_bf16_to_f32(const uint16_t* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = f_of(in[i]);
}

/* a*b + c exactly as every product-then-sum below is evaluated.  With the
 * required flags this is two roundings; a fused multiply-add would give one. */
float orc_probe_mul_add(float a, float b, float c) { return a * b + c; }

/* ------------------------------------------------------------------------ */
/* Welford-128 statistics (readings R2-R4)                                  */
/* ------------------------------------------------------------------------ */

typedef struct {
    float mean;
    float m2;
    float n; /* element count, an exact small integer */
} welford_t;

static void welford_push(welford_t* w, float x) {
    w->n = w->n + 1.0f;
    float d = x - w->mean;
    w->mean = w->mean + d / w->n;
    w->m2 = w->m2 + d * (x - w->mean);
}

/* Chan et al. pairwise combine; a keeps the lower lane index. */
static welford_t welford_combine(welford_t a, welford_t b) {
    if (b.n == 0.0f) return a;
    if (a.n == 0.0f) return b;
    welford_t c;
    c.n = a.n + b.n;
    float d = b.mean - a.mean;
    float r = b.n / c.n;
    c.mean = a.mean + d * r;
    c.m2 = (a.m2 + b.m2) + (d * d) * (a.n * r);
    return c;
}

/* Statistics of one row of D bf16 values under the fixed 128-lane order. */
void orc_welford128(const uint16_t* x, int64_t D, float* mean, float* m2, float* n) {
    welford_t L[ORC_LANES];
    for (int l = 0; l < ORC_LANES; ++l) {
        L[l].mean = 0.0f;
        L[l].m2 = 0.0f;
        L[l].n = 0.0f;
        for (int64_t c = l; c * ORC_CHUNK < D; c += ORC_LANES)
            for (int64_t e = c * ORC_CHUNK; e < c * ORC_CHUNK + ORC_CHUNK && e < D; ++e)
                welford_push(&L[l], f_of(x[e]));
    }
    for (int s = ORC_LANES / 2; s >= 1; s /= 2)
        for (int l = 0; l < s; ++l) L[l] = welford_combine(L[l], L[l + s]);
    *mean = L[0].mean;
    *m2 = L[0].m2;
    *n = L[0].n;
}

/* Reading R6: binary32 sum of bf16(x*x) over the same lanes and tree. */
void orc_sum128_sq(const uint16_t* x, int64_t D, float* sum) {
    float L[ORC_LANES];
    for (int l = 0; l < ORC_LANES; ++l) {
        L[l] = 0.0f;
        for (int64_t c = l; c * ORC_CHUNK < D; c += ORC_LANES)
            for (int64_t e = c * ORC_CHUNK; e < c * ORC_CHUNK + ORC_CHUNK && e < D; ++e) {
                float v = f_of(x[e]);
                L[l] = L[l] + fb(v * v);
            }
    }
    for (int s = ORC_LANES / 2; s >= 1; s /= 2)
        for (int l = 0; l < s; ++l) L[l] = L[l] + L[l + s];
    *sum = L[0];
}

/* Reading R5: (mean, rstd) of a LayerNorm row. */
static void ln_row_stats(const uint16_t* x, int64_t D, float eps, float* mean, float* rstd) {
    float m2, n;
    orc_welford128(x, D, mean, &m2, &n);
    float var = m2 / (float)D;
    *rstd = 1.0f / sqrtf(var + eps);
}

/* The BF16-native RMSNorm scalar: rstd = bf16(1/sqrt(bf16(bf16(S/D) + eps))). */
static float rms_row_rstd(const uint16_t* x, int64_t D, float eps) {
    float S;
    orc_sum128_sq(x, D, &S);
    float ms = fb(S / (float)D);
    float inner = fb(ms + eps);
    return fb(1.0f / sqrtf(inner));
}

/* ------------------------------------------------------------------------ */
/* Operations                                                               */
/* ------------------------------------------------------------------------ */

/* Row r of a [rows, D] tensor uses modulation row r / (rows / mod_rows). */
static int64_t mod_row(int64_t r, int64_t rows, int64_t mod_rows) {
    return r / (rows / mod_rows);
}

/* LayerNorm (no affine) + AdaLN modulate, bit-exact eager chain [AdaLN]:
 *   n   = bf16((x - mean) * rstd)          BF16 store between LN and modulate
 *   t   = bf16(1 + scale)
 *   u   = bf16(n * t)
 *   out = bf16(u + shift)                                                    */
void orc_ln_modulate(uint16_t* out, int64_t out_stride, const uint16_t* x, int64_t x_stride,
                     int64_t rows, int64_t D, const uint16_t* scale, int64_t scale_stride,
                     const uint16_t* shift, int64_t shift_stride, int64_t mod_rows, float eps) {
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* xr = x + r * x_stride;
        int64_t m = mod_row(r, rows, mod_rows);
        const uint16_t* sc = scale + m * scale_stride;
        const uint16_t* sh = shift + m * shift_stride;
        float mean, rstd;
        ln_row_stats(xr, D, eps, &mean, &rstd);
        for (int64_t e = 0; e < D; ++e) {
            float n = fb((f_of(xr[e]) - mean) * rstd);
            float t = fb(1.0f + f_of(sc[e]));
            float u = fb(n * t);
            out[r * out_stride + e] = bf16_of(u + f_of(sh[e]));
        }
    }
}

/* BF16-native RMSNorm * weight * scale [RMS]:
 *   out = bf16(bf16(bf16(x * rstd) * w) * scale)                             */
void orc_rmsnorm_scale(uint16_t* out, int64_t out_stride, const uint16_t* x, int64_t x_stride,
                       int64_t rows, int64_t D, const uint16_t* weight, const uint16_t* scale,
                       int64_t scale_stride, int64_t mod_rows, float eps) {
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* xr = x + r * x_stride;
        const uint16_t* sc = scale + mod_row(r, rows, mod_rows) * scale_stride;
        float rstd = rms_row_rstd(xr, D, eps);
        for (int64_t e = 0; e < D; ++e) {
            float a = fb(f_of(xr[e]) * rstd);
            float b = fb(a * f_of(weight[e]));
            out[r * out_stride + e] = bf16_of(b * f_of(sc[e]));
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Correctly rounded bfloat16 tanh (reading R7)                             */
/* ------------------------------------------------------------------------ */

/* Round a binary64 value in the normal bfloat16 range to bfloat16,
 * nearest-even, directly (no intermediate binary32 rounding). */
static uint16_t bf16_of_double_normal(double v) {
    uint64_t u;
    memcpy(&u, &v, sizeof u);
    uint64_t sign = u >> 63;
    uint64_t mag = u & 0x7fffffffffffffffull;
    /* keep 1 + 7 significand bits: drop the low 45 of the 52-bit fraction */
    uint64_t kept = mag >> 45;
    uint64_t rest = mag & ((1ull << 45) - 1);
    uint64_t half = 1ull << 44;
    if (rest > half || (rest == half && (kept & 1ull))) kept += 1;
    /* kept is the binary64 pattern >> 45; rebuild and narrow exactly */
    uint64_t back = kept << 45;
    double d;
    memcpy(&d, &back, sizeof d);
    float f = (float)d; /* exact: d has 8 significant bits, in float range */
    uint32_t fu;
    memcpy(&fu, &f, sizeof fu);
    return (uint16_t)((fu >> 16) | (uint32_t)(sign << 15));
}

/* tanh_bf16(g): the bfloat16 nearest to tanh(g).  For |g| < 2^-8 the answer is
 * g itself: |tanh(g) - g| <= |g|^3/3 < 2^-10 |g|, below half the bfloat16 gap
 * under |g| (this also covers zeros and subnormals).  Otherwise tanh is
 * evaluated in binary64 and rounded once. */
static uint16_t tanh_bf16(uint16_t g) {
    uint32_t a = g & 0x7fffu;
    if (a > 0x7f80u) return 0x7fff;                  /* NaN */
    if (a == 0x7f80u) return (g & 0x8000u) | 0x3f80u; /* +-inf -> +-1 */
    float x = f_of(g);
    if (fabsf(x) < 0.00390625f) return g;
    return bf16_of_double_normal(tanh((double)x));
}

void orc_tanh_bf16_table(uint16_t* table) {
    for (uint32_t g = 0; g < 65536u; ++g) table[g] = tanh_bf16((uint16_t)g);
}

/* RMSNorm -> tanh-gated residual [RMS], BF16-native:
 *   n   = bf16(bf16(x * rstd) * w)
 *   p   = bf16(tanh_bf16(g) * n)
 *   out = bf16(r + p)                                                        */
void orc_rmsnorm_tanh_residual(uint16_t* out, int64_t out_stride, const uint16_t* x,
                               int64_t x_stride, int64_t rows, int64_t D, const uint16_t* gate,
                               int64_t gate_stride, int64_t gate_rows, const uint16_t* residual,
                               int64_t res_stride, const uint16_t* weight, float eps) {
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* xr = x + r * x_stride;
        const uint16_t* gr = gate + mod_row(r, rows, gate_rows) * gate_stride;
        const uint16_t* rr = residual + r * res_stride;
        float rstd = rms_row_rstd(xr, D, eps);
        for (int64_t e = 0; e < D; ++e) {
            float a = fb(f_of(xr[e]) * rstd);
            float n = fb(a * f_of(weight[e]));
            float p = fb(f_of(tanh_bf16(gr[e])) * n);
            out[r * out_stride + e] = bf16_of(f_of(rr[e]) + p);
        }
    }
}

/* Gated residual add [RMS] item 3:  out = bf16(x + bf16(gate * y)). */
void orc_residual_gate_add(uint16_t* out, int64_t out_stride, const uint16_t* x, int64_t x_stride,
                           int64_t rows, int64_t D, const uint16_t* gate, int64_t gate_stride,
                           int64_t gate_rows, const uint16_t* y, int64_t y_stride) {
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* gr = gate + mod_row(r, rows, gate_rows) * gate_stride;
        for (int64_t e = 0; e < D; ++e) {
            float gy = fb(f_of(gr[e]) * f_of(y[r * y_stride + e]));
            out[r * out_stride + e] = bf16_of(f_of(x[r * x_stride + e]) + gy);
        }
    }
}

/* Gated residual fused into LayerNorm + AdaLN modulate [NVFP4 producer chain]:
 * tahou.com article, section Qwen-Image FP8和NVFP4优化 (the chain PR #37129
 * fuses, without its FP4 quantisation):
 *   a   = update, or bf16(update + bias) when a bias row is given
 *   r'  = bf16(residual + bf16(gate * a))        the new residual stream
 *   out = the LN + modulate chain of orc_ln_modulate applied to r'
 * gate, scale and shift share mod_rows.  Writes r' and out. */
void orc_gated_residual_ln_modulate(uint16_t* res_out, uint16_t* out, const uint16_t* residual,
                                    int64_t res_stride, int64_t rows, int64_t D,
                                    const uint16_t* update, int64_t upd_stride,
                                    const uint16_t* bias, const uint16_t* gate,
                                    int64_t gate_stride, const uint16_t* scale,
                                    int64_t scale_stride, const uint16_t* shift,
                                    int64_t shift_stride, int64_t mod_rows, float eps) {
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* gr = gate + mod_row(r, rows, mod_rows) * gate_stride;
        uint16_t* dst = res_out + r * D;
        for (int64_t e = 0; e < D; ++e) {
            float a = f_of(update[r * upd_stride + e]);
            if (bias) a = fb(a + f_of(bias[e]));
            float ga = fb(f_of(gr[e]) * a);
            dst[e] = bf16_of(f_of(residual[r * res_stride + e]) + ga);
        }
    }
    orc_ln_modulate(out, D, res_out, D, rows, D, scale, scale_stride, shift, shift_stride, mod_rows, eps);
}

/* ------------------------------------------------------------------------ */
/* Static E4M3 quantisation [FP8]                                           */
/* ------------------------------------------------------------------------ */

/* binary32 -> FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits;
 * no infinities; S.1111.111 is NaN; largest finite 448 = 1.75 * 2^8).
 * Round to nearest, ties to even, on the exact value; a finite result beyond
 * 448 and an infinity saturate to +-448 (the "satfinite" conversion of the
 * FP8 producers); every NaN becomes 0x7F.  Signed zeros are kept. */
static uint8_t e4m3_of(float v) {
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7f;
    const uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
    float a = fabsf(v);
    if (a >= 448.0f) return (uint8_t)(sign | 0x7e);
    if (a < 0x1p-6f) {
        /* subnormal range: multiples of 2^-9; 8 * 2^-9 is the smallest normal,
         * whose encoding continues the count (exponent field 1, mantissa 0) */
        float q = rintf(a * 512.0f); /* exact scaling, then nearest-even */
        return (uint8_t)(sign | (uint8_t)q);
    }
    int e;
    frexpf(a, &e); /* a = f * 2^e, f in [0.5, 1): the binade is [2^(e-1), 2^e) */
    e -= 1;
    float q = rintf(ldexpf(a, 3 - e)); /* a / 2^(e-3): 8 <= q <= 16, exact scaling */
    if (q == 16.0f) {
        q = 8.0f;
        e += 1;
    }
    return (uint8_t)(sign | (uint8_t)((e + 7) << 3) | (uint8_t)((int)q - 8));
}

/* The value of an E4M3 code (NaN for 0x7F/0xFF). */
static float e4m3_value(uint8_t c) {
    const int e = (c >> 3) & 0xf, m = c & 7;
    float v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexpf((float)m, -9);
    else v = ldexpf((float)(8 + m), e - 10);
    return (c & 0x80) ? -v : v;
}

void orc_f32_to_e4m3(const float* in, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_of(in[i]);
}

/* The static quantiser applied to a BF16 output: q = e4m3(float(y) * inv) with
 * inv = 1 / scale, a correctly rounded binary32 division (the pages compute
 * it with div.full.f32, an approximation that a CPU cannot reproduce; see the
 * reading in the design notes), and one rounded multiply. */
void orc_quant_e4m3(uint8_t* out, int64_t out_stride, const uint16_t* y, int64_t y_stride,
                    int64_t rows, int64_t D, float scale) {
    const float inv = 1.0f / scale;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t e = 0; e < D; ++e) out[r * out_stride + e] = e4m3_of(f_of(y[r * y_stride + e]) * inv);
}

/* ------------------------------------------------------------------------ */
/* NVFP4 quantisation [FP4]                                                 */
/* ------------------------------------------------------------------------ */

/* binary32 -> FP4 E2M1 code (1 sign bit, 2 exponent bits with bias 1, 1
 * mantissa bit; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; no infinity or NaN).
 * Nearest on the exact value, ties to the even code (mantissa 0); beyond 6
 * (and +-inf) saturates to +-6; NaN gives +6 (0x7).  Signed zero kept. */
static uint8_t e2m1_of(float v) {
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7;
    const uint8_t sign = (uint8_t)((u >> 28) & 0x8u);
    const float a = fabsf(v);
    /* the eight magnitudes and the midpoints between neighbours; at a midpoint
     * the code with mantissa bit 0 (even) wins */
    static const float mag[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
    uint8_t code = 7;
    for (uint8_t c = 0; c < 7; ++c) {
        const float mid = (mag[c] + mag[c + 1]) * 0.5f; /* exact: few significant bits */
        if (a < mid || (a == mid && (c & 1u) == 0)) {
            code = c;
            break;
        }
    }
    return (uint8_t)(sign | code);
}

void orc_f32_to_e2m1(const float* in, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = e2m1_of(in[i]);
}

/* Byte offset of the scale of (row r, block b) in the 128x4-swizzled layout:
 * the [rows, D/16] scale matrix is cut into tiles of 128 rows x 4 blocks (512
 * bytes, tiles in row-major order over the padded matrix); inside a tile, row
 * r sits in one of four 32-row bands, and (r mod 32, band, b mod 4) are laid
 * out in that order (16 bytes per r mod 32). */
int64_t orc_nvfp4_sf_offset(int64_t r, int64_t b, int64_t blocks_per_row) {
    const int64_t col_tiles = (blocks_per_row + 3) / 4;
    const int64_t tile = (r / 128) * col_tiles + b / 4;
    return tile * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (b % 4);
}

/* NVFP4 copy of a bfloat16 output y [rows, D] (D a multiple of 16), with the
 * per-tensor global scale gs (the factor that maps the tensor's range onto
 * E2M1 x E4M3, e.g. 448*6/amax).  Readings (the pages name the output only):
 *   block      16 consecutive elements of a row; amax = max |y| over them
 *   scale      s = e4m3(RN(RN(amax * gs) / 6))           (one E4M3 byte)
 *   elements   q = e2m1(RN(y * RN(gs / float(s))))      (s > 0)
 *              q = 0 for every element of a block whose s is zero
 *   packing    out_fp4[r][i] = q[2i] | q[2i+1] << 4
 *   scales     at orc_nvfp4_sf_offset(r, block); padding bytes untouched
 * Every division and product is one correctly rounded binary32 operation. */
void orc_quant_nvfp4(uint8_t* out_fp4, int64_t fp4_stride, uint8_t* out_sf, const uint16_t* y,
                     int64_t y_stride, int64_t rows, int64_t D, float gs) {
    const int64_t blocks = D / 16;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < blocks; ++b) {
            const uint16_t* blk = y + r * y_stride + b * 16;
            float amax = 0.0f; /* a NaN anywhere makes amax NaN */
            for (int i = 0; i < 16; ++i) {
                const float a = fabsf(f_of(blk[i]));
                if (a != a || amax != amax) amax = NAN;
                else if (a > amax) amax = a;
            }
            const float sf = (amax * gs) / 6.0f;
            const uint8_t s = e4m3_of(sf);
            out_sf[orc_nvfp4_sf_offset(r, b, blocks)] = s;
            const float sv = e4m3_value(s);
            uint8_t* dst = out_fp4 + r * fp4_stride + b * 8;
            for (int i = 0; i < 8; ++i) {
                uint8_t lo = 0, hi = 0;
                if (sv != 0.0f) {
                    const float esc = gs / sv;
                    lo = e2m1_of(f_of(blk[2 * i]) * esc);
                    hi = e2m1_of(f_of(blk[2 * i + 1]) * esc);
                }
                dst[i] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Per-token modulation table [WAN]                                         */
/* ------------------------------------------------------------------------ */

/* Element (r, e) of a bfloat16 (is_f32 == 0) or binary32 row-major matrix,
 * widened exactly to binary32. */
static float elem_f32(const void* base, int is_f32, int64_t stride, int64_t r, int64_t e) {
    if (is_f32) return ((const float*)base)[r * stride + e];
    return f_of(((const uint16_t*)base)[r * stride + e]);
}

/* out[k*rows + r][d] = float(table[k][d]) + float(temb[r][k*D + d]) for the six
 * chunks k = 0..5 of the eager (table.unsqueeze(0) + temb.float()).chunk(6, 2):
 * table [6, D], temb [rows, 6*D] (B*S token rows), out binary32 [6*rows, D]
 * (plane k is rows k*rows .. k*rows + rows - 1).  One binary32 addition per
 * element, in the eager order (table first). */
void orc_modulation_table_add(float* out, int64_t out_stride, const void* table,
                              int64_t table_stride, int table_f32, const void* temb,
                              int64_t temb_stride, int temb_f32, int64_t rows, int64_t D) {
    for (int k = 0; k < 6; ++k)
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t d = 0; d < D; ++d) {
                float t = elem_f32(table, table_f32, table_stride, k, d);
                float e = elem_f32(temb, temb_f32, temb_stride, r, (int64_t)k * D + d);
                out[((int64_t)k * rows + r) * out_stride + d] = t + e;
            }
}

/* ------------------------------------------------------------------------ */
/* Fused QKV epilogue [QKV]                                                 */
/* ------------------------------------------------------------------------ */

/* One head of Q or K: BF16-native RMSNorm (the rmsnorm chain without the
 * scale), then interleaved RoPE on the pairs (2i, 2i+1):
 *   o0 = bf16(n0*c - n1*s),  o1 = bf16(n0*s + n1*c)
 * with c = cosv[i], s = sinv[i] (binary32 table entries).                    */
static void qk_head(uint16_t* dst, const uint16_t* src, int64_t hd, const uint16_t* w,
                    const float* cosv, const float* sinv, float eps) {
    float rstd = rms_row_rstd(src, hd, eps);
    for (int64_t i = 0; i < hd / 2; ++i) {
        float n0 = fb(fb(f_of(src[2 * i]) * rstd) * f_of(w[2 * i]));
        float n1 = fb(fb(f_of(src[2 * i + 1]) * rstd) * f_of(w[2 * i + 1]));
        float c = cosv[i], s = sinv[i];
        dst[2 * i] = bf16_of(n0 * c - n1 * s);
        dst[2 * i + 1] = bf16_of(n0 * s + n1 * c);
    }
}

/* Rows of one branch (text or image): [B * S, 3*H*hd] with row stride
 * `stride`; q = columns [0, H*hd), k = [H*hd, 2*H*hd), v = [2*H*hd, 3*H*hd).
 * Token s of batch b lands at joint[b, part, h, s_off + s, :], where joint is
 * the contiguous [B, 3, H, S_tot, hd] buffer.  Tables are [S, hd/2]. */
static void qkv_branch(uint16_t* joint, int64_t s_tot, int64_t s_off, const uint16_t* src,
                       int64_t stride, int64_t S, int64_t B, int64_t H, int64_t hd,
                       const uint16_t* wq, const uint16_t* wk, const float* cosv,
                       const float* sinv, float eps) {
    for (int64_t b = 0; b < B; ++b)
        for (int64_t s = 0; s < S; ++s) {
            const uint16_t* row = src + (b * S + s) * stride;
            for (int64_t part = 0; part < 3; ++part)
                for (int64_t h = 0; h < H; ++h) {
                    const uint16_t* in = row + (part * H + h) * hd;
                    uint16_t* dst = joint + (((b * 3 + part) * H + h) * s_tot + s_off + s) * hd;
                    if (part == 2) {
                        memcpy(dst, in, (size_t)hd * sizeof(uint16_t)); /* V: bit copy */
                    } else {
                        qk_head(dst, in, hd, part == 0 ? wq : wk, cosv + s * (hd / 2),
                                sinv + s * (hd / 2), eps);
                    }
                }
        }
}

/* Text tokens first (s_off = 0), image tokens after them (s_off = S_txt). */
void orc_qkv_epilogue(uint16_t* joint, const uint16_t* txt, int64_t txt_stride, int64_t s_txt,
                      const uint16_t* img, int64_t img_stride, int64_t s_img, int64_t B,
                      int64_t H, int64_t hd, const uint16_t* wq_txt, const uint16_t* wk_txt,
                      const uint16_t* wq_img, const uint16_t* wk_img, const float* cos_txt,
                      const float* sin_txt, const float* cos_img, const float* sin_img,
                      float eps) {
    int64_t s_tot = s_txt + s_img;
    if (s_txt > 0)
        qkv_branch(joint, s_tot, 0, txt, txt_stride, s_txt, B, H, hd, wq_txt, wk_txt, cos_txt,
                   sin_txt, eps);
    if (s_img > 0)
        qkv_branch(joint, s_tot, s_txt, img, img_stride, s_img, B, H, hd, wq_img, wk_img,
                   cos_img, sin_img, eps);
}

/* ------------------------------------------------------------------------ */
/* Binary64 references for the single-pass "high" variants                  */
/* ------------------------------------------------------------------------ */
/* Each writes the unrounded real-number result (in binary64) and `mag`, the
 * largest magnitude among the terms of the final sum, which sets the scale of
 * the tolerance (a number of bfloat16 ulps of mag). */

void orc_ln_modulate_f64(double* out, double* mag, const uint16_t* x, int64_t x_stride,
                         int64_t rows, int64_t D, const uint16_t* scale, int64_t scale_stride,
                         const uint16_t* shift, int64_t shift_stride, int64_t mod_rows,
                         float eps) {
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* xr = x + r * x_stride;
        int64_t m = mod_row(r, rows, mod_rows);
        double s1 = 0.0, s2 = 0.0;
        for (int64_t e = 0; e < D; ++e) s1 += (double)f_of(xr[e]);
        double mean = s1 / (double)D;
        for (int64_t e = 0; e < D; ++e) {
            double d = (double)f_of(xr[e]) - mean;
            s2 += d * d;
        }
        double rstd = 1.0 / sqrt(s2 / (double)D + (double)eps);
        for (int64_t e = 0; e < D; ++e) {
            double u = ((double)f_of(xr[e]) - mean) * rstd *
                       (1.0 + (double)f_of(scale[m * scale_stride + e]));
            double sh = (double)f_of(shift[m * shift_stride + e]);
            double o = u + sh;
            out[r * D + e] = o;
            double a = fabs(u) > fabs(sh) ? fabs(u) : fabs(sh);
            mag[r * D + e] = a > fabs(o) ? a : fabs(o);
        }
    }
}

static double rms_rstd_f64(const uint16_t* xr, int64_t D, float eps) {
    double s = 0.0;
    for (int64_t e = 0; e < D; ++e) {
        double v = (double)f_of(xr[e]);
        s += v * v;
    }
    return 1.0 / sqrt(s / (double)D + (double)eps);
}

void orc_rmsnorm_scale_f64(double* out, double* mag, const uint16_t* x, int64_t x_stride,
                           int64_t rows, int64_t D, const uint16_t* weight, const uint16_t* scale,
                           int64_t scale_stride, int64_t mod_rows, float eps) {
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* xr = x + r * x_stride;
        const uint16_t* sc = scale + mod_row(r, rows, mod_rows) * scale_stride;
        double rstd = rms_rstd_f64(xr, D, eps);
        for (int64_t e = 0; e < D; ++e) {
            double o = (double)f_of(xr[e]) * rstd * (double)f_of(weight[e]) * (double)f_of(sc[e]);
            out[r * D + e] = o;
            mag[r * D + e] = fabs(o);
        }
    }
}

void orc_rmsnorm_tanh_residual_f64(double* out, double* mag, const uint16_t* x, int64_t x_stride,
                                   int64_t rows, int64_t D, const uint16_t* gate,
                                   int64_t gate_stride, int64_t gate_rows,
                                   const uint16_t* residual, int64_t res_stride,
                                   const uint16_t* weight, float eps) {
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* xr = x + r * x_stride;
        const uint16_t* gr = gate + mod_row(r, rows, gate_rows) * gate_stride;
        double rstd = rms_rstd_f64(xr, D, eps);
        for (int64_t e = 0; e < D; ++e) {
            double p = tanh((double)f_of(gr[e])) * ((double)f_of(xr[e]) * rstd *
                                                    (double)f_of(weight[e]));
            double rv = (double)f_of(residual[r * res_stride + e]);
            double o = rv + p;
            out[r * D + e] = o;
            double a = fabs(p) > fabs(rv) ? fabs(p) : fabs(rv);
            mag[r * D + e] = a > fabs(o) ? a : fabs(o);
        }
    }
}

void orc_residual_gate_add_f64(double* out, double* mag, const uint16_t* x, int64_t x_stride,
                               int64_t rows, int64_t D, const uint16_t* gate, int64_t gate_stride,
                               int64_t gate_rows, const uint16_t* y, int64_t y_stride) {
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* gr = gate + mod_row(r, rows, gate_rows) * gate_stride;
        for (int64_t e = 0; e < D; ++e) {
            double gy = (double)f_of(gr[e]) * (double)f_of(y[r * y_stride + e]);
            double xv = (double)f_of(x[r * x_stride + e]);
            double o = xv + gy;
            out[r * D + e] = o;
            double a = fabs(gy) > fabs(xv) ? fabs(gy) : fabs(xv);
            mag[r * D + e] = a > fabs(o) ? a : fabs(o);
        }
    }
}

/* Q/K heads only (V is a bit copy in both variants): the binary64 value of
 * the normalised, weighted and rotated pair, per element of one head row. */
void orc_qk_head_f64(double* out, double* mag, const uint16_t* src, int64_t hd,
                     const uint16_t* w, const float* cosv, const float* sinv, float eps) {
    double rstd = rms_rstd_f64(src, hd, eps);
    for (int64_t i = 0; i < hd / 2; ++i) {
        double n0 = (double)f_of(src[2 * i]) * rstd * (double)f_of(w[2 * i]);
        double n1 = (double)f_of(src[2 * i + 1]) * rstd * (double)f_of(w[2 * i + 1]);
        double c = (double)cosv[i], s = (double)sinv[i];
        out[2 * i] = n0 * c - n1 * s;
        out[2 * i + 1] = n0 * s + n1 * c;
        double a = fabs(n0) > fabs(n1) ? fabs(n0) : fabs(n1);
        mag[2 * i] = a;
        mag[2 * i + 1] = a;
    }
}
