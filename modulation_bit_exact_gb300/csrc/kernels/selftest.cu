// selftest.cu -- exhaustive checks of the arithmetic building blocks that the
// lossless kernels rely on, against the GPU's own correctly rounded binary32
// operations:
//   0: div_k<K>(d) (two-word reciprocal: a multiply and a fused multiply-add) ==
//      div.rn(d, K) for K = 1..64 and every finite binary32 d;
//   1: mul.rn.bf16x2 == binary32 multiply then round, every operand pair;
//   2: add.rn.bf16x2 == binary32 add then round, every operand pair;
//   3: div_k_fast<K>(d) (no guard) == div.rn(d, K) for K = 1..64, every
//      binary32 d with |d| >= 2^-100, and d = +0;
//   4: the QKV epilogue's rstd table == bf16(div.rn(1, sqrt.rn(v))) for every
//      non-negative bfloat16 v (finite and +inf);
//   5: the hardware binary32 -> E4M3 conversion of the FP8 producers
//      (cvt.rn.satfinite.e4m3x2.f32) == the E4M3 definition (nearest even on
//      the exact value, saturation to +-448, NaN -> 0x7F) for every binary32
//      pattern; NaN inputs whose byte is not 0x7F are counted apart;
//   6: the hardware binary32 -> FP4 E2M1 conversion of the NVFP4 producers
//      (cvt.rn.satfinite.e2m1x2.f32) == the E2M1 definition (nearest, ties to
//      the code with mantissa 0, saturation to +-6) for every binary32
//      pattern; NaN inputs whose code is not 0x7 are counted apart.
// A mismatch where either result is a NaN is counted apart from the others:
// NaN payloads never reach a bfloat16 output except as the canonical NaN.
#include "launch.h"
#include "numerics.cuh"
#include "rstd_bf16_table.inc"

namespace mbx {

__device__ __forceinline__ bool is_nan32(uint32_t u) { return (u & 0x7fffffffu) > 0x7f800000u; }
__device__ __forceinline__ bool is_nan16(uint32_t h) { return (h & 0x7fffu) > 0x7f80u; }

template <bool FAST>
__global__ void selftest_div_kernel(unsigned long long* counts) {
    unsigned long long bad = 0, bad_nan = 0;
    const uint64_t total = 1ull << 32;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (uint64_t)gridDim.x * blockDim.x) {
        const float d = __uint_as_float((uint32_t)i);
        if (!isfinite(d)) continue;  // finite numerators only (see numerics.cuh)
        if (FAST && fabsf(d) < 0x1p-100f && (uint32_t)i != 0u) continue;  // fast form: |d| >= 2^-100 or +0
        static_for<1, 65>([&](auto kc) {
            constexpr int K = decltype(kc)::value;
            uint32_t got = __float_as_uint(FAST ? div_k_fast<K>(d) : div_k<K>(d));
            uint32_t want = __float_as_uint(__fdiv_rn(d, (float)K));
            if (got != want) {
                if (is_nan32(got) || is_nan32(want)) ++bad_nan;
                else ++bad;
            }
        });
    }
    if (bad) atomicAdd(&counts[0], bad);
    if (bad_nan) atomicAdd(&counts[1], bad_nan);
}

// Every (a, b) pair of bfloat16 operands: a = i >> 16, b = i & 0xffff packed
// as (a,b) and (b,a) in the two halves, so both halves see every pair.
template <bool MUL>
__global__ void selftest_bf16x2_kernel(unsigned long long* counts) {
    unsigned long long bad = 0, bad_nan = 0;
    const uint64_t total = 1ull << 32;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t a = (uint32_t)(i >> 16), b = (uint32_t)(i & 0xffffu);
        const uint32_t A = a | (b << 16), B = b | (a << 16);
        const uint32_t got = MUL ? bmul(A, B) : badd(A, B);
        const uint32_t want = MUL ? bmul_ref(A, B) : badd_ref(A, B);
        if (got != want) {
            uint32_t x = got ^ want;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t sh = 16 * h;
                if ((x >> sh) & 0xffffu) {
                    if (is_nan16((got >> sh) & 0xffffu) || is_nan16((want >> sh) & 0xffffu)) ++bad_nan;
                    else ++bad;
                }
            }
        }
    }
    if (bad) atomicAdd(&counts[0], bad);
    if (bad_nan) atomicAdd(&counts[1], bad_nan);
}

// The rstd table of the QKV epilogue vs bf16(div.rn(1, sqrt.rn(v))) for
// every bfloat16 pattern v with a non-negative finite or +inf value.
__global__ void selftest_rstd_kernel(unsigned long long* counts) {
    unsigned long long bad = 0;
    for (uint32_t v = blockIdx.x * blockDim.x + threadIdx.x; v <= 0x7f80u; v += gridDim.x * blockDim.x) {
        const float x = __uint_as_float(v << 16);
        const uint32_t want = pack_rn(__fdiv_rn(1.0f, __fsqrt_rn(x)), 0.0f) & 0xffffu;
        if ((uint32_t)kRstdBf16[v] != want) ++bad;
    }
    if (bad) atomicAdd(&counts[0], bad);
}

// E4M3 from its definition: 1 sign, 4 exponent bits (bias 7), 3 mantissa
// bits, largest finite 1.75 * 2^8; multiples of 2^-9 below 2^-6.
__device__ uint32_t e4m3_by_definition(float v) {
    const uint32_t u = __float_as_uint(v);
    if (is_nan32(u)) return 0x7fu;
    const uint32_t sign = (u >> 24) & 0x80u;
    const float a = fabsf(v);
    if (a >= 448.0f) return sign | 0x7eu;  // 464 ties to 448 (even); beyond saturates
    if (a < 0x1p-6f) return sign | (uint32_t)rintf(a * 512.0f);
    const int e = (int)((__float_as_uint(a) >> 23) & 0xffu) - 127;  // a is normal here
    float q = rintf(a * __uint_as_float((uint32_t)(127 + 3 - e) << 23));  // a / 2^(e-3), exact
    int ee = e;
    if (q == 16.0f) {
        q = 8.0f;
        ++ee;
    }
    return sign | ((uint32_t)(ee + 7) << 3) | ((uint32_t)q - 8u);
}

__global__ void selftest_e4m3_kernel(unsigned long long* counts) {
    unsigned long long bad = 0, bad_nan = 0;
    const uint64_t total = 1ull << 32;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (uint64_t)gridDim.x * blockDim.x) {
        const float v = __uint_as_float((uint32_t)i);
        const uint32_t got = e4m3x2(0.0f, v) & 0xffu;
        if (is_nan32((uint32_t)i)) {
            if (got != 0x7fu) ++bad_nan;
        } else if (got != e4m3_by_definition(v)) {
            ++bad;
        }
    }
    if (bad) atomicAdd(&counts[0], bad);
    if (bad_nan) atomicAdd(&counts[1], bad_nan);
}

// E2M1 from its definition: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 (codes
// 0..7); the decision points are the midpoints, each tie going to the code
// whose mantissa bit is 0.
__device__ uint32_t e2m1_by_definition(float v) {
    const uint32_t u = __float_as_uint(v);
    if (is_nan32(u)) return 0x7u;
    const uint32_t sign = (u >> 28) & 0x8u;
    const float a = fabsf(v);
    uint32_t c;
    if (a <= 0.25f) c = 0;
    else if (a < 0.75f) c = 1;
    else if (a <= 1.25f) c = 2;
    else if (a < 1.75f) c = 3;
    else if (a <= 2.5f) c = 4;
    else if (a < 3.5f) c = 5;
    else if (a <= 5.0f) c = 6;
    else c = 7;
    return sign | c;
}

__global__ void selftest_e2m1_kernel(unsigned long long* counts) {
    unsigned long long bad = 0, bad_nan = 0;
    const uint64_t total = 1ull << 32;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (uint64_t)gridDim.x * blockDim.x) {
        const float v = __uint_as_float((uint32_t)i);
        const float v8[8] = {v, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        const uint32_t got = e2m1x8(v8) & 0xfu;
        if (is_nan32((uint32_t)i)) {
            if (got != 0x7u) ++bad_nan;
        } else if (got != e2m1_by_definition(v)) {
            ++bad;
        }
    }
    if (bad) atomicAdd(&counts[0], bad);
    if (bad_nan) atomicAdd(&counts[1], bad_nan);
}

cudaError_t launch_selftest(int which, unsigned long long* counts, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(counts, 0, 2 * sizeof(unsigned long long), s);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int grid = sms * 8, block = 256;
    switch (which) {
        case 0: selftest_div_kernel<false><<<grid, block, 0, s>>>(counts); break;
        case 3: selftest_div_kernel<true><<<grid, block, 0, s>>>(counts); break;
        case 4: selftest_rstd_kernel<<<grid, block, 0, s>>>(counts); break;
        case 5: selftest_e4m3_kernel<<<grid, block, 0, s>>>(counts); break;
        case 6: selftest_e2m1_kernel<<<grid, block, 0, s>>>(counts); break;
        case 1: selftest_bf16x2_kernel<true><<<grid, block, 0, s>>>(counts); break;
        case 2: selftest_bf16x2_kernel<false><<<grid, block, 0, s>>>(counts); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace mbx
