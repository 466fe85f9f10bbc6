// modtable.cu -- per-token modulation table written in the (6, rows, D) layout.
//
// "Agent-assisted SGLang diffusion kernel optimisation: Qwen-Image, FLUX.2 and
// video models" (tahou.com), section Wan视频模型的数据搬运优化: a Wan block's
// eager (table.unsqueeze(0) + temb.float()).chunk(6, dim=2) materialises a
// binary32 [B, S, 6, D] temporary (about 8 GB at 704p, 121 frames) and hands
// out six strided views that later need .contiguous().  Here one pass reads
// temb once and writes the six chunks as contiguous planes:
//   out[k*rows + r][d] = float(table[k][d]) + float(temb[r][k*D + d])
// one binary32 addition per element, as in the eager expression, so the
// result is the same bits.
//
// Layout: a CTA takes a token row at a time (grid-stride); its threads walk the
// row's 6*D/8 eight-element chunks in order, so loads of temb and stores of
// each plane are coalesced 16-byte accesses.  Each thread issues the loads of
// kUnroll chunks before it computes and stores them.  The [6, D] table is
// read through L1 (every row of a CTA uses all of it).
#include "launch.h"
#include "rowops.cuh"

namespace mbx {

constexpr int kTabThreads = 256;
constexpr int kUnroll = 4;
// chunks in flight per thread in the flat kernel: eight for binary32 temb
// (measured 9% faster there), four for bf16 temb (eight measured 13% slower)
template <bool EMB_F32>
constexpr int kFlatUnroll = EMB_F32 ? 8 : 4;

__device__ __forceinline__ unsigned div_by(unsigned n, const FastDiv& f) {
    return (unsigned)(((unsigned long long)n * f.m) >> f.shift);
}

__device__ __forceinline__ uint4 ld_l1(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Eight consecutive elements at element offset `e` of a bf16 or binary32 row,
// widened exactly to binary32.  STREAM: read once (no L1 allocation).
template <bool F32, bool STREAM>
__device__ __forceinline__ void load8(const void* row, int64_t e, float (&v)[8]) {
    if constexpr (F32) {
        const float* p = static_cast<const float*>(row) + e;
        const uint4 a = STREAM ? ld_stream(p) : ld_l1(p);
        const uint4 b = STREAM ? ld_stream(p + 4) : ld_l1(p + 4);
        v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
        v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
        v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
        v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
    } else {
        const uint16_t* p = static_cast<const uint16_t*>(row) + e;
        const uint4 a = STREAM ? ld_stream(p) : ld_l1(p);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = lo_f(w_of(a, i));
            v[2 * i + 1] = hi_f(w_of(a, i));
        }
    }
}

template <bool TAB_F32, bool EMB_F32>
__global__ void __launch_bounds__(kTabThreads) modtable_vec_kernel(ModTableParams p) {
    grid_dep_wait();  // launched programmatically: the previous kernel has finished
    grid_dep_launch();
    const int nch = p.D / kChunk;
    const unsigned per_row = 6u * (unsigned)nch;
    const int64_t esz = EMB_F32 ? 4 : 2, tsz = TAB_F32 ? 4 : 2;
    for (int64_t r = blockIdx.x; r < p.rows; r += gridDim.x) {
        const void* erow = static_cast<const char*>(p.temb) + r * p.temb_stride * esz;
        for (unsigned i0 = threadIdx.x; i0 < per_row; i0 += kTabThreads * kUnroll) {
            float e[kUnroll][8];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const unsigned i = i0 + u * kTabThreads;
                if (i < per_row) load8<EMB_F32, true>(erow, (int64_t)i * kChunk, e[u]);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const unsigned i = i0 + u * kTabThreads;
                if (i >= per_row) continue;
                const unsigned k = div_by(i, p.by_nch);
                const unsigned c = i - k * (unsigned)nch;
                float t[8];
                load8<TAB_F32, false>(static_cast<const char*>(p.table) + (int64_t)k * p.table_stride * tsz,
                                      (int64_t)c * kChunk, t);
                uint4 o0, o1;
                o0.x = __float_as_uint(__fadd_rn(t[0], e[u][0]));
                o0.y = __float_as_uint(__fadd_rn(t[1], e[u][1]));
                o0.z = __float_as_uint(__fadd_rn(t[2], e[u][2]));
                o0.w = __float_as_uint(__fadd_rn(t[3], e[u][3]));
                o1.x = __float_as_uint(__fadd_rn(t[4], e[u][4]));
                o1.y = __float_as_uint(__fadd_rn(t[5], e[u][5]));
                o1.z = __float_as_uint(__fadd_rn(t[6], e[u][6]));
                o1.w = __float_as_uint(__fadd_rn(t[7], e[u][7]));
                float* dst = p.out + ((int64_t)k * p.rows + r) * p.out_stride + (int64_t)c * kChunk;
                st_v4(dst, o0);
                st_v4(dst + 4, o1);
            }
        }
    }
}

// The same with the whole output as one list of chunks (token rows back to
// back, 6*D/8 chunks each), so that every thread holds within one chunk of
// the same share; used while that index fits in 32 bits.
template <bool TAB_F32, bool EMB_F32>
__global__ void __launch_bounds__(kTabThreads) modtable_flat_kernel(ModTableParams p, FastDiv by_row,
                                                                    unsigned total) {
    grid_dep_wait();  // launched programmatically: the previous kernel has finished
    grid_dep_launch();
    const unsigned nch = (unsigned)p.D / kChunk, per_row = 6u * nch;
    const int64_t esz = EMB_F32 ? 4 : 2, tsz = TAB_F32 ? 4 : 2;
    constexpr int kU = kFlatUnroll<EMB_F32>;
    const unsigned stride = gridDim.x * kTabThreads * kU;
    for (unsigned base = blockIdx.x * kTabThreads * kU + threadIdx.x; base < total; base += stride) {
        float e[kU][8];
        unsigned row[kU], idx[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const unsigned q = base + u * kTabThreads;
            if (q >= total) continue;
            row[u] = div_by(q, by_row);
            idx[u] = q - row[u] * per_row;
            load8<EMB_F32, true>(static_cast<const char*>(p.temb) + (int64_t)row[u] * p.temb_stride * esz,
                                 (int64_t)idx[u] * kChunk, e[u]);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const unsigned q = base + u * kTabThreads;
            if (q >= total) continue;
            const unsigned k = div_by(idx[u], p.by_nch);
            const unsigned c = idx[u] - k * nch;
            float t[8];
            load8<TAB_F32, false>(static_cast<const char*>(p.table) + (int64_t)k * p.table_stride * tsz,
                                  (int64_t)c * kChunk, t);
            uint4 o0, o1;
            o0.x = __float_as_uint(__fadd_rn(t[0], e[u][0]));
            o0.y = __float_as_uint(__fadd_rn(t[1], e[u][1]));
            o0.z = __float_as_uint(__fadd_rn(t[2], e[u][2]));
            o0.w = __float_as_uint(__fadd_rn(t[3], e[u][3]));
            o1.x = __float_as_uint(__fadd_rn(t[4], e[u][4]));
            o1.y = __float_as_uint(__fadd_rn(t[5], e[u][5]));
            o1.z = __float_as_uint(__fadd_rn(t[6], e[u][6]));
            o1.w = __float_as_uint(__fadd_rn(t[7], e[u][7]));
            float* dst = p.out + ((int64_t)k * p.rows + row[u]) * p.out_stride + (int64_t)c * kChunk;
            st_v4(dst, o0);
            st_v4(dst + 4, o1);
        }
    }
}

template <bool F32>
__device__ __forceinline__ float elem(const void* base, int64_t i) {
    if constexpr (F32) return static_cast<const float*>(base)[i];
    else return __uint_as_float((uint32_t)static_cast<const uint16_t*>(base)[i] << 16);
}

// Any alignment, any D: one element per step, the same addition.
template <bool TAB_F32, bool EMB_F32>
__global__ void __launch_bounds__(kTabThreads) modtable_scalar_kernel(ModTableParams p, FastDiv by_d) {
    grid_dep_wait();  // launched programmatically: the previous kernel has finished
    grid_dep_launch();
    const unsigned per_row = 6u * (unsigned)p.D;
    for (int64_t r = blockIdx.x; r < p.rows; r += gridDim.x) {
        for (unsigned i = threadIdx.x; i < per_row; i += kTabThreads) {
            const unsigned k = div_by(i, by_d);
            const unsigned d = i - k * (unsigned)p.D;
            const float t = elem<TAB_F32>(p.table, (int64_t)k * p.table_stride + d);
            const float e = elem<EMB_F32>(p.temb, r * p.temb_stride + i);
            p.out[((int64_t)k * p.rows + r) * p.out_stride + d] = __fadd_rn(t, e);
        }
    }
}

template <bool TAB_F32, bool EMB_F32>
static cudaError_t launch_t(const ModTableParams& p0, bool vec, cudaStream_t s) {
    ModTableParams p = p0;
    const int64_t total = p.rows * 6 * (p.D / kChunk);
    if (vec && total < (1ll << 31)) {
        auto k = modtable_flat_kernel<TAB_F32, EMB_F32>;
        p.by_nch = make_fastdiv((unsigned)(p.D / kChunk));
        const int grid = grid_for_rows(reinterpret_cast<const void*>(k),
                                       (total + kTabThreads * kFlatUnroll<EMB_F32> - 1) / (kTabThreads * kFlatUnroll<EMB_F32>), 1,
                                       kTabThreads);
        if (grid < 0) return cudaErrorUnknown;
        return launch_pdl(k, grid, kTabThreads, 0, s, p, make_fastdiv((unsigned)(6 * (p.D / kChunk))), (unsigned)total);
    } else if (vec) {
        auto k = modtable_vec_kernel<TAB_F32, EMB_F32>;
        p.by_nch = make_fastdiv((unsigned)(p.D / kChunk));
        const int grid = grid_for_rows(reinterpret_cast<const void*>(k), p.rows, 1, kTabThreads);
        if (grid < 0) return cudaErrorUnknown;
        return launch_pdl(k, grid, kTabThreads, 0, s, p);
    } else {
        auto k = modtable_scalar_kernel<TAB_F32, EMB_F32>;
        const int grid = grid_for_rows(reinterpret_cast<const void*>(k), p.rows, 1, kTabThreads);
        if (grid < 0) return cudaErrorUnknown;
        return launch_pdl(k, grid, kTabThreads, 0, s, p, make_fastdiv((unsigned)p.D));
    }
}

cudaError_t launch_modulation_table_add(const ModTableParams& p, bool vec, cudaStream_t s) {
    if (p.table_f32)
        return p.temb_f32 ? launch_t<true, true>(p, vec, s) : launch_t<true, false>(p, vec, s);
    return p.temb_f32 ? launch_t<false, true>(p, vec, s) : launch_t<false, false>(p, vec, s);
}

}  // namespace mbx
