// rowops.cuh -- the row machinery shared by the norm kernels.
//
// A row of D bfloat16 values is cut into 8-element chunks (16 bytes); chunk c
// belongs to logical lane c mod 128, and a lane visits its chunks in
// ascending order.  A group of TPR threads (32, 64 or 128) owns one row at a
// time: thread t holds the M = 128/TPR lanes t, t+TPR, ..., so for every
// chunk index j the group's loads cover TPR consecutive chunks (coalesced
// 128-bit accesses).  Per-lane results are combined by the fixed halving tree
//   for s = 64, 32, ..., 1:  L[l] = combine(L[l], L[l+s])   (l < s)
// realised as: levels s >= TPR inside a thread, 32 <= s < TPR through shared
// memory between the group's warps, s < 32 by warp shuffles.  Every
// realisation performs the same operations on the same operands, so the
// result does not depend on TPR.
//
// The lane/chunk order and the tree follow the bit-exact LayerNorm
// description of "Agent-assisted SGLang diffusion kernel optimisation:
// Qwen-Image, FLUX.2 and video models" (tahou.com), section
// 扩散Kernel对数值精度的敏感性 (a 128-thread Welford and a fixed shuffle tree).
#pragma once

#include "numerics.cuh"

namespace mbx {

constexpr int kLanes = 128;
constexpr int kChunk = 8;
constexpr int kBlock = 256;  // threads per CTA of the row kernels

template <int TPR_, int J_, bool VEC_>
struct RowCfg {
    static constexpr int TPR = TPR_;          // threads per row group
    static constexpr int J = J_;              // chunks per lane (max)
    static constexpr int M = kLanes / TPR_;   // lanes per thread
    static constexpr bool VEC = VEC_;         // 128-bit accesses allowed
    static constexpr int RPC = kBlock / TPR_; // row groups per CTA
    static_assert(TPR_ == 32 || TPR_ == 64 || TPR_ == 128, "TPR");
};

// Shared memory of one row group for the cross-warp tree levels.
struct TreeSmem {
    float a64[3][64];
    float a32[3][32];
    float bcast[4];
};

__device__ __forceinline__ void group_bar(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Chunk c of a row: 8 elements, zero-filled past D.  RW: the row may be
// overwritten by this kernel (an in-place residual), so it is read with
// coherent loads.
template <bool VEC, bool RW = false>
__device__ __forceinline__ uint4 load_chunk(const uint16_t* row, int c, int D, bool stream) {
    if constexpr (VEC) {
        const uint16_t* p = row + (int64_t)c * kChunk;
        if constexpr (RW) return ld_stream_rw(p);
        return stream ? ld_stream(p) : ld_shared_row(p);
    } else {
        uint4 v = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int e0 = c * kChunk + 2 * i;
            uint32_t lo = e0 < D ? (RW ? ld_u16_rw(row + e0) : ld_u16(row + e0)) : 0u;
            uint32_t hi = e0 + 1 < D ? (RW ? ld_u16_rw(row + e0 + 1) : ld_u16(row + e0 + 1)) : 0u;
            w_set(v, i, lo | (hi << 16));
        }
        return v;
    }
}

template <bool VEC>
__device__ __forceinline__ void store_chunk(uint16_t* row, int c, int D, uint4 v) {
    if constexpr (VEC) {
        st_v4(row + (int64_t)c * kChunk, v);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int e0 = c * kChunk + 2 * i;
            uint32_t w = w_of(v, i);
            if (e0 < D) st_u16(row + e0, (uint16_t)(w & 0xffffu));
            if (e0 + 1 < D) st_u16(row + e0 + 1, (uint16_t)(w >> 16));
        }
    }
}

// Elements of chunk c that exist (0..8).
__device__ __forceinline__ int chunk_len(int c, int D) {
    int n = D - c * kChunk;
    return n <= 0 ? 0 : (n >= kChunk ? kChunk : n);
}

// Number of elements of lane l (its count in the Welford / sum).
__device__ __forceinline__ int lane_count(int l, int D) {
    int nch = (D + kChunk - 1) / kChunk;
    if (l >= nch) return 0;
    int full = (nch - 1 - l) / kLanes;  // chunks of lane l before its last one
    return full * kChunk + chunk_len(l + full * kLanes, D);
}

// Load every chunk of the row owned by this thread: v[m][j] is chunk
// t + TPR*m + 128*j.
template <class C>
__device__ __forceinline__ void load_row(uint4 (&v)[C::M][C::J], const uint16_t* row, int t, int D,
                                         bool stream) {
    const int nch = (D + kChunk - 1) / kChunk;
#pragma unroll
    for (int j = 0; j < C::J; ++j)
#pragma unroll
        for (int m = 0; m < C::M; ++m) {
            int c = t + C::TPR * m + kLanes * j;
            v[m][j] = c < nch ? load_chunk<C::VEC>(row, c, D, stream) : make_uint4(0, 0, 0, 0);
        }
}

// True when every element this thread owns has |x| >= 2^-60 (bfloat16
// exponent field >= 67; inf and NaN pass).  Then, in each of its lanes, every
// Welford difference d = x - mean is +0 or |d| >= 2^-85: x is a multiple of
// 2^-67; if |mean| >= 2^-62 both are multiples of 2^-85 and x - mean is 0 or
// at least 2^-85 (exact below 2^-62), else |x - mean| > 2^-61.  That is the
// range where the unguarded division by the count is exact.
template <class C>
__device__ __forceinline__ bool lanes_plain(const uint4 (&v)[C::M][C::J], int t, int nch) {
    if constexpr (!C::VEC) {
        return false;  // the scalar path zero-fills partial chunks: use the guard
    } else {
        uint32_t acc = 0xffffffffu;
#pragma unroll
        for (int j = 0; j < C::J; ++j)
#pragma unroll
            for (int m = 0; m < C::M; ++m) {
                int c = t + C::TPR * m + kLanes * j;
                if (c < nch) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc = min_u16x2(acc, w_of(v[m][j], i) & 0x7f807f80u);
                }
            }
        uint32_t lo = acc & 0xffffu, hi = acc >> 16;
        return (lo < hi ? lo : hi) >= 0x2180u;
    }
}

// ------------------------------------------------------------------ cp.async ring

// 16-byte asynchronous global -> shared copy, L1 bypassed (streamed data).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ uint4 lds16(const uint4* p) {
    uint4 v;
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

// A row group's ring of NS stages; a stage holds NOPS rows (x and the
// per-token operands), each laid out by chunk index (16 bytes per chunk, 128*J
// chunks).  Thread t of the group copies exactly the chunks it later reads
// (t + TPR*m + 128*j), so its own cp.async.wait_group is the only
// synchronisation the ring needs.
template <class C, int NS, int NOPS>
struct Ring {
    static constexpr int kRowChunks = kLanes * C::J;
    static constexpr int kBytes = NS * NOPS * kRowChunks * 16;
    uint4* base;
    __device__ __forceinline__ uint4* at(int s, int o, int c) const {
        return base + ((s * NOPS + o) * kRowChunks + c);
    }
    // copy this thread's chunks of `src` into stage s, operand o
    __device__ __forceinline__ void issue(int s, int o, const uint16_t* src, int t, int nch) const {
#pragma unroll
        for (int j = 0; j < C::J; ++j)
#pragma unroll
            for (int m = 0; m < C::M; ++m) {
                int c = t + C::TPR * m + kLanes * j;
                if (c < nch) cp_async16(at(s, o, c), src + (int64_t)c * kChunk);
            }
    }
};

// row / seq along a sequence of rows advancing by a fixed step, without a
// 64-bit division per row: the quotient and remainder are carried along.
struct RowDiv {
    int64_t q, r, seq, dq, dr;
    __device__ __forceinline__ RowDiv(int64_t row, int64_t step, int64_t seq_) : seq(seq_) {
        q = row / seq;
        r = row - q * seq;
        dq = step / seq;
        dr = step - dq * seq;
    }
    __device__ __forceinline__ void advance() {
        q += dq;
        r += dr;
        if (r >= seq) {
            r -= seq;
            ++q;
        }
    }
};

// ------------------------------------------------------------------ tree

__device__ __forceinline__ float sum_combine(float a, float b) { return __fadd_rn(a, b); }

__device__ __forceinline__ float shfl_down_t(float v, int s) { return __shfl_down_sync(0xffffffffu, v, s); }
__device__ __forceinline__ Wf shfl_down_t(Wf v, int s) { return wf_shfl_down(v, s); }

__device__ __forceinline__ void smem_put(float (&a)[3][64], int i, float v) { a[0][i] = v; }
__device__ __forceinline__ void smem_put(float (&a)[3][64], int i, Wf v) {
    a[0][i] = v.mean; a[1][i] = v.m2; a[2][i] = v.n;
}
__device__ __forceinline__ void smem_get(const float (&a)[3][64], int i, float& v) { v = a[0][i]; }
__device__ __forceinline__ void smem_get(const float (&a)[3][64], int i, Wf& v) {
    v.mean = a[0][i]; v.m2 = a[1][i]; v.n = a[2][i];
}
__device__ __forceinline__ void smem_put32(float (&a)[3][32], int i, float v) { a[0][i] = v; }
__device__ __forceinline__ void smem_put32(float (&a)[3][32], int i, Wf v) {
    a[0][i] = v.mean; a[1][i] = v.m2; a[2][i] = v.n;
}
__device__ __forceinline__ void smem_get32(const float (&a)[3][32], int i, float& v) { v = a[0][i]; }
__device__ __forceinline__ void smem_get32(const float (&a)[3][32], int i, Wf& v) {
    v.mean = a[0][i]; v.m2 = a[1][i]; v.n = a[2][i];
}

// Reduce the M per-lane values of every thread of the group along the fixed
// tree.  The returned value is meaningful in group thread 0 only.
template <class C, class T, class Comb>
__device__ __forceinline__ T tree_reduce(T (&L)[C::M], int t, TreeSmem& sm, int bar_id, Comb comb) {
    // levels inside the thread: lane t+TPR*m with lane t+TPR*(m + s/TPR)
#pragma unroll
    for (int s = 64; s >= C::TPR; s /= 2) {
#pragma unroll
        for (int m = 0; m < s / C::TPR; ++m) L[m] = comb(L[m], L[m + s / C::TPR]);
    }
    T v = L[0];
    // levels between warps of the group
    if constexpr (C::TPR == 128) {
        if (t >= 64) smem_put(sm.a64, t - 64, v);
        group_bar(bar_id, C::TPR);
        if (t < 64) {
            T o;
            smem_get(sm.a64, t, o);
            v = comb(v, o);
        }
        if (t >= 32 && t < 64) smem_put32(sm.a32, t - 32, v);
        group_bar(bar_id, C::TPR);
        if (t < 32) {
            T o;
            smem_get32(sm.a32, t, o);
            v = comb(v, o);
        }
    } else if constexpr (C::TPR == 64) {
        if (t >= 32) smem_put32(sm.a32, t - 32, v);
        group_bar(bar_id, C::TPR);
        if (t < 32) {
            T o;
            smem_get32(sm.a32, t, o);
            v = comb(v, o);
        }
    }
    // levels inside the first warp
    if (t < 32) {
#pragma unroll
        for (int s = 16; s >= 1; s /= 2) v = comb(v, shfl_down_t(v, s));
    }
    return v;
}

// Make two floats computed by group thread 0 visible to the whole group.
template <class C>
__device__ __forceinline__ void group_bcast(float& a, float& b, int t, TreeSmem& sm, int bar_id) {
    if constexpr (C::TPR == 32) {
        a = __shfl_sync(0xffffffffu, a, 0);
        b = __shfl_sync(0xffffffffu, b, 0);
    } else {
        if (t == 0) {
            sm.bcast[0] = a;
            sm.bcast[1] = b;
        }
        group_bar(bar_id, C::TPR);
        a = sm.bcast[0];
        b = sm.bcast[1];
    }
}

// ------------------------------------------------------------------ single-barrier tree
//
// The same tree with its result in every thread of the group, at one barrier
// per row.  After the levels inside each thread, every thread publishes its
// lane value; after one barrier each warp reads the values it needs and
// computes the cross-warp levels itself (warp w's thread i forms the same
// combine(L[l], L[l+s]) that warp 0's thread i forms, with the same operands,
// so every warp holds the same bits), runs the shuffle levels, and takes the
// result from its lane 0.  The published values are double-buffered by row
// parity: a slot is written again two rows later, after the next row's
// barrier, which every reader of the older row has passed.

template <int TPR>
struct TreeAll {
    float v[2][2][TPR];  // [row parity][mean | m2, or the sum][thread]
};
template <>
struct TreeAll<32> {  // one warp per row: shuffles only
    float unused[4];
};
// The kernels place 16-byte-aligned arrays (modulation, ring stages) right
// after the groups' tree buffers.
static_assert(sizeof(TreeAll<32>) % 16 == 0 && sizeof(TreeAll<64>) % 16 == 0 && sizeof(TreeAll<128>) % 16 == 0,
              "tree buffers keep the 16-byte alignment of what follows them");

// Published values.  A Wf's count is not stored: the reader recomputes it from
// the publishing thread's lanes (n_of).
template <int N>
__device__ __forceinline__ void tall_put(float (&a)[2][N], int i, float v) { a[0][i] = v; }
template <int N>
__device__ __forceinline__ void tall_put(float (&a)[2][N], int i, Wf v) {
    a[0][i] = v.mean; a[1][i] = v.m2;
}
template <int N>
__device__ __forceinline__ void tall_get(const float (&a)[2][N], int i, float& v, float) { v = a[0][i]; }
template <int N>
__device__ __forceinline__ void tall_get(const float (&a)[2][N], int i, Wf& v, float n) {
    v.mean = a[0][i]; v.m2 = a[1][i]; v.n = n;
}
__device__ __forceinline__ float shfl_idx0(float v) { return __shfl_sync(0xffffffffu, v, 0); }
__device__ __forceinline__ Wf shfl_idx0(Wf v) {
    return Wf{__shfl_sync(0xffffffffu, v.mean, 0), __shfl_sync(0xffffffffu, v.m2, 0),
              __shfl_sync(0xffffffffu, v.n, 0)};
}

// The cross-warp levels and the shuffle levels of the tree, after the levels
// inside each thread (v = this thread's lane value, lane t), with the result
// returned in every thread, as described above.  PUT(i, x) publishes thread
// i's value, GET(i) reads it, COMB at level S combines, SHFL(x, s) shuffles
// down, BCAST(x) takes lane 0's value.
template <int TPR, class T, class Put, class Get, class Comb, class Shfl, class Bcast>
__device__ __forceinline__ T tree_cross(T v, int t, int bar_id, Put put, Get get, Comb comb, Shfl shfl, Bcast bcast) {
    if constexpr (TPR == 64) {
        put(t, v);
        group_bar(bar_id, TPR);
        const T o = get(t ^ 32);
        v = t < 32 ? comb(std::integral_constant<int, 32>{}, v, o) : comb(std::integral_constant<int, 32>{}, o, v);
    } else if constexpr (TPR == 128) {
        put(t, v);
        group_bar(bar_id, TPR);
        const int lo = t & 31;
        const T a = get(lo), b = get(lo + 32), c = get(lo + 64), d = get(lo + 96);
        // s = 64 for lanes lo and lo + 32, then s = 32
        v = comb(std::integral_constant<int, 32>{}, comb(std::integral_constant<int, 64>{}, a, c),
                 comb(std::integral_constant<int, 64>{}, b, d));
    }
    static_for<0, 5>([&](auto lc) {
        constexpr int S = 16 >> decltype(lc)::value;
        v = comb(std::integral_constant<int, S>{}, v, shfl(v, S));
    });
    return bcast(v);
}

// D: the row length, for the element counts of published Welford values
// (thread i holds lanes i + TPR*m after the levels inside the thread).
template <class C, class T, class Comb>
__device__ __forceinline__ T tree_allreduce(T (&L)[C::M], int t, TreeAll<C::TPR>& sm, int bar_id, int par, int D,
                                            Comb comb) {
#pragma unroll
    for (int s = 64; s >= C::TPR; s /= 2) {
#pragma unroll
        for (int m = 0; m < s / C::TPR; ++m) L[m] = comb(L[m], L[m + s / C::TPR]);
    }
    return tree_cross<C::TPR>(
        L[0], t, bar_id,
        [&](int i, T x) {
            if constexpr (C::TPR > 32) tall_put(sm.v[par], i, x);
        },
        [&](int i) {
            T x{};
            if constexpr (C::TPR > 32) {
                float n = 0.0f;
                if constexpr (std::is_same<T, Wf>::value) {
#pragma unroll
                    for (int m = 0; m < C::M; ++m) n += (float)lane_count(i + C::TPR * m, D);
                }
                tall_get(sm.v[par], i, x, n);
            }
            return x;
        },
        [&](auto, T a, T b) { return comb(a, b); }, [](T x, int s) { return shfl_down_t(x, s); },
        [](T x) { return shfl_idx0(x); });
}

// The Welford tree of a full row (every lane holds N0 = 8*J elements) with
// its result in every thread: at level s both operands hold N0*64/s elements,
// so wf_combine_eq's counts are compile-time constants (na/2 exact), and only
// mean and M2 are published and shuffled.  Same operations on the same
// operands as tree_reduce with wf_combine_eq: the same bits.
template <int NA2>
__device__ __forceinline__ Wf wf_combine_k(Wf a, Wf b) {
    const float d = __fsub_rn(b.mean, a.mean);
    return Wf{__fadd_rn(a.mean, __fmul_rn(d, 0.5f)),
              __fadd_rn(__fadd_rn(a.m2, b.m2), __fmul_rn(__fmul_rn(d, d), (float)NA2)), 0.0f};
}

// The other realisation: warp 0 alone computes the cross-warp and shuffle
// levels (a barrier per cross-warp level), thread 0 applies FIN to the result
// (a scalar chain such as the RMSNorm rstd) and publishes two floats, and a
// last barrier hands them to the group.  Fewer instructions than every warp
// computing the tree and FIN, more waiting; measured faster for the RMSNorm
// kernels and for the short-row two-pass statistics.
template <int TPR, class T, class Put, class Get, class Comb, class Shfl, class Fin>
__device__ __forceinline__ float2 tree_w0(T v, int t, int bar_id, Put put, Get get, Comb comb, Shfl shfl, Fin fin,
                                          float* pub) {
    if constexpr (TPR == 128) {
        if (t >= 64) put(t, v);
        group_bar(bar_id, TPR);
        if (t < 64) v = comb(std::integral_constant<int, 64>{}, v, get(t + 64));
        if (t >= 32 && t < 64) put(t, v);
        group_bar(bar_id, TPR);
        if (t < 32) v = comb(std::integral_constant<int, 32>{}, v, get(t + 32));
    } else if constexpr (TPR == 64) {
        if (t >= 32) put(t, v);
        group_bar(bar_id, TPR);
        if (t < 32) v = comb(std::integral_constant<int, 32>{}, v, get(t + 32));
    }
    float2 r = make_float2(0.0f, 0.0f);
    if (t < 32) {
        static_for<0, 5>([&](auto lc) {
            constexpr int S = 16 >> decltype(lc)::value;
            v = comb(std::integral_constant<int, S>{}, v, shfl(v, S));
        });
        if (t == 0) r = fin(v);
    }
    if constexpr (TPR == 32) {
        return make_float2(__shfl_sync(0xffffffffu, r.x, 0), __shfl_sync(0xffffffffu, r.y, 0));
    } else {
        if (t == 0) {
            pub[0] = r.x;
            pub[1] = r.y;
        }
        group_bar(bar_id, TPR);
        return make_float2(pub[0], pub[1]);
    }
}

template <class C, class Fin>
__device__ __forceinline__ float2 tree_w0_sum(float (&L)[C::M], int t, TreeAll<C::TPR>& sm, int bar_id, int par, Fin fin) {
#pragma unroll
    for (int s = 64; s >= C::TPR; s /= 2) {
#pragma unroll
        for (int m = 0; m < s / C::TPR; ++m) L[m] = sum_combine(L[m], L[m + s / C::TPR]);
    }
    float* pub = nullptr;
    if constexpr (C::TPR > 32) pub = &sm.v[par][1][0];  // a sum uses only the first row
    return tree_w0<C::TPR>(
        L[0], t, bar_id,
        [&](int i, float x) {
            if constexpr (C::TPR > 32) sm.v[par][0][i] = x;
        },
        [&](int i) {
            float x = 0.0f;
            if constexpr (C::TPR > 32) x = sm.v[par][0][i];
            return x;
        },
        [](auto, float a, float b) { return sum_combine(a, b); }, [](float x, int s) { return shfl_down_t(x, s); },
        fin, pub);
}

template <class C>
__device__ __forceinline__ Wf tree_allreduce_full(Wf (&L)[C::M], int t, TreeAll<C::TPR>& sm, int bar_id, int par) {
    constexpr int N0 = kChunk * C::J;
    static_for<0, 7>([&](auto lc) {  // levels s = 64 >> lc kept inside the thread
        constexpr int S = 64 >> decltype(lc)::value;
        if constexpr (S >= C::TPR) {
#pragma unroll
            for (int m = 0; m < S / C::TPR; ++m) L[m] = wf_combine_k<N0 * 32 / S>(L[m], L[m + S / C::TPR]);
        }
    });
    Wf r = tree_cross<C::TPR>(
        L[0], t, bar_id,
        [&](int i, Wf x) {
            if constexpr (C::TPR > 32) {
                sm.v[par][0][i] = x.mean;
                sm.v[par][1][i] = x.m2;
            }
        },
        [&](int i) {
            Wf x{0.0f, 0.0f, 0.0f};
            if constexpr (C::TPR > 32) x = Wf{sm.v[par][0][i], sm.v[par][1][i], 0.0f};
            return x;
        },
        [](auto sc, Wf a, Wf b) { return wf_combine_k<N0 * 32 / decltype(sc)::value>(a, b); },
        [](Wf x, int s) {
            return Wf{__shfl_down_sync(0xffffffffu, x.mean, s), __shfl_down_sync(0xffffffffu, x.m2, s), 0.0f};
        },
        [](Wf x) { return Wf{__shfl_sync(0xffffffffu, x.mean, 0), __shfl_sync(0xffffffffu, x.m2, 0), 0.0f}; });
    r.n = (float)(kLanes * N0);
    return r;
}

// Grid-wide row-group loop parameters.
struct RowLoop {
    int t;       // thread index within the row group
    int group;   // row group within the CTA
    int bar_id;  // named barrier of the group (1..RPC)
    int64_t first, step;
};

template <class C>
__device__ __forceinline__ RowLoop row_loop() {
    RowLoop r;
    r.t = threadIdx.x % C::TPR;
    r.group = threadIdx.x / C::TPR;
    r.bar_id = 1 + r.group;
    r.first = (int64_t)blockIdx.x * C::RPC + r.group;
    r.step = (int64_t)gridDim.x * C::RPC;
    return r;
}

}  // namespace mbx
