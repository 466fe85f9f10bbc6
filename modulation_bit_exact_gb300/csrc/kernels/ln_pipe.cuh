// ln_pipe.cuh -- the pipelined (shared-memory ring) LayerNorm + AdaLN
// modulate kernel and its launch helpers, shared by the translation units
// that instantiate it (ln_modulate.cu: plain, gated and FP8 outputs;
// ln_nvfp4.cu: the NVFP4 output).
//
// The operation and its lossless rounding order are defined at the top of
// ln_modulate.cu ("Agent-assisted SGLang diffusion kernel optimisation"
// (tahou.com), section 扩散Kernel对数值精度的敏感性); the gated front pass and
// the FP8/NVFP4 stores follow the section 将FP8量化融合到前序算子 and the
// gated-residual chain of section Qwen-Image FP8和NVFP4优化 of the same article.
#pragma once
#include <algorithm>

#include "launch.h"
#include "rowops.cuh"

namespace mbx {

__device__ __forceinline__ u64 sel2(bool a, bool b, u64 n, u64 o) {
    return f2(a ? f2lo(n) : f2lo(o), b ? f2hi(n) : f2hi(o));
}

// ------------------------------------------------------------------ pipelined path
//
// For 16-byte-aligned rows (D % 8 == 0): one CTA per SM holds several row
// groups; each group streams its next rows into a ring of shared-memory
// stages with cp.async (each thread copies exactly the chunks it will read),
// so loads stay in flight while the group computes.  Same lanes, same order,
// same tree as above: the results are the same bits.

// Every element of the chunk has |x| >= 2^-60 (bf16 exponent field >= 67).
__device__ __forceinline__ bool chunk_plain(const uint4& v) {
    uint32_t a = min_u16x2(min_u16x2(v.x & 0x7f807f80u, v.y & 0x7f807f80u),
                           min_u16x2(v.z & 0x7f807f80u, v.w & 0x7f807f80u));
    uint32_t lo = a & 0xffffu, hi = a >> 16;
    return (lo < hi ? lo : hi) >= 0x2180u;
}

struct WPair {
    u64 mean, m2;
};

// Welford over one chunk of lane A (low halves) and one of lane B (high
// halves), counts k0+1..k0+8, with plain correctly rounded division: the rare
// path for chunks holding zeros or values below 2^-60.  na / nb: elements of
// each chunk that exist (0 or 8).
static __device__ __noinline__ WPair welford_chunk_exact(uint4 a, uint4 b, int k0, int na, int nb, WPair st) {
    float ma = f2lo(st.mean), qa = f2lo(st.m2), mb = f2hi(st.mean), qb = f2hi(st.m2);
    for (int e = 0; e < kChunk; ++e) {
        const float k = (float)(k0 + e + 1);
        const uint32_t wa = w_of(a, e >> 1), wb = w_of(b, e >> 1);
        const float xa = (e & 1) ? hi_f(wa) : lo_f(wa), xb = (e & 1) ? hi_f(wb) : lo_f(wb);
        if (e < na) {
            float d = __fsub_rn(xa, ma);
            ma = __fadd_rn(ma, __fdiv_rn(d, k));
            qa = __fadd_rn(qa, __fmul_rn(d, __fsub_rn(xa, ma)));
        }
        if (e < nb) {
            float d = __fsub_rn(xb, mb);
            mb = __fadd_rn(mb, __fdiv_rn(d, k));
            qb = __fadd_rn(qb, __fmul_rn(d, __fsub_rn(xb, mb)));
        }
    }
    return WPair{f2(ma, mb), f2(qa, qb)};
}

// Welford of every lane this thread owns, reading its chunks from ring stage
// s.  For each chunk index j one branch decides, for all the thread's lanes at
// once, between the fast division (every element plain) and the exact one,
// so the lane pairs' dependency chains interleave.  `full` (every lane has
// all J chunks) removes the per-step selects of the last chunk.
// ROWCHECK: for full rows, decide fast-or-exact once for all of the thread's
// chunks (measured faster for the unfused kernel at J = 1 and 3; slower at
// even J and in the fused kernel, where the extra live chunks cost more).
template <class C, bool ROWCHECK, class RingT>
__device__ __forceinline__ void welford_stage(const RingT& ring, int s, int t, int nch, bool full,
                                              Wf (&L)[C::M], u64 nz) {
    if constexpr (C::M >= 2) {
        constexpr int P = C::M / 2;
        u64 mean[P], m2[P];
#pragma unroll
        for (int p = 0; p < P; ++p) mean[p] = m2[p] = f2(0.0f, 0.0f);
        if (ROWCHECK && full) {
            // Common case: every lane has all J chunks.  One check for all of
            // this thread's elements (the smallest exponent field over every
            // chunk), then the fast division throughout, both lane pairs'
            // chains interleaved.
            uint4 A[C::J][P], B[C::J][P];
            uint32_t lowest = 0xffffffffu;
#pragma unroll
            for (int j = 0; j < C::J; ++j)
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    const int ca = t + C::TPR * p + kLanes * j;
                    A[j][p] = lds16(ring.at(s, 0, ca));
                    B[j][p] = lds16(ring.at(s, 0, ca + C::TPR * P));
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        lowest = min_u16x2(lowest, w_of(A[j][p], i) & 0x7f807f80u);
                        lowest = min_u16x2(lowest, w_of(B[j][p], i) & 0x7f807f80u);
                    }
                }
            const uint32_t lo = lowest & 0xffffu, hi = lowest >> 16;
            if ((lo < hi ? lo : hi) >= 0x2180u) {
                static_for<0, C::J>([&](auto jc) {
                    constexpr int j = decltype(jc)::value;
                    static_for<0, kChunk>([&](auto ec) {
                        constexpr int e = decltype(ec)::value;
                        constexpr int K = kChunk * j + e + 1;
#pragma unroll
                        for (int p = 0; p < P; ++p)
                            welford_step2<K, false>(pair_elem(w_of(A[j][p], e / 2), w_of(B[j][p], e / 2), e & 1),
                                                    mean[p], m2[p], nz);
                    });
                });
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    L[p].mean = f2lo(mean[p]);
                    L[p].m2 = f2lo(m2[p]);
                    L[p + P].mean = f2hi(mean[p]);
                    L[p + P].m2 = f2hi(m2[p]);
                    L[p].n = L[p + P].n = (float)(kChunk * C::J);
                }
                return;
            }
        }
        static_for<0, C::J>([&](auto jc) {
            constexpr int j = decltype(jc)::value;
            uint4 A[P], B[P];
            bool va[P], vb[P];
            bool plain = true;
#pragma unroll
            for (int p = 0; p < P; ++p) {
                const int ca = t + C::TPR * p + kLanes * j, cb = ca + C::TPR * P;
                va[p] = ca < nch;
                vb[p] = cb < nch;
                A[p] = va[p] ? lds16(ring.at(s, 0, ca)) : make_uint4(0, 0, 0, 0);
                B[p] = vb[p] ? lds16(ring.at(s, 0, cb)) : make_uint4(0, 0, 0, 0);
                plain = plain && (!va[p] || chunk_plain(A[p])) && (!vb[p] || chunk_plain(B[p]));
            }
            if (plain && (j < C::J - 1 || full)) {
                static_for<0, kChunk>([&](auto ec) {
                    constexpr int e = decltype(ec)::value;
                    constexpr int K = kChunk * j + e + 1;
#pragma unroll
                    for (int p = 0; p < P; ++p)
                        welford_step2<K, false>(pair_elem(w_of(A[p], e / 2), w_of(B[p], e / 2), e & 1), mean[p], m2[p], nz);
                });
            } else if (plain) {  // last chunk, some lanes without it
                static_for<0, kChunk>([&](auto ec) {
                    constexpr int e = decltype(ec)::value;
                    constexpr int K = kChunk * j + e + 1;
#pragma unroll
                    for (int p = 0; p < P; ++p) {
                        u64 mn = mean[p], q = m2[p];
                        welford_step2<K, false>(pair_elem(w_of(A[p], e / 2), w_of(B[p], e / 2), e & 1), mn, q, nz);
                        mean[p] = sel2(va[p], vb[p], mn, mean[p]);
                        m2[p] = sel2(va[p], vb[p], q, m2[p]);
                    }
                });
            } else {
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    WPair r = welford_chunk_exact(A[p], B[p], kChunk * j, va[p] ? kChunk : 0, vb[p] ? kChunk : 0,
                                                  WPair{mean[p], m2[p]});
                    mean[p] = r.mean;
                    m2[p] = r.m2;
                }
            }
        });
#pragma unroll
        for (int p = 0; p < P; ++p) {
            L[p].mean = f2lo(mean[p]);
            L[p].m2 = f2lo(m2[p]);
            L[p + P].mean = f2hi(mean[p]);
            L[p + P].m2 = f2hi(m2[p]);
        }
    } else {
        u64 st = f2(0.0f, 0.0f), sq = f2(0.0f, 0.0f);  // lane in the low halves
        static_for<0, C::J>([&](auto jc) {
            constexpr int j = decltype(jc)::value;
            const int c = t + kLanes * j;
            if (c >= nch) return;
            const uint4 A = lds16(ring.at(s, 0, c));
            if (chunk_plain(A)) {
                float mean = f2lo(st), m2 = f2lo(sq);
                static_for<0, kChunk>([&](auto ec) {
                    constexpr int e = decltype(ec)::value;
                    constexpr int K = kChunk * j + e + 1;
                    const uint32_t w = w_of(A, e / 2);
                    welford_step<K, false>((e & 1) ? hi_f(w) : lo_f(w), mean, m2);
                });
                st = f2(mean, 0.0f);
                sq = f2(m2, 0.0f);
            } else {
                WPair r = welford_chunk_exact(A, make_uint4(0, 0, 0, 0), kChunk * j, kChunk, 0, WPair{st, sq});
                st = r.mean;
                sq = r.m2;
            }
        });
        L[0].mean = f2lo(st);
        L[0].m2 = f2lo(sq);
    }
#pragma unroll
    for (int m = 0; m < C::M; ++m) {
        const int c_last = t + C::TPR * m + kLanes * (C::J - 1);
        L[m].n = (float)(kChunk * (C::J - 1) + (c_last < nch ? kChunk : 0));
    }
}

// Modulation modes of the pipelined kernel:
//   kModRing:   each row reads its own modulation row (per-token modulation,
//               or samples that change within a CTA's rows): loaded into
//               registers, or carried in the ring (see LnOps);
//   kModStaged: a CTA's rows span at most two samples; their bf16(1+scale)
//               (lossless) or scale (high) and shift are staged in shared
//               memory once.
//   kModL1:     the gated kernel on rows too wide to stage the per-sample
//               vectors beside a two-operand ring: gate, scale, shift and the
//               bias are read from global memory where they are used (a
//               sample's vectors are shared by all its rows, so they stay in
//               L1 and L2), leaving shared memory to the ring.
enum { kModRing = 0, kModStaged = 1, kModL1 = 2 };

// Ring operands of the pipelined kernel: x (the residual when FUSED), then,
// in ring mode, the gate (FUSED) and, for fused rows of more than 4096
// elements, scale and shift.  The fused kernel's update is read once, by the
// front pass, so it has a single stage of its own: the next row's update is
// copied in right after the front pass has consumed the current one, and
// lands while the statistics and the output pass run.  That frees a ring
// operand's second stage, so more row groups fit.
//
// Per-row modulation is otherwise read from global memory into registers when
// the row's data has landed (its latency hides behind the statistics), so it
// takes no ring stages and more row groups fit in shared memory.  The fused
// kernel's gate, used by its front pass at once, stays in the ring; so do its
// scale and shift where the registers they would hold cost more than the ring
// stages (measured): J >= 5, and the high variant at J = 4.
constexpr bool ln_fused_direct(int J, bool high) { return J <= 3 || (J == 4 && !high); }
// Whether the fused kernel's update takes the one-stage buffer (measured per
// row width: faster except at 4096 and 5120 elements, where the update keeps
// its two ring stages).
constexpr bool ln_update_one_stage(int J) { return J != 4 && J != 5; }
constexpr int ln_ring_ops(bool fused, int mode, int J, bool high) {
    const int u = fused && !ln_update_one_stage(J) ? 1 : 0;
    return u + (mode != kModRing ? 1 : !fused ? 1 : ln_fused_direct(J, high) ? 2 : 4);
}

template <bool FUSED, int MODE, int J, bool HIGH>
struct LnOps {
    static constexpr bool DIRECT = MODE == kModRing && (!FUSED || ln_fused_direct(J, HIGH));
    static constexpr bool RING_MOD = MODE == kModRing && FUSED && !DIRECT;  // scale, shift in the ring
    static constexpr bool USTAGE = FUSED && ln_update_one_stage(J);  // update in its own one-stage buffer
    static constexpr int U = FUSED && !USTAGE ? 1 : -1;                 // else in the ring, after x
    static constexpr int B = U > 0 ? 2 : 1;                              // first modulation operand
    static constexpr int SC = RING_MOD ? B : -1;
    static constexpr int SH = RING_MOD ? B + 1 : -1;
    static constexpr int G = MODE == kModRing && FUSED ? (RING_MOD ? B + 2 : B) : -1;
    static constexpr int N = ln_ring_ops(FUSED, MODE, J, HIGH);
    static constexpr int SLOT = FUSED ? 3 : 2;  // staged arrays per sample: t, shift[, gate]
    static_assert(N == 1 + (U > 0 ? 1 : 0) + (G >= 0 ? 1 : 0) + (RING_MOD ? 2 : 0), "ring operands");
};

__device__ __forceinline__ void sts16(uint4* p, uint4 v) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// rows per group brought into L2 before the wait on the previous kernel
constexpr int kPrefetchRows = 2;

template <int TPR, int J, int NS, bool HIGH, int MODE, bool FUSED, bool FP4>
__global__ void __launch_bounds__(512, 1) ln_modulate_pipe_kernel(LnModParams p, int64_t rows_per_cta) {
    using C = RowCfg<TPR, J, true>;
    using O = LnOps<FUSED, MODE, J, HIGH>;
    constexpr int NOPS = O::N;
    using R = Ring<C, NS, NOPS>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int groups = blockDim.x / TPR;
    const int g = threadIdx.x / TPR, t = threadIdx.x % TPR;
    const int D = p.D;
    const int nch = D / kChunk;
    TreeAll<TPR>& sm = reinterpret_cast<TreeAll<TPR>*>(smem_raw)[g];
    uint4* mod = reinterpret_cast<uint4*>(smem_raw + groups * sizeof(TreeAll<TPR>));  // [2 slots][t|shift[|gate]][nch]
    const int mod_chunks = MODE == kModStaged ? 2 * O::SLOT * nch : 0;
    uint4* bias_sm = mod + mod_chunks;  // [nch] when FUSED with a bias
    const int bias_chunks = FUSED && MODE != kModL1 && p.bias != nullptr ? nch : 0;
    const R ring{bias_sm + bias_chunks + (size_t)g * (R::kBytes / 16)};
    // the fused kernel's one-stage update buffers, after every group's ring
    const Ring<C, 1, 1> ustage{bias_sm + bias_chunks + (size_t)groups * (R::kBytes / 16) +
                               (size_t)g * (O::USTAGE ? Ring<C, 1, 1>::kBytes / 16 : 0)};
    const int bar_id = 1 + g;
    const int64_t r0 = (int64_t)blockIdx.x * rows_per_cta;
    const int64_t r1 = r0 + rows_per_cta < p.rows ? r0 + rows_per_cta : p.rows;
    const int64_t m0 = r0 / p.seq;
    const int64_t split = (m0 + 1) * p.seq;  // staged: rows from here use slot 1
    // rows go to the groups in reverse order, so a block's extra rows (its row
    // count mod the groups) fall to the highest-numbered groups, whose warps
    // the schedulers serve first (measured: they finish a round earliest)
    const int64_t first = r0 + (groups - 1 - g);
    RowDiv next(first, groups, p.seq);  // modulation row of the next row to issue
    RowDiv here(first, groups, p.seq);  // modulation row of the row being processed
    // (advanced per row in the modes that read a row's modulation from global memory)
    constexpr bool kHere = O::DIRECT || MODE == kModL1;
    // while the previous kernel in the stream drains, bring the per-sample
    // vectors of this block's rows (first: every row group needs them before
    // its first row) and this group's first rows into L2; then wait for it
    // before reading anything it may write
    if (t == 0 && g == 0 && MODE != kModRing && r1 > r0) {
        const int64_t m_last = (r1 - 1) / p.seq;
        for (int64_t m = m0; m <= m_last && m <= m0 + 1; ++m) {
            prefetch_l2_bulk(p.scale + m * p.scale_stride, (uint32_t)D * 2);
            prefetch_l2_bulk(p.shift + m * p.shift_stride, (uint32_t)D * 2);
            if constexpr (FUSED) prefetch_l2_bulk(p.gate + m * p.gate_stride, (uint32_t)D * 2);
        }
    }
    if (FUSED && t == 0 && g == 0 && p.bias != nullptr) prefetch_l2_bulk(p.bias, (uint32_t)D * 2);
    if (t == 0)
#pragma unroll
        for (int s = 0; s < kPrefetchRows; ++s) {
            const int64_t r = first + s * groups;
            if (r >= r1) break;
            prefetch_l2_bulk(p.x + r * p.x_stride, (uint32_t)D * 2);
            if constexpr (FUSED) prefetch_l2_bulk(p.update + r * p.update_stride, (uint32_t)D * 2);
            if constexpr (O::DIRECT) {
                prefetch_l2_bulk(p.scale + r / p.seq * p.scale_stride, (uint32_t)D * 2);
                prefetch_l2_bulk(p.shift + r / p.seq * p.shift_stride, (uint32_t)D * 2);
            }
        }
    grid_dep_wait();
    grid_dep_launch();
    // FP8 producer: 1/scale correctly rounded, once per thread
    const float inv8 = p.out_fp8 != nullptr ? __fdiv_rn(1.0f, __ldg(p.fp8_scale)) : 0.0f;
    // NVFP4 copy: the global scale, and gs / value(s) for every E4M3 code s
    const float gs4 = FP4 ? __ldg(p.fp4_scale) : 0.0f;
    __shared__ float fp4_tab[FP4 ? 256 : 1];
    if constexpr (FP4) nvfp4_fill_table(fp4_tab, gs4);

    auto issue = [&](int s, int64_t row) {
        ring.issue(s, 0, p.x + row * p.x_stride, t, nch);
        if constexpr (O::U > 0) ring.issue(s, O::U, p.update + row * p.update_stride, t, nch);
        if constexpr (O::RING_MOD) {
            ring.issue(s, O::SC > 0 ? O::SC : 0, p.scale + next.q * p.scale_stride, t, nch);
            ring.issue(s, O::SH > 0 ? O::SH : 0, p.shift + next.q * p.shift_stride, t, nch);
        }
        if constexpr (MODE == kModRing && FUSED) ring.issue(s, O::G > 0 ? O::G : 0, p.gate + next.q * p.gate_stride, t, nch);
    };
#pragma unroll
    for (int s = 0; s < NS - 1; ++s) {
        const int64_t r = first + s * groups;
        if (r < r1) issue(s, r);
        if constexpr (MODE == kModRing) next.advance();
        cp_async_commit();
    }
    if constexpr (O::USTAGE) {  // the first row's update, a commit group of its own
        if (first < r1) ustage.issue(0, 0, p.update + first * p.update_stride, t, nch);
        cp_async_commit();
    }
    // the first rows are on their way; stage the modulation meanwhile
    if constexpr (MODE == kModStaged) {
        const int64_t m_last = (r1 - 1) / p.seq;
        const int slots = (int)(m_last - m0 + 1);  // 1 or 2 (host guarantees)
        for (int i = threadIdx.x; i < slots * nch; i += blockDim.x) {
            const int slot = i / nch, c = i - slot * nch;
            const uint4 sc = ld_shared_row(p.scale + (m0 + slot) * p.scale_stride + (int64_t)c * kChunk);
            const uint4 sh = ld_shared_row(p.shift + (m0 + slot) * p.shift_stride + (int64_t)c * kChunk);
            uint4 tv;
            if constexpr (!HIGH) {
                tv.x = badd(0x3f803f80u, sc.x);  // bf16(1 + scale), as the eager chain rounds it
                tv.y = badd(0x3f803f80u, sc.y);
                tv.z = badd(0x3f803f80u, sc.z);
                tv.w = badd(0x3f803f80u, sc.w);
            } else {
                tv = sc;
            }
            mod[(slot * O::SLOT + 0) * nch + c] = tv;
            mod[(slot * O::SLOT + 1) * nch + c] = sh;
            if constexpr (FUSED)
                mod[(slot * O::SLOT + 2) * nch + c] = ld_shared_row(p.gate + (m0 + slot) * p.gate_stride + (int64_t)c * kChunk);
        }
    }
    if constexpr (FUSED) {
        for (int c = threadIdx.x; c < bias_chunks; c += blockDim.x)
            bias_sm[c] = ld_shared_row(p.bias + (int64_t)c * kChunk);
    }
    if constexpr (MODE == kModStaged || FUSED || FP4) __syncthreads();

    int cur = 0, par = 0;
    for (int64_t row = first; row < r1; row += groups) {
        const int64_t rn = row + (NS - 1) * groups;
        const int sn = cur == 0 ? NS - 1 : cur - 1;
        if (rn < r1) issue(sn, rn);
        if constexpr (MODE == kModRing) next.advance();
        cp_async_commit();
        cp_async_wait<NS - 1>();
        const int slot = row >= split ? 1 : 0;
        // DIRECT: this row's scale and shift chunks, in flight during the statistics
        uint4 dT[O::DIRECT ? C::J : 1][O::DIRECT ? C::M : 1], dSH[O::DIRECT ? C::J : 1][O::DIRECT ? C::M : 1];
        if constexpr (O::DIRECT) {
            const uint16_t* sc_row = p.scale + here.q * p.scale_stride;
            const uint16_t* sh_row = p.shift + here.q * p.shift_stride;
#pragma unroll
            for (int j = 0; j < C::J; ++j)
#pragma unroll
                for (int m = 0; m < C::M; ++m) {
                    const int c = t + C::TPR * m + kLanes * j;
                    const bool ok = c < nch;
                    dT[j][m] = ok ? ld_stream(sc_row + (int64_t)c * kChunk) : make_uint4(0, 0, 0, 0);
                    dSH[j][m] = ok ? ld_stream(sh_row + (int64_t)c * kChunk) : make_uint4(0, 0, 0, 0);
                }
        }

        if constexpr (FUSED) {
            // front pass: the new residual r' = bf16(x + bf16(gate * a)), written
            // out and back over x in this thread's own ring chunks
            const uint4* gm = MODE == kModStaged ? mod + (slot * O::SLOT + 2) * nch : nullptr;
            const uint16_t* g_row = MODE == kModL1 ? p.gate + here.q * p.gate_stride : nullptr;
            uint16_t* res_row = p.res_out + row * p.res_out_stride;
#pragma unroll
            for (int j = 0; j < C::J; ++j)
#pragma unroll
                for (int m = 0; m < C::M; ++m) {
                    const int c = t + C::TPR * m + kLanes * j;
                    if (c >= nch) continue;
                    const uint4 X = lds16(ring.at(cur, 0, c));
                    uint4 U = O::USTAGE ? lds16(ustage.at(0, 0, c)) : lds16(ring.at(cur, O::U > 0 ? O::U : 0, c));
                    if (MODE == kModL1 ? p.bias != nullptr : bias_chunks != 0) {
                        const uint4 B = MODE == kModL1 ? ld_shared_row(p.bias + (int64_t)c * kChunk) : lds16(bias_sm + c);
                        U = make_uint4(badd(U.x, B.x), badd(U.y, B.y), badd(U.z, B.z), badd(U.w, B.w));
                    }
                    uint4 G;
                    if constexpr (MODE == kModStaged) G = lds16(gm + c);
                    else if constexpr (MODE == kModL1) G = ld_shared_row(g_row + (int64_t)c * kChunk);
                    else G = lds16(ring.at(cur, O::G > 0 ? O::G : 0, c));
                    const uint4 Y = make_uint4(badd(X.x, bmul(G.x, U.x)), badd(X.y, bmul(G.y, U.y)),
                                               badd(X.z, bmul(G.z, U.z)), badd(X.w, bmul(G.w, U.w)));
                    st_v4(res_row + (int64_t)c * kChunk, Y);
                    sts16(ring.at(cur, 0, c), Y);
                }
            if constexpr (O::USTAGE) {
                // this thread has consumed its update chunks: copy the next row's in
                // (the commit group the next row's wait completes together with x)
                if (row + groups < r1) ustage.issue(0, 0, p.update + (row + groups) * p.update_stride, t, nch);
                cp_async_commit();
            }
        }

        float mean = 0.0f, rstd = 0.0f;
        if constexpr (!HIGH) {
            Wf L[C::M];
            const bool full = nch == kLanes * C::J;
            welford_stage<C, !FUSED && (J == 1 || J == 3)>(ring, cur, t, nch, full, L, f2(p.neg_zero, p.neg_zero));
            const Wf s = full ? tree_allreduce_full<C>(L, t, sm, bar_id, par)
                              : tree_allreduce<C>(L, t, sm, bar_id, par, D, wf_combine);
            mean = s.mean;
            const float var = __fdiv_rn(s.m2, (float)D);
            rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(var, p.eps)));
        } else {
            if constexpr (C::J <= 2 && C::TPR == 32) {
                // short rows, one warp per row: two passes (mean, then squared
                // deviations), two trees
                float acc[C::M];
#pragma unroll
                for (int m = 0; m < C::M; ++m) {
                    acc[m] = 0.0f;
#pragma unroll
                    for (int j = 0; j < C::J; ++j) {
                        const int c = t + C::TPR * m + kLanes * j;
                        if (c >= nch) continue;
                        const uint4 v = lds16(ring.at(cur, 0, c));
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[m] += lo_f(w_of(v, i)) + hi_f(w_of(v, i));
                    }
                }
                // (one warp per row: both trees are shuffles only)
                mean = tree_w0_sum<C>(acc, t, sm, bar_id, par, [&](float S) {
                    return make_float2(S / (float)D, 0.0f);
                }).x;
#pragma unroll
                for (int m = 0; m < C::M; ++m) {
                    acc[m] = 0.0f;
#pragma unroll
                    for (int j = 0; j < C::J; ++j) {
                        const int c = t + C::TPR * m + kLanes * j;
                        if (c >= nch) continue;
                        const uint4 v = lds16(ring.at(cur, 0, c));
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float d0 = lo_f(w_of(v, i)) - mean, d1 = hi_f(w_of(v, i)) - mean;
                            acc[m] += d0 * d0 + d1 * d1;
                        }
                    }
                }
                rstd = tree_w0_sum<C>(acc, t, sm, bar_id, par, [&](float q) {
                    return make_float2(rsqrtf(q / (float)D + p.eps), 0.0f);
                }).x;
            } else {
                // longer rows, or more than one warp per row: each lane's mean
                // and sum of squared deviations from its own elements (two
                // passes over the lane's chunks), then one tree of Chan
                // combines (measured faster from J = 3)
                // (element pairs of a word in f32x2, two accumulators per pass:
                // short dependency chains)
                Wf L[C::M];
#pragma unroll
                for (int m = 0; m < C::M; ++m) {
                    u64 s2[2] = {f2(0.0f, 0.0f), f2(0.0f, 0.0f)};
                    int n = 0;
#pragma unroll
                    for (int j = 0; j < C::J; ++j) {
                        const int c = t + C::TPR * m + kLanes * j;
                        if (c >= nch) continue;
                        const uint4 v = lds16(ring.at(cur, 0, c));
                        n += kChunk;
#pragma unroll
                        for (int i = 0; i < 4; ++i) s2[i & 1] = add2(s2[i & 1], widen2(w_of(v, i)));
                    }
                    const u64 sum = add2(s2[0], s2[1]);
                    const float lm = n ? (f2lo(sum) + f2hi(sum)) / (float)n : 0.0f;
                    const u64 lm2 = f2(lm, lm);
                    u64 q2[2] = {f2(0.0f, 0.0f), f2(0.0f, 0.0f)};
#pragma unroll
                    for (int j = 0; j < C::J; ++j) {
                        const int c = t + C::TPR * m + kLanes * j;
                        if (c >= nch) continue;
                        const uint4 v = lds16(ring.at(cur, 0, c));
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const u64 d = sub2(widen2(w_of(v, i)), lm2);
                            q2[i & 1] = fma2(d, d, q2[i & 1]);
                        }
                    }
                    const u64 q = add2(q2[0], q2[1]);
                    L[m] = Wf{lm, f2lo(q) + f2hi(q), (float)n};
                }
                const bool full = nch == kLanes * C::J;
                const Wf st = full ? tree_allreduce_full<C>(L, t, sm, bar_id, par)
                                   : tree_allreduce<C>(L, t, sm, bar_id, par, D, wf_combine);
                mean = st.mean;
                rstd = rsqrtf(st.m2 / (float)D + p.eps);
            }
            }

        const uint4* tm = MODE == kModStaged ? mod + (slot * O::SLOT + 0) * nch : nullptr;
        const uint4* sh = MODE == kModStaged ? tm + nch : nullptr;
        const uint16_t* sc_l1 = MODE == kModL1 ? p.scale + here.q * p.scale_stride : nullptr;
        const uint16_t* sh_l1 = MODE == kModL1 ? p.shift + here.q * p.shift_stride : nullptr;
        uint16_t* out_row = p.out + row * p.out_stride;
        uint8_t* const q_row = FP4 ? p.out_fp4 + row * p.out_fp4_stride : nullptr;
        uint8_t* const sf_row = FP4 ? p.out_sf + nvfp4_sf_row(row, p.sf_col_tiles) : nullptr;
        const u64 mean2 = f2(mean, mean), rstd2 = f2(rstd, rstd);
#pragma unroll
        for (int j = 0; j < C::J; ++j)
#pragma unroll
            for (int m = 0; m < C::M; ++m) {
                const int c = t + C::TPR * m + kLanes * j;
                // FP4 and L1 modes: a chunk past the end of a short row is
                // computed from whatever its ring slot holds with only its
                // stores skipped (no branch: every lane takes part in the FP4
                // block shuffle, and the L1 loads can be issued early).
                // Otherwise each chunk is tested and a missing one skipped:
                // measured faster there (the compiler then keeps each chunk's
                // loads beside its use).
                constexpr bool kNoBranch = FP4 || MODE == kModL1;
                if constexpr (!kNoBranch) {
                    if (c >= nch) continue;
                }
                const bool valid = !kNoBranch || j < C::J - 1 || c < nch;
                const int cv = valid ? c : 0;  // FP4 reads of a missing chunk stay in its row's slots
                const uint4 X = lds16(ring.at(cur, 0, c));
                uint4 T, SH;
                if constexpr (MODE == kModStaged) {
                    T = lds16(tm + cv);
                    SH = lds16(sh + cv);
                } else if constexpr (MODE == kModL1) {
                    T = ld_shared_row(sc_l1 + (int64_t)cv * kChunk);
                    SH = ld_shared_row(sh_l1 + (int64_t)cv * kChunk);
                } else if constexpr (O::DIRECT) {
                    T = dT[O::DIRECT ? j : 0][O::DIRECT ? m : 0];
                    SH = dSH[O::DIRECT ? j : 0][O::DIRECT ? m : 0];
                } else {
                    T = lds16(ring.at(cur, O::SC > 0 ? O::SC : 0, c));
                    SH = lds16(ring.at(cur, O::SH > 0 ? O::SH : 0, c));
                }
                uint4 o;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t xw = w_of(X, i), tw = w_of(T, i), hw = w_of(SH, i);
                    uint32_t ow;
                    if constexpr (!HIGH) {
                        const uint32_t nrm = pack2_rn(mul2(sub2(widen2(xw), mean2), rstd2));
                        // ring and L1 modes carry scale itself: round 1 + scale here
                        const uint32_t tt = MODE == kModStaged ? tw : badd(0x3f803f80u, tw);
                        ow = badd(bmul(nrm, tt), hw);
                    } else {
                        const u64 nrm = mul2(sub2(widen2(xw), mean2), rstd2);
                        ow = pack2_rn(fma2(nrm, add2(widen2(tw), f2(1.0f, 1.0f)), widen2(hw)));
                    }
                    w_set(o, i, ow);
                }
                if (!kNoBranch || valid) {
                    st_v4(out_row + (int64_t)c * kChunk, o);
                    if (p.out_fp8 != nullptr)
                        st_v2(p.out_fp8 + row * p.out_fp8_stride + (int64_t)c * kChunk, e4m3x4_of_bf16(o.x, o.y, inv8),
                              e4m3x4_of_bf16(o.z, o.w, inv8));
                }
                if constexpr (FP4) {
                    // a 16-element block is chunks 2b and 2b+1, held by lanes
                    // t and t^1 of the same warp
                    const float a8 = valid ? amax8_bf16(o) : 0.0f;
                    const float a16 = max_nan(a8, __shfl_xor_sync(0xffffffffu, a8, 1));
                    float esc;
                    const uint32_t sc = nvfp4_block_scale_tab(a16, gs4, fp4_tab, esc);
                    const uint32_t q = nvfp4_codes_esc(o, sc, esc);
                    if (valid) st_u32(q_row + c * 4, q);
                    if (valid && (c & 1) == 0) sf_row[nvfp4_sf_block(c >> 1)] = (uint8_t)sc;
                }
            }
        cur = cur + 1 == NS ? 0 : cur + 1;
        par ^= 1;
        if constexpr (kHere) here.advance();
    }
    cp_async_wait<0>();
}

// ------------------------------------------------------------------ launch helpers

template <int TPR, int J, int NS, bool HIGH, int MODE, bool FUSED, bool FP4>
static cudaError_t launch_pipe(const LnModParams& p, cudaStream_t s) {
    auto k = ln_modulate_pipe_kernel<TPR, J, NS, HIGH, MODE, FUSED, FP4>;
    using C = RowCfg<TPR, J, true>;
    using O = LnOps<FUSED, MODE, J, HIGH>;
    using R = Ring<C, NS, O::N>;
    const int nch = p.D / kChunk;
    const int fixed = (MODE == kModStaged ? 2 * O::SLOT * nch * 16 : 0) + (FUSED && MODE != kModL1 && p.bias ? nch * 16 : 0);
    PipeShape sh;
    const int per_group = (int)sizeof(TreeAll<TPR>) + R::kBytes + (O::USTAGE ? Ring<C, 1, 1>::kBytes : 0);
    if (!pipe_shape(reinterpret_cast<const void*>(k), TPR, per_group, fixed, p.rows, &sh))
        return cudaErrorInvalidConfiguration;
    return launch_pdl(k, sh.grid, sh.groups * TPR, sh.smem, s, p, sh.rows_per_cta);
}

// Threads per row of the ring kernel for rows of J chunks per lane, measured
// per row width and kind of kernel (plain LN and its FP8 copy share one
// kernel; the NVFP4 copy and the fused gated kernel have their own):
//   J = 1 (D <= 1024):  fused 64; otherwise 32
//   J = 2 (D <= 2048):  plain lossless and FP8 64; otherwise 32
//   J = 3 (D <= 3072):  fused 128; FP8 128 from 32768 rows; otherwise 64
//   J = 4 (D <= 4096):  plain and FP8 128; otherwise 64
//   J = 5 (D <= 5120):  fused high with per-row modulation 64; otherwise 128
//   J >= 6:             128
// One warp per row keeps the high variant's short rows on two shuffle-only
// trees (plain LN, J <= 2); with more warps it takes the lane two-pass form of
// longer rows.  `ring`: each row reads its own modulation row (kModRing).
static int ln_tpr(int J, bool fused, bool fp4, bool fp8, bool high, int64_t rows, bool ring) {
    const bool plain = !fused && !fp4;
    switch (J) {
        case 1: return fused ? 64 : 32;
        case 2: return plain && (fp8 || !high) ? 64 : 32;
        case 3: return fused || (plain && fp8 && rows >= 32768) ? 128 : 64;
        case 4: return plain ? 128 : 64;
        case 5: return fused && !fp4 && high && ring ? 64 : 128;
        default: return 128;
    }
}

// Row groups of the fused kernel that fit in shared memory in a modulation
// mode: its stages carry the residual and the update (per token also the
// gate, and scale and shift where they are not loaded directly); staged
// per-sample modulation, gate and bias take a fixed share.  Same arithmetic
// as launch_pipe.
static int fused_groups(const LnModParams& p, bool high, int mode, bool fp4) {
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    const int J = chunks_per_lane(p.D), nch = p.D / kChunk;
    const int nops = ln_ring_ops(true, mode, J, high);
    const int tpr = ln_tpr(J, true, fp4, false, high, p.rows, mode == kModRing);  // as launch_pipe_d chooses
    const int tree = tpr == 32 ? (int)sizeof(TreeAll<32>) : tpr == 64 ? (int)sizeof(TreeAll<64>) : (int)sizeof(TreeAll<128>);
    const int per_group = tree + (2 * nops + (ln_update_one_stage(J) ? 1 : 0)) * kLanes * J * 16;  // + the update's one stage
    const int fixed = (mode == kModStaged ? 2 * LnOps<true, kModStaged, 1, false>::SLOT * nch * 16 : 0) +
                      (mode != kModL1 && p.bias ? nch * 16 : 0);
    return (optin - 8 * 1024 - fixed) / per_group;
}

// The fused kernel's modulation mode, or -1 when no mode keeps at least two
// row groups per SM (then two launches, gated add and LN, run faster).
// Per-sample rows stage their vectors unless reading them from L1 fits at
// least twice the row groups (rows of more than 4096 elements).
static int fused_mode(const LnModParams& p, bool high, bool fp4) {
    const bool staged = pipe_rows_per_cta(p.rows) <= p.seq;
    if (!staged) return fused_groups(p, high, kModRing, fp4) >= 2 ? kModRing : -1;
    const int cap = 512 / ln_tpr(chunks_per_lane(p.D), true, fp4, false, high, p.rows, false);  // 512 threads per CTA
    const int gs = std::min(fused_groups(p, high, kModStaged, fp4), cap);
    const int gl = chunks_per_lane(p.D) >= 5 ? std::min(fused_groups(p, high, kModL1, fp4), cap) : 0;
    // the L1 mode's global reads cost more than the staged form's shared ones:
    // taken where it fits at least twice the row groups (measured)
    if (gs >= 2 && gl < 2 * gs) return kModStaged;
    return gl >= 2 ? kModL1 : -1;
}

// fp4: the kernel with the NVFP4 store (its threads per row may differ)
static bool fused_fits(const LnModParams& p, bool high, bool fp4) { return fused_mode(p, high, fp4) >= 0; }

template <int TPR, int J, int NS, bool FUSED, bool FP4>
static cudaError_t launch_pipe_v(const LnModParams& p, bool high, cudaStream_t s) {
    // stage the modulation when each CTA's block of rows spans at most two
    // samples (rows per CTA <= seq); otherwise read it per row
    const bool staged = pipe_rows_per_cta(p.rows) <= p.seq;
    if constexpr (FUSED && J >= 5) {
        if (staged && fused_mode(p, high, FP4) == kModL1)
            return high ? launch_pipe<TPR, J, NS, true, kModL1, FUSED, FP4>(p, s)
                        : launch_pipe<TPR, J, NS, false, kModL1, FUSED, FP4>(p, s);
    }
    if (high)
        return staged ? launch_pipe<TPR, J, NS, true, kModStaged, FUSED, FP4>(p, s)
                      : launch_pipe<TPR, J, NS, true, kModRing, FUSED, FP4>(p, s);
    return staged ? launch_pipe<TPR, J, NS, false, kModStaged, FUSED, FP4>(p, s)
                  : launch_pipe<TPR, J, NS, false, kModRing, FUSED, FP4>(p, s);
}

template <bool FUSED, bool FP4>
static cudaError_t launch_pipe_d(const LnModParams& p, bool high, cudaStream_t s) {
    // threads per row from ln_tpr; `if constexpr` keeps each kind of kernel to
    // the instantiations its table entries name
    constexpr bool kPlain = !FUSED && !FP4;
    const int J = chunks_per_lane(p.D);
    const bool ring = pipe_rows_per_cta(p.rows) > p.seq;  // as launch_pipe_v decides
    const int tpr = ln_tpr(J, FUSED, FP4, p.out_fp8 != nullptr, high, p.rows, ring);
    switch (J) {
        case 1:
            if constexpr (FUSED) return launch_pipe_v<64, 1, 2, FUSED, FP4>(p, high, s);
            else return launch_pipe_v<32, 1, 2, FUSED, FP4>(p, high, s);
        case 2:
            if constexpr (kPlain) {
                if (tpr == 64) return launch_pipe_v<64, 2, 2, FUSED, FP4>(p, high, s);
            }
            return launch_pipe_v<32, 2, 2, FUSED, FP4>(p, high, s);
        case 3:
            if constexpr (FUSED) {
                return launch_pipe_v<128, 3, 2, FUSED, FP4>(p, high, s);
            } else {
                if constexpr (kPlain) {
                    if (tpr == 128) return launch_pipe_v<128, 3, 2, FUSED, FP4>(p, high, s);
                }
                return launch_pipe_v<64, 3, 2, FUSED, FP4>(p, high, s);
            }
        case 4:
            if constexpr (kPlain) return launch_pipe_v<128, 4, 2, FUSED, FP4>(p, high, s);
            else return launch_pipe_v<64, 4, 2, FUSED, FP4>(p, high, s);
        case 5:
            if constexpr (FUSED && !FP4) {
                if (tpr == 64) return launch_pipe<64, 5, 2, true, kModRing, FUSED, FP4>(p, s);
            }
            return launch_pipe_v<128, 5, 2, FUSED, FP4>(p, high, s);
        case 6: return launch_pipe_v<128, 6, 2, FUSED, FP4>(p, high, s);
        case 7: return launch_pipe_v<128, 7, 2, FUSED, FP4>(p, high, s);
        case 8:
            // the FP8 copy at 8192 takes a third ring stage from 32768 rows
            // (measured +6..8% at 65536 rows, -6% at 4096; slower for the
            // plain LN and the NVFP4 copy)
            if constexpr (kPlain) {
                if (p.out_fp8 != nullptr && p.rows >= 32768) return launch_pipe_v<128, 8, 3, FUSED, FP4>(p, high, s);
            }
            return launch_pipe_v<128, 8, 2, FUSED, FP4>(p, high, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mbx
