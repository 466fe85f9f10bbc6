// mbx_api.cu -- the C ABI of libmbx.so: argument validation and dispatch.
//
// Validation order (the first failing check decides the status):
//   1. pure host checks: NULL, dtype, empty, hidden size, shapes, strides,
//      element alignment, variant, eps, overlap between outputs and inputs;
//   2. device checks: every pointer is device (or managed) memory of the
//      current device, and every view lies inside one allocation
//      (cuMemGetAddressRange, looked up through the runtime so that the
//      library loads on machines without a driver).
// Nothing is launched unless every check passes.  The guard set follows the
// BF16-native RMSNorm wrapper of "#34085 [diffusion] Clean up kernels and
// shared fast paths" (prhub.com.cn), sections 实现拆解 item 2 and 关键源码片段.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "mbx.h"
#include "kernels/launch.h"

namespace {

constexpr int64_t kMaxHidden = 8192;  // MAX_HIDDEN_SIZE of the pages' guard

struct V {  // a view in one form, for the checks
    const void* data;
    int64_t rows, cols, stride;
    int32_t dtype;
};

V of(const mbx_cview* v) { return V{v->data, v->rows, v->cols, v->row_stride, v->dtype}; }
V of(const mbx_view* v) { return V{v->data, v->rows, v->cols, v->row_stride, v->dtype}; }

int64_t esize(int32_t dtype) { return dtype == MBX_F32 ? 4 : (dtype == MBX_E4M3 || dtype == MBX_E2M1X2) ? 1 : 2; }

// Bytes from a view's first element to one past its last.  Only called on
// views that extent_ok() accepted, so nothing here can overflow.
int64_t extent_bytes(const V& v) {
    return ((v.rows > 1 ? (v.rows - 1) * v.stride : 0) + v.cols) * esize(v.dtype);
}

// A view whose extent does not fit in 63 bits, or whose end address would
// wrap around, cannot lie inside any allocation: refused as out of bounds
// before any other check does arithmetic on it.  rows, cols > 0 and
// stride >= cols (for rows > 1) are checked first.
int extent_ok(const V& v) {
    int64_t span = 0, elems = 0, bytes = 0;
    uintptr_t end = 0;
    if (v.rows > 1 && __builtin_mul_overflow(v.rows - 1, v.stride, &span)) return MBX_E_BOUNDS;
    if (__builtin_add_overflow(span, v.cols, &elems)) return MBX_E_BOUNDS;
    if (__builtin_mul_overflow(elems, esize(v.dtype), &bytes)) return MBX_E_BOUNDS;
    if (__builtin_add_overflow(reinterpret_cast<uintptr_t>(v.data), (uintptr_t)bytes, &end))
        return MBX_E_BOUNDS;
    return MBX_OK;
}

// Step 1 of a view: dtype, non-empty, stride, alignment, extent.
int basic(const V& v) {
    if (v.data == nullptr) return MBX_E_NULL;
    if (v.dtype != MBX_BF16) return MBX_E_DTYPE;
    if (v.rows <= 0 || v.cols <= 0) return MBX_E_EMPTY;
    if (v.rows > 1 && v.stride < v.cols) return MBX_E_STRIDE;
    if (reinterpret_cast<uintptr_t>(v.data) % 2) return MBX_E_ALIGN;
    return extent_ok(v);
}

bool overlaps(const V& a, const V& b) {
    uintptr_t a0 = reinterpret_cast<uintptr_t>(a.data), b0 = reinterpret_cast<uintptr_t>(b.data);
    uintptr_t a1 = a0 + (uintptr_t)extent_bytes(a), b1 = b0 + (uintptr_t)extent_bytes(b);
    return a0 < b1 && b0 < a1;
}

bool same_view(const V& a, const V& b) {
    return a.data == b.data && a.rows == b.rows && a.cols == b.cols &&
           (a.rows == 1 || a.stride == b.stride);
}

bool aligned16(const V& v) {
    return reinterpret_cast<uintptr_t>(v.data) % 16 == 0 && (v.rows == 1 || (v.stride * esize(v.dtype)) % 16 == 0);
}

// basic() for an operand that may be bfloat16 or binary32.
int basic_any(const V& v) {
    if (v.data == nullptr) return MBX_E_NULL;
    if (v.dtype != MBX_BF16 && v.dtype != MBX_F32) return MBX_E_DTYPE;
    if (v.rows <= 0 || v.cols <= 0) return MBX_E_EMPTY;
    if (v.rows > 1 && v.stride < v.cols) return MBX_E_STRIDE;
    if (reinterpret_cast<uintptr_t>(v.data) % esize(v.dtype)) return MBX_E_ALIGN;
    return extent_ok(v);
}

int check_variant_eps(int variant, float eps) {
    if (variant != MBX_LOSSLESS && variant != MBX_HIGH) return MBX_E_VARIANT;
    if (!(eps >= 0.0f) || !std::isfinite(eps)) return MBX_E_ARG;
    return MBX_OK;
}

// ---------------------------------------------------------------- device checks

typedef CUresult (*AddrRangeFn)(CUdeviceptr*, size_t*, CUdeviceptr);

AddrRangeFn addr_range_fn() {
    static AddrRangeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<AddrRangeFn>(p);
        cudaGetLastError();
    });
    return fn;
}

int device_ok(const void* ptr, int64_t bytes, int dev) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();
        return MBX_E_DEVICE;
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) return MBX_E_DEVICE;
    if (a.type == cudaMemoryTypeDevice && a.device != dev) return MBX_E_DEVICE;
    AddrRangeFn fn = addr_range_fn();
    if (fn == nullptr) return MBX_E_DEVICE;
    CUdeviceptr base = 0;
    size_t size = 0;
    if (fn(&base, &size, reinterpret_cast<CUdeviceptr>(ptr)) != CUDA_SUCCESS) {
        return a.type == cudaMemoryTypeManaged ? MBX_OK : MBX_E_BOUNDS;
    }
    // base <= ptr < base + size; compare the remaining room, never a sum
    uintptr_t p0 = reinterpret_cast<uintptr_t>(ptr), b0 = (uintptr_t)base;
    if (p0 < b0 || bytes < 0 || (uintptr_t)bytes > b0 + size - p0) return MBX_E_BOUNDS;
    return MBX_OK;
}

int current_device(int* dev) {
    if (cudaGetDevice(dev) != cudaSuccess) {
        cudaGetLastError();
        return MBX_E_DEVICE;
    }
    return MBX_OK;
}

int views_on_device(const V* vs, int n) {
    int dev = 0;
    if (int st = current_device(&dev)) return st;
    for (int i = 0; i < n; ++i)
        if (int st = device_ok(vs[i].data, extent_bytes(vs[i]), dev)) return st;
    return MBX_OK;
}

int raw_on_device(const void* p, int64_t bytes) {
    int dev = 0;
    if (int st = current_device(&dev)) return st;
    return device_ok(p, bytes, dev);
}

#define MBX_TRY(expr)                   \
    do {                                \
        int _st = (expr);               \
        if (_st != MBX_OK) return _st;  \
    } while (0)

// Modulation view m against x: same width, rows of x a multiple of its rows.
int check_mod(const V& m, const V& x) {
    if (m.cols != x.cols) return MBX_E_SHAPE;
    if (x.rows % m.rows != 0) return MBX_E_SHAPE;
    return MBX_OK;
}

int check_weight(const V& w, const V& x) {
    if (w.rows != 1 || w.cols != x.cols) return MBX_E_SHAPE;
    return MBX_OK;
}

// ---------------------------------------------------------------- per op

int check_ln_modulate(const mbx_view* out, const mbx_cview* x, const mbx_cview* scale,
                      const mbx_cview* shift, float eps, int variant, bool dev) {
    if (!out || !x || !scale || !shift) return MBX_E_NULL;
    V o = of(out), xv = of(x), sc = of(scale), sh = of(shift);
    if (!o.data || !xv.data || !sc.data || !sh.data) return MBX_E_NULL;
    for (const V* v : {&o, &xv, &sc, &sh})
        if (v->dtype != MBX_BF16) return MBX_E_DTYPE;
    for (const V* v : {&o, &xv, &sc, &sh}) MBX_TRY(basic(*v));
    if (xv.cols > kMaxHidden) return MBX_E_DIM_TOO_LARGE;
    if (o.rows != xv.rows || o.cols != xv.cols) return MBX_E_SHAPE;
    MBX_TRY(check_mod(sc, xv));
    MBX_TRY(check_mod(sh, xv));
    if (sc.rows != sh.rows) return MBX_E_SHAPE;
    MBX_TRY(check_variant_eps(variant, eps));
    for (const V* v : {&xv, &sc, &sh})
        if (overlaps(o, *v)) return MBX_E_ALIAS;
    if (dev) {
        V all[4] = {o, xv, sc, sh};
        MBX_TRY(views_on_device(all, 4));
    }
    return MBX_OK;
}

int check_rmsnorm_scale(const mbx_view* out, const mbx_cview* x, const mbx_cview* weight,
                        const mbx_cview* scale, float eps, int variant, bool dev) {
    if (!out || !x || !weight || !scale) return MBX_E_NULL;
    V o = of(out), xv = of(x), w = of(weight), sc = of(scale);
    if (!o.data || !xv.data || !w.data || !sc.data) return MBX_E_NULL;
    for (const V* v : {&o, &xv, &w, &sc})
        if (v->dtype != MBX_BF16) return MBX_E_DTYPE;
    for (const V* v : {&o, &xv, &w, &sc}) MBX_TRY(basic(*v));
    if (xv.cols > kMaxHidden) return MBX_E_DIM_TOO_LARGE;
    if (o.rows != xv.rows || o.cols != xv.cols) return MBX_E_SHAPE;
    MBX_TRY(check_weight(w, xv));
    MBX_TRY(check_mod(sc, xv));
    MBX_TRY(check_variant_eps(variant, eps));
    for (const V* v : {&xv, &w, &sc})
        if (overlaps(o, *v)) return MBX_E_ALIAS;
    if (dev) {
        V all[4] = {o, xv, w, sc};
        MBX_TRY(views_on_device(all, 4));
    }
    return MBX_OK;
}

int check_rmsnorm_tanh_residual(const mbx_view* out, const mbx_cview* x, const mbx_cview* gate,
                                const mbx_cview* residual, const mbx_cview* weight, float eps,
                                int variant, bool dev) {
    if (!out || !x || !gate || !residual || !weight) return MBX_E_NULL;
    V o = of(out), xv = of(x), g = of(gate), r = of(residual), w = of(weight);
    if (!o.data || !xv.data || !g.data || !r.data || !w.data) return MBX_E_NULL;
    for (const V* v : {&o, &xv, &g, &r, &w})
        if (v->dtype != MBX_BF16) return MBX_E_DTYPE;
    for (const V* v : {&o, &xv, &g, &r, &w}) MBX_TRY(basic(*v));
    if (xv.cols > kMaxHidden) return MBX_E_DIM_TOO_LARGE;
    if (o.rows != xv.rows || o.cols != xv.cols) return MBX_E_SHAPE;
    if (r.rows != xv.rows || r.cols != xv.cols) return MBX_E_SHAPE;
    MBX_TRY(check_mod(g, xv));
    MBX_TRY(check_weight(w, xv));
    MBX_TRY(check_variant_eps(variant, eps));
    for (const V* v : {&xv, &g, &w})
        if (overlaps(o, *v)) return MBX_E_ALIAS;
    if (overlaps(o, r) && !same_view(o, r)) return MBX_E_ALIAS;  // in place on residual only
    if (dev) {
        V all[5] = {o, xv, g, r, w};
        MBX_TRY(views_on_device(all, 5));
    }
    return MBX_OK;
}

int check_residual_gate_add(const mbx_view* out, const mbx_cview* x, const mbx_cview* gate,
                            const mbx_cview* y, int variant, bool dev) {
    if (!out || !x || !gate || !y) return MBX_E_NULL;
    V o = of(out), xv = of(x), g = of(gate), yv = of(y);
    if (!o.data || !xv.data || !g.data || !yv.data) return MBX_E_NULL;
    for (const V* v : {&o, &xv, &g, &yv})
        if (v->dtype != MBX_BF16) return MBX_E_DTYPE;
    for (const V* v : {&o, &xv, &g, &yv}) MBX_TRY(basic(*v));
    if (xv.cols > kMaxHidden) return MBX_E_DIM_TOO_LARGE;
    if (o.rows != xv.rows || o.cols != xv.cols) return MBX_E_SHAPE;
    if (yv.rows != xv.rows || yv.cols != xv.cols) return MBX_E_SHAPE;
    MBX_TRY(check_mod(g, xv));
    MBX_TRY(check_variant_eps(variant, 0.0f));
    for (const V* v : {&g, &yv})
        if (overlaps(o, *v)) return MBX_E_ALIAS;
    if (overlaps(o, xv) && !same_view(o, xv)) return MBX_E_ALIAS;  // in place on x only
    if (dev) {
        V all[4] = {o, xv, g, yv};
        MBX_TRY(views_on_device(all, 4));
    }
    return MBX_OK;
}

int check_gated(const mbx_view* res_out, const mbx_view* out, const mbx_cview* residual,
                const mbx_cview* gate, const mbx_cview* update, const mbx_cview* bias,
                const mbx_cview* scale, const mbx_cview* shift, float eps, int variant, bool dev) {
    if (!res_out || !out || !residual || !gate || !update || !scale || !shift) return MBX_E_NULL;
    V ro = of(res_out), o = of(out), r = of(residual), g = of(gate), u = of(update), sc = of(scale),
      sh = of(shift);
    const bool has_b = bias != nullptr;
    V b = has_b ? of(bias) : V{nullptr, 0, 0, 0, MBX_BF16};
    if (!ro.data || !o.data || !r.data || !g.data || !u.data || !sc.data || !sh.data) return MBX_E_NULL;
    if (has_b && !b.data) return MBX_E_NULL;
    for (const V* v : {&ro, &o, &r, &g, &u, &sc, &sh})
        if (v->dtype != MBX_BF16) return MBX_E_DTYPE;
    if (has_b && b.dtype != MBX_BF16) return MBX_E_DTYPE;
    for (const V* v : {&ro, &o, &r, &g, &u, &sc, &sh}) MBX_TRY(basic(*v));
    if (has_b) MBX_TRY(basic(b));
    if (r.cols > kMaxHidden) return MBX_E_DIM_TOO_LARGE;
    for (const V* v : {&ro, &o, &u})
        if (v->rows != r.rows || v->cols != r.cols) return MBX_E_SHAPE;
    MBX_TRY(check_mod(g, r));
    MBX_TRY(check_mod(sc, r));
    MBX_TRY(check_mod(sh, r));
    if (g.rows != sc.rows || sc.rows != sh.rows) return MBX_E_SHAPE;
    if (has_b) MBX_TRY(check_weight(b, r));
    MBX_TRY(check_variant_eps(variant, eps));
    for (const V* v : {&r, &g, &u, &sc, &sh, &ro})
        if (overlaps(o, *v)) return MBX_E_ALIAS;
    if (has_b && overlaps(o, b)) return MBX_E_ALIAS;
    for (const V* v : {&g, &u, &sc, &sh})
        if (overlaps(ro, *v)) return MBX_E_ALIAS;
    if (has_b && overlaps(ro, b)) return MBX_E_ALIAS;
    if (overlaps(ro, r) && !same_view(ro, r)) return MBX_E_ALIAS;  // in place on the residual only
    if (dev) {
        V all[8] = {ro, o, r, g, u, sc, sh, b};
        MBX_TRY(views_on_device(all, has_b ? 8 : 7));
    }
    return MBX_OK;
}

// The FP8 producers' extra output and scale: E4M3 [rows, D] like `out`,
// overlapping none of the other views; the scale one device binary32.
int check_fp8(const mbx_view* out_fp8, const float* fp8_scale, const V* others, int n, bool dev) {
    if (!out_fp8 || !out_fp8->data || !fp8_scale) return MBX_E_NULL;
    V q = of(out_fp8);
    if (q.dtype != MBX_E4M3) return MBX_E_DTYPE;
    if (q.rows <= 0 || q.cols <= 0) return MBX_E_EMPTY;
    if (q.rows > 1 && q.stride < q.cols) return MBX_E_STRIDE;
    MBX_TRY(extent_ok(q));
    if (reinterpret_cast<uintptr_t>(fp8_scale) % 4) return MBX_E_ALIGN;
    if (q.rows != others[0].rows || q.cols != others[0].cols) return MBX_E_SHAPE;  // others[0] = out
    for (int i = 0; i < n; ++i)
        if (overlaps(q, others[i])) return MBX_E_ALIAS;
    if (dev) {
        MBX_TRY(views_on_device(&q, 1));
        MBX_TRY(raw_on_device(fp8_scale, 4));
    }
    return MBX_OK;
}

// The NVFP4 producers' outputs: packed values [rows, D/2] (MBX_E2M1X2) and the
// swizzled block scales [pad128(rows), pad4(D/16)] (MBX_E4M3, contiguous).
int check_fp4(const mbx_view* out_fp4, const mbx_view* out_sf, const float* fp4_scale, const V* others,
              int n, bool dev) {
    if (!out_fp4 || !out_fp4->data || !out_sf || !out_sf->data || !fp4_scale) return MBX_E_NULL;
    V q = of(out_fp4), f = of(out_sf);
    if (q.dtype != MBX_E2M1X2 || f.dtype != MBX_E4M3) return MBX_E_DTYPE;
    if (q.rows <= 0 || q.cols <= 0 || f.rows <= 0 || f.cols <= 0) return MBX_E_EMPTY;
    if ((q.rows > 1 && q.stride < q.cols) || (f.rows > 1 && f.stride != f.cols)) return MBX_E_STRIDE;
    MBX_TRY(extent_ok(q));
    MBX_TRY(extent_ok(f));
    if (reinterpret_cast<uintptr_t>(fp4_scale) % 4) return MBX_E_ALIGN;
    const int64_t rows = others[0].rows, D = others[0].cols;  // others[0] = out
    if (D % 16) return MBX_E_SHAPE;
    if (q.rows != rows || q.cols != D / 2) return MBX_E_SHAPE;
    if (f.rows != (rows + 127) / 128 * 128 || f.cols != (D / 16 + 3) / 4 * 4) return MBX_E_SHAPE;
    if (overlaps(q, f)) return MBX_E_ALIAS;
    for (int i = 0; i < n; ++i)
        if (overlaps(q, others[i]) || overlaps(f, others[i])) return MBX_E_ALIAS;
    if (dev) {
        V all[2] = {q, f};
        MBX_TRY(views_on_device(all, 2));
        MBX_TRY(raw_on_device(fp4_scale, 4));
    }
    return MBX_OK;
}

void set_fp4(mbx::LnModParams& p, const mbx_view* out_fp4, const mbx_view* out_sf, const float* fp4_scale) {
    p.out_fp4 = static_cast<uint8_t*>(out_fp4->data);
    p.out_fp4_stride = out_fp4->row_stride;
    p.out_sf = static_cast<uint8_t*>(out_sf->data);
    p.sf_col_tiles = (int)(out_sf->cols / 4);
    p.fp4_scale = fp4_scale;
}

bool aligned4_fp4(const mbx_view* q) {
    return reinterpret_cast<uintptr_t>(q->data) % 4 == 0 && (q->rows == 1 || q->row_stride % 4 == 0);
}

bool aligned8_fp8(const mbx_view* q) {
    return reinterpret_cast<uintptr_t>(q->data) % 8 == 0 && (q->rows == 1 || q->row_stride % 8 == 0);
}

mbx::LnModParams gated_params(const mbx_view* residual_out, const mbx_view* out, const mbx_cview* residual,
                              const mbx_cview* gate, const mbx_cview* update, const mbx_cview* bias,
                              const mbx_cview* scale, const mbx_cview* shift, float eps) {
    mbx::LnModParams p;
    p.out = static_cast<uint16_t*>(out->data);
    p.out_stride = out->row_stride;
    p.x = static_cast<const uint16_t*>(residual->data);
    p.x_stride = residual->row_stride;
    p.scale = static_cast<const uint16_t*>(scale->data);
    p.scale_stride = scale->row_stride;
    p.shift = static_cast<const uint16_t*>(shift->data);
    p.shift_stride = shift->row_stride;
    p.rows = residual->rows;
    p.D = (int)residual->cols;
    p.seq = residual->rows / scale->rows;
    p.eps = eps;
    p.update = static_cast<const uint16_t*>(update->data);
    p.update_stride = update->row_stride;
    p.gate = static_cast<const uint16_t*>(gate->data);
    p.gate_stride = gate->row_stride;
    p.bias = bias ? static_cast<const uint16_t*>(bias->data) : nullptr;
    p.res_out = static_cast<uint16_t*>(residual_out->data);
    p.res_out_stride = residual_out->row_stride;
    return p;
}

bool gated_vec(const mbx::LnModParams& p, const mbx_view* residual_out, const mbx_view* out,
               const mbx_cview* residual, const mbx_cview* gate, const mbx_cview* update,
               const mbx_cview* bias, const mbx_cview* scale, const mbx_cview* shift) {
    bool vec = p.D % 8 == 0 && aligned16(of(residual_out)) && aligned16(of(out)) && aligned16(of(residual)) &&
               aligned16(of(gate)) && aligned16(of(update)) && aligned16(of(scale)) && aligned16(of(shift));
    if (bias) vec = vec && aligned16(of(bias));
    return vec;
}

int check_modtable(const mbx_view* out, const mbx_cview* table, const mbx_cview* temb, bool dev) {
    if (!out || !table || !temb) return MBX_E_NULL;
    V o = of(out), t = of(table), e = of(temb);
    MBX_TRY(basic_any(o));
    MBX_TRY(basic_any(t));
    MBX_TRY(basic_any(e));
    if (o.dtype != MBX_F32) return MBX_E_DTYPE;
    const int64_t D = t.cols;
    if (D > (int64_t)0x7fffffff / 6) return MBX_E_DIM_TOO_LARGE;
    if (t.rows != 6 || e.cols != 6 * D || o.cols != D || o.rows != 6 * e.rows) return MBX_E_SHAPE;
    if (overlaps(o, t) || overlaps(o, e)) return MBX_E_ALIAS;
    if (dev) {
        V all[3] = {o, t, e};
        MBX_TRY(views_on_device(all, 3));
    }
    return MBX_OK;
}

int check_qkv(const mbx_view* joint, const mbx_cview* txt, const mbx_cview* img, int64_t batch,
              int64_t heads, const mbx_cview* wq_txt, const mbx_cview* wk_txt,
              const mbx_cview* wq_img, const mbx_cview* wk_img, const float* cos_txt,
              const float* sin_txt, const float* cos_img, const float* sin_img, float eps,
              int variant, bool dev, int64_t* s_txt_out, int64_t* s_img_out) {
    if (!joint || !txt || !img || !wq_txt || !wk_txt || !wq_img || !wk_img) return MBX_E_NULL;
    V j = of(joint), t = of(txt), im = of(img);
    V w[4] = {of(wq_txt), of(wk_txt), of(wq_img), of(wk_img)};
    if (!j.data) return MBX_E_NULL;
    for (const V* v : {&j, &t, &im, &w[0], &w[1], &w[2], &w[3]})
        if (v->dtype != MBX_BF16) return MBX_E_DTYPE;
    if (batch <= 0 || heads <= 0) return MBX_E_ARG;
    if (batch >= (int64_t(1) << 31) || heads > (int64_t(1) << 20)) return MBX_E_ARG;  // no overflow below
    const int64_t hd = j.cols;
    if (hd != 64 && hd != 128 && hd != 256) return MBX_E_ARG;
    const int64_t width = 3 * heads * hd;
    // a branch may be empty (rows == 0, any data); otherwise a full view
    const bool has_t = t.rows != 0, has_i = im.rows != 0;
    if (!has_t && !has_i) return MBX_E_EMPTY;
    if (t.rows < 0 || im.rows < 0) return MBX_E_EMPTY;
    if (has_t && (!t.data || !cos_txt || !sin_txt)) return MBX_E_NULL;
    if (has_i && (!im.data || !cos_img || !sin_img)) return MBX_E_NULL;
    if (has_t) MBX_TRY(basic(t));
    if (has_i) MBX_TRY(basic(im));
    MBX_TRY(basic(j));
    for (int i = 0; i < 4; ++i) {
        if (!w[i].data) return MBX_E_NULL;
        MBX_TRY(basic(w[i]));
        if (w[i].rows != 1 || w[i].cols != hd) return MBX_E_SHAPE;
    }
    if (has_t && (t.cols != width || t.rows % batch)) return MBX_E_SHAPE;
    if (has_i && (im.cols != width || im.rows % batch)) return MBX_E_SHAPE;
    const int64_t s_txt = t.rows / batch, s_img = im.rows / batch;
    if (s_txt + s_img > ((int64_t(1) << 31) - 1) / (batch * heads)) return MBX_E_ARG;  // 32-bit unit index
    if (j.rows != batch * 3 * heads * (s_txt + s_img)) return MBX_E_SHAPE;
    if (j.rows > 1 && j.stride != hd) return MBX_E_STRIDE;  // joint is contiguous
    // 128-bit paths only: every row start 16-byte aligned
    if (!aligned16(j)) return MBX_E_ALIGN;
    if (has_t && !aligned16(t)) return MBX_E_ALIGN;
    if (has_i && !aligned16(im)) return MBX_E_ALIGN;
    for (int i = 0; i < 4; ++i)
        if (!aligned16(w[i])) return MBX_E_ALIGN;
    for (const float* f : {cos_txt, sin_txt, cos_img, sin_img})
        if (f && reinterpret_cast<uintptr_t>(f) % 16) return MBX_E_ALIGN;
    MBX_TRY(check_variant_eps(variant, eps));
    if ((has_t && overlaps(j, t)) || (has_i && overlaps(j, im))) return MBX_E_ALIAS;
    for (int i = 0; i < 4; ++i)
        if (overlaps(j, w[i])) return MBX_E_ALIAS;
    const int64_t tab_t = s_txt * (hd / 2) * 4, tab_i = s_img * (hd / 2) * 4;
    const uintptr_t j0 = reinterpret_cast<uintptr_t>(j.data), j1 = j0 + extent_bytes(j);
    for (int k = 0; k < 4; ++k) {
        const float* f = k == 0 ? cos_txt : k == 1 ? sin_txt : k == 2 ? cos_img : sin_img;
        int64_t n = k < 2 ? tab_t : tab_i;
        if (!f || n == 0) continue;
        uintptr_t f0 = reinterpret_cast<uintptr_t>(f);
        if (f0 < j1 && j0 < f0 + (uintptr_t)n) return MBX_E_ALIAS;
    }
    if (dev) {
        MBX_TRY(views_on_device(&j, 1));
        if (has_t) MBX_TRY(views_on_device(&t, 1));
        if (has_i) MBX_TRY(views_on_device(&im, 1));
        MBX_TRY(views_on_device(w, 4));
        if (has_t) {
            MBX_TRY(raw_on_device(cos_txt, tab_t));
            MBX_TRY(raw_on_device(sin_txt, tab_t));
        }
        if (has_i) {
            MBX_TRY(raw_on_device(cos_img, tab_i));
            MBX_TRY(raw_on_device(sin_img, tab_i));
        }
    }
    if (s_txt_out) *s_txt_out = s_txt;
    if (s_img_out) *s_img_out = s_img;
    return MBX_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MBX_OK : MBX_E_CUDA; }

}  // namespace

// ---------------------------------------------------------------- occupancy

namespace mbx {

int grid_for_rows(const void* kernel, int64_t units, int units_per_block, int block) {
    struct Entry {
        const void* k;
        int dev, block, per_sm;
    };
    static Entry cache[256];
    static int n_cache = 0;
    static int sms[64] = {0};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
    int per_sm = -1, nsm = 0;
    {
        std::lock_guard<std::mutex> g(mu);
        if (sms[dev] == 0) cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
        nsm = sms[dev];
        for (int i = 0; i < n_cache; ++i)
            if (cache[i].k == kernel && cache[i].dev == dev && cache[i].block == block) per_sm = cache[i].per_sm;
        if (per_sm < 0) {
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, block, 0) != cudaSuccess)
                return -1;
            if (n_cache < 256) cache[n_cache++] = Entry{kernel, dev, block, per_sm};
        }
    }
    if (per_sm < 1 || nsm < 1) return -1;
    int64_t need = (units + units_per_block - 1) / units_per_block;
    int64_t cap = (int64_t)nsm * per_sm;
    return (int)(need < cap ? need : cap);
}

static int device_sms() {
    static int sms[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (sms[dev] == 0) cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
    return sms[dev];
}

int64_t pipe_rows_per_cta(int64_t rows) {
    const int sms = device_sms();
    if (sms < 1) return rows;
    return (rows + sms - 1) / sms;
}

bool pipe_shape(const void* kernel, int tpr, int smem_per_group, int smem_fixed, int64_t rows,
                PipeShape* out) {
    struct Entry {
        const void* k;
        int dev, smem;
    };
    static Entry done[256];
    static int n_done = 0;
    static std::mutex mu;
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const int sms = device_sms();
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    const int64_t per_cta = pipe_rows_per_cta(rows);
    const int budget = optin - 8 * 1024 - smem_fixed;  // leave some shared memory to L1
    int groups = budget / smem_per_group;
    const int cap = tpr > 32 ? 15 : 512 / tpr;
    if (groups > cap) groups = cap;
    if (groups * tpr > 512) groups = 512 / tpr;  // pipelined kernels launch <= 512 threads
    if ((int64_t)groups > per_cta) groups = (int)per_cta;
    if (groups < 1 || sms < 1) return false;
    const int smem = smem_fixed + groups * smem_per_group;
    {
        std::lock_guard<std::mutex> g(mu);
        bool seen = false;
        for (int i = 0; i < n_done; ++i)
            if (done[i].k == kernel && done[i].dev == dev && done[i].smem >= smem) seen = true;
        if (!seen) {
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
                return false;
            if (n_done < 256) done[n_done++] = Entry{kernel, dev, smem};
        }
    }
    out->grid = (int)((rows + per_cta - 1) / per_cta);
    out->groups = groups;
    out->smem = smem;
    out->rows_per_cta = per_cta;
    return true;
}

}  // namespace mbx

// ---------------------------------------------------------------- C ABI

extern "C" {

MBX_API int mbx_check_ln_modulate(const mbx_view* out, const mbx_cview* x, const mbx_cview* scale,
                                  const mbx_cview* shift, float eps, int variant) {
    return check_ln_modulate(out, x, scale, shift, eps, variant, true);
}

MBX_API int mbx_ln_modulate(const mbx_view* out, const mbx_cview* x, const mbx_cview* scale,
                            const mbx_cview* shift, float eps, int variant, void* stream) {
    MBX_TRY(check_ln_modulate(out, x, scale, shift, eps, variant, true));
    mbx::LnModParams p;
    p.out = static_cast<uint16_t*>(out->data);
    p.out_stride = out->row_stride;
    p.x = static_cast<const uint16_t*>(x->data);
    p.x_stride = x->row_stride;
    p.scale = static_cast<const uint16_t*>(scale->data);
    p.scale_stride = scale->row_stride;
    p.shift = static_cast<const uint16_t*>(shift->data);
    p.shift_stride = shift->row_stride;
    p.rows = x->rows;
    p.D = (int)x->cols;
    p.seq = x->rows / scale->rows;
    p.eps = eps;
    const bool vec = p.D % 8 == 0 && aligned16(of(out)) && aligned16(of(x)) &&
                     aligned16(of(scale)) && aligned16(of(shift));
    return cuda_status(mbx::launch_ln_modulate(p, vec, variant == MBX_HIGH, (cudaStream_t)stream));
}

MBX_API int mbx_check_ln_modulate_fp8(const mbx_view* out, const mbx_view* out_fp8,
                                      const mbx_cview* x, const mbx_cview* scale,
                                      const mbx_cview* shift, const float* fp8_scale, float eps,
                                      int variant) {
    // every host check of both parts before any device check
    for (bool dev : {false, true}) {
        MBX_TRY(check_ln_modulate(out, x, scale, shift, eps, variant, dev));
        V vs[4] = {of(out), of(x), of(scale), of(shift)};
        MBX_TRY(check_fp8(out_fp8, fp8_scale, vs, 4, dev));
    }
    return MBX_OK;
}

MBX_API int mbx_ln_modulate_fp8(const mbx_view* out, const mbx_view* out_fp8, const mbx_cview* x,
                                const mbx_cview* scale, const mbx_cview* shift,
                                const float* fp8_scale, float eps, int variant, void* stream) {
    MBX_TRY(mbx_check_ln_modulate_fp8(out, out_fp8, x, scale, shift, fp8_scale, eps, variant));
    mbx::LnModParams p;
    p.out = static_cast<uint16_t*>(out->data);
    p.out_stride = out->row_stride;
    p.x = static_cast<const uint16_t*>(x->data);
    p.x_stride = x->row_stride;
    p.scale = static_cast<const uint16_t*>(scale->data);
    p.scale_stride = scale->row_stride;
    p.shift = static_cast<const uint16_t*>(shift->data);
    p.shift_stride = shift->row_stride;
    p.rows = x->rows;
    p.D = (int)x->cols;
    p.seq = x->rows / scale->rows;
    p.eps = eps;
    p.out_fp8 = static_cast<uint8_t*>(out_fp8->data);
    p.out_fp8_stride = out_fp8->row_stride;
    p.fp8_scale = fp8_scale;
    const bool vec = p.D % 8 == 0 && aligned16(of(out)) && aligned16(of(x)) && aligned16(of(scale)) &&
                     aligned16(of(shift)) && aligned8_fp8(out_fp8);
    return cuda_status(mbx::launch_ln_modulate_fp8(p, vec, variant == MBX_HIGH, (cudaStream_t)stream));
}

MBX_API int mbx_check_ln_modulate_nvfp4(const mbx_view* out, const mbx_view* out_fp4,
                                        const mbx_view* out_sf, const mbx_cview* x,
                                        const mbx_cview* scale, const mbx_cview* shift,
                                        const float* fp4_scale, float eps, int variant) {
    for (bool dev : {false, true}) {
        MBX_TRY(check_ln_modulate(out, x, scale, shift, eps, variant, dev));
        V vs[4] = {of(out), of(x), of(scale), of(shift)};
        MBX_TRY(check_fp4(out_fp4, out_sf, fp4_scale, vs, 4, dev));
    }
    return MBX_OK;
}

MBX_API int mbx_ln_modulate_nvfp4(const mbx_view* out, const mbx_view* out_fp4, const mbx_view* out_sf,
                                  const mbx_cview* x, const mbx_cview* scale, const mbx_cview* shift,
                                  const float* fp4_scale, float eps, int variant, void* stream) {
    MBX_TRY(mbx_check_ln_modulate_nvfp4(out, out_fp4, out_sf, x, scale, shift, fp4_scale, eps, variant));
    mbx::LnModParams p;
    p.out = static_cast<uint16_t*>(out->data);
    p.out_stride = out->row_stride;
    p.x = static_cast<const uint16_t*>(x->data);
    p.x_stride = x->row_stride;
    p.scale = static_cast<const uint16_t*>(scale->data);
    p.scale_stride = scale->row_stride;
    p.shift = static_cast<const uint16_t*>(shift->data);
    p.shift_stride = shift->row_stride;
    p.rows = x->rows;
    p.D = (int)x->cols;
    p.seq = x->rows / scale->rows;
    p.eps = eps;
    set_fp4(p, out_fp4, out_sf, fp4_scale);
    const bool vec = p.D % 8 == 0 && aligned16(of(out)) && aligned16(of(x)) && aligned16(of(scale)) &&
                     aligned16(of(shift)) && aligned4_fp4(out_fp4);
    return cuda_status(mbx::launch_ln_modulate_nvfp4(p, vec, variant == MBX_HIGH, (cudaStream_t)stream));
}

MBX_API int mbx_check_rmsnorm_scale(const mbx_view* out, const mbx_cview* x,
                                    const mbx_cview* weight, const mbx_cview* scale, float eps,
                                    int variant) {
    return check_rmsnorm_scale(out, x, weight, scale, eps, variant, true);
}

MBX_API int mbx_rmsnorm_scale(const mbx_view* out, const mbx_cview* x, const mbx_cview* weight,
                              const mbx_cview* scale, float eps, int variant, void* stream) {
    MBX_TRY(check_rmsnorm_scale(out, x, weight, scale, eps, variant, true));
    mbx::RmsScaleParams p;
    p.out = static_cast<uint16_t*>(out->data);
    p.out_stride = out->row_stride;
    p.x = static_cast<const uint16_t*>(x->data);
    p.x_stride = x->row_stride;
    p.weight = static_cast<const uint16_t*>(weight->data);
    p.scale = static_cast<const uint16_t*>(scale->data);
    p.scale_stride = scale->row_stride;
    p.rows = x->rows;
    p.D = (int)x->cols;
    p.seq = x->rows / scale->rows;
    p.eps = eps;
    const bool vec = p.D % 8 == 0 && aligned16(of(out)) && aligned16(of(x)) &&
                     aligned16(of(weight)) && aligned16(of(scale));
    return cuda_status(mbx::launch_rmsnorm_scale(p, vec, variant == MBX_HIGH, (cudaStream_t)stream));
}

MBX_API int mbx_check_rmsnorm_tanh_residual(const mbx_view* out, const mbx_cview* x,
                                            const mbx_cview* gate, const mbx_cview* residual,
                                            const mbx_cview* weight, float eps, int variant) {
    return check_rmsnorm_tanh_residual(out, x, gate, residual, weight, eps, variant, true);
}

MBX_API int mbx_rmsnorm_tanh_residual(const mbx_view* out, const mbx_cview* x,
                                      const mbx_cview* gate, const mbx_cview* residual,
                                      const mbx_cview* weight, float eps, int variant,
                                      void* stream) {
    MBX_TRY(check_rmsnorm_tanh_residual(out, x, gate, residual, weight, eps, variant, true));
    mbx::RmsTanhParams p;
    p.out = static_cast<uint16_t*>(out->data);
    p.out_stride = out->row_stride;
    p.x = static_cast<const uint16_t*>(x->data);
    p.x_stride = x->row_stride;
    p.gate = static_cast<const uint16_t*>(gate->data);
    p.gate_stride = gate->row_stride;
    p.residual = static_cast<const uint16_t*>(residual->data);
    p.res_stride = residual->row_stride;
    p.weight = static_cast<const uint16_t*>(weight->data);
    p.rows = x->rows;
    p.D = (int)x->cols;
    p.seq = x->rows / gate->rows;
    p.eps = eps;
    const bool vec = p.D % 8 == 0 && aligned16(of(out)) && aligned16(of(x)) && aligned16(of(gate)) &&
                     aligned16(of(residual)) && aligned16(of(weight));
    return cuda_status(
        mbx::launch_rmsnorm_tanh_residual(p, vec, variant == MBX_HIGH, (cudaStream_t)stream));
}

MBX_API int mbx_check_residual_gate_add(const mbx_view* out, const mbx_cview* x,
                                        const mbx_cview* gate, const mbx_cview* y, int variant) {
    return check_residual_gate_add(out, x, gate, y, variant, true);
}

MBX_API int mbx_residual_gate_add(const mbx_view* out, const mbx_cview* x, const mbx_cview* gate,
                                  const mbx_cview* y, int variant, void* stream) {
    MBX_TRY(check_residual_gate_add(out, x, gate, y, variant, true));
    mbx::GateAddParams p;
    p.out = static_cast<uint16_t*>(out->data);
    p.out_stride = out->row_stride;
    p.x = static_cast<const uint16_t*>(x->data);
    p.x_stride = x->row_stride;
    p.gate = static_cast<const uint16_t*>(gate->data);
    p.gate_stride = gate->row_stride;
    p.y = static_cast<const uint16_t*>(y->data);
    p.y_stride = y->row_stride;
    p.rows = x->rows;
    p.D = (int)x->cols;
    p.seq = x->rows / gate->rows;
    const bool vec = p.D % 8 == 0 && aligned16(of(out)) && aligned16(of(x)) && aligned16(of(gate)) &&
                     aligned16(of(y));
    return cuda_status(
        mbx::launch_residual_gate_add(p, vec, variant == MBX_HIGH, (cudaStream_t)stream));
}

MBX_API int mbx_check_gated_residual_ln_modulate_fp8(
    const mbx_view* residual_out, const mbx_view* out, const mbx_view* out_fp8,
    const mbx_cview* residual, const mbx_cview* gate, const mbx_cview* update,
    const mbx_cview* bias, const mbx_cview* scale, const mbx_cview* shift,
    const float* fp8_scale, float eps, int variant) {
    for (bool dev : {false, true}) {
        MBX_TRY(check_gated(residual_out, out, residual, gate, update, bias, scale, shift, eps, variant, dev));
        V vs[8] = {of(out), of(residual_out), of(residual), of(gate), of(update), of(scale), of(shift),
                   bias ? of(bias) : of(gate)};
        MBX_TRY(check_fp8(out_fp8, fp8_scale, vs, 8, dev));
    }
    return MBX_OK;
}

MBX_API int mbx_gated_residual_ln_modulate_fp8(const mbx_view* residual_out, const mbx_view* out,
                                               const mbx_view* out_fp8, const mbx_cview* residual,
                                               const mbx_cview* gate, const mbx_cview* update,
                                               const mbx_cview* bias, const mbx_cview* scale,
                                               const mbx_cview* shift, const float* fp8_scale,
                                               float eps, int variant, void* stream) {
    MBX_TRY(mbx_check_gated_residual_ln_modulate_fp8(residual_out, out, out_fp8, residual, gate, update,
                                                     bias, scale, shift, fp8_scale, eps, variant));
    mbx::LnModParams p = gated_params(residual_out, out, residual, gate, update, bias, scale, shift, eps);
    p.out_fp8 = static_cast<uint8_t*>(out_fp8->data);
    p.out_fp8_stride = out_fp8->row_stride;
    p.fp8_scale = fp8_scale;
    const bool vec = gated_vec(p, residual_out, out, residual, gate, update, bias, scale, shift) &&
                     aligned8_fp8(out_fp8);
    return cuda_status(mbx::launch_gated_residual_ln_modulate_fp8(p, vec, variant == MBX_HIGH, (cudaStream_t)stream));
}

MBX_API int mbx_check_gated_residual_ln_modulate_nvfp4(
    const mbx_view* residual_out, const mbx_view* out, const mbx_view* out_fp4, const mbx_view* out_sf,
    const mbx_cview* residual, const mbx_cview* gate, const mbx_cview* update, const mbx_cview* bias,
    const mbx_cview* scale, const mbx_cview* shift, const float* fp4_scale, float eps, int variant) {
    for (bool dev : {false, true}) {
        MBX_TRY(check_gated(residual_out, out, residual, gate, update, bias, scale, shift, eps, variant, dev));
        V vs[8] = {of(out), of(residual_out), of(residual), of(gate), of(update), of(scale), of(shift),
                   bias ? of(bias) : of(gate)};
        MBX_TRY(check_fp4(out_fp4, out_sf, fp4_scale, vs, 8, dev));
    }
    return MBX_OK;
}

MBX_API int mbx_gated_residual_ln_modulate_nvfp4(
    const mbx_view* residual_out, const mbx_view* out, const mbx_view* out_fp4, const mbx_view* out_sf,
    const mbx_cview* residual, const mbx_cview* gate, const mbx_cview* update, const mbx_cview* bias,
    const mbx_cview* scale, const mbx_cview* shift, const float* fp4_scale, float eps, int variant,
    void* stream) {
    MBX_TRY(mbx_check_gated_residual_ln_modulate_nvfp4(residual_out, out, out_fp4, out_sf, residual, gate,
                                                       update, bias, scale, shift, fp4_scale, eps, variant));
    mbx::LnModParams p = gated_params(residual_out, out, residual, gate, update, bias, scale, shift, eps);
    set_fp4(p, out_fp4, out_sf, fp4_scale);
    const bool vec = gated_vec(p, residual_out, out, residual, gate, update, bias, scale, shift) &&
                     aligned4_fp4(out_fp4);
    return cuda_status(
        mbx::launch_gated_residual_ln_modulate_nvfp4(p, vec, variant == MBX_HIGH, (cudaStream_t)stream));
}

MBX_API int mbx_check_modulation_table_add(const mbx_view* out, const mbx_cview* table,
                                           const mbx_cview* temb) {
    return check_modtable(out, table, temb, true);
}

MBX_API int mbx_modulation_table_add(const mbx_view* out, const mbx_cview* table,
                                     const mbx_cview* temb, void* stream) {
    MBX_TRY(check_modtable(out, table, temb, true));
    mbx::ModTableParams p;
    p.out = static_cast<float*>(out->data);
    p.out_stride = out->row_stride;
    p.table = table->data;
    p.table_stride = table->row_stride;
    p.table_f32 = table->dtype == MBX_F32;
    p.temb = temb->data;
    p.temb_stride = temb->row_stride;
    p.temb_f32 = temb->dtype == MBX_F32;
    p.rows = temb->rows;
    p.D = (int)table->cols;
    const bool vec = p.D % 8 == 0 && aligned16(of(out)) && aligned16(of(table)) && aligned16(of(temb));
    return cuda_status(mbx::launch_modulation_table_add(p, vec, (cudaStream_t)stream));
}

MBX_API int mbx_check_gated_residual_ln_modulate(const mbx_view* residual_out,
                                                 const mbx_view* out, const mbx_cview* residual,
                                                 const mbx_cview* gate, const mbx_cview* update,
                                                 const mbx_cview* bias, const mbx_cview* scale,
                                                 const mbx_cview* shift, float eps, int variant) {
    return check_gated(residual_out, out, residual, gate, update, bias, scale, shift, eps, variant, true);
}

MBX_API int mbx_gated_residual_ln_modulate(const mbx_view* residual_out, const mbx_view* out,
                                           const mbx_cview* residual, const mbx_cview* gate,
                                           const mbx_cview* update, const mbx_cview* bias,
                                           const mbx_cview* scale, const mbx_cview* shift,
                                           float eps, int variant, void* stream) {
    MBX_TRY(check_gated(residual_out, out, residual, gate, update, bias, scale, shift, eps, variant, true));
    const mbx::LnModParams p = gated_params(residual_out, out, residual, gate, update, bias, scale, shift, eps);
    const bool vec = gated_vec(p, residual_out, out, residual, gate, update, bias, scale, shift);
    return cuda_status(mbx::launch_gated_residual_ln_modulate(p, vec, variant == MBX_HIGH, (cudaStream_t)stream));
}

MBX_API int mbx_check_qk_norm_rope_qkv_epilogue(
    const mbx_view* joint, const mbx_cview* txt_qkv, const mbx_cview* img_qkv, int64_t batch,
    int64_t heads, const mbx_cview* wq_txt, const mbx_cview* wk_txt, const mbx_cview* wq_img,
    const mbx_cview* wk_img, const float* cos_txt, const float* sin_txt, const float* cos_img,
    const float* sin_img, float eps, int variant) {
    return check_qkv(joint, txt_qkv, img_qkv, batch, heads, wq_txt, wk_txt, wq_img, wk_img, cos_txt,
                     sin_txt, cos_img, sin_img, eps, variant, true, nullptr, nullptr);
}

MBX_API int mbx_qk_norm_rope_qkv_epilogue(const mbx_view* joint, const mbx_cview* txt_qkv,
                                          const mbx_cview* img_qkv, int64_t batch, int64_t heads,
                                          const mbx_cview* wq_txt, const mbx_cview* wk_txt,
                                          const mbx_cview* wq_img, const mbx_cview* wk_img,
                                          const float* cos_txt, const float* sin_txt,
                                          const float* cos_img, const float* sin_img, float eps,
                                          int variant, void* stream) {
    int64_t s_txt = 0, s_img = 0;
    MBX_TRY(check_qkv(joint, txt_qkv, img_qkv, batch, heads, wq_txt, wk_txt, wq_img, wk_img,
                      cos_txt, sin_txt, cos_img, sin_img, eps, variant, true, &s_txt, &s_img));
    mbx::QkvParams p;
    p.joint = static_cast<uint16_t*>(joint->data);
    p.txt = static_cast<const uint16_t*>(txt_qkv->data);
    p.txt_stride = txt_qkv->row_stride;
    p.img = static_cast<const uint16_t*>(img_qkv->data);
    p.img_stride = img_qkv->row_stride;
    p.s_txt = s_txt;
    p.s_img = s_img;
    p.batch = batch;
    p.heads = (int)heads;
    p.head_dim = (int)joint->cols;
    p.wq_txt = static_cast<const uint16_t*>(wq_txt->data);
    p.wk_txt = static_cast<const uint16_t*>(wk_txt->data);
    p.wq_img = static_cast<const uint16_t*>(wq_img->data);
    p.wk_img = static_cast<const uint16_t*>(wk_img->data);
    p.cos_txt = cos_txt;
    p.sin_txt = sin_txt;
    p.cos_img = cos_img;
    p.sin_img = sin_img;
    p.eps = eps;
    return cuda_status(mbx::launch_qkv_epilogue(p, variant == MBX_HIGH, (cudaStream_t)stream));
}

MBX_API int mbx_selftest(int which, unsigned long long* counts, void* stream) {
    if (!counts) return MBX_E_NULL;
    if (which < 0 || which > 6) return MBX_E_ARG;
    if (reinterpret_cast<uintptr_t>(counts) % 8) return MBX_E_ALIGN;
    MBX_TRY(raw_on_device(counts, 16));
    return cuda_status(mbx::launch_selftest(which, counts, (cudaStream_t)stream));
}

MBX_API const char* mbx_status_string(int status) {
    switch (status) {
        case MBX_OK: return "MBX_OK";
        case MBX_E_NULL: return "MBX_E_NULL: a required pointer is NULL";
        case MBX_E_DTYPE: return "MBX_E_DTYPE: every operand must be bfloat16";
        case MBX_E_EMPTY: return "MBX_E_EMPTY: empty input";
        case MBX_E_DIM_TOO_LARGE: return "MBX_E_DIM_TOO_LARGE: hidden size above 8192";
        case MBX_E_SHAPE: return "MBX_E_SHAPE: shapes disagree (or rows % modulation rows != 0)";
        case MBX_E_STRIDE: return "MBX_E_STRIDE: row stride smaller than the row, or not flat";
        case MBX_E_ALIGN: return "MBX_E_ALIGN: misaligned pointer or row";
        case MBX_E_ALIAS: return "MBX_E_ALIAS: output overlaps an input";
        case MBX_E_DEVICE: return "MBX_E_DEVICE: pointer is not device memory of the current device";
        case MBX_E_BOUNDS: return "MBX_E_BOUNDS: view extends past its allocation";
        case MBX_E_VARIANT: return "MBX_E_VARIANT: variant must be MBX_LOSSLESS or MBX_HIGH";
        case MBX_E_ARG: return "MBX_E_ARG: argument out of range";
        case MBX_E_CUDA: return "MBX_E_CUDA: CUDA runtime error";
        default: return "MBX_E_UNKNOWN: unknown status";
    }
}

MBX_API int mbx_abi_version(void) { return MBX_ABI_VERSION; }

}  // extern "C"
