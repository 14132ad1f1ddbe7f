// C-ABI entry points of the sg library: argument validation, the layout
// handle, and dispatch to the tensor-core or CUDA-core engine.  The operations
// themselves are defined in include/sg.h.
#include <cmath>

#include "sg_internal.cuh"

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

namespace {

thread_local char g_err[512];

// Every layout between a successful sg_layout_build and its sg_layout_free,
// in creation order, so that sg_device_status can read their status words.
std::mutex g_live_mu;
std::vector<sg_layout *> g_live;

void live_add(sg_layout *lo)
{
    std::lock_guard<std::mutex> lk(g_live_mu);
    g_live.push_back(lo);
}

void live_remove(sg_layout *lo)
{
    std::lock_guard<std::mutex> lk(g_live_mu);
    for (size_t i = 0; i < g_live.size(); ++i)
        if (g_live[i] == lo) {
            g_live.erase(g_live.begin() + (long)i);
            return;
        }
}

// Makes the layout's device current for the duration of a call.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            ok = false;
            return;
        }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess)
            ok = false;
    }
    ~DeviceGuard()
    {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev)
            cudaSetDevice(prev);
    }
};

#define FAIL(code, ...)               \
    do {                              \
        sg_set_error(__VA_ARGS__);    \
        return code;                  \
    } while (0)

sg_status check_call(const sg_layout *lo, int32_t B, const char *fn)
{
    if (!lo)
        FAIL(SG_ERR_INVALID, "%s: layout is NULL", fn);
    if (B < 1)
        FAIL(SG_ERR_INVALID, "%s: B must be >= 1 (got %d)", fn, B);
    if (B > lo->max_B)
        FAIL(SG_ERR_INVALID, "%s: B=%d exceeds the layout's max_B=%d", fn, B,
             lo->max_B);
    return SG_OK;
}

sg_status check_pos(const sg_layout *lo, const int32_t *rowptr,
                    const int32_t *labels, int64_t nnz, const char *fn)
{
    if (!rowptr)
        FAIL(SG_ERR_INVALID, "%s: pos_rowptr is NULL", fn);
    if (nnz < 0)
        FAIL(SG_ERR_INVALID, "%s: nnz must be >= 0", fn);
    if (nnz > 0 && !labels)
        FAIL(SG_ERR_INVALID, "%s: pos_label is NULL", fn);
    if (nnz > lo->max_nnz)
        FAIL(SG_ERR_INVALID, "%s: nnz=%lld exceeds the layout's max_nnz=%lld",
             fn, (long long)nnz, (long long)lo->max_nnz);
    return SG_OK;
}

#define REQUIRE(ptr, fn)                                                   \
    do {                                                                   \
        if (!(ptr))                                                        \
            FAIL(SG_ERR_INVALID, "%s: %s is NULL", fn, #ptr);              \
    } while (0)

#define TRY(expr)                  \
    do {                           \
        sg_status rc_ = (expr);    \
        if (rc_ != SG_OK)          \
            return rc_;            \
    } while (0)

// Which engine runs `stage` for a batch of B: the tensor-core engine unless the
// layout is pinned to CUDA cores or the shape is outside what it supports.  A
// layout pinned to the tensor-core engine fails instead of switching.
sg_status pick_tc(const sg_layout *lo, int stage, int32_t B, bool *tc, const char *fn)
{
    *tc = false;
    if (lo->engine == SG_ENGINE_SIMT)
        return SG_OK;
    const bool ok = lo->tc_ok && tc_stage_ok(lo, stage, B);
    if (!ok && (lo->engine == SG_ENGINE_TC || lo->engine == SG_ENGINE_FUSED))
        FAIL(SG_ERR_UNSUPPORTED, "%s: this shape (B=%d G=%d F=%d H=%d) is outside the "
             "tensor-core engine", fn, B, lo->G, lo->F, lo->H);
    *tc = ok;
    return SG_OK;
}

void timer_release(sg_layout::Timer &t)
{
    if (t.ev) {
        for (int i = 0; i < 2 * t.cap; ++i)
            cudaEventDestroy(t.ev[i]);
        delete[] t.ev;
    }
    delete[] t.kind;
    t = sg_layout::Timer();
}

void free_layout(sg_layout *lo)
{
    if (!lo)
        return;
    timer_release(lo->timer);
    void *bufs[] = {lo->slot_of_label, lo->label_of_slot, lo->idx_s, lo->hT,
                    lo->gcount, lo->gptr, lo->gent, lo->tsorted, lo->tslots,
                    lo->rowcnt, lo->loss_part, lo->status, lo->dZ_ws, lo->scan_part, lo->wmax,
                    lo->ht_ws, lo->rw_ws};
    for (void *p : bufs)
        if (p)
            cudaFree(p);
    delete lo;
}

template <typename T>
sg_status dev_alloc(T **p, size_t n, const char *what)
{
    size_t bytes = n * sizeof(T);
    if (bytes == 0)
        bytes = sizeof(T);
    if (cudaMalloc((void **)p, bytes) != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        FAIL(SG_ERR_OOM, "sg_layout_build: cudaMalloc of %zu bytes for %s failed",
             bytes, what);
    }
    return SG_OK;
}

sg_status ensure_dz_ws(sg_layout *lo)
{
    // two planes of [B][L], or K group tiles of 2 x roundup(B, 128) x G
    size_t need = 2 * (size_t)lo->ldB * (size_t)lo->L;
    if (lo->dZ_ws && lo->dZ_ws_elems >= need)
        return SG_OK;
    if (lo->dZ_ws)
        cudaFree(lo->dZ_ws);
    lo->dZ_ws = nullptr;
    if (cudaMalloc((void **)&lo->dZ_ws, need * 2) != cudaSuccess) {
        cudaGetLastError();
        FAIL(SG_ERR_OOM, "sg_step: cudaMalloc of %zu bytes of dZ scratch failed",
             need * 2);
    }
    lo->dZ_ws_elems = need;
    return SG_OK;
}

}  // namespace

void sg_set_error(const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
}

extern "C" {

const char *sg_last_error(void) { return g_err; }

int32_t sg_abi_version(void) { return SG_ABI_VERSION; }

const char *sg_status_string(int32_t s)
{
    switch (s) {
    case SG_OK: return "SG_OK";
    case SG_ERR_INVALID: return "SG_ERR_INVALID";
    case SG_ERR_UNSUPPORTED: return "SG_ERR_UNSUPPORTED";
    case SG_ERR_CUDA: return "SG_ERR_CUDA";
    case SG_ERR_OOM: return "SG_ERR_OOM";
    case SG_ERR_TIMEOUT: return "SG_ERR_TIMEOUT";
    case SG_ERR_DATA: return "SG_ERR_DATA";
    default: return "SG_ERR_UNKNOWN";
    }
}

// ---------------------------------------------------------------- layout
sg_status sg_layout_build(const int32_t *groups, int64_t L, int32_t G,
                          const int32_t *idx, int32_t F, int32_t H,
                          int32_t max_B, int64_t max_nnz, void *stream,
                          sg_layout **out)
{
    const char *fn = "sg_layout_build";
    NvtxRange nvtx_(fn);
    if (!out)
        FAIL(SG_ERR_INVALID, "%s: out is NULL", fn);
    *out = nullptr;
    REQUIRE(groups, fn);
    REQUIRE(idx, fn);
    if (L < 1 || G < 1 || F < 1 || H < 1 || max_B < 1 || max_nnz < 0)
        FAIL(SG_ERR_INVALID, "%s: sizes must be positive (L=%lld G=%d F=%d H=%d "
             "max_B=%d max_nnz=%lld)", fn, (long long)L, G, F, H, max_B,
             (long long)max_nnz);
    if (L % G != 0)
        FAIL(SG_ERR_INVALID, "%s: L=%lld is not a multiple of G=%d", fn,
             (long long)L, G);
    if (F > H)
        FAIL(SG_ERR_INVALID, "%s: F=%d exceeds H=%d", fn, F, H);
    if (G > SG_MAX_G || F > SG_MAX_F || H > SG_MAX_H || max_B > SG_MAX_B)
        FAIL(SG_ERR_UNSUPPORTED, "%s: outside the supported range (G<=%d, F<=%d, "
             "H<=%d, max_B<=%d)", fn, SG_MAX_G, SG_MAX_F, SG_MAX_H, SG_MAX_B);
    if (L > (int64_t)INT32_MAX || max_nnz > (int64_t)INT32_MAX)
        FAIL(SG_ERR_UNSUPPORTED, "%s: L and max_nnz must fit in int32", fn);

    sg_layout *lo = new (std::nothrow) sg_layout();
    if (!lo)
        FAIL(SG_ERR_OOM, "%s: host allocation failed", fn);
    lo->L = L;
    lo->G = G;
    lo->K = L / G;
    lo->F = F;
    lo->H = H;
    lo->max_B = max_B;
    lo->max_nnz = max_nnz;
    lo->ldB = (int32_t)(ceil_div(max_B, 128) * 128);
    cudaStream_t st = (cudaStream_t)stream;

    sg_status rc = SG_OK;
    cudaDeviceProp prop;
    if (cudaGetDevice(&lo->device) != cudaSuccess ||
        cudaGetDeviceProperties(&prop, lo->device) != cudaSuccess) {
        sg_set_error("%s: no usable CUDA device (%s)", fn,
                     cudaGetErrorString(cudaGetLastError()));
        delete lo;
        return SG_ERR_CUDA;
    }
    lo->num_sms = prop.multiProcessorCount;
    lo->loss_part_n = 8192;

#define ALLOC(field, n)                                                    \
    do {                                                                   \
        rc = dev_alloc(&lo->field, (size_t)(n), #field);                   \
        if (rc != SG_OK) {                                                 \
            free_layout(lo);                                               \
            return rc;                                                     \
        }                                                                  \
    } while (0)
    ALLOC(slot_of_label, L);
    ALLOC(label_of_slot, L);
    ALLOC(idx_s, lo->K * F);
    ALLOC(hT, (size_t)H * lo->ldB);
    ALLOC(gcount, lo->K + 1);
    ALLOC(gptr, lo->K + 1);
    ALLOC(scan_part, (lo->K + 4095) / 4096 + 1);
    ALLOC(gent, max_nnz);
    ALLOC(tsorted, max_nnz);
    ALLOC(tslots, max_nnz);
    ALLOC(rowcnt, max_B);
    ALLOC(loss_part, lo->loss_part_n);
    ALLOC(status, 1);
#undef ALLOC
    if (cudaMemsetAsync(lo->gcount, 0, sizeof(int32_t) * (lo->K + 1), st) != cudaSuccess ||
        cudaMemsetAsync(lo->status, 0, sizeof(int32_t), st) != cudaSuccess ||
        cudaMemsetAsync(lo->hT, 0, (size_t)H * lo->ldB * 2, st) != cudaSuccess) {
        sg_set_error("%s: %s", fn, cudaGetErrorString(cudaGetLastError()));
        free_layout(lo);
        return SG_ERR_CUDA;
    }
    rc = sg_layout_kernels(lo, groups, idx, st);
    if (rc != SG_OK) {
        free_layout(lo);
        return rc;
    }
    lo->tc_ok = tc_supported(lo) || tc_step_ok(lo, max_B < 128 ? max_B : 128);
    live_add(lo);
    *out = lo;
    return SG_OK;
}

sg_status sg_layout_export(const sg_layout *lo, int32_t *slot_of_label,
                           int32_t *label_of_slot, uint16_t *idx_sorted,
                           void *stream)
{
    const char *fn = "sg_layout_export";
    NvtxRange nvtx_(fn);
    if (!lo)
        FAIL(SG_ERR_INVALID, "%s: layout is NULL", fn);
    DeviceGuard dg(lo->device);
    cudaStream_t st = (cudaStream_t)stream;
    if (slot_of_label)
        SG_TRY_CUDA(cudaMemcpyAsync(slot_of_label, lo->slot_of_label, 4 * lo->L,
                                    cudaMemcpyDeviceToDevice, st));
    if (label_of_slot)
        SG_TRY_CUDA(cudaMemcpyAsync(label_of_slot, lo->label_of_slot, 4 * lo->L,
                                    cudaMemcpyDeviceToDevice, st));
    if (idx_sorted)
        SG_TRY_CUDA(cudaMemcpyAsync(idx_sorted, lo->idx_s, 2 * lo->K * lo->F,
                                    cudaMemcpyDeviceToDevice, st));
    SG_TRY_CUDA(cudaStreamSynchronize(st));
    return SG_OK;
}

void sg_layout_free(sg_layout *lo)
{
    if (!lo)
        return;
    live_remove(lo);
    DeviceGuard dg(lo->device);
    cudaDeviceSynchronize();
    free_layout(lo);
}

sg_status sg_layout_set_engine(sg_layout *lo, int32_t engine)
{
    const char *fn = "sg_layout_set_engine";
    if (!lo)
        FAIL(SG_ERR_INVALID, "%s: layout is NULL", fn);
    if (engine != SG_ENGINE_AUTO && engine != SG_ENGINE_SIMT && engine != SG_ENGINE_TC &&
        engine != SG_ENGINE_FUSED)
        FAIL(SG_ERR_INVALID, "%s: unknown engine %d", fn, engine);
    if ((engine == SG_ENGINE_TC || engine == SG_ENGINE_FUSED) && !lo->tc_ok)
        FAIL(SG_ERR_UNSUPPORTED, "%s: the tensor-core engine needs G in {16, 32} or a multiple of 64, "
             "F %% 16 == 0, and the group's tiles within shared memory and TMEM (G=%d, F=%d, max_B=%d)",
             fn, lo->G, lo->F, lo->max_B);
    lo->engine = engine;
    return SG_OK;
}

sg_status sg_layout_info(const sg_layout *lo, int64_t *L, int32_t *G,
                         int32_t *F, int32_t *H, int64_t *K)
{
    if (!lo)
        FAIL(SG_ERR_INVALID, "sg_layout_info: layout is NULL");
    if (L) *L = lo->L;
    if (G) *G = lo->G;
    if (F) *F = lo->F;
    if (H) *H = lo->H;
    if (K) *K = lo->K;
    return SG_OK;
}

sg_status sg_layout_status(sg_layout *lo, int32_t *code, int32_t clear)
{
    const char *fn = "sg_layout_status";
    NvtxRange nvtx_(fn);
    if (!lo)
        FAIL(SG_ERR_INVALID, "%s: layout is NULL", fn);
    REQUIRE(code, fn);
    DeviceGuard dg(lo->device);
    SG_TRY_CUDA(cudaDeviceSynchronize());
    SG_TRY_CUDA(cudaMemcpy(code, lo->status, sizeof(int32_t), cudaMemcpyDeviceToHost));
    if (clear)
        SG_TRY_CUDA(cudaMemset(lo->status, 0, sizeof(int32_t)));
    SG_TRY_CUDA(cudaDeviceSynchronize());
    return SG_OK;
}

sg_status sg_device_status(int32_t *code)
{
    const char *fn = "sg_device_status";
    NvtxRange nvtx_(fn);
    REQUIRE(code, fn);
    *code = SG_OK;
    int dev = 0;
    SG_TRY_CUDA(cudaGetDevice(&dev));
    SG_TRY_CUDA(cudaDeviceSynchronize());
    std::lock_guard<std::mutex> lk(g_live_mu);
    for (sg_layout *lo : g_live) {
        if (lo->device != dev)
            continue;
        int32_t c = 0;
        SG_TRY_CUDA(cudaMemcpy(&c, lo->status, sizeof(int32_t), cudaMemcpyDeviceToHost));
        if (c != SG_OK) {
            *code = c;
            break;
        }
    }
    return SG_OK;
}

// ---------------------------------------------------------------- positives
sg_status sg_pos_export(sg_layout *lo, int32_t B, const int32_t *pos_rowptr,
                        const int32_t *pos_label, int64_t nnz,
                        int32_t *out_rowptr, int32_t *out_slots,
                        int32_t *out_gptr, int32_t *out_gentry, void *stream)
{
    const char *fn = "sg_pos_export";
    NvtxRange nvtx_(fn);
    TRY(check_call(lo, B, fn));
    TRY(check_pos(lo, pos_rowptr, pos_label, nnz, fn));
    DeviceGuard dg(lo->device);
    cudaStream_t st = (cudaStream_t)stream;
    TRY(sg_pos_prepare(lo, B, pos_rowptr, pos_label, nnz, st));
    if (out_rowptr || out_slots) {
        int32_t *orp = out_rowptr;
        if (!orp)
            FAIL(SG_ERR_INVALID, "%s: out_slots needs out_rowptr", fn);
        TRY(sg_pos_compact(lo, B, pos_rowptr, orp, out_slots, st));
    }
    if (out_gptr)
        SG_TRY_CUDA(cudaMemcpyAsync(out_gptr, lo->gptr, 4 * (lo->K + 1),
                                    cudaMemcpyDeviceToDevice, st));
    if (out_gentry && nnz > 0)
        SG_TRY_CUDA(cudaMemcpyAsync(out_gentry, lo->gent, 4 * nnz,
                                    cudaMemcpyDeviceToDevice, st));
    return SG_OK;
}

// ---------------------------------------------------------------- forward
sg_status sg_fwd(sg_layout *lo, const sg_bf16 *h, int32_t B, const sg_bf16 *W,
                 sg_bf16 *Z, void *stream)
{
    const char *fn = "sg_fwd";
    NvtxRange nvtx_(fn);
    TRY(check_call(lo, B, fn));
    REQUIRE(h, fn);
    REQUIRE(W, fn);
    REQUIRE(Z, fn);
    DeviceGuard dg(lo->device);
    cudaStream_t st = (cudaStream_t)stream;
    bool tc = false;
    TRY(pick_tc(lo, SG_KIND_FWD, B, &tc, fn));
    TRY(simt_transpose_h(lo, h, B, st));
    if (tc)
        return tc_fwd(lo, B, W, Z, nullptr, nullptr, nullptr, nullptr, st);
    return simt_fwd(lo, B, W, Z, nullptr, nullptr, nullptr, st);
}

sg_status sg_bce_grad(sg_layout *lo, const sg_bf16 *Z, int32_t B,
                      const int32_t *pos_rowptr, const int32_t *pos_label,
                      int64_t nnz, sg_bf16 *dZ, double *loss, void *stream)
{
    const char *fn = "sg_bce_grad";
    NvtxRange nvtx_(fn);
    TRY(check_call(lo, B, fn));
    TRY(check_pos(lo, pos_rowptr, pos_label, nnz, fn));
    REQUIRE(Z, fn);
    REQUIRE(dZ, fn);
    REQUIRE(loss, fn);
    DeviceGuard dg(lo->device);
    cudaStream_t st = (cudaStream_t)stream;
    TRY(sg_pos_prepare(lo, B, pos_rowptr, pos_label, nnz, st));
    return simt_bce(lo, Z, B, dZ, loss, st);
}

sg_status sg_fwd_bce(sg_layout *lo, const sg_bf16 *h, int32_t B,
                     const sg_bf16 *W, const int32_t *pos_rowptr,
                     const int32_t *pos_label, int64_t nnz, sg_bf16 *dZ,
                     double *loss, sg_bf16 *Z_or_null, void *stream)
{
    const char *fn = "sg_fwd_bce";
    NvtxRange nvtx_(fn);
    TRY(check_call(lo, B, fn));
    TRY(check_pos(lo, pos_rowptr, pos_label, nnz, fn));
    REQUIRE(h, fn);
    REQUIRE(W, fn);
    REQUIRE(dZ, fn);
    REQUIRE(loss, fn);
    DeviceGuard dg(lo->device);
    cudaStream_t st = (cudaStream_t)stream;
    bool tc = false;
    TRY(pick_tc(lo, SG_KIND_FWD, B, &tc, fn));
    TRY(sg_step_prepare(lo, h, B, pos_rowptr, pos_label, nnz, st));
    if (tc)
        return tc_fwd(lo, B, W, Z_or_null, dZ, nullptr, nullptr, loss, st);
    return simt_fwd(lo, B, W, Z_or_null, dZ, nullptr, loss, st);
}

// ---------------------------------------------------------------- backward
sg_status sg_bwd_dW(sg_layout *lo, const sg_bf16 *dZ, const sg_bf16 *h,
                    int32_t B, sg_bf16 *dW, void *stream)
{
    const char *fn = "sg_bwd_dW";
    NvtxRange nvtx_(fn);
    TRY(check_call(lo, B, fn));
    REQUIRE(dZ, fn);
    REQUIRE(h, fn);
    REQUIRE(dW, fn);
    DeviceGuard dg(lo->device);
    cudaStream_t st = (cudaStream_t)stream;
    bool tc = false;
    TRY(pick_tc(lo, SG_KIND_DW, B, &tc, fn));
    TRY(simt_transpose_h(lo, h, B, st));
    if (tc)
        return tc_dW(lo, dZ, nullptr, nullptr, B, dW, st);
    return simt_dW(lo, dZ, nullptr, B, dW, st);
}

sg_status sg_bwd_dh(sg_layout *lo, const sg_bf16 *dZ, int32_t B,
                    const sg_bf16 *W, float *dh, void *stream)
{
    const char *fn = "sg_bwd_dh";
    NvtxRange nvtx_(fn);
    TRY(check_call(lo, B, fn));
    REQUIRE(dZ, fn);
    REQUIRE(W, fn);
    REQUIRE(dh, fn);
    DeviceGuard dg(lo->device);
    cudaStream_t st = (cudaStream_t)stream;
    bool tc = false;
    TRY(pick_tc(lo, SG_KIND_DH, B, &tc, fn));
    if (tc)
        return tc_dh(lo, dZ, nullptr, nullptr, false, B, W, dh, st);
    return simt_dh(lo, dZ, nullptr, B, W, dh, st);
}

sg_status sg_bwd(sg_layout *lo, const sg_bf16 *dZ, const sg_bf16 *h, int32_t B,
                 const sg_bf16 *W, sg_bf16 *dW, float *dh, void *stream)
{
    const char *fn = "sg_bwd";
    NvtxRange nvtx_(fn);
    TRY(check_call(lo, B, fn));
    REQUIRE(dZ, fn);
    REQUIRE(h, fn);
    REQUIRE(W, fn);
    REQUIRE(dW, fn);
    REQUIRE(dh, fn);
    TRY(sg_bwd_dW(lo, dZ, h, B, dW, stream));
    return sg_bwd_dh(lo, dZ, B, W, dh, stream);
}

// ---------------------------------------------------------------- step
namespace {

// Which kernels a step of B samples runs: the whole step in one kernel on
// CTA clusters, the fused forward + BCE + dW kernel then dh, or one kernel per
// phase on the engine each phase fits.
struct StepPath {
    int single = 0, fused = 0, tc_f = 0, tc_w = 0, tc_h = 0;
};

sg_status step_path(const sg_layout *lo, int32_t B, bool sgd, StepPath *p, const char *fn)
{
    *p = StepPath();
    // shapes the fused forward + BCE + dW kernel and the dh kernel cannot run
    // (e.g. F not a multiple of 64) take the whole step in one kernel on CTA
    // clusters, where it fits: dZ never leaves the chip there, but on the
    // shapes both paths run it measures slower than the two-kernel path
    const bool two_kernel = lo->engine != SG_ENGINE_SIMT && tc_fwdw_ok(lo, B) && tc_stage_ok(lo, SG_KIND_DH, B);
    if (!sgd && lo->engine != SG_ENGINE_SIMT && (!two_kernel || lo->engine == SG_ENGINE_FUSED) &&
        tc_step_ok(lo, B)) {
        p->single = p->tc_f = p->tc_w = p->tc_h = 1;
        return SG_OK;
    }
    // the fused forward + BCE + dW kernel and the tensor-core dh, with dZ in
    // the group-tiled workspace, whenever the shape fits them
    if (lo->engine != SG_ENGINE_SIMT && lo->tc_ok && two_kernel) {
        p->fused = p->tc_f = p->tc_w = p->tc_h = 1;
        return SG_OK;
    }
    bool f = false, w = false, h = false;
    TRY(pick_tc(lo, SG_KIND_FWD, B, &f, fn));
    TRY(pick_tc(lo, SG_KIND_DW, B, &w, fn));
    TRY(pick_tc(lo, SG_KIND_DH, B, &h, fn));
    p->tc_f = f;
    p->tc_w = w;
    p->tc_h = h;
    return SG_OK;
}

// the step after argument checks; with sgd, dW receives the updated weights
sg_status step_impl(sg_layout *lo, const sg_bf16 *h, int32_t B, const sg_bf16 *W,
                    const int32_t *pos_rowptr, const int32_t *pos_label, int64_t nnz, sg_bf16 *dW,
                    float *dh, double *loss, const sg_sgd *sgd, cudaStream_t st, const char *fn)
{
    StepPath path;
    TRY(step_path(lo, B, sgd != nullptr, &path, fn));
    if (path.single) {
        TRY(sg_step_prepare(lo, h, B, pos_rowptr, pos_label, nnz, st));
        return tc_step(lo, B, W, dW, dh, loss, st);
    }
    const bool fused = path.fused != 0;
    const bool tc_f = path.tc_f, tc_w = path.tc_w, tc_h = path.tc_h;
    TRY(sg_step_prepare(lo, h, B, pos_rowptr, pos_label, nnz, st));
    // forward + BCE into dZ scratch, then dW and dh from it.  Outside the
    // fused kernel dZ is kept as two bf16 planes (hi + lo): a single bf16
    // rounding of dZ, summed over B samples (dW) or over every label (dh),
    // would move results by more than 2e-2 (1 + |ref|) against the exact
    // gradient.
    TRY(ensure_dz_ws(lo));
    if (fused || (tc_f && tc_w && tc_h && tc_tiled_ok(lo, B))) {
        // all three on the tensor cores: dZ in the group-tiled workspace
        uint8_t *dZt = reinterpret_cast<uint8_t *>(lo->dZ_ws);
        if (fused) {
            // the fused kernel leaves dZ as one fp16 plane and max |W| for dh
            // (and applies the optimiser step to dW in its epilogue)
            TRY(tc_fwdw(lo, B, W, dZt, dW, sgd, loss, dh, st));
            return tc_dh(lo, nullptr, nullptr, dZt, true, B, W, dh, st);
        }
        TRY(tc_fwd(lo, B, W, nullptr, nullptr, nullptr, dZt, loss, st));
        TRY(tc_dW(lo, nullptr, nullptr, dZt, B, dW, st));
        TRY(tc_dh(lo, nullptr, nullptr, dZt, false, B, W, dh, st));
        return sgd ? sgd_update(lo, W, dW, *sgd, st) : SG_OK;
    }
    uint16_t *dZ = lo->dZ_ws;
    uint16_t *dZlo = lo->dZ_ws + (size_t)B * lo->L;
    TRY(tc_f ? tc_fwd(lo, B, W, nullptr, dZ, dZlo, nullptr, loss, st)
             : simt_fwd(lo, B, W, nullptr, dZ, dZlo, loss, st));
    TRY(tc_w ? tc_dW(lo, dZ, dZlo, nullptr, B, dW, st) : simt_dW(lo, dZ, dZlo, B, dW, st));
    TRY(tc_h ? tc_dh(lo, dZ, dZlo, nullptr, false, B, W, dh, st) : simt_dh(lo, dZ, dZlo, B, W, dh, st));
    return sgd ? sgd_update(lo, W, dW, *sgd, st) : SG_OK;
}

}  // namespace

sg_status sg_step_plan(const sg_layout *lo, int32_t B, int32_t sgd, int32_t *plan)
{
    const char *fn = "sg_step_plan";
    NvtxRange nvtx_(fn);
    if (!lo || !plan)
        FAIL(SG_ERR_INVALID, "%s: layout or plan is NULL", fn);
    if (B < 1 || B > lo->max_B)
        FAIL(SG_ERR_INVALID, "%s: B=%d outside [1, max_B=%d]", fn, B, lo->max_B);
    StepPath p;
    TRY(step_path(lo, B, sgd != 0, &p, fn));
    plan[0] = p.single ? SG_PLAN_ONE_KERNEL : p.fused ? SG_PLAN_FUSED_FWDW : SG_PLAN_PER_PHASE;
    plan[1] = p.tc_f;
    plan[2] = p.tc_w;
    plan[3] = p.tc_h;
    return SG_OK;
}

sg_status sg_step(sg_layout *lo, const sg_bf16 *h, int32_t B, const sg_bf16 *W,
                  const int32_t *pos_rowptr, const int32_t *pos_label,
                  int64_t nnz, sg_bf16 *dW, float *dh, double *loss,
                  void *stream)
{
    const char *fn = "sg_step";
    NvtxRange nvtx_(fn);
    TRY(check_call(lo, B, fn));
    TRY(check_pos(lo, pos_rowptr, pos_label, nnz, fn));
    REQUIRE(h, fn);
    REQUIRE(W, fn);
    REQUIRE(dW, fn);
    REQUIRE(dh, fn);
    REQUIRE(loss, fn);
    DeviceGuard dg(lo->device);
    return step_impl(lo, h, B, W, pos_rowptr, pos_label, nnz, dW, dh, loss, nullptr,
                     (cudaStream_t)stream, fn);
}

sg_status sg_step_sgd(sg_layout *lo, const sg_bf16 *h, int32_t B, const sg_bf16 *W_in,
                      const int32_t *pos_rowptr, const int32_t *pos_label, int64_t nnz, float lr,
                      float mu, float *mom, sg_bf16 *W_out, float *dh, double *loss, void *stream)
{
    const char *fn = "sg_step_sgd";
    NvtxRange nvtx_(fn);
    TRY(check_call(lo, B, fn));
    TRY(check_pos(lo, pos_rowptr, pos_label, nnz, fn));
    REQUIRE(h, fn);
    REQUIRE(W_in, fn);
    REQUIRE(W_out, fn);
    REQUIRE(mom, fn);
    REQUIRE(dh, fn);
    REQUIRE(loss, fn);
    if (!std::isfinite(lr) || !std::isfinite(mu))
        FAIL(SG_ERR_INVALID, "%s: lr and mu must be finite", fn);
    // dh is taken at W_in after the update has started writing W_out
    const uintptr_t in0 = (uintptr_t)W_in, out0 = (uintptr_t)W_out;
    const uintptr_t bytes = (uintptr_t)lo->L * (uintptr_t)lo->F * sizeof(sg_bf16);
    if (in0 < out0 + bytes && out0 < in0 + bytes)
        FAIL(SG_ERR_INVALID, "%s: W_out overlaps W_in", fn);
    DeviceGuard dg(lo->device);
    const sg_sgd sgd{mom, lr, mu};
    return step_impl(lo, h, B, W_in, pos_rowptr, pos_label, nnz, W_out, dh, loss, &sgd,
                     (cudaStream_t)stream, fn);
}

// ---------------------------------------------------------------- timing
sg_status sg_timing_start(sg_layout *lo, int32_t capacity)
{
    const char *fn = "sg_timing_start";
    NvtxRange nvtx_(fn);
    if (!lo)
        FAIL(SG_ERR_INVALID, "%s: layout is NULL", fn);
    if (capacity < 0 || capacity > (1 << 20))
        FAIL(SG_ERR_INVALID, "%s: capacity %d out of range", fn, capacity);
    DeviceGuard dg(lo->device);
    sg_layout::Timer &t = lo->timer;
    if (t.cap < capacity) {
        timer_release(t);
        t.ev = new (std::nothrow) cudaEvent_t[2 * (size_t)capacity];
        t.kind = new (std::nothrow) int[capacity];
        if (!t.ev || !t.kind) {
            timer_release(t);
            FAIL(SG_ERR_OOM, "%s: host allocation failed", fn);
        }
        for (int i = 0; i < 2 * capacity; ++i) {
            if (cudaEventCreate(&t.ev[i]) != cudaSuccess) {
                for (int j = 0; j < i; ++j)
                    cudaEventDestroy(t.ev[j]);
                delete[] t.ev;
                t.ev = nullptr;
                timer_release(t);
                FAIL(SG_ERR_CUDA, "%s: cudaEventCreate failed", fn);
            }
        }
        t.cap = capacity;
    }
    t.n = 0;
    t.pending = false;
    for (int i = 0; i < SG_KIND_COUNT; ++i)
        t.counts[i] = 0;
    t.on = true;
    return SG_OK;
}

sg_status sg_timing_stop(sg_layout *lo, double *ms_per_kind,
                         int32_t *launches_per_kind)
{
    const char *fn = "sg_timing_stop";
    NvtxRange nvtx_(fn);
    if (!lo)
        FAIL(SG_ERR_INVALID, "%s: layout is NULL", fn);
    DeviceGuard dg(lo->device);
    sg_layout::Timer &t = lo->timer;
    t.on = false;
    double ms[SG_KIND_COUNT] = {};
    if (t.n > 0)
        SG_TRY_CUDA(cudaEventSynchronize(t.ev[2 * t.n - 1]));
    for (int i = 0; i < t.n; ++i) {
        float e = 0.f;
        SG_TRY_CUDA(cudaEventElapsedTime(&e, t.ev[2 * i], t.ev[2 * i + 1]));
        ms[t.kind[i]] += e;
    }
    for (int k = 0; k < SG_KIND_COUNT; ++k) {
        if (ms_per_kind)
            ms_per_kind[k] = ms[k];
        if (launches_per_kind)
            launches_per_kind[k] = t.counts[k];
    }
    return SG_OK;
}

}  // extern "C"
