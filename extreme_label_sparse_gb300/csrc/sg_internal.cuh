// Internal declarations of the sg library (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "../../include/sg.h"

// ----------------------------------------------------------------- limits
constexpr int SG_MAX_B = 256;
constexpr int SG_MAX_F = 256;
constexpr int SG_MAX_H = 65535;  // idx is u16
constexpr int SG_MAX_G = 256;

// ----------------------------------------------------------------- layout
struct sg_layout {
    int64_t L = 0, K = 0;
    int32_t G = 0, F = 0, H = 0, max_B = 0;
    int64_t max_nnz = 0;
    int32_t engine = SG_ENGINE_AUTO;
    int32_t device = 0;
    int32_t num_sms = 0;
    bool tc_ok = false;  // the tensor-core engine can run this layout

    // canonical layout (device)
    int32_t *slot_of_label = nullptr;  // [L]
    int32_t *label_of_slot = nullptr;  // [L]
    uint16_t *idx_s = nullptr;         // [K][F] ascending

    // per-call scratch (device)
    uint16_t *hT = nullptr;  // [H][ldB] bf16, transposed h, zero padded
    int32_t ldB = 0;         // roundup(max_B, 128)
    int32_t *gcount = nullptr;  // [K+1], all zero between calls
    int32_t *gptr = nullptr;    // [K+1]
    int32_t *scan_part = nullptr;  // per-tile sums of the group-count scan
    int32_t *gent = nullptr;    // [max_nnz]  (b << 16) | j
    int32_t *tsorted = nullptr; // [max_nnz]  per-row slots, sorted (with dups)
    int32_t *tslots = nullptr;  // [max_nnz]  per-row slots, sorted, deduplicated
    int32_t *rowcnt = nullptr;  // [max_B]    kept entries per row
    double *loss_part = nullptr;
    int32_t loss_part_n = 0;
    int32_t *status = nullptr;  // sticky device status word

    // dZ scratch of the composed step (hi and lo bf16 planes of max_B x L),
    // allocated on first use
    uint16_t *dZ_ws = nullptr;
    size_t dZ_ws_elems = 0;
    // the step's max |W| as bf16 magnitude bits (scale of dh's fp16 operands),
    // in two slots used by alternate fused launches (each launch clears the
    // other slot for the next), then the fused kernel's loss ticket; zeroed
    // once when allocated.  wmax_slot: the slot the last fused launch wrote.
    uint32_t *wmax = nullptr;
    int32_t wmax_slot = 0;

    // scratch of sg_headtail_step when this layout is the tail (allocated on
    // first use): projected activations, both branches' dh, bf16 planes
    void *ht_ws = nullptr;
    size_t ht_ws_bytes = 0;
    // grow scores of sg_rewire ([K][H] fp32, allocated on first use)
    float *rw_ws = nullptr;
    size_t rw_ws_bytes = 0;

    // resident clusters of the fused step kernel for the shape keyed by
    // step_ncl_key (0 until the first call)
    int64_t step_ncl = 0, step_ncl_key = 0;

    // per-kernel event timing (sg_timing_start / sg_timing_stop)
    struct Timer {
        bool on = false;
        bool pending = false;
        int cap = 0, n = 0;
        cudaEvent_t *ev = nullptr;  // [2 * cap]
        int *kind = nullptr;        // [cap]
        int32_t counts[SG_KIND_COUNT] = {};
    } timer;
};

// Bracket one kernel launch with timing events (no-op unless enabled).
inline void sg_tick(sg_layout *lo, int kind, cudaStream_t st)
{
    sg_layout::Timer &t = lo->timer;
    if (!t.on)
        return;
    t.counts[kind] += 1;
    t.pending = t.n < t.cap;
    if (t.pending) {
        t.kind[t.n] = kind;
        cudaEventRecord(t.ev[2 * t.n], st);
    }
}

inline void sg_tock(sg_layout *lo, cudaStream_t st)
{
    sg_layout::Timer &t = lo->timer;
    if (!t.on || !t.pending)
        return;
    cudaEventRecord(t.ev[2 * t.n + 1], st);
    t.n += 1;
    t.pending = false;
}

#define SG_LAUNCH(lo, kind, st, ...)   \
    do {                               \
        sg_tick((lo), (kind), (st));   \
        __VA_ARGS__;                   \
        sg_tock((lo), (st));           \
    } while (0)

// ----------------------------------------------------------------- errors
void sg_set_error(const char *fmt, ...);
#define SG_TRY_CUDA(expr)                                                   \
    do {                                                                    \
        cudaError_t e_ = (expr);                                            \
        if (e_ != cudaSuccess) {                                            \
            sg_set_error("%s failed: %s (%s:%d)", #expr,                    \
                         cudaGetErrorString(e_), __FILE__, __LINE__);       \
            cudaGetLastError(); /* a later call must not see it again */    \
            return SG_ERR_CUDA;                                             \
        }                                                                   \
    } while (0)

// First error wins: a later error never overwrites an earlier one.
__device__ __forceinline__ void sg_flag(int32_t *status, int32_t code)
{
    atomicCAS(status, 0, code);
}

// ----------------------------------------------------------------- bf16
__device__ __forceinline__ float bf2f(uint16_t v)
{
    return __uint_as_float(((uint32_t)v) << 16);
}

// fp32 -> bf16 bits, round to nearest even (finite inputs; NaN kept quiet)
__device__ __forceinline__ uint16_t f2bf(float x)
{
    uint32_t u = __float_as_uint(x);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu))
        return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

// ----------------------------------------------------------------- BCE
// loss term max(z,0) - y z + log(1 + e^-|z|) and gradient sigmoid(z) - y,
// in fp32 with CUDA's expf/log1pf.
__device__ __forceinline__ float bce_grad_loss(float z, int y, float *loss)
{
    float e = expf(-fabsf(z));
    float r = 1.0f / (1.0f + e);
    float sig = z >= 0.f ? r : e * r;
    *loss = fmaxf(z, 0.f) - (y ? z : 0.f) + log1pf(e);
    return sig - (float)y;
}

// ----------------------------------------------------------------- launchers
// layout.cu
sg_status sg_layout_kernels(sg_layout *lo, const int32_t *groups,
                            const int32_t *idx, cudaStream_t st);
// pos.cu: build the per-group positive lists (gptr/gent) for one call
sg_status sg_pos_prepare(sg_layout *lo, int32_t B, const int32_t *rowptr,
                         const int32_t *labels, int64_t nnz, cudaStream_t st);
sg_status sg_pos_compact(sg_layout *lo, int32_t B, const int32_t *rowptr,
                         int32_t *out_rowptr, int32_t *out_slots,
                         cudaStream_t st);
// An NVTX range around a public entry point, named after it (a profiler shows
// the library's calls on its timeline; without one attached the calls cost
// nothing beyond a branch)
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

// per-label fan-in (G = 1) kernels of the CUDA-core engine (g1.cu)
bool g1_ok(const sg_layout *lo);
sg_status g1_fwd(sg_layout *lo, int32_t B, const uint16_t *W, uint16_t *Z, uint16_t *dZ, uint16_t *dZ_lo,
                 double *loss, cudaStream_t st);
sg_status g1_dW(sg_layout *lo, const uint16_t *dZ, const uint16_t *dZ_lo, int32_t B, uint16_t *dW, cudaStream_t st);
sg_status g1_dh(sg_layout *lo, const uint16_t *dZ, const uint16_t *dZ_lo, int32_t B, const uint16_t *W, float *dh,
                cudaStream_t st);

sg_status sg_loss_finalize(sg_layout *lo, int32_t nparts, double *loss,
                           cudaStream_t st);
// simt.cu
// One 32 x 32 tile of h^T: rows i0 .. i0 + 31 (features), columns b0 ..
// b0 + 31 (samples; zero past B, up to ldB), by 256 threads (tx = thread
// mod 32, ty = thread / 32) through a padded shared tile.  Every thread of the
// block calls it.
__device__ __forceinline__ void transpose_h_tile(const uint16_t *__restrict__ h, int B, int H, int ldB,
                                                 uint16_t *__restrict__ hT, int i0, int b0, int tx, int ty,
                                                 uint16_t (*tile)[34])
{
    for (int r = ty; r < 32; r += 8) {
        const int b = b0 + r, i = i0 + tx;
        tile[r][tx] = (b < B && i < H) ? h[(int64_t)b * H + i] : (uint16_t)0;
    }
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {
        const int i = i0 + r, b = b0 + tx;
        if (i < H && b < ldB)
            hT[(int64_t)i * ldB + b] = tile[tx][r];
    }
}

// The step's preparation in three fewer launches than the transpose plus
// sg_pos_prepare: one kernel runs the positive rows and the transpose of h
// side by side, then the group scan and the bucketing.
sg_status sg_step_prepare(sg_layout *lo, const uint16_t *h, int32_t B, const int32_t *rowptr,
                          const int32_t *labels, int64_t nnz, cudaStream_t st);
sg_status simt_transpose_h(sg_layout *lo, const uint16_t *h, int32_t B,
                           cudaStream_t st);
// dZ_lo (optional): second bf16 plane with dZ - bf16(dZ), so that hi + lo
// carries dZ to about 16 significant bits between the forward and backward
sg_status simt_fwd(sg_layout *lo, int32_t B, const uint16_t *W, uint16_t *Z,
                   uint16_t *dZ, uint16_t *dZ_lo, double *loss, cudaStream_t st);
sg_status simt_bce(sg_layout *lo, const uint16_t *Z, int32_t B, uint16_t *dZ,
                   double *loss, cudaStream_t st);
sg_status simt_dW(sg_layout *lo, const uint16_t *dZ, const uint16_t *dZ_lo,
                  int32_t B, uint16_t *dW, cudaStream_t st);
sg_status simt_dh(sg_layout *lo, const uint16_t *dZ, const uint16_t *dZ_lo,
                  int32_t B, const uint16_t *W, float *dh, cudaStream_t st);
// tc.cu
bool tc_supported(const sg_layout *lo);
bool tc_stage_ok(const sg_layout *lo, int stage, int B);
// dZ is either caller-layout [B][L] (dZ, optional residual plane dZ_lo) or
// the step's group-tiled workspace dZt (both planes; see tc.cu)
sg_status tc_fwd(sg_layout *lo, int32_t B, const uint16_t *W, uint16_t *Z,
                 uint16_t *dZ, uint16_t *dZ_lo, uint8_t *dZt, double *loss, cudaStream_t st);
sg_status tc_dW(sg_layout *lo, const uint16_t *dZ, const uint16_t *dZ_lo, const uint8_t *dZt,
                int32_t B, uint16_t *dW, cudaStream_t st);
// dzt_f16: the tiled dZ is the fused kernel's single fp16 plane (fp16 MMA
// operands, W scaled by the step's max |W| that kernel recorded)
sg_status tc_dh(sg_layout *lo, const uint16_t *dZ, const uint16_t *dZ_lo, const uint8_t *dZt,
                bool dzt_f16, int32_t B, const uint16_t *W, float *dh, cudaStream_t st);
sg_status tc_ensure_wmax(sg_layout *lo);
// bytes of one group's dZ tile, and whether fwd, dW and dh all run on the
// tensor cores with the tiled workspace for this batch size
uint64_t tc_dz_tile_bytes(const sg_layout *lo, int32_t B);
bool tc_tiled_ok(const sg_layout *lo, int32_t B);
// fused forward + BCE + dW into the tiled workspace (one pass over the groups)
bool tc_fwdw_ok(const sg_layout *lo, int32_t B);
// momentum SGD of the output layer: m <- mu m + dW, W_out <- bf16(W - lr m)
struct sg_sgd {
    float *mom;  // [L][F] fp32, read and written
    float lr, mu;
};
// with sgd, dW receives the updated weights instead of the gradient
// dh_zero: the feature gradient the following tc_dh (fp16 workspace) adds
// into, cleared by this kernel (B x H floats), or nullptr
sg_status tc_fwdw(sg_layout *lo, int32_t B, const uint16_t *W, uint8_t *dZt, uint16_t *dW,
                  const sg_sgd *sgd, double *loss, float *dh_zero, cudaStream_t st);
// the same update from a stored bf16 dW (in place: W_out holds dW on entry)
sg_status sgd_update(sg_layout *lo, const uint16_t *W, uint16_t *W_out, const sg_sgd &sgd, cudaStream_t st);

// step.cu: the whole step (forward, BCE, dW, dh) in one kernel on clusters
// of CTAs that split dh's columns (B <= 128, G in {16, 32, 64}, F % 16 == 0,
// F <= 128)
bool tc_step_ok(const sg_layout *lo, int32_t B);
sg_status tc_step(sg_layout *lo, int32_t B, const uint16_t *W, uint16_t *dW, float *dh, double *loss,
                  cudaStream_t st);

static inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
