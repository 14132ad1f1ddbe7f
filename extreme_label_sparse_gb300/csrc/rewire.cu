// Rewiring of the groups' fan-in sets (HASTE, "Method / overall framework"
// and "Loss and training strategy": a periodic discrete phase re-selects each
// I_k by the RigL protocol, |I_k| = F).  The selection rule is not on the
// pages; this is the RigL reading for group-shared fan-in:
//   prune score of an active index f:  m_k(f) = sum over the group of |W[l][f]|
//   grow score of a feature j:         g_k(j) = sum over the group of
//                                               |sum_b dZ[b][l] h[b][j]|
// drop the n_drop smallest m (ties: smaller feature), grow the n_drop largest g
// outside the old I_k (ties: smaller feature); kept columns keep their
// weights, grown ones start at zero, the new I_k is sorted ascending.
//
// The grow scores of every (group, feature) are one tcgen05 GEMM, h^T dZ,
// whose epilogue sums |.| over each group's labels (gemm.cu: the labels
// streamed past a resident tile of h; groups below 16 labels take the tiled
// form dZ^T h); the selection is one warp per group.
#include "sg_internal.cuh"

sg_status gemm_group_abs(const uint16_t *A, int64_t lda, int M, const uint16_t *B, int64_t ldb, int N, int K, int G,
                         float *out, int32_t *status, cudaStream_t st);
sg_status gemm_group_abs_t(const uint16_t *A, int64_t lda, int M, const uint16_t *B, int64_t ldb, int64_t L, int K,
                           int G, float *out, int num_sms, int32_t *status, cudaStream_t st);

namespace {

constexpr int kRwWarps = 4;
constexpr int kRwMaxF = 256;
constexpr int kRwRegs = 32;  // grow-score registers per lane (H <= 1024 held in registers)

__device__ __forceinline__ float bfv(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }

// warp-wide best of (value, feature): larger value first (grow) or smaller
// value first (prune); ties to the smaller feature
__device__ __forceinline__ void warp_best(float &v, int &j, bool largest)
{
    for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
        const int j2 = __shfl_xor_sync(0xffffffffu, j, o);
        const bool take = j2 >= 0 && (j < 0 || (largest ? v2 > v : v2 < v) || (v2 == v && j2 < j));
        if (take) {
            v = v2;
            j = j2;
        }
    }
}

// one warp per group k
__global__ void __launch_bounds__(32 * kRwWarps)
    k_rewire_select(int64_t K, int32_t G, int32_t F, int32_t H, int32_t n_drop, const uint16_t *__restrict__ idx_s,
                    const uint16_t *__restrict__ W, float *__restrict__ score, int32_t *__restrict__ idx_out,
                    uint16_t *__restrict__ W_out)
{
    __shared__ int32_t sh_drop[kRwWarps][kRwMaxF];
    __shared__ int32_t sh_grow[kRwWarps][kRwMaxF];
    const int lane = threadIdx.x & 31, wl = threadIdx.x / 32;
    const int64_t k = (int64_t)blockIdx.x * kRwWarps + wl;
    if (k >= K)
        return;
    const uint16_t *I = idx_s + k * F;
    const uint16_t *Wk = W + k * G * F;
    float *sc = score + k * (int64_t)H;
    int32_t *drop = sh_drop[wl], *grow = sh_grow[wl];
    constexpr int FT = kRwMaxF / 32;  // f slots per lane
    // prune scores of this lane's f = lane + 32 t, summed over the group's rows
    float m[FT];
    bool dropped[FT];
#pragma unroll
    for (int t = 0; t < FT; ++t) {
        const int f = lane + 32 * t;
        float s = 0.f;
        if (f < F)
            for (int g = 0; g < G; ++g)
                s += fabsf(bfv(Wk[(int64_t)g * F + f]));
        m[t] = s;
        dropped[t] = false;
    }
    // drop the n_drop smallest.  Each lane keeps the best of its own slots
    // (smallest m, then smallest feature); a round takes the warp's best and
    // only the lane that held it looks at its slots again.  Slot loops stop
    // at the slots that hold features (a warp-uniform bound).
    const int ftn = (F + 31) / 32;
    int feat[FT];
#pragma unroll
    for (int t = 0; t < FT; ++t) {
        const int f = lane + 32 * t;
        feat[t] = t < ftn && f < F ? (int)I[f] : -1;
    }
    float dv = 0.f;
    int dj = -1, dt = -1;
    auto drop_best = [&]() {
        dv = 0.f;
        dj = -1;
        dt = -1;
#pragma unroll
        for (int t = 0; t < FT; ++t) {
            if (t >= ftn)
                break;
            if (feat[t] >= 0 && !dropped[t] && (dj < 0 || m[t] < dv || (m[t] == dv && feat[t] < dj))) {
                dv = m[t];
                dj = feat[t];
                dt = t;
            }
        }
    };
    drop_best();
    for (int r = 0; r < n_drop; ++r) {
        float v = dv;
        int j = dj;
        warp_best(v, j, false);
        if (j >= 0 && dj == j) {  // this lane held it (features of a group are distinct)
#pragma unroll
            for (int t = 0; t < FT; ++t)
                if (t == dt)
                    dropped[t] = true;
            drop_best();
        }
        if (lane == 0)
            drop[r] = j;
    }
    // the old members are no candidates
    for (int f = lane; f < F; f += 32)
        sc[I[f]] = -1.f;
    __syncwarp();
    // grow the n_drop largest: the row in registers (feature x = lane + 32 t)
    // when it fits, else scanned from memory each time; as for the drop, a
    // lane keeps its best (largest, then smallest x) and only the lane that
    // held a round's winner looks again
    if (H <= 32 * kRwRegs) {
        const int htn = (H + 31) / 32;
        float rv[kRwRegs];
#pragma unroll
        for (int t = 0; t < kRwRegs; ++t) {
            const int x = lane + 32 * t;
            rv[t] = t < htn && x < H ? sc[x] : -1.f;
        }
        float gv = -1.f;
        int gj = -1, gt = -1;
        auto grow_best = [&]() {
            gv = -1.f;
            gj = -1;
            gt = -1;
#pragma unroll
            for (int t = 0; t < kRwRegs; ++t) {
                if (t >= htn)
                    break;
                if (rv[t] >= 0.f && (gj < 0 || rv[t] > gv)) {  // ascending x: ties keep the smaller
                    gv = rv[t];
                    gj = lane + 32 * t;
                    gt = t;
                }
            }
        };
        grow_best();
        for (int r = 0; r < n_drop; ++r) {
            float v = gv;
            int j = gj;
            warp_best(v, j, true);
            if (j >= 0 && gj == j) {
#pragma unroll
                for (int t = 0; t < kRwRegs; ++t)
                    if (t == gt)
                        rv[t] = -1.f;
                grow_best();
            }
            if (lane == 0)
                grow[r] = j;
        }
    } else {
        for (int r = 0; r < n_drop; ++r) {
            float v = -1.f;
            int j = -1;
            for (int x = lane; x < H; x += 32) {
                const float s = sc[x];
                if (s >= 0.f && (j < 0 || s > v))  // ascending x: ties keep the smaller
                    v = s, j = x;
            }
            warp_best(v, j, true);
            if (lane == 0) {
                grow[r] = j;
                if (j >= 0)
                    sc[j] = -1.f;
            }
            __syncwarp();
        }
    }
    __syncwarp();
    // the new set, ascending: a kept index at old position p lands at
    // (#kept below it) + (#grown below it); a grown one at
    // (#old below it) - (#dropped below it) + (#grown below it)
    unsigned below = 0;  // kept positions before this chunk
#pragma unroll
    for (int t = 0; t < FT; ++t) {
        const int f = lane + 32 * t;
        const bool keep = f < F && !dropped[t];
        const unsigned bal = __ballot_sync(0xffffffffu, keep);
        if (keep) {
            const int v = I[f];
            int pos = (int)below + __popc(bal & ((1u << lane) - 1u));
            for (int r = 0; r < n_drop; ++r)
                pos += grow[r] < v ? 1 : 0;
            idx_out[k * F + pos] = v;
            for (int g = 0; g < G; ++g)
                W_out[(k * G + g) * F + pos] = Wk[(int64_t)g * F + f];
        }
        below += __popc(bal);
    }
    for (int r = lane; r < n_drop; r += 32) {
        const int v = grow[r];
        int lo = 0, hi = F;  // old members below v
        while (lo < hi) {
            const int mid = (lo + hi) / 2;
            if ((int)I[mid] < v)
                lo = mid + 1;
            else
                hi = mid;
        }
        int pos = lo;
        for (int q = 0; q < n_drop; ++q) {
            pos -= drop[q] < v ? 1 : 0;
            pos += grow[q] < v ? 1 : 0;
        }
        idx_out[k * F + pos] = v;
        for (int g = 0; g < G; ++g)
            W_out[(k * G + g) * F + pos] = 0;
    }
}

}  // namespace

extern "C" sg_status sg_rewire(sg_layout *lo, const sg_bf16 *h, int32_t B, const sg_bf16 *dZ, const sg_bf16 *W,
                               int32_t n_drop, int32_t *idx_out, sg_bf16 *W_out, void *stream)
{
    const char *fn = "sg_rewire";
    NvtxRange nvtx_(fn);
    if (!lo || !h || !dZ || !W || !idx_out || !W_out) {
        sg_set_error("%s: a required pointer is NULL", fn);
        return SG_ERR_INVALID;
    }
    if (B < 1 || n_drop < 0 || n_drop > lo->F || n_drop > lo->H - lo->F) {
        sg_set_error("%s: need B >= 1 and 0 <= n_drop <= min(F, H - F) (B=%d n_drop=%d)", fn, B, n_drop);
        return SG_ERR_INVALID;
    }
    const int G = lo->G;
    if (G > 128 || (G & (G - 1)) != 0 || lo->F > kRwMaxF || lo->L % 8 != 0 || lo->H % 8 != 0 ||
        lo->L > INT32_MAX / 2) {
        sg_set_error("%s: needs G a power of two <= 128, F <= %d, L and H multiples of 8 (G=%d F=%d L=%lld H=%d)",
                     fn, kRwMaxF, G, lo->F, (long long)lo->L, lo->H);
        return SG_ERR_UNSUPPORTED;
    }
    const uintptr_t w0 = (uintptr_t)W, w1 = w0 + (uintptr_t)lo->L * lo->F * 2, o0 = (uintptr_t)W_out,
                    o1 = o0 + (uintptr_t)lo->L * lo->F * 2;
    if (w0 < o1 && o0 < w1) {
        sg_set_error("%s: W_out overlaps W", fn);
        return SG_ERR_INVALID;
    }
    int prev = -1;
    cudaGetDevice(&prev);
    if (prev != lo->device)
        cudaSetDevice(lo->device);
    cudaStream_t st = (cudaStream_t)stream;
    sg_status rc = SG_OK;
    const size_t need = sizeof(float) * (size_t)lo->K * lo->H;
    if (lo->rw_ws_bytes < need) {
        if (lo->rw_ws)
            cudaFree(lo->rw_ws);
        lo->rw_ws = nullptr;
        lo->rw_ws_bytes = 0;
        if (cudaMalloc((void **)&lo->rw_ws, need) != cudaSuccess) {
            cudaGetLastError();
            sg_set_error("%s: cudaMalloc of %zu bytes of grow scores failed", fn, need);
            rc = SG_ERR_OOM;
        } else {
            lo->rw_ws_bytes = need;
        }
    }
    // grow scores: the labels streamed past a resident tile of h (A = h,
    // MN-major, M = H; B = dZ, MN-major, the L labels; K = samples), or for
    // groups below 16 labels A = dZ^T (M = L) against B = h^T (N = H)
    if (rc == SG_OK) {
        if (G >= 16 && B <= 256 && lo->L <= INT32_MAX)
            rc = gemm_group_abs_t(h, lo->H, lo->H, dZ, lo->L, lo->L, B, G, lo->rw_ws, lo->num_sms, lo->status, st);
        else
            rc = SG_ERR_UNSUPPORTED;
        if (rc == SG_ERR_UNSUPPORTED)
            rc = gemm_group_abs(dZ, lo->L, (int)lo->L, h, lo->H, lo->H, B, G, lo->rw_ws, lo->status, st);
    }
    if (rc == SG_OK) {
        const unsigned grid = (unsigned)((lo->K + kRwWarps - 1) / kRwWarps);
        k_rewire_select<<<grid, 32 * kRwWarps, 0, st>>>(lo->K, G, lo->F, lo->H, n_drop, lo->idx_s, W, lo->rw_ws,
                                                       idx_out, W_out);
        if (cudaGetLastError() != cudaSuccess) {
            sg_set_error("%s: launch failed", fn);
            rc = SG_ERR_CUDA;
        }
    }
    if (prev >= 0 && prev != lo->device)
        cudaSetDevice(prev);
    return rc;
}
