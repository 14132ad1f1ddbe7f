// CUDA-core engine: every group size G (G = 1 is per-label fixed fan-in),
// FP32 accumulation.  It follows the same dataflow as the tensor-core engine
// (HASTE, key design "gather-once + dense MMA kernel"): the block gathers the
// group's H_k tile once into shared memory and every label of the group reuses
// it; dh is a Split-K over label chunks with a CTA-local partial in shared
// memory, flushed to global memory with atomics once per CTA.
#include "sg_internal.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kWLD = 33;     // row stride (floats) of the transposed W chunk
constexpr int kBT = 32;      // samples per dh tile (one per lane)

__host__ __device__ inline int align16(int x) { return (x + 15) & ~15; }

// ------------------------------------------------------------ h transpose
// hT[i][b] = h[b][i], zero for b >= B (hT has ldB >= B columns).
__global__ void k_transpose_h(const uint16_t *__restrict__ h, int B, int H,
                              int ldB, uint16_t *__restrict__ hT)
{
    __shared__ uint16_t tile[32][34];
    transpose_h_tile(h, B, H, ldB, hT, blockIdx.x * 32, blockIdx.y * 32, threadIdx.x, threadIdx.y, tile);
}

__device__ __forceinline__ void block_sum_to(double v, double *dst)
{
    __shared__ double red[kThreads / 32];
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_down_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        double s = 0.0;
        for (int w = 0; w < kThreads / 32; ++w)
            s += red[w];
        *dst = s;
    }
}

// positives of sample b among slots j0 .. j0+n-1 of group k, as a bit mask
__device__ __forceinline__ uint32_t pos_mask(const int32_t *__restrict__ gptr,
                                             const int32_t *__restrict__ gent,
                                             int64_t k, int b, int j0, int n)
{
    uint32_t y = 0;
    const int e1 = gptr[k + 1];
    for (int e = gptr[k]; e < e1; ++e) {
        int v = gent[e];
        int jj = (v & 0xffff) - j0;
        if ((v >> 16) == b && jj >= 0 && jj < n)
            y |= 1u << jj;
    }
    return y;
}

// gather H_k = h[:, I_k] from hT: rows I_k[f] of hT (ldB bf16 each) into
// Hs[f][0..ldB) with row stride ld (elements); 16-byte loads.
__device__ __forceinline__ void gather_rows(const uint16_t *__restrict__ hT,
                                            int ldB, const int *idxs, int F,
                                            uint16_t *Hs, int ld)
{
    const int nch = ldB >> 3;
    for (int e = threadIdx.x; e < F * nch; e += kThreads) {
        int f = e / nch, c = e - f * nch;
        uint4 v = __ldg(reinterpret_cast<const uint4 *>(hT + (int64_t)idxs[f] * ldB) + c);
        uint32_t *d = reinterpret_cast<uint32_t *>(Hs + f * ld + c * 8);
        d[0] = v.x;
        d[1] = v.y;
        d[2] = v.z;
        d[3] = v.w;
    }
}

// ------------------------------------------------------------ forward
struct FwdArgs {
    const uint16_t *hT, *W, *idx_s;
    uint16_t *Z, *dZ, *dZ_lo;
    const int32_t *gptr, *gent;
    double *loss_part;
    int64_t K, L;
    int32_t B, ldB, G, F;
};

template <int JT, bool BCE>
__global__ void __launch_bounds__(kThreads) k_simt_fwd(FwdArgs a)
{
    extern __shared__ __align__(16) unsigned char smem[];
    const int F = a.F, ldB = a.ldB, B = a.B, G = a.G;
    uint16_t *Hs = reinterpret_cast<uint16_t *>(smem);
    float *Ws = reinterpret_cast<float *>(smem + align16(F * ldB * 2));
    int *idxs = reinterpret_cast<int *>(Ws + F * kWLD);
    const int tid = threadIdx.x;
    const int GC = G < 32 ? G : 32;
    double lacc = 0.0;

    for (int64_t k = blockIdx.x; k < a.K; k += gridDim.x) {
        for (int f = tid; f < F; f += kThreads)
            idxs[f] = a.idx_s[k * F + f];
        __syncthreads();
        gather_rows(a.hT, ldB, idxs, F, Hs, ldB);
        for (int j0 = 0; j0 < G; j0 += GC) {
            const int gc = min(GC, G - j0);
            for (int e = tid; e < gc * F; e += kThreads) {
                int j = e / F, f = e - j * F;
                Ws[f * kWLD + j] = bf2f(a.W[(k * G + j0 + j) * (int64_t)F + f]);
            }
            __syncthreads();
            const int ntask = B * (gc / JT);
            for (int t = tid; t < ntask; t += kThreads) {
                const int b = t % B, jt = t / B;
                float acc[JT];
#pragma unroll
                for (int u = 0; u < JT; ++u)
                    acc[u] = 0.f;
                const float *wp = Ws + jt * JT;
                const uint16_t *hp = Hs + b;
                for (int f = 0; f < F; ++f) {
                    float hv = bf2f(hp[f * ldB]);
#pragma unroll
                    for (int u = 0; u < JT; ++u)
                        acc[u] = fmaf(hv, wp[f * kWLD + u], acc[u]);
                }
                const int64_t s0 = k * G + j0 + jt * JT;
                if (a.Z) {
                    uint16_t *zr = a.Z + (int64_t)b * a.L + s0;
#pragma unroll
                    for (int u = 0; u < JT; ++u)
                        zr[u] = f2bf(acc[u]);
                }
                if (BCE) {
                    uint32_t y = pos_mask(a.gptr, a.gent, k, b, j0 + jt * JT, JT);
                    uint16_t *dr = a.dZ + (int64_t)b * a.L + s0;
                    float l = 0.f;
#pragma unroll
                    for (int u = 0; u < JT; ++u) {
                        float lt;
                        float d = bce_grad_loss(acc[u], (y >> u) & 1u, &lt);
                        l += lt;
                        const uint16_t hi = f2bf(d);
                        dr[u] = hi;
                        if (a.dZ_lo)
                            a.dZ_lo[(int64_t)b * a.L + s0 + u] = f2bf(d - bf2f(hi));
                    }
                    lacc += l;
                }
            }
            __syncthreads();
        }
    }
    if (BCE)
        block_sum_to(lacc, a.loss_part + blockIdx.x);
}

// ------------------------------------------------------------ BCE from Z
__global__ void __launch_bounds__(kThreads)
    k_simt_bce(const uint16_t *__restrict__ Z, int B, int64_t L, int G,
               const int32_t *__restrict__ gptr, const int32_t *__restrict__ gent,
               uint16_t *__restrict__ dZ, double *loss_part)
{
    const int64_t cpr = (L + 7) / 8;
    const int64_t total = (int64_t)B * cpr;
    double lacc = 0.0;
    for (int64_t c = blockIdx.x * (int64_t)kThreads + threadIdx.x; c < total;
         c += (int64_t)gridDim.x * kThreads) {
        const int b = (int)(c / cpr);
        const int64_t s0 = (c - (int64_t)b * cpr) * 8;
        const int n = (int)min((int64_t)8, L - s0);
        const uint16_t *zr = Z + (int64_t)b * L + s0;
        uint16_t *dr = dZ + (int64_t)b * L + s0;
        int64_t k = s0 / G;
        int j = (int)(s0 - k * G);
        float l = 0.f;
        for (int u = 0; u < n; ++u) {
            int y = (int)pos_mask(gptr, gent, k, b, j, 1);
            float lt;
            float d = bce_grad_loss(bf2f(zr[u]), y, &lt);
            l += lt;
            dr[u] = f2bf(d);
            if (++j == G) {
                j = 0;
                ++k;
            }
        }
        lacc += l;
    }
    block_sum_to(lacc, loss_part + blockIdx.x);
}

// ------------------------------------------------------------ dW
struct DWArgs {
    const uint16_t *hT, *dZ, *dZ_lo, *idx_s;
    uint16_t *dW;
    int64_t K, L;
    int32_t B, ldB, G, F;
};

template <int JT>
__global__ void __launch_bounds__(kThreads) k_simt_dW(DWArgs a)
{
    extern __shared__ __align__(16) unsigned char smem[];
    const int F = a.F, ldB = a.ldB, B = a.B, G = a.G;
    const int ldp = ldB + 2;  // odd word stride: conflict-free column reads
    uint16_t *Hs = reinterpret_cast<uint16_t *>(smem);
    float *dZs = reinterpret_cast<float *>(smem + align16(F * ldp * 2));  // [B][32]
    int *idxs = reinterpret_cast<int *>(dZs + B * 32);
    const int tid = threadIdx.x;
    const int GC = G < 32 ? G : 32;

    for (int64_t k = blockIdx.x; k < a.K; k += gridDim.x) {
        for (int f = tid; f < F; f += kThreads)
            idxs[f] = a.idx_s[k * F + f];
        __syncthreads();
        gather_rows(a.hT, ldB, idxs, F, Hs, ldp);
        for (int j0 = 0; j0 < G; j0 += GC) {
            const int gc = min(GC, G - j0);
            for (int e = tid; e < B * gc; e += kThreads) {
                int b = e / gc, j = e - b * gc;
                const int64_t at = (int64_t)b * a.L + k * G + j0 + j;
                dZs[b * 32 + j] = bf2f(a.dZ[at]) + (a.dZ_lo ? bf2f(a.dZ_lo[at]) : 0.f);
            }
            __syncthreads();
            const int ntask = F * (gc / JT);
            for (int t = tid; t < ntask; t += kThreads) {
                const int f = t % F, jt = t / F;
                float acc[JT];
#pragma unroll
                for (int u = 0; u < JT; ++u)
                    acc[u] = 0.f;
                const uint16_t *hp = Hs + f * ldp;
                const float *dp = dZs + jt * JT;
                for (int b = 0; b < B; ++b) {
                    float hv = bf2f(hp[b]);
#pragma unroll
                    for (int u = 0; u < JT; ++u)
                        acc[u] = fmaf(hv, dp[b * 32 + u], acc[u]);
                }
                const int64_t s0 = k * G + j0 + jt * JT;
#pragma unroll
                for (int u = 0; u < JT; ++u)
                    a.dW[(s0 + u) * F + f] = f2bf(acc[u]);
            }
            __syncthreads();
        }
    }
}

// ------------------------------------------------------------ dh
// CTA (tile bt, part c): samples [32 bt, 32 bt + 32) x slot chunks
// [c0, c1) of 32 slots.  For each group piece in a chunk the lane (= sample)
// forms dH[b][f] = sum_j dZ[b][j] W[j][f] and adds it into the CTA partial
// part[b][I_k[f]] (shared-memory atomics; groups overlap).  The partial is
// added to dh once at the end.
struct DhArgs {
    const uint16_t *dZ, *dZ_lo, *W, *idx_s;
    float *dh;
    int64_t K, L;
    int32_t B, G, F, H;
    int32_t nbt;      // sample tiles
    int64_t nchunk;   // slot chunks in total
    int32_t nct;      // CTAs per (sample tile, column window)
    int32_t hw, ncw;  // dh columns per window, windows
};

__global__ void __launch_bounds__(kThreads) k_simt_dh(DhArgs a)
{
    extern __shared__ __align__(16) unsigned char smem[];
    const int F = a.F, H = a.H, G = a.G;
    const int ldp = a.hw + 1;
    float *part = reinterpret_cast<float *>(smem);                 // [32][hw+1]
    float *Ws = part + kBT * ldp;                                  // [32][F]
    float *dZs = Ws + 32 * F;                                      // [32][33]
    uint16_t *idxc = reinterpret_cast<uint16_t *>(dZs + kBT * 33); // [32][F]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int bt = blockIdx.x % a.nbt;
    const int cw = (blockIdx.x / a.nbt) % a.ncw;  // this CTA's window of dh columns
    const int c = blockIdx.x / (a.nbt * a.ncw);
    const int brow0 = bt * kBT;
    const int j0 = cw * a.hw;
    const int jn = H - j0 < a.hw ? H - j0 : a.hw;
    const int64_t q0 = a.nchunk * c / a.nct, q1 = a.nchunk * (c + 1) / a.nct;

    for (int e = tid; e < kBT * ldp; e += kThreads)
        part[e] = 0.f;
    for (int64_t q = q0; q < q1; ++q) {
        const int64_t s0 = q * 32;
        const int ns = (int)min((int64_t)32, a.L - s0);
        const int64_t kfirst = s0 / G, klast = (s0 + ns - 1) / G;
        const int ng = (int)(klast - kfirst + 1);
        __syncthreads();
        for (int e = tid; e < 32 * F; e += kThreads) {
            int s = e / F, f = e - s * F;
            Ws[e] = s < ns ? bf2f(a.W[(s0 + s) * F + f]) : 0.f;
        }
        for (int e = tid; e < kBT * 32; e += kThreads) {
            int b = e >> 5, s = e & 31;
            int row = brow0 + b;
            float v = 0.f;
            if (s < ns && row < a.B) {
                const int64_t at = (int64_t)row * a.L + s0 + s;
                v = bf2f(a.dZ[at]) + (a.dZ_lo ? bf2f(a.dZ_lo[at]) : 0.f);
            }
            dZs[b * 33 + s] = v;
        }
        for (int e = tid; e < ng * F; e += kThreads)
            idxc[e] = a.idx_s[kfirst * F + e];
        __syncthreads();
        for (int it = warp; it < ng * F; it += kThreads / 32) {
            const int j = (int)idxc[it] - j0;  // the same for the whole warp
            if (j < 0 || j >= jn)
                continue;
            const int g = it / F, f = it - g * F;
            const int64_t kb = (kfirst + g) * G;
            const int sa = (int)(max(kb, s0) - s0);
            const int sb = (int)(min(kb + G, s0 + ns) - s0);
            float acc = 0.f;
            for (int s = sa; s < sb; ++s)
                acc = fmaf(dZs[lane * 33 + s], Ws[s * F + f], acc);
            atomicAdd(&part[lane * ldp + j], acc);
        }
    }
    __syncthreads();
    for (int e = tid; e < kBT * jn; e += kThreads) {
        int b = e / jn, i = e - b * jn;
        int row = brow0 + b;
        if (row < a.B)
            atomicAdd(&a.dh[(int64_t)row * H + j0 + i], part[b * ldp + i]);
    }
}

int pick_jt(int G)
{
    int gc = G < 32 ? G : 32;
    if (G % 8 == 0 && gc % 8 == 0)
        return 8;
    if (G % 4 == 0)
        return 4;
    if (G % 2 == 0)
        return 2;
    return 1;
}

int persistent_grid(const sg_layout *lo, int64_t work, int per_sm)
{
    int64_t g = (int64_t)lo->num_sms * per_sm;
    if (g > work)
        g = work;
    if (g < 1)
        g = 1;
    if (g > lo->loss_part_n)
        g = lo->loss_part_n;
    return (int)g;
}

}  // namespace

sg_status simt_transpose_h(sg_layout *lo, const uint16_t *h, int32_t B,
                           cudaStream_t st)
{
    dim3 grid((unsigned)ceil_div(lo->H, 32), (unsigned)ceil_div(lo->ldB, 32));
    SG_LAUNCH(lo, SG_KIND_PREP, st, k_transpose_h<<<grid, dim3(32, 8), 0, st>>>(h, B, lo->H, lo->ldB, lo->hT));
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}

#define SG_SET_SMEM(kern, bytes)                                            \
    SG_TRY_CUDA(cudaFuncSetAttribute(kern,                                  \
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                     (int)(bytes)))

sg_status simt_fwd(sg_layout *lo, int32_t B, const uint16_t *W, uint16_t *Z,
                   uint16_t *dZ, uint16_t *dZ_lo, double *loss, cudaStream_t st)
{
    if (g1_ok(lo))  // per-label fan-in: its own kernels (g1.cu)
        return g1_fwd(lo, B, W, Z, dZ, dZ_lo, loss, st);
    FwdArgs a;
    a.hT = lo->hT;
    a.W = W;
    a.idx_s = lo->idx_s;
    a.Z = Z;
    a.dZ = dZ;
    a.dZ_lo = dZ_lo;
    a.gptr = lo->gptr;
    a.gent = lo->gent;
    a.loss_part = lo->loss_part;
    a.K = lo->K;
    a.L = lo->L;
    a.B = B;
    a.ldB = lo->ldB;  // row stride of hT as the transpose wrote it
    a.G = lo->G;
    a.F = lo->F;
    const size_t smem = align16(a.F * a.ldB * 2) + (size_t)a.F * kWLD * 4 + a.F * 4;
    const int grid = persistent_grid(lo, lo->K, 2);
    const bool bce = dZ != nullptr;
    void (*kern)(FwdArgs) = nullptr;
    switch (pick_jt(lo->G)) {
    case 1: kern = bce ? k_simt_fwd<1, true> : k_simt_fwd<1, false>; break;
    case 2: kern = bce ? k_simt_fwd<2, true> : k_simt_fwd<2, false>; break;
    case 4: kern = bce ? k_simt_fwd<4, true> : k_simt_fwd<4, false>; break;
    default: kern = bce ? k_simt_fwd<8, true> : k_simt_fwd<8, false>; break;
    }
    SG_SET_SMEM(kern, smem);
    SG_LAUNCH(lo, SG_KIND_FWD, st, kern<<<grid, kThreads, smem, st>>>(a));
    SG_TRY_CUDA(cudaGetLastError());
    if (bce)
        return sg_loss_finalize(lo, grid, loss, st);
    return SG_OK;
}

sg_status simt_bce(sg_layout *lo, const uint16_t *Z, int32_t B, uint16_t *dZ,
                   double *loss, cudaStream_t st)
{
    const int64_t chunks = (int64_t)B * ceil_div(lo->L, 8);
    const int grid = persistent_grid(lo, ceil_div(chunks, kThreads), 8);
    SG_LAUNCH(lo, SG_KIND_BCE, st,
              k_simt_bce<<<grid, kThreads, 0, st>>>(Z, B, lo->L, lo->G, lo->gptr,
                                                    lo->gent, dZ, lo->loss_part));
    SG_TRY_CUDA(cudaGetLastError());
    return sg_loss_finalize(lo, grid, loss, st);
}

sg_status simt_dW(sg_layout *lo, const uint16_t *dZ, const uint16_t *dZ_lo,
                  int32_t B, uint16_t *dW, cudaStream_t st)
{
    if (g1_ok(lo))
        return g1_dW(lo, dZ, dZ_lo, B, dW, st);
    DWArgs a;
    a.hT = lo->hT;
    a.dZ = dZ;
    a.dZ_lo = dZ_lo;
    a.idx_s = lo->idx_s;
    a.dW = dW;
    a.K = lo->K;
    a.L = lo->L;
    a.B = B;
    a.ldB = lo->ldB;
    a.G = lo->G;
    a.F = lo->F;
    const size_t smem = align16(a.F * (a.ldB + 2) * 2) + (size_t)B * 32 * 4 + a.F * 4;
    const int grid = persistent_grid(lo, lo->K, 2);
    void (*kern)(DWArgs) = nullptr;
    switch (pick_jt(lo->G)) {
    case 1: kern = k_simt_dW<1>; break;
    case 2: kern = k_simt_dW<2>; break;
    case 4: kern = k_simt_dW<4>; break;
    default: kern = k_simt_dW<8>; break;
    }
    SG_SET_SMEM(kern, smem);
    SG_LAUNCH(lo, SG_KIND_DW, st, kern<<<grid, kThreads, smem, st>>>(a));
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}

sg_status simt_dh(sg_layout *lo, const uint16_t *dZ, const uint16_t *dZ_lo,
                  int32_t B, const uint16_t *W, float *dh, cudaStream_t st)
{
    if (g1_ok(lo))
        return g1_dh(lo, dZ, dZ_lo, B, W, dh, st);
    DhArgs a;
    a.dZ = dZ;
    a.dZ_lo = dZ_lo;
    a.W = W;
    a.idx_s = lo->idx_s;
    a.dh = dh;
    a.K = lo->K;
    a.L = lo->L;
    a.B = B;
    a.G = lo->G;
    a.F = lo->F;
    a.H = lo->H;
    a.nbt = (int)ceil_div(B, kBT);
    a.nchunk = ceil_div(lo->L, 32);
    // windows of at most 1024 dh columns (the CTA's shared-memory partial);
    // every window scans all slots and keeps the products that land in it
    a.ncw = (int)ceil_div(a.H, 1024);
    a.hw = (int)ceil_div(a.H, a.ncw);
    int64_t nct = ((int64_t)lo->num_sms * 2 + (int64_t)a.nbt * a.ncw - 1) / ((int64_t)a.nbt * a.ncw);
    if (nct > a.nchunk)
        nct = a.nchunk;
    if (nct < 1)
        nct = 1;
    a.nct = (int)nct;
    const size_t smem = (size_t)kBT * (a.hw + 1) * 4 + 32 * a.F * 4 + kBT * 33 * 4 +
                        32 * a.F * 2;
    SG_TRY_CUDA(cudaMemsetAsync(dh, 0, sizeof(float) * B * a.H, st));
    SG_SET_SMEM(k_simt_dh, smem);
    SG_LAUNCH(lo, SG_KIND_DH, st,
              k_simt_dh<<<(unsigned)((int64_t)a.nbt * a.ncw * a.nct), kThreads, smem, st>>>(a));
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}

// ---------------------------------------------------------------- optimiser
// Momentum SGD of the output layer from a stored bf16 dW (the unfused step):
// W_out holds dW on entry and the updated weights on return,
//     m <- mu m + dW,   W_out <- bf16(W - lr m).
__global__ void __launch_bounds__(256) k_sgd_update(const uint16_t *__restrict__ W, uint16_t *W_out,
                                                    float *mom, float lr, float mu, int64_t n)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float m = fmaf(mu, mom[i], bf2f(W_out[i]));
        mom[i] = m;
        W_out[i] = f2bf(bf2f(W[i]) - lr * m);
    }
}

sg_status sgd_update(sg_layout *lo, const uint16_t *W, uint16_t *W_out, const sg_sgd &sgd, cudaStream_t st)
{
    const int64_t n = lo->L * (int64_t)lo->F;
    int64_t grid = ceil_div(n, 256);
    if (grid > (int64_t)lo->num_sms * 8)
        grid = (int64_t)lo->num_sms * 8;
    SG_LAUNCH(lo, SG_KIND_DW, st, k_sgd_update<<<(unsigned)grid, 256, 0, st>>>(W, W_out, sgd.mom, sgd.lr, sgd.mu, n));
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}
