// Per-label fixed fan-in (G = 1) on CUDA cores: the comparator the group-shared
// layer is measured against (HASTE, "Key findings": the per-label form has no
// shared feature tile, so every label is a thin dot product of F gathered
// features).  Each kernel keeps what it reuses in shared memory and streams the
// labels past it:
//   forward: a 64-sample tile of h^T (every feature, two samples per 32-bit
//            word) stays in shared memory; a warp takes one label at a time,
//            lane l computing the logits of samples 2l and 2l + 1 from the
//            label's F (index, weight) pairs; the BCE follows in registers and
//            dZ leaves through a shared-memory staging tile in 128-byte rows.
//   dW:      per 64-label chunk and 64-sample tile, the h^T tile and the dZ
//            tile in shared memory; a warp owns 8 labels, lane l the features
//            f = l + 32 q, accumulating over every sample tile in registers.
//   dh:      a CTA holds a 32-sample dh partial; warp w owns a window of
//            dh columns and lane l sample l, so every thread adds into its own
//            entries (no atomics per product); a CTA streams a contiguous
//            range of labels and adds its partial to dh once.
#include "sg_internal.cuh"

namespace {

constexpr int kG1T = 256;  // threads (8 warps)
constexpr int kSB = 64;    // samples per tile
constexpr int kLC = 64;    // labels per staged round / dW chunk

__device__ __forceinline__ float lo_bf(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ double g1_block_sum(double v)
{
    __shared__ double red[kG1T / 32];
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_down_sync(0xffffffffu, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = v;
    __syncthreads();
    double s = 0.0;
    if (threadIdx.x == 0)
        for (int w = 0; w < kG1T / 32; ++w)
            s += red[w];
    return s;
}

struct G1Fwd {
    const uint16_t *hT, *W, *idx_s;
    uint16_t *Z, *dZ, *dZ_lo;
    const int32_t *gptr, *gent;
    double *loss_part;
    int64_t L, lchunk;
    int32_t B, ldB, F, H, ntile;
};

// CTA: sample tile blockIdx % ntile, labels [chunk * lchunk, +lchunk)
template <bool BCE>
__global__ void __launch_bounds__(kG1T) k_g1_fwd(G1Fwd a)
{
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t *hs = reinterpret_cast<uint32_t *>(smem);  // [H][32]: samples (2w, 2w + 1) of the tile
    float *zt = reinterpret_cast<float *>(smem + (size_t)a.H * 128);  // [kSB][kLC + 1] logits
    float *dt = zt + kSB * (kLC + 1);                                 // [kSB][kLC + 1] dZ
    uint16_t *is = reinterpret_cast<uint16_t *>(dt + kSB * (kLC + 1));  // [kLC][F] the round's I_l
    uint16_t *wsm = is + kLC * a.F;                                     // [kLC][F] the round's w_l
    __shared__ int32_t gp[kLC + 1];  // the round's positive-list bounds
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int tile = blockIdx.x % a.ntile;
    const int64_t chunk = blockIdx.x / a.ntile;
    const int b0 = tile * kSB;
    for (int e = threadIdx.x; e < a.H * 32; e += kG1T) {
        const int j = e >> 5, w = e & 31;
        hs[e] = *reinterpret_cast<const uint32_t *>(a.hT + (int64_t)j * a.ldB + b0 + 2 * w);
    }
    __syncthreads();
    const int F = a.F;
    const int64_t l_begin = chunk * a.lchunk;
    const int64_t l_end = min(a.L, l_begin + a.lchunk);
    const int bA = b0 + 2 * lane, bB = bA + 1;
    double lacc = 0.0;
    for (int64_t r0 = l_begin; r0 < l_end; r0 += kLC) {
        const int nl = (int)min((int64_t)kLC, l_end - r0);
        float lf = 0.f;
        // the round's index rows and weights, all loads in flight at once
        for (int e = threadIdx.x; e < nl * F / 8; e += kG1T) {
            reinterpret_cast<uint4 *>(is)[e] = __ldg(reinterpret_cast<const uint4 *>(a.idx_s + r0 * F) + e);
            reinterpret_cast<uint4 *>(wsm)[e] = __ldg(reinterpret_cast<const uint4 *>(a.W + r0 * F) + e);
        }
        if (BCE)
            for (int e = threadIdx.x; e <= nl; e += kG1T)
                gp[e] = a.gptr[r0 + e];
        __syncthreads();
        for (int li = warp; li < nl; li += kG1T / 32) {
            const uint4 *I = reinterpret_cast<const uint4 *>(is + li * F);
            const uint4 *Wl = reinterpret_cast<const uint4 *>(wsm + li * F);
            float z0 = 0.f, z1 = 0.f;
#pragma unroll 2
            for (int f8 = 0; f8 < F / 8; ++f8) {
                const uint4 iv = I[f8], wv = Wl[f8];
                const uint32_t ii[4] = {iv.x, iv.y, iv.z, iv.w}, ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t h0 = hs[(ii[q] & 0xffffu) * 32 + lane];
                    const uint32_t h1 = hs[(ii[q] >> 16) * 32 + lane];
                    const float w0 = lo_bf(ww[q]), w1 = hi_bf(ww[q]);
                    z0 = fmaf(lo_bf(h0), w0, z0);
                    z1 = fmaf(hi_bf(h0), w0, z1);
                    z0 = fmaf(lo_bf(h1), w1, z0);
                    z1 = fmaf(hi_bf(h1), w1, z1);
                }
            }
            zt[(2 * lane) * (kLC + 1) + li] = z0;
            zt[(2 * lane + 1) * (kLC + 1) + li] = z1;
            if (BCE) {
                int y0 = 0, y1 = 0;
                const int e1 = gp[li + 1];
                for (int e = gp[li]; e < e1; ++e) {
                    const int b = a.gent[e] >> 16;
                    y0 |= b == bA;
                    y1 |= b == bB;
                }
                float l0, l1;
                const float d0 = bce_grad_loss(z0, y0, &l0), d1 = bce_grad_loss(z1, y1, &l1);
                lf += (bA < a.B ? l0 : 0.f) + (bB < a.B ? l1 : 0.f);
                dt[(2 * lane) * (kLC + 1) + li] = d0;
                dt[(2 * lane + 1) * (kLC + 1) + li] = d1;
            }
        }
        lacc += (double)lf;
        __syncthreads();
        // rows of nl labels per sample, 2 bytes each: consecutive threads,
        // consecutive labels
        for (int e = threadIdx.x; e < kSB * kLC; e += kG1T) {
            const int rb = e / kLC, c = e - rb * kLC;
            const int b = b0 + rb;
            if (c >= nl || b >= a.B)
                continue;
            const int64_t at = (int64_t)b * a.L + r0 + c;
            if (a.Z)
                a.Z[at] = f2bf(zt[rb * (kLC + 1) + c]);
            if (BCE) {
                const float d = dt[rb * (kLC + 1) + c];
                const uint16_t hi = f2bf(d);
                a.dZ[at] = hi;
                if (a.dZ_lo)
                    a.dZ_lo[at] = f2bf(d - bf2f(hi));
            }
        }
        __syncthreads();
    }
    if (BCE) {
        const double s = g1_block_sum(lacc);
        if (threadIdx.x == 0)
            a.loss_part[blockIdx.x] = s;
    }
}

struct G1DW {
    const uint16_t *hT, *dZ, *dZ_lo, *idx_s;
    uint16_t *dW;
    int64_t L;
    int32_t B, ldB, F, H;
};

// CTA loops over 64-label chunks; FQ = F / 32 features per lane
template <int FQ>
__global__ void __launch_bounds__(kG1T) k_g1_dW(G1DW a)
{
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int HLD = 33;  // words per h^T row (odd: rows of different j spread over banks)
    uint32_t *hs = reinterpret_cast<uint32_t *>(smem);                 // [H][33]
    float *dzs = reinterpret_cast<float *>(smem + (size_t)a.H * HLD * 4);  // [kSB][kLC + 1]
    uint16_t *is = reinterpret_cast<uint16_t *>(dzs + kSB * (kLC + 1));   // [kLC][F]
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int F = a.F;
    const int ntile = (a.B + kSB - 1) / kSB;
    const int64_t nchunk = (a.L + kLC - 1) / kLC;
    for (int64_t ch = blockIdx.x; ch < nchunk; ch += gridDim.x) {
        const int64_t r0 = ch * kLC;
        const int nl = (int)min((int64_t)kLC, a.L - r0);
        __syncthreads();
        for (int e = threadIdx.x; e < nl * F; e += kG1T)
            is[e] = a.idx_s[r0 * F + e];
        float acc[8][FQ];
#pragma unroll
        for (int t = 0; t < 8; ++t)
#pragma unroll
            for (int q = 0; q < FQ; ++q)
                acc[t][q] = 0.f;
        for (int tile = 0; tile < ntile; ++tile) {
            const int b0 = tile * kSB;
            __syncthreads();
            for (int e = threadIdx.x; e < a.H * 32; e += kG1T) {
                const int j = e >> 5, w = e & 31;
                hs[j * HLD + w] = *reinterpret_cast<const uint32_t *>(a.hT + (int64_t)j * a.ldB + b0 + 2 * w);
            }
            for (int e = threadIdx.x; e < kSB * kLC; e += kG1T) {
                const int rb = e / kLC, c = e - rb * kLC;
                const int b = b0 + rb;
                float v = 0.f;
                if (c < nl && b < a.B) {
                    const int64_t at = (int64_t)b * a.L + r0 + c;
                    v = bf2f(a.dZ[at]) + (a.dZ_lo ? bf2f(a.dZ_lo[at]) : 0.f);
                }
                dzs[rb * (kLC + 1) + c] = v;
            }
            __syncthreads();
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const int li = warp + 8 * t;
                if (li >= nl)
                    break;
                int j[FQ];
#pragma unroll
                for (int q = 0; q < FQ; ++q)
                    j[q] = is[li * F + q * 32 + lane] * HLD;
#pragma unroll 4
                for (int w = 0; w < 32; ++w) {
                    const float d0 = dzs[(2 * w) * (kLC + 1) + li], d1 = dzs[(2 * w + 1) * (kLC + 1) + li];
#pragma unroll
                    for (int q = 0; q < FQ; ++q) {
                        const uint32_t h = hs[j[q] + w];
                        acc[t][q] = fmaf(lo_bf(h), d0, acc[t][q]);
                        acc[t][q] = fmaf(hi_bf(h), d1, acc[t][q]);
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int li = warp + 8 * t;
            if (li < nl)
#pragma unroll
                for (int q = 0; q < FQ; ++q)
                    a.dW[(r0 + li) * F + q * 32 + lane] = f2bf(acc[t][q]);
        }
    }
}

struct G1Dh {
    const uint16_t *dZ, *dZ_lo, *W, *idx_s;
    float *dh;
    int64_t L, lchunk;
    int32_t B, F, H, ntile, hw;
};

// CTA: 32 samples (tile blockIdx % ntile) x labels [chunk * lchunk, +lchunk).
// Warp w owns the dh columns [w hw, w hw + hw) and lane l sample l: each
// thread adds into its own part of its own row, so no two threads ever meet
// on an entry and there is no atomic per product.  The round's index rows are
// sorted, so a warp finds its window's entries by binary search.
__global__ void __launch_bounds__(kG1T) k_g1_dh(G1Dh a)
{
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int SB = 32;
    const int ldp = a.H + 1;  // odd row stride: a warp's 32 rows on distinct banks
    float *part = reinterpret_cast<float *>(smem);                     // [SB][H + 1]
    float *dzs = part + (size_t)SB * ldp;                              // [SB][kLC + 1]
    uint16_t *is = reinterpret_cast<uint16_t *>(dzs + SB * (kLC + 1));  // [kLC][F]
    uint16_t *wsm = is + kLC * a.F;                                     // [kLC][F]
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int tile = blockIdx.x % a.ntile;
    const int64_t chunk = blockIdx.x / a.ntile;
    const int b0 = tile * SB;
    const int F = a.F;
    const int j0 = warp * a.hw, j1 = min(a.H, j0 + a.hw);
    for (int e = threadIdx.x; e < SB * ldp; e += kG1T)
        part[e] = 0.f;
    const int64_t l_begin = chunk * a.lchunk;
    const int64_t l_end = min(a.L, l_begin + a.lchunk);
    float *prow = part + (size_t)lane * ldp;
    for (int64_t r0 = l_begin; r0 < l_end; r0 += kLC) {
        const int nl = (int)min((int64_t)kLC, l_end - r0);
        __syncthreads();
        for (int e = threadIdx.x; e < SB * kLC; e += kG1T) {
            const int r = e / kLC, c = e - r * kLC;
            const int b = b0 + r;
            float v = 0.f;
            if (c < nl && b < a.B) {
                const int64_t at = (int64_t)b * a.L + r0 + c;
                v = bf2f(a.dZ[at]) + (a.dZ_lo ? bf2f(a.dZ_lo[at]) : 0.f);
            }
            dzs[r * (kLC + 1) + c] = v;
        }
        for (int e = threadIdx.x; e < nl * F / 8; e += kG1T) {
            reinterpret_cast<uint4 *>(is)[e] = __ldg(reinterpret_cast<const uint4 *>(a.idx_s + r0 * F) + e);
            reinterpret_cast<uint4 *>(wsm)[e] = __ldg(reinterpret_cast<const uint4 *>(a.W + r0 * F) + e);
        }
        __syncthreads();
        if (j0 >= j1)
            continue;
        for (int li = 0; li < nl; ++li) {
            const uint16_t *I = is + li * F;
            // entries [fa, fb) of the sorted row fall in the window: count
            // the entries below each bound, 32 at a time (no load chain)
            int fa = 0, fb = 0;
            for (int f0 = 0; f0 < F; f0 += 32) {
                const int v = I[f0 + lane];
                fa += __popc(__ballot_sync(0xffffffffu, v < j0));
                fb += __popc(__ballot_sync(0xffffffffu, v < j1));
            }
            const float dz = dzs[lane * (kLC + 1) + li];
            const uint16_t *Wl = wsm + li * F;
            // a label's indices are distinct: eight updates at a time with
            // their loads in flight together
            for (int f0 = fa; f0 < fb; f0 += 8) {
                int j[8];
                float w[8], p[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int f = f0 + u < fb ? f0 + u : fa;
                    j[u] = I[f];
                    w[u] = f0 + u < fb ? bf2f(Wl[f]) : 0.f;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    p[u] = prow[j[u]];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (f0 + u < fb)
                        prow[j[u]] = fmaf(dz, w[u], p[u]);
            }
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < SB * a.H; e += kG1T) {
        const int r = e / a.H, i = e - r * a.H;
        const int b = b0 + r;
        if (b < a.B)
            atomicAdd(a.dh + (int64_t)b * a.H + i, part[(size_t)r * ldp + i]);
    }
}

int g1_grid(const sg_layout *lo)
{
    int g = lo->num_sms;
    if (g > lo->loss_part_n)
        g = lo->loss_part_n;
    return g < 1 ? 1 : g;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15) == 0; }

size_t g1_fwd_smem(const sg_layout *lo)
{
    return (size_t)lo->H * 128 + 2 * (size_t)kSB * (kLC + 1) * 4 + 2 * (size_t)kLC * lo->F * 2;
}
size_t g1_dW_smem(const sg_layout *lo)
{
    return (size_t)lo->H * 33 * 4 + (size_t)kSB * (kLC + 1) * 4 + (size_t)kLC * lo->F * 2;
}
size_t g1_dh_smem(const sg_layout *lo)
{
    return (size_t)32 * (lo->H + 1) * 4 + (size_t)32 * (kLC + 1) * 4 + 2 * (size_t)kLC * lo->F * 2;
}

}  // namespace

// The per-label kernels take F % 32 == 0 (F <= 256) and an h^T tile of every
// feature in shared memory; other shapes keep the general CUDA-core kernels.
bool g1_ok(const sg_layout *lo)
{
    constexpr size_t kMax = 220 * 1024;
    return lo->G == 1 && lo->F % 32 == 0 && lo->F <= 256 && lo->ldB % 64 == 0 && g1_fwd_smem(lo) <= kMax &&
           g1_dW_smem(lo) <= kMax && g1_dh_smem(lo) <= kMax;
}

sg_status g1_fwd(sg_layout *lo, int32_t B, const uint16_t *W, uint16_t *Z, uint16_t *dZ, uint16_t *dZ_lo,
                 double *loss, cudaStream_t st)
{
    if (!aligned16(W)) {
        sg_set_error("W: device pointer must be 16-byte aligned");
        return SG_ERR_INVALID;
    }
    G1Fwd a;
    a.hT = lo->hT;
    a.W = W;
    a.idx_s = lo->idx_s;
    a.Z = Z;
    a.dZ = dZ;
    a.dZ_lo = dZ_lo;
    a.gptr = lo->gptr;
    a.gent = lo->gent;
    a.loss_part = lo->loss_part;
    a.L = lo->L;
    a.B = B;
    a.ldB = lo->ldB;
    a.F = lo->F;
    a.H = lo->H;
    a.ntile = (B + kSB - 1) / kSB;
    int grid = g1_grid(lo);
    int chunks = grid / a.ntile;
    if (chunks < 1)
        chunks = 1;
    a.lchunk = (lo->L + chunks - 1) / chunks;
    grid = (int)((lo->L + a.lchunk - 1) / a.lchunk) * a.ntile;
    const size_t smem = g1_fwd_smem(lo);
    const bool bce = dZ != nullptr;
    void (*kern)(G1Fwd) = bce ? k_g1_fwd<true> : k_g1_fwd<false>;
    SG_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    SG_LAUNCH(lo, SG_KIND_FWD, st, kern<<<grid, kG1T, smem, st>>>(a));
    SG_TRY_CUDA(cudaGetLastError());
    if (bce)
        return sg_loss_finalize(lo, grid, loss, st);
    return SG_OK;
}

sg_status g1_dW(sg_layout *lo, const uint16_t *dZ, const uint16_t *dZ_lo, int32_t B, uint16_t *dW, cudaStream_t st)
{
    G1DW a;
    a.hT = lo->hT;
    a.dZ = dZ;
    a.dZ_lo = dZ_lo;
    a.idx_s = lo->idx_s;
    a.dW = dW;
    a.L = lo->L;
    a.B = B;
    a.ldB = lo->ldB;
    a.F = lo->F;
    a.H = lo->H;
    const size_t smem = g1_dW_smem(lo);
    void (*kern)(G1DW) = nullptr;
    switch (lo->F / 32) {
    case 1: kern = k_g1_dW<1>; break;
    case 2: kern = k_g1_dW<2>; break;
    case 3: kern = k_g1_dW<3>; break;
    case 4: kern = k_g1_dW<4>; break;
    case 5: kern = k_g1_dW<5>; break;
    case 6: kern = k_g1_dW<6>; break;
    case 7: kern = k_g1_dW<7>; break;
    default: kern = k_g1_dW<8>; break;
    }
    int64_t nchunk = (lo->L + kLC - 1) / kLC;
    int grid = lo->num_sms;
    if (grid > nchunk)
        grid = (int)nchunk;
    SG_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    SG_LAUNCH(lo, SG_KIND_DW, st, kern<<<grid, kG1T, smem, st>>>(a));
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}

sg_status g1_dh(sg_layout *lo, const uint16_t *dZ, const uint16_t *dZ_lo, int32_t B, const uint16_t *W, float *dh,
                cudaStream_t st)
{
    if (!aligned16(W)) {
        sg_set_error("W: device pointer must be 16-byte aligned");
        return SG_ERR_INVALID;
    }
    G1Dh a;
    a.dZ = dZ;
    a.dZ_lo = dZ_lo;
    a.W = W;
    a.idx_s = lo->idx_s;
    a.dh = dh;
    a.L = lo->L;
    a.B = B;
    a.F = lo->F;
    a.H = lo->H;
    a.hw = (lo->H + kG1T / 32 - 1) / (kG1T / 32);  // one window of columns per warp
    a.ntile = (B + 31) / 32;
    int chunks = lo->num_sms / a.ntile;
    if (chunks < 1)
        chunks = 1;
    a.lchunk = (lo->L + chunks - 1) / chunks;
    const int grid = (int)((lo->L + a.lchunk - 1) / a.lchunk) * a.ntile;
    const size_t smem = g1_dh_smem(lo);
    SG_TRY_CUDA(cudaFuncSetAttribute(k_g1_dh, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    SG_TRY_CUDA(cudaMemsetAsync(dh, 0, sizeof(float) * B * lo->H, st));
    SG_LAUNCH(lo, SG_KIND_DH, st, k_g1_dh<<<grid, kG1T, smem, st>>>(a));
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}
