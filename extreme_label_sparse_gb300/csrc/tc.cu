// Tensor-core engine (sm_103a): tcgen05 MMA with TMEM accumulators, operands
// staged in shared memory by TMA (tile loads for W_k and dZ_k, gather4 loads
// for H_k).  HASTE, key design "gather-once + dense MMA kernel":
//   forward   Z_k    = H_k W_k^T          M = samples, N = G, K = F
//   weights   dW_k^T = H_k^T dZ_k         M = F,       N = G, K = samples
//   features  dH_k   = dZ_k W_k, scattered into the columns I_k of dh
//             (Split-K over groups: each CTA keeps a partial of one band of
//             dh columns in TMEM and adds it to dh once at the end).
//
// Shared-memory operand layouts (all 1024-byte aligned):
//   H_k  : gathered rows hT[I_k[f]] -> [b-chunk of 64][f][64 b], 128-byte
//          swizzle.  Read as MN-major A (M = b) by the forward and as K-major A
//          (M = f, K = b) by the weight gradient.
//   W_k  : TMA box {64 f, G rows} per 64-wide f chunk, 128-byte swizzle:
//          K-major B (N = j, K = f) of the forward, MN-major B (N = f, K = j)
//          of the feature gradient.
//   dZ_k : TMA box {min(G,64) j, rows b}, swizzle = row width: MN-major B
//          (N = j, K = b) of the weight gradient, K-major A (M = b, K = j) of
//          the feature gradient.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "sg_internal.cuh"
#include "tc_ptx.cuh"

using namespace tc;

namespace {

constexpr int kMaxStages = 8;
constexpr int kSmemBudget = 220 * 1024;  // dynamic shared memory we plan with
constexpr int kEpiWarps = 8;   // two per TMEM lane quarter
constexpr int kProdWarps = 4;  // cp.async gather + TMA issue
// forward / dW: producers, two MMA-issuing warps, epilogue
constexpr int kFwdThreads = 32 * (kProdWarps + 2 + kEpiWarps);
constexpr int kFirstEpi = kProdWarps + 2;
// dh: one TMA producer, one MMA warp, epilogue
constexpr int kDhThreads = 32 * (2 + kEpiWarps);

// ------------------------------------------------------------------ plans
struct FwdPlan {
    bool ok = false;
    int MT = 0, nk = 0, S = 0, issuers = 0;
    uint32_t a_bytes = 0, w_bytes = 0, stage_bytes = 0, tmem_cols = 0;
};

struct DWPlan {
    bool ok = false;
    int MT = 0, FT = 0, S = 0, nzc = 0, zsw = 0, issuers = 0;
    int planes = 0;   // dZ planes in smem (2 with the lo residual)
    int ncat = 0;     // 1: the planes are concatenated along N in one pass
    int Nacc = 0;     // accumulator columns per (f tile, group)
    uint32_t a_bytes = 0, z_bytes = 0, stage_bytes = 0, tmem_cols = 0;
};

struct DhPlan {
    bool ok = false;
    int MT = 0, nk = 0, S = 0, nzc = 0, zsw = 0, nbands = 0, band_w = 0, win = 0;
    uint32_t z_bytes = 0, w_bytes = 0, i_bytes = 0, stage_bytes = 0, tmem_cols = 0;
};

uint32_t pow2_cols(int n)
{
    uint32_t c = 32;
    while ((int)c < n)
        c <<= 1;
    return c;
}

bool shape_ok(const sg_layout *lo)
{
    return lo->G % 16 == 0 && lo->G <= 256 && lo->F % 64 == 0 && lo->F <= 256 &&
           lo->L % 8 == 0 && lo->ldB % 128 == 0;
}

int stages_for(uint32_t stage_bytes)
{
    int S = (int)(kSmemBudget / stage_bytes);
    return S > 6 ? 6 : S;
}

FwdPlan plan_fwd(const sg_layout *lo, int B)
{
    FwdPlan p;
    if (!shape_ok(lo) || B < 1 || B > 256)
        return p;
    p.MT = (B + 127) / 128;
    if (p.MT * 128 > lo->ldB)
        return p;
    p.nk = lo->F / 64;
    p.a_bytes = (uint32_t)p.MT * 2 * lo->F * 128;
    p.w_bytes = (uint32_t)p.nk * lo->G * 128;
    p.stage_bytes = p.a_bytes + p.w_bytes;
    p.S = stages_for(p.stage_bytes);
    if (p.S < 3)
        return p;
    const int per = p.MT * lo->G;  // accumulator columns of one group
    p.issuers = 4 * per <= 512 ? 2 : 1;
    if (2 * p.issuers * per > 512)
        return p;
    p.tmem_cols = pow2_cols(2 * p.issuers * per);
    p.ok = true;
    return p;
}

int dz_swizzle(int G) { return G * 2 >= 128 ? 128 : G * 2; }

DWPlan plan_dW(const sg_layout *lo, int B, bool split)
{
    DWPlan p;
    if (!shape_ok(lo) || lo->F % 128 != 0 || B < 1 || B > 256)
        return p;
    p.MT = (B + 127) / 128;
    if (p.MT * 128 > lo->ldB)
        return p;
    p.FT = lo->F / 128;
    p.zsw = dz_swizzle(lo->G);
    p.nzc = lo->G * 2 > 128 ? lo->G / 64 : 1;
    p.planes = split ? 2 : 1;
    p.ncat = (split && 2 * lo->G <= 256) ? 1 : 0;
    p.Nacc = p.ncat ? 2 * lo->G : lo->G;
    p.a_bytes = (uint32_t)p.MT * 2 * lo->F * 128;
    p.z_bytes = (uint32_t)p.planes * p.nzc * p.MT * 128 * p.zsw;
    p.stage_bytes = p.a_bytes + p.z_bytes;
    p.S = stages_for(p.stage_bytes);
    if (p.S < 3)
        return p;
    const int per = p.FT * p.Nacc;
    p.issuers = 4 * per <= 512 ? 2 : 1;
    if (2 * p.issuers * per > 512)
        return p;
    p.tmem_cols = pow2_cols(2 * p.issuers * per);
    p.ok = true;
    return p;
}

DhPlan plan_dh(const sg_layout *lo, int B, bool split)
{
    DhPlan p;
    if (!shape_ok(lo) || lo->F > 128 || B < 1 || B > 256)
        return p;
    p.MT = (B + 127) / 128;
    p.nk = lo->F / 64;
    p.zsw = dz_swizzle(lo->G);
    p.nzc = lo->G * 2 > 128 ? lo->G / 64 : 1;
    // TMEM: [0, band_w) partial, then two dH windows of F columns
    p.win = lo->F;
    const int wmax = 512 - 2 * p.win;
    p.nbands = (lo->H + wmax - 1) / wmax;
    p.band_w = (lo->H + p.nbands - 1) / p.nbands;
    p.band_w = (p.band_w + 31) / 32 * 32;
    if (p.band_w + 2 * p.win > 512)
        return p;
    p.z_bytes = (uint32_t)(split ? 2 : 1) * p.nzc * 128 * p.zsw;
    p.w_bytes = (uint32_t)p.nk * lo->G * 128;
    p.i_bytes = (uint32_t)((lo->F * 2 + 1023) / 1024 * 1024);
    p.stage_bytes = p.z_bytes + p.w_bytes + p.i_bytes;
    p.S = stages_for(p.stage_bytes);
    if (p.S < 2)
        return p;
    p.tmem_cols = 512;
    p.ok = true;
    return p;
}

// ------------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

sg_status get_encode()
{
    if (g_encode)
        return SG_OK;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
        sg_set_error("cuTensorMapEncodeTiled is not available from the driver");
        return SG_ERR_CUDA;
    }
    g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    return SG_OK;
}

sg_status make_map_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer,
                      uint32_t box_inner, uint32_t box_outer, int swizzle_bytes,
                      const char *what)
{
    sg_status rc = get_encode();
    if (rc != SG_OK)
        return rc;
    if (((uintptr_t)base & 15) != 0) {
        sg_set_error("%s: device pointer must be 16-byte aligned", what);
        return SG_ERR_INVALID;
    }
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUtensorMapSwizzle sw = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                            : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                            : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                  : CU_TENSOR_MAP_SWIZZLE_NONE;
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        sg_set_error("%s: cuTensorMapEncodeTiled failed (%d)", what, (int)r);
        return SG_ERR_CUDA;
    }
    return SG_OK;
}

// ------------------------------------------------------------------ common
constexpr int kMaxAcc = 4;  // accumulator slots: two per MMA-issuing warp

struct Ctl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tfull[kMaxAcc];
    uint64_t tempty[kMaxAcc];
    uint64_t drain[2];  // one per MMA-issuing warp
    uint32_t tmem;
    int abort_flag;
    double red[kEpiWarps];
};

__device__ __forceinline__ uint32_t bar_addr(const uint64_t &b) { return smem_u32(&b); }

// two floats -> packed bf16x2 (a in the low half), round to nearest even
__device__ __forceinline__ uint32_t pack2(float a, float b)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float lo_half(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_half(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// store N (multiple of 8) floats as bf16 to 16-byte aligned global memory;
// with `lo`, also store the rounding residual v - bf16(v) as a second plane
template <int N>
__device__ __forceinline__ void store_bf16_row(uint16_t *dst, uint16_t *lo, const float (&v)[N])
{
#pragma unroll
    for (int i = 0; i < N; i += 8) {
        uint4 q;
        q.x = pack2(v[i + 0], v[i + 1]);
        q.y = pack2(v[i + 2], v[i + 3]);
        q.z = pack2(v[i + 4], v[i + 5]);
        q.w = pack2(v[i + 6], v[i + 7]);
        *reinterpret_cast<uint4 *>(dst + i) = q;
        if (lo) {
            uint4 r;
            r.x = pack2(v[i + 0] - lo_half(q.x), v[i + 1] - hi_half(q.x));
            r.y = pack2(v[i + 2] - lo_half(q.y), v[i + 3] - hi_half(q.y));
            r.z = pack2(v[i + 4] - lo_half(q.z), v[i + 5] - hi_half(q.z));
            r.w = pack2(v[i + 6] - lo_half(q.w), v[i + 7] - hi_half(q.w));
            *reinterpret_cast<uint4 *>(lo + i) = r;
        }
    }
}

template <int CH>
__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, float (&v)[CH])
{
    if constexpr (CH == 32) {
        uint32_t r[32];
        tmem_ld32(taddr, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i)
            v[i] = __uint_as_float(r[i]);
    } else {
        uint32_t r[16];
        tmem_ld16(taddr, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i)
            v[i] = __uint_as_float(r[i]);
    }
}

// positives of sample b among columns c0 .. c0+n-1 of a group whose entries
// are gent[e0 .. e1)
__device__ __forceinline__ uint32_t group_pos_mask(const int32_t *__restrict__ gent, int e0,
                                                   int e1, int b, int c0, int n)
{
    uint32_t y = 0;
    for (int e = e0; e < e1; ++e) {
        const int v = __ldg(gent + e);
        const int jj = (v & 0xffff) - c0;
        if ((v >> 16) == b && jj >= 0 && jj < n)
            y |= 1u << jj;
    }
    return y;
}

// BCE on a chunk of logits in place: v[i] <- sigmoid(v[i]) - y_i; returns the
// chunk's loss sum(max(z,0) - y z + log(1 + e^-|z|)).  The log of the product
// of the (1 + e^-|z|) factors (each in (1, 2], so at most 2^32 for 32 of
// them) replaces one log per element.
template <int CH>
__device__ __forceinline__ float bce_chunk(float (&v)[CH], uint32_t y)
{
    float prod = 1.f, lin = 0.f;
#pragma unroll
    for (int i = 0; i < CH; ++i) {
        const float z = v[i];
        const float e = __expf(-fabsf(z));
        const float one_e = 1.f + e;
        const float r = __fdividef(1.f, one_e);
        const float sig = z >= 0.f ? r : e * r;
        const bool yi = (y >> i) & 1u;
        lin += fmaxf(z, 0.f) - (yi ? z : 0.f);
        prod *= one_e;
        v[i] = sig - (yi ? 1.f : 0.f);
    }
    return lin + __logf(prod);
}

// After an abort, wait (bounded) until the loads of the last stages issued
// have landed, so no TMA write is still in flight when the CTA exits.  In a
// normal run every one of these phases has already completed.
__device__ __forceinline__ void drain_loads(Ctl &c, int issued, int S)
{
    if (!c.abort_flag)
        return;
    for (int i = issued - S < 0 ? 0 : issued - S; i < issued; ++i)
        mbar_wait_drain(bar_addr(c.full[i % S]), (uint32_t)(i / S) & 1u);
}

// sum of one double per thread over the epilogue threads (warps first_epi ..)
__device__ __forceinline__ void epi_sum_to(double v, Ctl &c, double *dst, int first_epi)
{
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_down_sync(0xffffffffu, v, o);
    const int ew = threadIdx.x / 32 - first_epi;
    if ((threadIdx.x & 31) == 0)
        c.red[ew] = v;
    named_bar(1, kEpiWarps * 32);
    if (ew == 0 && (threadIdx.x & 31) == 0) {
        double s = 0.0;
        for (int i = 0; i < kEpiWarps; ++i)
            s += c.red[i];
        *dst = s;
    }
}

// ------------------------------------------------------------------ gather
// H_k = rows I_k[f] of hT, copied with 16-byte cp.async by the producer
// threads into the 128-byte-swizzled layout [b-chunk of 64][f][64 b]: unit u
// (16 B) of row f lands at chunk(u/8) * F*128 + f*128 + ((u%8) ^ (f%8))*16.
// Thread t copies the units u of rows f = t mod F (every unit of its row when
// F = 128); its row indices are loaded one group ahead.
struct GatherRows {
    int f0, f1;   // rows of this thread (f1 = -1 if one row)
    int i0, i1;   // their indices in hT
};

__device__ __forceinline__ GatherRows gather_rows_of(const uint16_t *idx_s, int64_t k, int F, int t)
{
    GatherRows g;
    g.f0 = t % F;
    g.f1 = F > kProdWarps * 32 ? t + kProdWarps * 32 : -1;
    const uint16_t *I = idx_s + k * F;
    g.i0 = __ldg(I + g.f0);
    g.i1 = g.f1 >= 0 ? __ldg(I + g.f1) : 0;
    return g;
}

__device__ __forceinline__ void issue_gather(const uint16_t *hT, int ldB, uint32_t A, int F,
                                             int units, const GatherRows &g, int t)
{
    // units = MT * 16 16-byte units per row; rows f0 (and f1) of this thread
    const int nthr = kProdWarps * 32;
    const int rows_per_pass = nthr < F ? nthr : F;     // threads sharing the rows
    const int u_step = nthr / rows_per_pass;           // threads per row
    const int u_first = t / rows_per_pass;
    for (int r = 0; r < 2; ++r) {
        const int f = r == 0 ? g.f0 : g.f1;
        if (f < 0)
            break;
        const uint16_t *src = hT + (size_t)(r == 0 ? g.i0 : g.i1) * ldB;
        const uint32_t rowbase = A + (uint32_t)f * 128;
        for (int u = u_first; u < units; u += u_step) {
            const int cch = u >> 3, w = u & 7;
            cp_async16(rowbase + (uint32_t)cch * F * 128 + (uint32_t)((w ^ (f & 7)) << 4), src + u * 8);
        }
    }
}

// Producer loop shared by the forward and the weight gradient: per group, one
// thread arms the stage barrier with the TMA bytes (`tma_bytes`, issued by
// `issue_tma`), every producer thread copies its share of H_k, and a copy
// group is signalled complete two groups later (wait_group, proxy fence,
// arrive) so each thread keeps three groups of copies in flight.
template <typename IssueTma>
__device__ __forceinline__ void producer_loop(Ctl &c, uint32_t stage0, uint32_t stage_bytes, int S,
                                              int64_t K, const uint16_t *idx_s, const uint16_t *hT,
                                              int ldB, int F, int MT, uint32_t tma_bytes,
                                              volatile int *abort_flag, int32_t *status,
                                              IssueTma issue_tma)
{
    constexpr int kLag = 2;
    const int t = threadIdx.x;  // producer threads are 0 .. kProdWarps*32-1
    const int units = MT * 16;
    int it = 0;
    GatherRows cur = {0, -1, 0, 0};
    if (blockIdx.x < K)
        cur = gather_rows_of(idx_s, blockIdx.x, F, t);
    for (int64_t k = blockIdx.x; k < K; k += gridDim.x, ++it) {
        const int s = it % S;
        const uint32_t ph = (uint32_t)(it / S) & 1u;
        GatherRows nxt = cur;
        if (k + gridDim.x < K)
            nxt = gather_rows_of(idx_s, k + gridDim.x, F, t);
        if (!mbar_wait(bar_addr(c.empty[s]), ph ^ 1u, abort_flag, status))
            break;
        const uint32_t A = stage0 + (uint32_t)s * stage_bytes;
        if (t == 0) {
            mbar_arrive_expect_tx(bar_addr(c.full[s]), tma_bytes);
            issue_tma(k, A, bar_addr(c.full[s]));
        }
        issue_gather(hT, ldB, A, F, units, cur, t);
        cp_async_commit();
        if (it >= kLag) {
            cp_async_wait<kLag>();
            fence_proxy_async();
            mbar_arrive(bar_addr(c.full[(it - kLag) % S]));
        }
        cur = nxt;
    }
    cp_async_wait<0>();
    fence_proxy_async();
    for (int j = it - kLag < 0 ? 0 : it - kLag; j < it; ++j)
        mbar_arrive(bar_addr(c.full[j % S]));
    if (*abort_flag) {
        // wait (bounded) for the TMA bytes of the stages still in flight
        for (int j = it - S < 0 ? 0 : it - S; j < it; ++j)
            mbar_wait_drain(bar_addr(c.full[j % S]), (uint32_t)(j / S) & 1u);
    }
}

__device__ __forceinline__ void setup_ctl(Ctl &c, int S, int nacc, uint32_t full_count,
                                          uint32_t empty_count)
{
    // the plans keep S <= kMaxStages and nacc <= kMaxAcc; never index past them
    if (S > kMaxStages)
        S = kMaxStages;
    if (nacc > kMaxAcc)
        nacc = kMaxAcc;
    c.abort_flag = 0;
    for (int s = 0; s < S; ++s) {
        mbar_init(bar_addr(c.full[s]), full_count);
        mbar_init(bar_addr(c.empty[s]), empty_count);
    }
    for (int i = 0; i < nacc; ++i) {
        mbar_init(bar_addr(c.tfull[i]), 1);
        mbar_init(bar_addr(c.tempty[i]), kEpiWarps * 32);
    }
    mbar_init(bar_addr(c.drain[0]), 1);
    mbar_init(bar_addr(c.drain[1]), 1);
    fence_mbar_init();
}

// Accumulator slot of the it-th group: the issuer is it mod `issuers`, each
// issuer owns two slots used alternately.
__device__ __forceinline__ int acc_slot(int it, int issuers)
{
    return issuers == 2 ? 2 * (it & 1) + ((it >> 1) & 1) : (it & 1);
}
__device__ __forceinline__ uint32_t acc_phase(int it, int issuers)
{
    return issuers == 2 ? (uint32_t)(it >> 2) & 1u : (uint32_t)(it >> 1) & 1u;
}

// ================================================================== forward
struct FwdArgs {
    const uint16_t *idx_s, *hT;
    uint16_t *Z, *dZ, *dZ_lo;
    const int32_t *gptr, *gent;
    double *loss_part;
    int32_t *status;
    int64_t K, L;
    int32_t B, G, F, MT, nk, S, issuers, ldB;
    uint32_t a_bytes, w_bytes, stage_bytes, tmem_cols;
};

template <bool BCE, int CH>
__global__ void __launch_bounds__(kFwdThreads, 1)
    k_tc_fwd(const __grid_constant__ CUtensorMap tm_w, const FwdArgs a)
{
    __shared__ Ctl c;
    extern __shared__ uint8_t dsm[];
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const uint32_t stage0 = (smem_u32(dsm) + 1023u) & ~1023u;
    const int G = a.G, F = a.F, S = a.S;
    const int nacc = 2 * a.issuers;
    const int per = a.MT * G;  // accumulator columns per group

    if (threadIdx.x == 0)
        setup_ctl(c, S, nacc, kProdWarps * 32 + 1, 1);
    if (warp == kProdWarps) {
        tmem_alloc(smem_u32(&c.tmem), a.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = c.tmem;
    volatile int *abort_flag = &c.abort_flag;

    if (warp < kProdWarps) {
        // ---------------------------------------------------------- producers
        producer_loop(c, stage0, a.stage_bytes, S, a.K, a.idx_s, a.hT, a.ldB, F, a.MT, a.w_bytes,
                      abort_flag, a.status, [&](int64_t k, uint32_t A, uint32_t fb) {
                          const uint32_t Wt = A + a.a_bytes;
                          for (int kc = 0; kc < a.nk; ++kc)
                              tma_load_2d(Wt + (uint32_t)kc * G * 128, &tm_w, kc * 64, (int)(k * G), fb);
                      });
    } else if (warp < kFirstEpi) {
        // ---------------------------------------------------------- MMA issue
        const int me = warp - kProdWarps;
        const uint32_t idesc = idesc_bf16(128, G, 1, 0);
        int it = 0;
        for (int64_t k = blockIdx.x; k < a.K; k += gridDim.x, ++it) {
            if (it % a.issuers != me)
                continue;
            const int s = it % S;
            const uint32_t ph = (uint32_t)(it / S) & 1u;
            const int acc = acc_slot(it, a.issuers);
            if (!mbar_wait(bar_addr(c.tempty[acc]), acc_phase(it, a.issuers) ^ 1u, abort_flag, a.status))
                break;
            tc_fence_after();
            if (!mbar_wait(bar_addr(c.full[s]), ph, abort_flag, a.status))
                break;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t A = stage0 + (uint32_t)s * a.stage_bytes;
                const uint32_t Wt = A + a.a_bytes;
                for (int t = 0; t < a.MT; ++t) {
                    const uint32_t d = tbase + (uint32_t)(acc * per + t * G);
                    for (int st = 0; st < F / 16; ++st) {
                        // A: H_k, MN-major; 8 f-rows per 1024-byte atom, b chunks F*128 apart
                        const uint64_t ad = sdesc(A + (uint32_t)t * 2 * F * 128 + (uint32_t)st * 2048,
                                                  (uint32_t)F * 128, 1024, kLayoutSW128);
                        // B: W_k, K-major; 32 bytes per 16 f inside a 128-byte row
                        const uint64_t bd = sdesc(Wt + (uint32_t)(st / 4) * G * 128 + (uint32_t)(st % 4) * 32,
                                                  16, 1024, kLayoutSW128);
                        mma_bf16(d, ad, bd, idesc, st > 0 ? 1u : 0u);
                    }
                }
                mma_commit(bar_addr(c.empty[s]));
                mma_commit(bar_addr(c.tfull[acc]));
            }
            __syncwarp();
        }
        // every MMA this warp issued has completed once its drain barrier flips
        if (lane == 0)
            mma_commit(bar_addr(c.drain[me]));
        __syncwarp();
        mbar_wait_drain(bar_addr(c.drain[me]), 0);
    } else {
        // ---------------------------------------------------------- epilogue
        // two warps per TMEM lane quarter; they split the (tile, chunk) units
        const int q = warp & 3;
        const int sub = (warp - kFirstEpi) / 4;
        const int units = a.MT * (G / CH);
        double lacc = 0.0;
        int it = 0;
        for (int64_t k = blockIdx.x; k < a.K; k += gridDim.x, ++it) {
            const int acc = acc_slot(it, a.issuers);
            int e0 = 0, e1 = 0;
            if (BCE) {
                e0 = __ldg(a.gptr + k);
                e1 = __ldg(a.gptr + k + 1);
            }
            if (!mbar_wait(bar_addr(c.tfull[acc]), acc_phase(it, a.issuers), abort_flag, a.status))
                break;
            tc_fence_after();
            for (int u = sub; u < units; u += 2) {
                const int t = u / (G / CH), c0 = (u % (G / CH)) * CH;
                const int b = t * 128 + q * 32 + lane;
                float v[CH];
                tmem_ld_chunk<CH>(tbase + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * per + t * G + c0), v);
                if (b >= a.B)
                    continue;
                const int64_t off = (int64_t)b * a.L + k * G + c0;
                if (a.Z)
                    store_bf16_row<CH>(a.Z + off, nullptr, v);
                if (BCE) {
                    const uint32_t y = e1 > e0 ? group_pos_mask(a.gent, e0, e1, b, c0, CH) : 0u;
                    lacc += bce_chunk<CH>(v, y);
                    store_bf16_row<CH>(a.dZ + off, a.dZ_lo ? a.dZ_lo + off : nullptr, v);
                }
            }
            tc_fence_before();
            mbar_arrive(bar_addr(c.tempty[acc]));
        }
        if (BCE)
            epi_sum_to(lacc, c, a.loss_part + blockIdx.x, kFirstEpi);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kProdWarps) {
        tc_fence_after();
        tmem_dealloc(tbase, a.tmem_cols);
    }
}

// ================================================================== dW
struct DWArgs {
    const uint16_t *idx_s, *hT;
    uint16_t *dW;
    int32_t *status;
    int64_t K, L;
    int32_t B, G, F, MT, FT, S, nzc, zsw, planes, ncat, Nacc, issuers, ldB;
    uint32_t a_bytes, z_bytes, stage_bytes, tmem_cols;
};

template <int CH>
__global__ void __launch_bounds__(kFwdThreads, 1)
    k_tc_dW(const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_zl,
            const DWArgs a)
{
    __shared__ Ctl c;
    extern __shared__ uint8_t dsm[];
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const uint32_t stage0 = (smem_u32(dsm) + 1023u) & ~1023u;
    const int G = a.G, F = a.F, S = a.S;
    const uint32_t zrows = (uint32_t)a.MT * 128;
    const uint32_t zchunk = zrows * (uint32_t)a.zsw;          // one dZ chunk (<= 64 j)
    const uint32_t zplane = (uint32_t)a.nzc * zchunk;         // all of G for hi or lo
    const int nacc = 2 * a.issuers;
    const int per = a.FT * a.Nacc;

    if (threadIdx.x == 0)
        setup_ctl(c, S, nacc, kProdWarps * 32 + 1, 1);
    if (warp == kProdWarps) {
        tmem_alloc(smem_u32(&c.tmem), a.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = c.tmem;
    volatile int *abort_flag = &c.abort_flag;

    if (warp < kProdWarps) {
        producer_loop(c, stage0, a.stage_bytes, S, a.K, a.idx_s, a.hT, a.ldB, F, a.MT, a.z_bytes,
                      abort_flag, a.status, [&](int64_t k, uint32_t A, uint32_t fb) {
                          const uint32_t Zs = A + a.a_bytes;
                          for (int cj = 0; cj < a.nzc; ++cj) {
                              tma_load_2d(Zs + (uint32_t)cj * zchunk, &tm_z, (int)(k * G + cj * 64), 0, fb);
                              if (a.planes > 1)
                                  tma_load_2d(Zs + zplane + (uint32_t)cj * zchunk, &tm_zl,
                                              (int)(k * G + cj * 64), 0, fb);
                          }
                      });
    } else if (warp < kFirstEpi) {
        const int me = warp - kProdWarps;
        const uint32_t zlayout = layout_for_swizzle(a.zsw);
        // N = Nacc columns: [hi | lo] along N when concatenated (chunks of
        // <= 64 j at a uniform stride zchunk), else G columns per pass
        const uint32_t idesc = idesc_bf16(128, a.Nacc, 0, 1);
        const int passes = a.ncat ? 1 : a.planes;
        int it = 0;
        for (int64_t k = blockIdx.x; k < a.K; k += gridDim.x, ++it) {
            if (it % a.issuers != me)
                continue;
            const int s = it % S;
            const uint32_t ph = (uint32_t)(it / S) & 1u;
            const int acc = acc_slot(it, a.issuers);
            if (!mbar_wait(bar_addr(c.tempty[acc]), acc_phase(it, a.issuers) ^ 1u, abort_flag, a.status))
                break;
            tc_fence_after();
            if (!mbar_wait(bar_addr(c.full[s]), ph, abort_flag, a.status))
                break;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t A = stage0 + (uint32_t)s * a.stage_bytes;
                const uint32_t Zs = A + a.a_bytes;
                for (int tf = 0; tf < a.FT; ++tf) {
                    const uint32_t d = tbase + (uint32_t)(acc * per + tf * a.Nacc);
                    for (int ps = 0; ps < passes; ++ps) {
                        for (int st = 0; st < a.MT * 8; ++st) {
                            // A: H_k^T, K-major (rows f, K = b): b chunk st/4, 32 B per 16 b
                            const uint64_t ad = sdesc(A + (uint32_t)(st / 4) * F * 128 +
                                                          (uint32_t)tf * 128 * 128 + (uint32_t)(st % 4) * 32,
                                                      16, 1024, kLayoutSW128);
                            // B: dZ_k, MN-major (N = j, K = b): 16 b rows per step
                            const uint64_t bd = sdesc(Zs + (uint32_t)ps * zplane + (uint32_t)st * 16 * a.zsw,
                                                      zchunk, 8 * a.zsw, zlayout);
                            mma_bf16(d, ad, bd, idesc, (ps > 0 || st > 0) ? 1u : 0u);
                        }
                    }
                }
                mma_commit(bar_addr(c.empty[s]));
                mma_commit(bar_addr(c.tfull[acc]));
            }
            __syncwarp();
        }
        if (lane == 0)
            mma_commit(bar_addr(c.drain[me]));
        __syncwarp();
        mbar_wait_drain(bar_addr(c.drain[me]), 0);
    } else {
        const int q = warp & 3;
        const int sub = (warp - kFirstEpi) / 4;
        const int units = a.FT * (G / CH);
        int it = 0;
        for (int64_t k = blockIdx.x; k < a.K; k += gridDim.x, ++it) {
            const int acc = acc_slot(it, a.issuers);
            if (!mbar_wait(bar_addr(c.tfull[acc]), acc_phase(it, a.issuers), abort_flag, a.status))
                break;
            tc_fence_after();
            for (int u = sub; u < units; u += 2) {
                const int tf = u / (G / CH), c0 = (u % (G / CH)) * CH;
                const int f = tf * 128 + q * 32 + lane;
                const uint32_t col = tbase + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * per + tf * a.Nacc + c0);
                float v[CH];
                tmem_ld_chunk<CH>(col, v);
                if (a.ncat) {  // add the lo half, G columns further on
                    float w[CH];
                    tmem_ld_chunk<CH>(col + (uint32_t)G, w);
#pragma unroll
                    for (int i = 0; i < CH; ++i)
                        v[i] += w[i];
                }
                uint16_t *dst = a.dW + (k * G + c0) * F + f;
#pragma unroll
                for (int i = 0; i < CH; ++i)
                    dst[(int64_t)i * F] = f2bf(v[i]);
            }
            tc_fence_before();
            mbar_arrive(bar_addr(c.tempty[acc]));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kProdWarps) {
        tc_fence_after();
        tmem_dealloc(tbase, a.tmem_cols);
    }
}

// ================================================================== dh
struct DhArgs {
    const uint16_t *idx_s;
    float *dh;
    int32_t *status;
    int64_t K, L;
    int32_t B, G, F, H, MT, nk, S, nzc, zsw, nbands, band_w, win, parts, npass;
    uint32_t z_bytes, w_bytes, i_bytes, stage_bytes, tmem_cols;
};

// first f with I[f] >= v (I ascending, n entries)
__device__ __forceinline__ int lower_bound_u16(const uint16_t *I, int n, int v)
{
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if ((int)I[mid] < v)
            lo = mid + 1;
        else
            hi = mid;
    }
    return lo;
}

// CTA (band, mtile, part): dh columns [i0, i1) of the band, samples
// [128 mt, 128 mt + 128), groups k = part, part + parts, ...  TMEM columns
// [0, band_w) hold the CTA's fp32 partial of dh; two windows of `win` columns
// after it receive dH_k = dZ_k W_k for the f range of the band (alternately,
// so the MMA of the next group overlaps the scatter of this one).
__global__ void __launch_bounds__(kDhThreads, 1)
    k_tc_dh(const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_zl,
            const __grid_constant__ CUtensorMap tm_w, const DhArgs a)
{
    __shared__ Ctl c;
    extern __shared__ uint8_t dsm[];
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const uint32_t stage0 = (smem_u32(dsm) + 1023u) & ~1023u;
    uint8_t *stage0_ptr = dsm + (stage0 - smem_u32(dsm));
    const int G = a.G, F = a.F, S = a.S;
    const int band = blockIdx.x % a.nbands;
    const int mt = (blockIdx.x / a.nbands) % a.MT;
    const int part = blockIdx.x / (a.nbands * a.MT);
    const int i0 = band * a.band_w;
    const int i1 = min(a.H, i0 + a.band_w);
    const uint32_t zrows = 128;
    const uint32_t zchunk = zrows * (uint32_t)a.zsw;
    const uint32_t zplane = (uint32_t)a.nzc * zchunk;

    if (threadIdx.x == 0)
        setup_ctl(c, S, 2, 1, kEpiWarps * 32);  // stages released by the epilogue
    if (warp == 1) {
        tmem_alloc(smem_u32(&c.tmem), a.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = c.tmem;
    volatile int *abort_flag = &c.abort_flag;

    if (warp == 0) {
        int it = 0;
        for (int64_t k = part; k < a.K; k += a.parts, ++it) {
            const int s = it % S;
            const uint32_t ph = (uint32_t)(it / S) & 1u;
            if (!mbar_wait(bar_addr(c.empty[s]), ph ^ 1u, abort_flag, a.status))
                break;
            const uint32_t Zs = stage0 + (uint32_t)s * a.stage_bytes;
            const uint32_t Wt = Zs + a.z_bytes;
            const uint32_t Is = Wt + a.w_bytes;
            const uint32_t fb = bar_addr(c.full[s]);
            if (lane == 0) {
                mbar_arrive_expect_tx(fb, a.z_bytes + a.w_bytes + (uint32_t)F * 2);
                for (int cj = 0; cj < a.nzc; ++cj) {
                    tma_load_2d(Zs + (uint32_t)cj * zchunk, &tm_z, (int)(k * G + cj * 64), mt * 128, fb);
                    if (a.npass > 1)
                        tma_load_2d(Zs + zplane + (uint32_t)cj * zchunk, &tm_zl, (int)(k * G + cj * 64),
                                    mt * 128, fb);
                }
                for (int kc = 0; kc < a.nk; ++kc)
                    tma_load_2d(Wt + (uint32_t)kc * G * 128, &tm_w, kc * 64, (int)(k * G), fb);
                bulk_load(Is, a.idx_s + k * F, (uint32_t)F * 2, fb);
            }
            __syncwarp();
        }
        drain_loads(c, it, S);
    } else if (warp == 1) {
        const uint32_t zlayout = layout_for_swizzle(a.zsw);
        const int nks = G / 16;
        int it = 0;
        for (int64_t k = part; k < a.K; k += a.parts, ++it) {
            const int s = it % S;
            const uint32_t ph = (uint32_t)(it / S) & 1u;
            const int wb = it & 1;
            if (!mbar_wait(bar_addr(c.tempty[wb]), ((uint32_t)(it >> 1) & 1u) ^ 1u, abort_flag, a.status))
                break;
            tc_fence_after();
            if (!mbar_wait(bar_addr(c.full[s]), ph, abort_flag, a.status))
                break;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t Zs = stage0 + (uint32_t)s * a.stage_bytes;
                const uint32_t Wt = Zs + a.z_bytes;
                const uint16_t *I = reinterpret_cast<const uint16_t *>(
                    stage0_ptr + (size_t)s * a.stage_bytes + a.z_bytes + a.w_bytes);
                // f range whose index falls in [i0, i1): I_k is ascending
                const int fa = lower_bound_u16(I, F, i0), fbnd = lower_bound_u16(I, F, i1);
                // whole 64-f chunks of W_k that hold part of the f range:
                // every window starts on a swizzle-atom boundary of the tile
                const uint32_t dbase = tbase + (uint32_t)(a.band_w + wb * a.win);
                if (fa < fbnd) {
                    const int c_first = fa / 64, c_last = (fbnd - 1) / 64;
                    const uint32_t idesc = idesc_bf16(128, 64, 0, 1);
                    for (int cc = c_first; cc <= c_last; ++cc) {
                        const uint32_t d = dbase + (uint32_t)((cc - c_first) * 64);
                        // K runs over j for dZ hi (and again for dZ lo) against W_k
                        for (int ks2 = 0; ks2 < a.npass * nks; ++ks2) {
                            const int ks = ks2 % nks;
                            const uint32_t za = Zs + (uint32_t)(ks2 / nks) * zplane +
                                                (uint32_t)(ks / 4) * zchunk + (uint32_t)(ks % 4) * 32;
                            const uint64_t ad = sdesc(za, 16, 8 * a.zsw, zlayout);
                            const uint64_t bd = sdesc(Wt + (uint32_t)cc * G * 128 + (uint32_t)ks * 2048,
                                                      (uint32_t)G * 128, 1024, kLayoutSW128);
                            mma_bf16(d, ad, bd, idesc, ks2 > 0 ? 1u : 0u);
                        }
                    }
                }
                mma_commit(bar_addr(c.tfull[wb]));
            }
            __syncwarp();
        }
        if (lane == 0)
            mma_commit(bar_addr(c.drain[0]));
        __syncwarp();
        mbar_wait_drain(bar_addr(c.drain[0]), 0);
    } else {
        // two warps per TMEM lane quarter.  They may be working on different
        // groups at the same time (the dH windows are double buffered), so
        // they own disjoint partial columns (column parity) rather than
        // disjoint pieces: no column is ever updated by both.
        const int q = warp & 3;
        const int sub = (warp - 2) / 4;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        for (int col = sub; col < a.band_w; col += 2)
            tmem_st1(tbase + lane_off + (uint32_t)col, 0u);
        tmem_st_wait();
        int it = 0;
        for (int64_t k = part; k < a.K; k += a.parts, ++it) {
            const int s = it % S;
            const uint32_t ph = (uint32_t)(it / S) & 1u;
            const int wb = it & 1;
            if (!mbar_wait(bar_addr(c.full[s]), ph, abort_flag, a.status))
                break;
            if (!mbar_wait(bar_addr(c.tfull[wb]), (uint32_t)(it >> 1) & 1u, abort_flag, a.status))
                break;
            tc_fence_after();
            const uint16_t *I = reinterpret_cast<const uint16_t *>(
                stage0_ptr + (size_t)s * a.stage_bytes + a.z_bytes + a.w_bytes);
            const int fa = lower_bound_u16(I, F, i0), fbnd = lower_bound_u16(I, F, i1);
            const int fbase = (fa / 64) * 64;  // first f of the first window
            const uint32_t dbase = tbase + lane_off + (uint32_t)(a.band_w + wb * a.win);
            for (int p = fa / 16; p * 16 < fbnd; ++p) {
                uint32_t r[16];
                tmem_ld16(dbase + (uint32_t)(p * 16 - fbase), r);
                uint32_t col[16], old[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int f = p * 16 + u;
                    const uint32_t cf = (f >= fa && f < fbnd) ? (uint32_t)(I[f] - i0) : 0xffffffffu;
                    col[u] = (cf != 0xffffffffu && (int)(cf & 1u) == sub) ? cf : 0xffffffffu;
                    old[u] = 0u;
                    if (col[u] != 0xffffffffu)
                        old[u] = tmem_ld1(tbase + lane_off + col[u]);
                }
                tmem_ld_wait();
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    if (col[u] != 0xffffffffu)
                        tmem_st1(tbase + lane_off + col[u],
                                 __float_as_uint(__uint_as_float(old[u]) + __uint_as_float(r[u])));
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar_addr(c.tempty[wb]));
            mbar_arrive(bar_addr(c.empty[s]));
        }
        // add the partial into dh, once both warps of every quarter are done
        named_bar(1, kEpiWarps * 32);
        const int b = mt * 128 + q * 32 + lane;
        for (int c0 = sub * 32; c0 < a.band_w; c0 += 64) {
            uint32_t r[32];
            tmem_ld32(tbase + lane_off + (uint32_t)c0, r);
            tmem_ld_wait();
            if (b < a.B) {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int colg = i0 + c0 + i;
                    if (colg < i1)
                        atomicAdd(a.dh + (int64_t)b * a.H + colg, __uint_as_float(r[i]));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, a.tmem_cols);
    }
}

template <typename K>
sg_status set_smem(K kern, size_t bytes)
{
    SG_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes));
    return SG_OK;
}

int persistent_grid(const sg_layout *lo, int64_t work)
{
    int64_t g = lo->num_sms;
    if (g > work)
        g = work;
    if (g < 1)
        g = 1;
    return (int)g;
}

}  // namespace

// ------------------------------------------------------------------ host side
bool tc_supported(const sg_layout *lo) { return plan_fwd(lo, lo->max_B).ok; }

bool tc_stage_ok(const sg_layout *lo, int stage, int B)
{
    switch (stage) {
    case SG_KIND_FWD: return plan_fwd(lo, B).ok;
    case SG_KIND_DW: return plan_dW(lo, B, true).ok;
    case SG_KIND_DH: return plan_dh(lo, B, true).ok;
    default: return false;
    }
}

sg_status tc_fwd(sg_layout *lo, int32_t B, const uint16_t *W, uint16_t *Z, uint16_t *dZ,
                 uint16_t *dZ_lo, double *loss, cudaStream_t st)
{
    const FwdPlan p = plan_fwd(lo, B);
    if (!p.ok) {
        sg_set_error("tc_fwd: shape not supported by the tensor-core engine");
        return SG_ERR_UNSUPPORTED;
    }
    CUtensorMap tm_w;
    sg_status rc = make_map_2d(&tm_w, W, (uint64_t)lo->F, (uint64_t)lo->L, 64, (uint32_t)lo->G, 128, "W");
    if (rc != SG_OK)
        return rc;
    FwdArgs a;
    a.idx_s = lo->idx_s;
    a.hT = lo->hT;
    a.Z = Z;
    a.dZ = dZ;
    a.dZ_lo = dZ_lo;
    a.gptr = lo->gptr;
    a.gent = lo->gent;
    a.loss_part = lo->loss_part;
    a.status = lo->status;
    a.K = lo->K;
    a.L = lo->L;
    a.B = B;
    a.G = lo->G;
    a.F = lo->F;
    a.MT = p.MT;
    a.nk = p.nk;
    a.S = p.S;
    a.issuers = p.issuers;
    a.ldB = lo->ldB;
    a.a_bytes = p.a_bytes;
    a.w_bytes = p.w_bytes;
    a.stage_bytes = p.stage_bytes;
    a.tmem_cols = p.tmem_cols;
    const size_t smem = (size_t)p.S * p.stage_bytes + 1024;
    const int grid = persistent_grid(lo, lo->K);
    const bool bce = dZ != nullptr;
    void (*kern)(CUtensorMap, FwdArgs);
    if (lo->G >= 64)
        kern = bce ? k_tc_fwd<true, 32> : k_tc_fwd<false, 32>;
    else
        kern = bce ? k_tc_fwd<true, 16> : k_tc_fwd<false, 16>;
    rc = set_smem(kern, smem);
    if (rc != SG_OK)
        return rc;
    SG_LAUNCH(lo, SG_KIND_FWD, st, kern<<<grid, kFwdThreads, smem, st>>>(tm_w, a));
    SG_TRY_CUDA(cudaGetLastError());
    if (bce)
        return sg_loss_finalize(lo, grid, loss, st);
    return SG_OK;
}

sg_status tc_dW(sg_layout *lo, const uint16_t *dZ, const uint16_t *dZ_lo, int32_t B,
                uint16_t *dW, cudaStream_t st)
{
    const DWPlan p = plan_dW(lo, B, dZ_lo != nullptr);
    if (!p.ok) {
        sg_set_error("tc_dW: shape not supported by the tensor-core engine");
        return SG_ERR_UNSUPPORTED;
    }
    CUtensorMap tm_z, tm_zl;
    const int zbox = lo->G < 64 ? lo->G : 64;
    sg_status rc = make_map_2d(&tm_z, dZ, (uint64_t)lo->L, (uint64_t)B, (uint32_t)zbox,
                               (uint32_t)(p.MT * 128), p.zsw, "dZ");
    if (rc != SG_OK)
        return rc;
    tm_zl = tm_z;
    if (dZ_lo) {
        rc = make_map_2d(&tm_zl, dZ_lo, (uint64_t)lo->L, (uint64_t)B, (uint32_t)zbox,
                         (uint32_t)(p.MT * 128), p.zsw, "dZ_lo");
        if (rc != SG_OK)
            return rc;
    }
    DWArgs a;
    a.idx_s = lo->idx_s;
    a.hT = lo->hT;
    a.dW = dW;
    a.status = lo->status;
    a.K = lo->K;
    a.L = lo->L;
    a.B = B;
    a.G = lo->G;
    a.F = lo->F;
    a.MT = p.MT;
    a.FT = p.FT;
    a.S = p.S;
    a.nzc = p.nzc;
    a.zsw = p.zsw;
    a.planes = p.planes;
    a.ncat = p.ncat;
    a.Nacc = p.Nacc;
    a.issuers = p.issuers;
    a.ldB = lo->ldB;
    a.a_bytes = p.a_bytes;
    a.z_bytes = p.z_bytes;
    a.stage_bytes = p.stage_bytes;
    a.tmem_cols = p.tmem_cols;
    const size_t smem = (size_t)p.S * p.stage_bytes + 1024;
    const int grid = persistent_grid(lo, lo->K);
    void (*kern)(CUtensorMap, CUtensorMap, DWArgs) = lo->G >= 64 ? k_tc_dW<32> : k_tc_dW<16>;
    rc = set_smem(kern, smem);
    if (rc != SG_OK)
        return rc;
    SG_LAUNCH(lo, SG_KIND_DW, st, kern<<<grid, kFwdThreads, smem, st>>>(tm_z, tm_zl, a));
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}

sg_status tc_dh(sg_layout *lo, const uint16_t *dZ, const uint16_t *dZ_lo, int32_t B,
                const uint16_t *W, float *dh, cudaStream_t st)
{
    const DhPlan p = plan_dh(lo, B, dZ_lo != nullptr);
    if (!p.ok) {
        sg_set_error("tc_dh: shape not supported by the tensor-core engine");
        return SG_ERR_UNSUPPORTED;
    }
    CUtensorMap tm_z, tm_zl, tm_w;
    const int zbox = lo->G < 64 ? lo->G : 64;
    sg_status rc = make_map_2d(&tm_z, dZ, (uint64_t)lo->L, (uint64_t)B, (uint32_t)zbox, 128,
                               p.zsw, "dZ");
    if (rc != SG_OK)
        return rc;
    tm_zl = tm_z;
    if (dZ_lo) {
        rc = make_map_2d(&tm_zl, dZ_lo, (uint64_t)lo->L, (uint64_t)B, (uint32_t)zbox, 128, p.zsw,
                         "dZ_lo");
        if (rc != SG_OK)
            return rc;
    }
    rc = make_map_2d(&tm_w, W, (uint64_t)lo->F, (uint64_t)lo->L, 64, (uint32_t)lo->G, 128, "W");
    if (rc != SG_OK)
        return rc;
    DhArgs a;
    a.idx_s = lo->idx_s;
    a.dh = dh;
    a.status = lo->status;
    a.K = lo->K;
    a.L = lo->L;
    a.B = B;
    a.G = lo->G;
    a.F = lo->F;
    a.H = lo->H;
    a.MT = p.MT;
    a.nk = p.nk;
    a.S = p.S;
    a.nzc = p.nzc;
    a.zsw = p.zsw;
    a.nbands = p.nbands;
    a.band_w = p.band_w;
    a.win = p.win;
    a.npass = dZ_lo ? 2 : 1;
    int parts = lo->num_sms / (p.nbands * p.MT);
    if (parts < 1)
        parts = 1;
    if (parts > lo->K)
        parts = (int)lo->K;
    a.parts = parts;
    a.z_bytes = p.z_bytes;
    a.w_bytes = p.w_bytes;
    a.i_bytes = p.i_bytes;
    a.stage_bytes = p.stage_bytes;
    a.tmem_cols = p.tmem_cols;
    const size_t smem = (size_t)p.S * p.stage_bytes + 1024;
    rc = set_smem(k_tc_dh, smem);
    if (rc != SG_OK)
        return rc;
    SG_TRY_CUDA(cudaMemsetAsync(dh, 0, sizeof(float) * B * lo->H, st));
    SG_LAUNCH(lo, SG_KIND_DH, st,
              k_tc_dh<<<p.nbands * p.MT * parts, kDhThreads, smem, st>>>(tm_z, tm_zl, tm_w, a));
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}

sg_status tc_step(sg_layout *lo, int32_t B, const uint16_t *W, uint16_t *dW, float *dh,
                  double *loss, cudaStream_t st)
{
    (void)lo; (void)B; (void)W; (void)dW; (void)dh; (void)loss; (void)st;
    sg_set_error("tc_step: the fused step kernel is not built yet");
    return SG_ERR_UNSUPPORTED;
}
