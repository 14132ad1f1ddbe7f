// Dense bf16 GEMM on the tensor cores (sm_103a) for the head-tail split's
// projections (HASTE, "Method / overall framework": h_head = h P_head^T,
// h_tail = h P_tail^T, and their backward).  One 128 x 128 output tile per
// CTA: a TMA producer warp streams 64-wide K blocks of A and B into a ring of
// shared-memory stages (128-byte swizzle), one thread issues tcgen05.mma into
// a TMEM accumulator, four warps write the tile out.
//
//   C[m][n] (+)= sum_k A[m][k] B[n][k]        (fp32 accumulation)
// A is K-major (A[m][k] at A + m lda + k) or MN-major (A + k lda + m); the
// same for B with n.  C is row-major fp32 or bf16 (RNE).  Loads past M, N or
// K read zeros (TMA fill); stores stop at M and N.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "sg_internal.cuh"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

using namespace tc;

namespace {

constexpr int kGS = 4;                // stages
constexpr int kGThreads = 32 * 6;     // producer, MMA, four epilogue warps
constexpr uint32_t kTileBytes = 16384;  // one 128 x 64 bf16 operand tile

struct GemmCtl {
    uint64_t full[kGS], empty[kGS];
    uint64_t tfull, drain;
    uint32_t tmem;
    int abort_flag;
};

struct GemmArgs {
    void *C;
    int64_t ldc;
    int32_t M, N, K, a_mn, b_mn, c_bf16, accumulate;
    int32_t *status;
};

__device__ __forceinline__ uint32_t bar_of(const uint64_t &b) { return smem_u32(&b); }

// one operand tile of 128 rows (m or n) x 64 k into shared memory at dst:
// K-major: one box {64 k, 128 rows}; MN-major: two boxes {64 rows, 64 k}
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap *map, int mn_major, int row0, int k0,
                                          uint32_t bar)
{
    if (!mn_major) {
        tma_load_2d(dst, map, k0, row0, bar);
    } else {
        tma_load_2d(dst, map, row0, k0, bar);
        tma_load_2d(dst + kTileBytes / 2, map, row0 + 64, k0, bar);
    }
}

// descriptor of k step ks (16 k) of a tile: K-major rows of 128 bytes in
// 1024-byte atoms of 8 rows; MN-major two chunks of 64 rows (k rows of 128
// bytes, 8 k per atom), the second kTileBytes / 2 further on
__device__ __forceinline__ uint64_t tile_desc(uint32_t tile, int mn_major, int ks)
{
    return mn_major ? sdesc(tile + (uint32_t)ks * 2048, kTileBytes / 2, 1024, kLayoutSW128)
                    : sdesc(tile + (uint32_t)ks * 32, 16, 1024, kLayoutSW128);
}

__global__ void __launch_bounds__(kGThreads, 1)
    k_gemm(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b, const GemmArgs a)
{
    __shared__ GemmCtl c;
    extern __shared__ uint8_t dsm[];
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const uint32_t base = (smem_u32(dsm) + 1023u) & ~1023u;
    const int m0 = blockIdx.y * 128, n0 = blockIdx.x * 128;
    const int nkb = (a.K + 63) / 64;
    if (threadIdx.x == 0) {
        c.abort_flag = 0;
        for (int s = 0; s < kGS; ++s) {
            mbar_init(bar_of(c.full[s]), 1);
            mbar_init(bar_of(c.empty[s]), 1);
        }
        mbar_init(bar_of(c.tfull), 1);
        mbar_init(bar_of(c.drain), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&c.tmem), 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = c.tmem;
    volatile int *abort_flag = &c.abort_flag;

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        int kb = 0;
        if (lane == 0) {
            for (; kb < nkb; ++kb) {
                const int s = kb % kGS;
                if (!mbar_wait(bar_of(c.empty[s]), ((uint32_t)(kb / kGS) & 1u) ^ 1u, abort_flag, a.status))
                    break;
                const uint32_t st = base + (uint32_t)s * 2 * kTileBytes;
                mbar_arrive_expect_tx(bar_of(c.full[s]), 2 * kTileBytes);
                load_tile(st, &tm_a, a.a_mn, m0, kb * 64, bar_of(c.full[s]));
                load_tile(st + kTileBytes, &tm_b, a.b_mn, n0, kb * 64, bar_of(c.full[s]));
            }
            if (*abort_flag)
                for (int j = kb - kGS < 0 ? 0 : kb - kGS; j < kb; ++j)
                    mbar_wait_drain(bar_of(c.full[j % kGS]), (uint32_t)(j / kGS) & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA
        const uint32_t idesc = idesc_bf16(128, 128, a.a_mn, a.b_mn);
        int kb = 0;
        for (; kb < nkb; ++kb) {
            const int s = kb % kGS;
            if (!__all_sync(0xffffffffu, mbar_wait(bar_of(c.full[s]), (uint32_t)(kb / kGS) & 1u, abort_flag,
                                                   a.status)))
                break;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t st = base + (uint32_t)s * 2 * kTileBytes;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tbase, tile_desc(st, a.a_mn, ks), tile_desc(st + kTileBytes, a.b_mn, ks), idesc,
                             (kb > 0 || ks > 0) ? 1u : 0u);
                mma_commit(bar_of(c.empty[s]));
            }
            __syncwarp();
        }
        if (lane == 0) {
            if (kb == nkb)
                mma_commit(bar_of(c.tfull));
            mma_commit(bar_of(c.drain));
        }
        __syncwarp();
        mbar_wait_drain(bar_of(c.drain), 0);
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quarter of this warp
        const int m = m0 + q * 32 + lane;
        if (__all_sync(0xffffffffu, mbar_wait(bar_of(c.tfull), 0, abort_flag, a.status))) {
            tc_fence_after();
            for (int cc = 0; cc < 128; cc += 32) {
                uint32_t r[32];
                tmem_ld32(tbase + ((uint32_t)(q * 32) << 16) + (uint32_t)cc, r);
                tmem_ld_wait();
                if (m >= a.M)
                    continue;
#pragma unroll
                for (int x = 0; x < 32; ++x) {
                    const int n = n0 + cc + x;
                    if (n >= a.N)
                        break;
                    float v = __uint_as_float(r[x]);
                    if (a.c_bf16) {
                        uint16_t *dst = reinterpret_cast<uint16_t *>(a.C) + (int64_t)m * a.ldc + n;
                        if (a.accumulate)
                            v += __uint_as_float((uint32_t)*dst << 16);
                        *dst = bf16_rn(v);
                    } else {
                        float *dst = reinterpret_cast<float *>(a.C) + (int64_t)m * a.ldc + n;
                        if (a.accumulate)
                            v += *dst;
                        *dst = v;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 128);
    }
}

// ---------------------------------------------------------------- group |.|-sum GEMM
// out[m / G][n] = sum over the G rows m of a group of |sum_k A[m][k] B[n][k]|
// (A and B MN-major, G a power of two <= 128, so a 128-row tile holds whole
// groups).  The same tile loop as k_gemm; the epilogue reduces |acc| over
// the group's TMEM lanes with shuffles (G <= 32) or across the four epilogue
// warps through shared memory (G = 64, 128).
__global__ void __launch_bounds__(kGThreads, 1)
    k_gemm_gabs(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b, float *out,
                int32_t M, int32_t N, int32_t K, int32_t G, int32_t NS, int32_t *status)
{
    __shared__ GemmCtl c;
    __shared__ float part[4][32];
    extern __shared__ uint8_t dsm[];
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const uint32_t base = (smem_u32(dsm) + 1023u) & ~1023u;
    const int m0 = blockIdx.y * 128, n0 = blockIdx.x * 128;
    const int nkb = (K + 63) / 64;
    if (threadIdx.x == 0) {
        c.abort_flag = 0;
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar_of(c.full[s]), 1);
            mbar_init(bar_of(c.empty[s]), 1);
        }
        mbar_init(bar_of(c.tfull), 1);
        mbar_init(bar_of(c.drain), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&c.tmem), 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = c.tmem;
    volatile int *abort_flag = &c.abort_flag;

    if (warp == 0) {
        int kb = 0;
        if (lane == 0) {
            for (; kb < nkb; ++kb) {
                const int s = kb % NS;
                if (!mbar_wait(bar_of(c.empty[s]), ((uint32_t)(kb / NS) & 1u) ^ 1u, abort_flag, status))
                    break;
                const uint32_t st = base + (uint32_t)s * 2 * kTileBytes;
                mbar_arrive_expect_tx(bar_of(c.full[s]), 2 * kTileBytes);
                load_tile(st, &tm_a, 1, m0, kb * 64, bar_of(c.full[s]));
                load_tile(st + kTileBytes, &tm_b, 1, n0, kb * 64, bar_of(c.full[s]));
            }
            if (*abort_flag)
                for (int j = kb - NS < 0 ? 0 : kb - NS; j < kb; ++j)
                    mbar_wait_drain(bar_of(c.full[j % NS]), (uint32_t)(j / NS) & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        const uint32_t idesc = idesc_bf16(128, 128, 1, 1);
        int kb = 0;
        for (; kb < nkb; ++kb) {
            const int s = kb % NS;
            if (!__all_sync(0xffffffffu, mbar_wait(bar_of(c.full[s]), (uint32_t)(kb / NS) & 1u, abort_flag,
                                                   status)))
                break;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t st = base + (uint32_t)s * 2 * kTileBytes;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tbase, tile_desc(st, 1, ks), tile_desc(st + kTileBytes, 1, ks), idesc,
                             (kb > 0 || ks > 0) ? 1u : 0u);
                mma_commit(bar_of(c.empty[s]));
            }
            __syncwarp();
        }
        if (lane == 0) {
            if (kb == nkb)
                mma_commit(bar_of(c.tfull));
            mma_commit(bar_of(c.drain));
        }
        __syncwarp();
        mbar_wait_drain(bar_of(c.drain), 0);
    } else {
        const int q = warp & 3;
        const int m = m0 + q * 32 + lane;
        const bool ok = __all_sync(0xffffffffu, mbar_wait(bar_of(c.tfull), 0, abort_flag, status));
        if (ok)
            tc_fence_after();
        for (int cc = 0; cc < 128; cc += 32) {
            float v[32];
#pragma unroll
            for (int x = 0; x < 32; ++x)
                v[x] = 0.f;
            if (ok) {
                uint32_t r[32];
                tmem_ld32(tbase + ((uint32_t)(q * 32) << 16) + (uint32_t)cc, r);
                tmem_ld_wait();
#pragma unroll
                for (int x = 0; x < 32; ++x)
                    v[x] = fabsf(__uint_as_float(r[x]));
            }
            const int gl = G < 32 ? G : 32;  // lanes of a group inside the warp
            for (int off = 1; off < gl; off <<= 1) {
#pragma unroll
                for (int x = 0; x < 32; ++x)
                    v[x] += __shfl_xor_sync(0xffffffffu, v[x], off);
            }
            if (G <= 32) {
                // lane i of a group writes the columns x = i (mod G)
                const int64_t k = m / G;
                if (ok && m < M) {
#pragma unroll
                    for (int x = 0; x < 32; ++x) {
                        const int n = n0 + cc + x;
                        if ((x & (G - 1)) == (lane & (G - 1)) && n < N)
                            out[k * N + n] = v[x];
                    }
                }
            } else {
                // warp sums to shared memory, then the first warp of each
                // group adds the group's warps (named barrier of the four)
#pragma unroll
                for (int x = 0; x < 32; ++x)
                    if (x == lane)
                        part[q][x] = v[x];
                asm volatile("bar.sync 1, 128;" ::: "memory");
                const int wpg = G / 32;  // warps per group
                if (ok && q % wpg == 0 && m0 + q * 32 < M) {
                    float sum = 0.f;
                    for (int w2 = q; w2 < q + wpg; ++w2)
                        sum += part[w2][lane];
                    const int n = n0 + cc + lane;
                    if (n < N)
                        out[(int64_t)((m0 + q * 32) / G) * N + n] = sum;
                }
                asm volatile("bar.sync 1, 128;" ::: "memory");
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 128);
    }
}

// ---------------------------------------------------------------- argmax GEMM
// For each row m of A (M x K, K-major) the column n of B (N x K, K-major) with
// the largest <A_m, B_n> (fp32 accumulation; ties to the smaller n).  One CTA
// per 128-row tile of A walks all 128-column tiles of B: the producer streams
// (n tile, k block) pairs of A and B tiles, one thread issues the MMAs into two
// TMEM accumulators used alternately, and each epilogue thread keeps its row's
// running best over the tiles in registers.
struct ArgmaxCtl {
    uint64_t full[kGS], empty[kGS];
    uint64_t tfull[2], tempty[2], drain;
    uint32_t tmem;
    int abort_flag;
};

struct ArgmaxArgs {
    int32_t *best_idx;
    float *best_val;
    int32_t M, N, K;
    int32_t *status;
};

__global__ void __launch_bounds__(kGThreads, 1)
    k_gemm_argmax(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                  const ArgmaxArgs a)
{
    __shared__ ArgmaxCtl c;
    extern __shared__ uint8_t dsm[];
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const uint32_t base = (smem_u32(dsm) + 1023u) & ~1023u;
    const int m0 = blockIdx.x * 128;
    const int nkb = (a.K + 63) / 64;
    const int ntiles = (a.N + 127) / 128;
    if (threadIdx.x == 0) {
        c.abort_flag = 0;
        for (int s = 0; s < kGS; ++s) {
            mbar_init(bar_of(c.full[s]), 1);
            mbar_init(bar_of(c.empty[s]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_of(c.tfull[i]), 1);
            mbar_init(bar_of(c.tempty[i]), 128);
        }
        mbar_init(bar_of(c.drain), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&c.tmem), 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = c.tmem;
    volatile int *abort_flag = &c.abort_flag;
    const int total = ntiles * nkb;

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        int it = 0;
        if (lane == 0) {
            for (; it < total; ++it) {
                const int s = it % kGS;
                if (!mbar_wait(bar_of(c.empty[s]), ((uint32_t)(it / kGS) & 1u) ^ 1u, abort_flag, a.status))
                    break;
                const int n = it / nkb, kb = it - n * nkb;
                const uint32_t st = base + (uint32_t)s * 2 * kTileBytes;
                mbar_arrive_expect_tx(bar_of(c.full[s]), 2 * kTileBytes);
                tma_load_2d(st, &tm_a, kb * 64, m0, bar_of(c.full[s]));
                tma_load_2d(st + kTileBytes, &tm_b, kb * 64, n * 128, bar_of(c.full[s]));
            }
            if (*abort_flag)
                for (int j = it - kGS < 0 ? 0 : it - kGS; j < it; ++j)
                    mbar_wait_drain(bar_of(c.full[j % kGS]), (uint32_t)(j / kGS) & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA
        const uint32_t idesc = idesc_bf16(128, 128, 0, 0);
        int it = 0;
        bool live = true;
        for (int n = 0; n < ntiles && live; ++n) {
            const int acc = n & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(bar_of(c.tempty[acc]), ((uint32_t)(n >> 1) & 1u) ^ 1u,
                                                   abort_flag, a.status)))
                break;
            tc_fence_after();
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const int s = it % kGS;
                if (!__all_sync(0xffffffffu, mbar_wait(bar_of(c.full[s]), (uint32_t)(it / kGS) & 1u, abort_flag,
                                                       a.status))) {
                    live = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t st = base + (uint32_t)s * 2 * kTileBytes;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16(tbase + (uint32_t)(acc * 128), tile_desc(st, 0, ks),
                                 tile_desc(st + kTileBytes, 0, ks), idesc, (kb > 0 || ks > 0) ? 1u : 0u);
                    mma_commit(bar_of(c.empty[s]));
                    if (kb == nkb - 1)
                        mma_commit(bar_of(c.tfull[acc]));
                }
                __syncwarp();
            }
        }
        if (lane == 0)
            mma_commit(bar_of(c.drain));
        __syncwarp();
        mbar_wait_drain(bar_of(c.drain), 0);
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int m = m0 + q * 32 + lane;
        float best = -INFINITY;
        int bidx = -1;
        bool ok = true;
        for (int n = 0; n < ntiles; ++n) {
            const int acc = n & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(bar_of(c.tfull[acc]), (uint32_t)(n >> 1) & 1u, abort_flag,
                                                   a.status))) {
                ok = false;
                break;
            }
            tc_fence_after();
            for (int cc = 0; cc < 128; cc += 32) {
                uint32_t r[32];
                tmem_ld32(tbase + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * 128 + cc), r);
                tmem_ld_wait();
#pragma unroll
                for (int x = 0; x < 32; ++x) {
                    const int col = n * 128 + cc + x;
                    const float v = __uint_as_float(r[x]);
                    if (col < a.N && v > best) {  // ascending columns: ties keep the smaller
                        best = v;
                        bidx = col;
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar_of(c.tempty[acc]));
        }
        if (ok && m < a.M) {
            a.best_idx[m] = bidx;
            if (a.best_val)
                a.best_val[m] = best;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 256);
    }
}

// fp32 -> bf16 value plane + residual plane (x - bf16(x), rounded to bf16):
// the pair carries about 16 significant bits into a bf16 GEMM
__global__ void k_split_hilo(const float *__restrict__ x, int64_t n, uint16_t *__restrict__ hi,
                             uint16_t *__restrict__ lo)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float v = x[i];
        const uint16_t h = bf16_rn(v);
        hi[i] = h;
        lo[i] = bf16_rn(v - __uint_as_float((uint32_t)h << 16));
    }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode_gemm = nullptr;

// 2D bf16 tensor map: `inner` contiguous elements per row, `outer` rows,
// row stride ld elements, box {box_inner, box_outer}, 128-byte swizzle
sg_status map_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t ld,
                 uint32_t box_inner, uint32_t box_outer, const char *what)
{
    if (!g_encode_gemm) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn) {
            sg_set_error("cuTensorMapEncodeTiled is not available from the driver");
            return SG_ERR_CUDA;
        }
        g_encode_gemm = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    }
    if (((uintptr_t)base & 15) != 0 || (ld * 2) % 16 != 0) {
        sg_set_error("%s: base must be 16-byte aligned and the row stride a multiple of 8 elements", what);
        return SG_ERR_INVALID;
    }
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode_gemm(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
                               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        sg_set_error("%s: cuTensorMapEncodeTiled failed (%d)", what, (int)r);
        return SG_ERR_CUDA;
    }
    return SG_OK;
}

}  // namespace

sg_status gemm_bf16(const uint16_t *A, int a_mn, int64_t lda, const uint16_t *B, int b_mn, int64_t ldb, int M,
                    int N, int K, void *C, int c_bf16, int64_t ldc, int accumulate, int32_t *status, cudaStream_t st)
{
    if (M < 1 || N < 1 || K < 1)
        return SG_OK;
    CUtensorMap ta, tb;
    // K-major: rows of K (inner), box {64 k, 128 rows}; MN-major: rows of M
    // or N (inner) for each k, box {64, 64 k}
    sg_status rc = a_mn ? map_2d(&ta, A, (uint64_t)M, (uint64_t)K, (uint64_t)lda, 64, 64, "A")
                        : map_2d(&ta, A, (uint64_t)K, (uint64_t)M, (uint64_t)lda, 64, 128, "A");
    if (rc != SG_OK)
        return rc;
    rc = b_mn ? map_2d(&tb, B, (uint64_t)N, (uint64_t)K, (uint64_t)ldb, 64, 64, "B")
              : map_2d(&tb, B, (uint64_t)K, (uint64_t)N, (uint64_t)ldb, 64, 128, "B");
    if (rc != SG_OK)
        return rc;
    GemmArgs a;
    a.C = C;
    a.ldc = ldc;
    a.M = M;
    a.N = N;
    a.K = K;
    a.a_mn = a_mn;
    a.b_mn = b_mn;
    a.c_bf16 = c_bf16;
    a.accumulate = accumulate;
    a.status = status;
    const size_t smem = (size_t)kGS * 2 * kTileBytes + 1024;
    SG_TRY_CUDA(cudaFuncSetAttribute(k_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    dim3 grid((unsigned)((N + 127) / 128), (unsigned)((M + 127) / 128));
    k_gemm<<<grid, kGThreads, smem, st>>>(ta, tb, a);
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}

sg_status gemm_argmax_bf16(const uint16_t *A, int64_t lda, int M, const uint16_t *B, int64_t ldb, int N, int K,
                           int32_t *best_idx, float *best_val, int32_t *status, cudaStream_t st)
{
    if (M < 1)
        return SG_OK;
    if (N < 1 || K < 1) {
        sg_set_error("argmax GEMM: N and K must be positive (N=%d K=%d)", N, K);
        return SG_ERR_INVALID;
    }
    CUtensorMap ta, tb;
    sg_status rc = map_2d(&ta, A, (uint64_t)K, (uint64_t)M, (uint64_t)lda, 64, 128, "A");
    if (rc != SG_OK)
        return rc;
    rc = map_2d(&tb, B, (uint64_t)K, (uint64_t)N, (uint64_t)ldb, 64, 128, "B");
    if (rc != SG_OK)
        return rc;
    ArgmaxArgs a;
    a.best_idx = best_idx;
    a.best_val = best_val;
    a.M = M;
    a.N = N;
    a.K = K;
    a.status = status;
    const size_t smem = (size_t)kGS * 2 * kTileBytes + 1024;
    SG_TRY_CUDA(cudaFuncSetAttribute(k_gemm_argmax, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    k_gemm_argmax<<<(unsigned)((M + 127) / 128), kGThreads, smem, st>>>(ta, tb, a);
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}

sg_status gemm_group_abs(const uint16_t *A, int64_t lda, int M, const uint16_t *B, int64_t ldb, int N, int K, int G,
                         float *out, int32_t *status, cudaStream_t st)
{
    if (M < 1 || N < 1 || K < 1)
        return SG_OK;
    if (G < 1 || G > 128 || (G & (G - 1)) != 0 || M % G != 0) {
        sg_set_error("group |.|-sum GEMM: G must be a power of two <= 128 dividing M (G=%d M=%d)", G, M);
        return SG_ERR_UNSUPPORTED;
    }
    CUtensorMap ta, tb;
    sg_status rc = map_2d(&ta, A, (uint64_t)M, (uint64_t)K, (uint64_t)lda, 64, 64, "A");
    if (rc != SG_OK)
        return rc;
    rc = map_2d(&tb, B, (uint64_t)N, (uint64_t)K, (uint64_t)ldb, 64, 64, "B");
    if (rc != SG_OK)
        return rc;
    // stages: no more than the K blocks (with few of them, several CTAs share an SM)
    const int nkb = (K + 63) / 64;
    const int NS = nkb < kGS ? nkb : kGS;
    const size_t smem = (size_t)NS * 2 * kTileBytes + 1024;
    SG_TRY_CUDA(cudaFuncSetAttribute(k_gemm_gabs, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    dim3 grid((unsigned)((N + 127) / 128), (unsigned)((M + 127) / 128));
    k_gemm_gabs<<<grid, kGThreads, smem, st>>>(ta, tb, out, M, N, K, G, NS, status);
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}

sg_status split_hilo(const float *x, int64_t n, uint16_t *hi, uint16_t *lo, cudaStream_t st)
{
    if (n <= 0)
        return SG_OK;
    int64_t blocks = ceil_div(n, 256);
    if (blocks > 4096)
        blocks = 4096;
    k_split_hilo<<<(int)blocks, 256, 0, st>>>(x, n, hi, lo);
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}
