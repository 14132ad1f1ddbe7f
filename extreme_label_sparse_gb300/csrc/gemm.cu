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

// ---------------------------------------------------------------- group |.|-sum GEMM, label-streaming form
// The same sums with the product transposed: out[l / G][m] = sum over the G
// labels l of a group of |sum_k A[m][k] B[l][k]|, A (M <= a few hundred rows,
// MN-major) resident in shared memory, B (the long label side, MN-major)
// streamed in chunks of NW = 256 (or 128) labels.  The accumulator's lanes
// are A's rows and its columns the chunk's labels, so a group's sum runs
// along one thread's registers (no shuffles) and 32 lanes store 32
// consecutive outputs.  CTA (mt, r): rows [128 mt, 128 mt + 128), chunks of
// label range r; the CTAs of one range follow each other's chunks closely,
// so each chunk comes from HBM once and from L2 to the other row tiles.
struct GabsTCtl {
    uint64_t full[4], empty[4];
    uint64_t afull, tfull[2], tempty[2], drain;
    uint32_t tmem;
    int abort_flag;
};

struct GabsTArgs {
    float *out;
    int32_t M, L, K, G, NW, S, nkb, mtiles;
    int64_t nchunks;
    int32_t *status;
};

template <int NW>
__global__ void __launch_bounds__(kGThreads, 1)
    k_gemm_gabs_t(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                  const GabsTArgs a)
{
    __shared__ GabsTCtl c;
    extern __shared__ uint8_t dsm[];
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const uint32_t base = (smem_u32(dsm) + 1023u) & ~1023u;
    const int mt = blockIdx.x % a.mtiles;
    const int r = blockIdx.x / a.mtiles;
    const int nr = gridDim.x / a.mtiles;
    const int64_t c0 = a.nchunks * r / nr, c1 = a.nchunks * (r + 1) / nr;  // this CTA's chunks
    const int m0 = mt * 128;
    const int S = a.S, nkb = a.nkb;
    constexpr uint32_t kChunkTile = (uint32_t)NW * 128;  // one K block of a chunk: NW labels x 64 k
    const uint32_t stage0 = base + (uint32_t)nkb * kTileBytes;  // A: nkb tiles of 128 rows x 64 k
    const uint32_t stage_bytes = (uint32_t)nkb * kChunkTile;
    if (threadIdx.x == 0) {
        c.abort_flag = 0;
        for (int i = 0; i < S; ++i) {
            mbar_init(bar_of(c.full[i]), 1);
            mbar_init(bar_of(c.empty[i]), 1);
        }
        mbar_init(bar_of(c.afull), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_of(c.tfull[i]), 1);
            mbar_init(bar_of(c.tempty[i]), 128);
        }
        mbar_init(bar_of(c.drain), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&c.tmem), 2 * NW);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = c.tmem;
    volatile int *abort_flag = &c.abort_flag;

    if (warp == 0) {
        // ---------------------------------------------------------- loads
        if (lane == 0) {
            mbar_arrive_expect_tx(bar_of(c.afull), (uint32_t)nkb * kTileBytes);
            for (int kb = 0; kb < nkb; ++kb)
                load_tile(base + (uint32_t)kb * kTileBytes, &tm_a, 1, m0, kb * 64, bar_of(c.afull));
            Ring rs;
            int64_t ch = c0;
            for (; ch < c1; ++ch, rs.next(S)) {
                if (!mbar_wait(bar_of(c.empty[rs.i]), rs.ph ^ 1u, abort_flag, a.status))
                    break;
                const uint32_t st = stage0 + (uint32_t)rs.i * stage_bytes;
                mbar_arrive_expect_tx(bar_of(c.full[rs.i]), stage_bytes);
                for (int kb = 0; kb < nkb; ++kb)
                    for (int q = 0; q < NW / 64; ++q)
                        tma_load_2d(st + (uint32_t)kb * kChunkTile + (uint32_t)q * (kTileBytes / 2), &tm_b,
                                    (int)(ch * NW) + 64 * q, kb * 64, bar_of(c.full[rs.i]));
            }
            // winding down after an abort: the loads in flight land first
            mbar_wait_drain(bar_of(c.afull), 0);
            if (*abort_flag) {
                Ring rd;
                for (int64_t j = c0; j < ch; ++j, rd.next(S))
                    if (j + S >= ch)
                        mbar_wait_drain(bar_of(c.full[rd.i]), rd.ph);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA
        // D[128 rows][NW labels] += A (MN-major, 128 rows) x B (MN-major, NW labels)
        const uint32_t idesc = idesc_bf16(128, NW, 1, 1);
        bool ok = __all_sync(0xffffffffu, mbar_wait(bar_of(c.afull), 0, abort_flag, a.status));
        Ring rs;
        int acc = 0;
        uint32_t aph = 0;
        for (int64_t ch = c0; ok && ch < c1; ++ch, rs.next(S)) {
            if (!__all_sync(0xffffffffu, mbar_wait(bar_of(c.tempty[acc]), aph ^ 1u, abort_flag, a.status)))
                break;
            if (!__all_sync(0xffffffffu, mbar_wait(bar_of(c.full[rs.i]), rs.ph, abort_flag, a.status)))
                break;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t st = stage0 + (uint32_t)rs.i * stage_bytes;
                const uint32_t d = tbase + (uint32_t)(acc * NW);
                for (int kb = 0; kb < nkb; ++kb) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16(d, tile_desc(base + (uint32_t)kb * kTileBytes, 1, ks),
                                 sdesc(st + (uint32_t)kb * kChunkTile + (uint32_t)ks * 2048, kTileBytes / 2, 1024,
                                       kLayoutSW128),
                                 idesc, (kb > 0 || ks > 0) ? 1u : 0u);
                }
                mma_commit(bar_of(c.empty[rs.i]));
                mma_commit(bar_of(c.tfull[acc]));
            }
            __syncwarp();
            if (++acc == 2) {
                acc = 0;
                aph ^= 1u;
            }
        }
        if (lane == 0)
            mma_commit(bar_of(c.drain));
        __syncwarp();
        mbar_wait_drain(bar_of(c.drain), 0);
    } else {
        // ---------------------------------------------------------- epilogue
        // warp w reads TMEM lanes 32 (w % 4) .. (its A rows); a group of G
        // labels is G consecutive columns of the accumulator
        const int q = warp & 3;
        const int m = m0 + q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const int64_t K = a.L / a.G;  // groups
        int acc = 0;
        uint32_t aph = 0;
        for (int64_t ch = c0; ch < c1; ++ch) {
            if (!__all_sync(0xffffffffu, mbar_wait(bar_of(c.tfull[acc]), aph, abort_flag, a.status)))
                break;
            tc_fence_after();
            // 128 columns per round: four loads in flight, one wait (a
            // load-wait pair per 32 columns left the epilogue the slowest
            // role); |.| summed in four independent chains
            float sum = 0.f;
            for (int cb = 0; cb < NW; cb += 128) {
                uint32_t v[4][32];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    tmem_ld32(tbase + lane_off + (uint32_t)(acc * NW + cb + 32 * j), v[j]);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int cc = cb + 32 * j;
                    if (a.G >= 32) {
                        float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
                        for (int x = 0; x < 32; x += 4) {
                            p0 += fabsf(__uint_as_float(v[j][x]));
                            p1 += fabsf(__uint_as_float(v[j][x + 1]));
                            p2 += fabsf(__uint_as_float(v[j][x + 2]));
                            p3 += fabsf(__uint_as_float(v[j][x + 3]));
                        }
                        sum += (p0 + p1) + (p2 + p3);
                        if (((cc + 32) & (a.G - 1)) == 0) {  // the group ends here
                            const int64_t k = (ch * NW + cc + 32) / a.G - 1;
                            if (k < K && m < a.M)
                                a.out[k * a.M + m] = sum;
                            sum = 0.f;
                        }
                    } else {  // G = 16: two groups per 32 columns
                        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
                        for (int x = 0; x < 16; x += 2) {
                            s0 += fabsf(__uint_as_float(v[j][x]));
                            s1 += fabsf(__uint_as_float(v[j][x + 1]));
                            s2 += fabsf(__uint_as_float(v[j][x + 16]));
                            s3 += fabsf(__uint_as_float(v[j][x + 17]));
                        }
                        const int64_t k = (ch * NW + cc) / 16;
                        if (m < a.M) {
                            if (k < K)
                                a.out[k * a.M + m] = s0 + s1;
                            if (k + 1 < K)
                                a.out[(k + 1) * a.M + m] = s2 + s3;
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar_of(c.tempty[acc]));
            if (++acc == 2) {
                acc = 0;
                aph ^= 1u;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 2 * NW);
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

// out[l / G][m] = sum over the G labels l of a group of |sum_k A[m][k] B[l][k]|
// (A: M x K MN-major, leading dimension lda; B: L x K MN-major, ldb), with
// G in {16, 32, 64, 128, 256} dividing L and K <= 256.  Returns
// SG_ERR_UNSUPPORTED for other shapes (the caller then takes gemm_group_abs).
sg_status gemm_group_abs_t(const uint16_t *A, int64_t lda, int M, const uint16_t *B, int64_t ldb, int64_t L, int K,
                           int G, float *out, int num_sms, int32_t *status, cudaStream_t st)
{
    if (M < 1 || L < 1 || K < 1)
        return SG_OK;
    if (G < 16 || G > 256 || (G & (G - 1)) != 0 || L % G != 0 || K > 256) {
        sg_set_error("label-streaming group |.|-sum GEMM: G in 16..256 a power of two dividing L, K <= 256");
        return SG_ERR_UNSUPPORTED;
    }
    const int nkb = (K + 63) / 64;
    // stages of NW labels x K: 256 labels while three stages fit, else 128
    const long budget = 227l * 1024 - 1024 - (long)nkb * kTileBytes;
    int NW = 256;
    int S = (int)(budget / ((long)nkb * NW * 128));
    if (S < 3) {
        NW = 128;
        S = (int)(budget / ((long)nkb * NW * 128));
    }
    if (S > 4)
        S = 4;
    if (S < 2 || G > NW) {
        sg_set_error("label-streaming group |.|-sum GEMM: no room for two stages of whole groups (K=%d G=%d)", K, G);
        return SG_ERR_UNSUPPORTED;
    }
    CUtensorMap ta, tb;
    sg_status rc = map_2d(&ta, A, (uint64_t)M, (uint64_t)K, (uint64_t)lda, 64, 64, "A");
    if (rc != SG_OK)
        return rc;
    rc = map_2d(&tb, B, (uint64_t)L, (uint64_t)K, (uint64_t)ldb, 64, 64, "B");
    if (rc != SG_OK)
        return rc;
    GabsTArgs a;
    a.out = out;
    a.M = M;
    a.L = (int32_t)L;
    a.K = K;
    a.G = G;
    a.NW = NW;
    a.S = S;
    a.nkb = nkb;
    a.mtiles = (M + 127) / 128;
    a.nchunks = (L + NW - 1) / NW;
    a.status = status;
    if (L > INT32_MAX) {
        sg_set_error("label-streaming group |.|-sum GEMM: L must fit 31 bits");
        return SG_ERR_UNSUPPORTED;
    }
    // ranges of chunks: the row tiles of one range run side by side
    int64_t ranges = num_sms / a.mtiles;
    if (ranges < 1)
        ranges = 1;
    if (ranges > a.nchunks)
        ranges = a.nchunks;
    const size_t smem = (size_t)nkb * kTileBytes + (size_t)S * nkb * NW * 128 + 1024;
    void (*kern)(CUtensorMap, CUtensorMap, GabsTArgs) = NW == 256 ? k_gemm_gabs_t<256> : k_gemm_gabs_t<128>;
    SG_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    kern<<<(unsigned)(ranges * a.mtiles), kGThreads, smem, st>>>(ta, tb, a);
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
