// The whole training step of the layer in one persistent kernel on clusters
// of C CTAs (sm_103a).  HASTE, key design "gather-once + dense MMA kernel":
// per group k the CTA that owns it
//   gathers H_k = h[:, I_k] once (cp.async of rows of the transposed h),
//   Z_k    = H_k W_k^T                (tcgen05, M = samples, N = G, K = F)
//   dZ_k   = sigmoid(Z_k) - Y_k       (BCE from TMEM, loss partials)
//   dW_k^T = H_k^T [dZ_hi | dZ_lo]    (tcgen05, M = F, N = 2G, K = samples)
// and every CTA of the cluster adds the group's feature gradient to its own
// band of dh columns, which stays in TMEM for the whole kernel:
//   dh[:, band] += dZ_k Ws_k,  Ws_k[j][i - i0] = W_k[j][f] where I_k[f] = i
// (the scatter-add into the columns I_k written as a product with W_k
// scattered into the band's rows; Split-K over groups kept on chip).  W_k is
// read from HBM once per step and dZ never leaves the chip: the owner writes
// its fp16 dZ tile into its shared memory and the other CTAs of the cluster
// copy it with distributed-shared-memory loads.
//
// A cluster works through "steps" of C consecutive groups (CTA r owns group
// C*step + r); every CTA loads the W_k and I_k of all C groups of a step (the
// other CTAs' rows come from L2: the owner loads them at the same time).
//
// Precision inside the step: dW takes dZ as two bf16 planes (value and
// rounding residual) against the bf16 H_k; dh takes dZ as one fp16 plane
// against W_k in fp16.  A group whose W_k holds a value of magnitude >= 2^15
// in a CTA's band (beyond what fp16 keeps exactly) adds that band's
// contribution with fp32 CUDA-core arithmetic and atomics instead.
//
// Shared memory (from a 1024-byte aligned base):
//   [S stages: H_k (2 sample chunks x F rows x 128 B, 128-byte swizzle),
//              W of the C groups (TMA boxes of CW columns x G rows),
//              I of the C groups]
//   [2 x dZ bf16 value + residual planes (dW operand)]
//   [2 x C fp16 dZ tiles (dh operand): slot g holds group C*step + g]
//   [2 x Ws (band rows of 2G bytes)]
// TMEM: dh band [0, BW), Z slots [BW, BW + 2G), dW slot [BW + 2G, BW + 4G).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "sg_internal.cuh"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

using namespace tc;

namespace {

constexpr int kP = 4;     // producer warps
constexpr int kBce = 8;   // BCE warps: two per TMEM lane quarter
constexpr int kDw = 4;    // dW store + tile copy warps: one per lane quarter
constexpr int kBld = 4;   // Ws builder warps: one thread per feature f
constexpr int kWA = kP;   // forward and dW MMA warp
constexpr int kWB = kP + 1;  // dh MMA warp
constexpr int kW0Bce = kP + 2;
constexpr int kW0Dw = kW0Bce + kBce;
constexpr int kW0Bld = kW0Dw + kDw;
constexpr int kWarps = kW0Bld + kBld;
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxC = 4;
constexpr int kMaxS = 4;
constexpr int kMaxF = 128;
// dynamic shared memory the plan may use (the opt-in maximum is 227 KB,
// less the static control block)
constexpr int kSmemBudget = 227 * 1024 - 1024;
// named barriers
constexpr int kBarBce = 1, kBarDw = 2, kBarBld = 3;

struct StepCtl {
    uint64_t full[kMaxS], empty[kMaxS];
    uint64_t zfull[2], zempty[2];      // Z slots
    uint64_t dzwfull[2], dzwempty[2];  // dZ bf16 planes (dW operand)
    uint64_t wfull, wempty;            // dW slot
    uint64_t dzhfull[2];               // the step's fp16 tiles are all in place
    uint64_t dzhdone[2];               // the local dh MMAs are done with them
    uint64_t dzready[2];               // the other CTAs wrote their tiles (cluster)
    uint64_t dzcopied[2];              // the other CTAs copied this CTA's tile (cluster)
    uint64_t wsfull[2], wsempty[2];    // Ws buffers
    uint64_t drainA, drainB;
    uint32_t tmem;
    int abort_flag;
    double red[kBce];
};

struct StepArgs {
    const uint16_t *idx_s, *hT;
    uint16_t *dW;
    float *dh;
    const int32_t *gptr, *gent;
    double *loss_part;
    int32_t *status;
    int64_t K, NPS;  // groups; steps of C groups
    int32_t B, F, H, ldB, C, BW, S, CW, nbc;
    uint32_t h_bytes, w_bytes, i_bytes, stage_bytes, dzw_bytes, ws_bytes;
    uint32_t off_dzw, off_dzh, off_ws;
};

__device__ __forceinline__ uint32_t bar_addr(const uint64_t &b) { return smem_u32(&b); }

// a bounded wait whose outcome every lane of the warp shares (the warp then
// takes the same branch around .sync.aligned TMEM accesses and __syncwarp)
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag, int32_t *status)
{
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, status));
}

template <int G_>
__global__ void __launch_bounds__(kThreads, 1) k_tc_step(const __grid_constant__ CUtensorMap tm_w, const StepArgs a)
{
    constexpr int G = G_;
    constexpr int ZSW = 2 * G >= 128 ? 128 : 2 * G;  // bytes of a dZ row
    constexpr uint32_t ZCH = 128u * ZSW;              // one dZ plane (128 sample rows)
    constexpr int RB = 2 * G;                         // bytes of a Ws row
    constexpr int CHB = G / 2;                        // BCE columns per warp
    constexpr int DCH = G < 32 ? G : 32;              // dW columns per TMEM load
    __shared__ StepCtl c;
    extern __shared__ uint8_t dsm[];
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const uint32_t base = (smem_u32(dsm) + 1023u) & ~1023u;
    uint8_t *bp = dsm + (base - smem_u32(dsm));
    const int C = a.C, S = a.S, BW = a.BW, F = a.F, CW = a.CW;
    const uint32_t WCH = (uint32_t)G * CW * 2;  // bytes of one TMA box of W
    const uint32_t rank = cluster_rank();
    const int64_t cl = cluster_index(), ncl = cluster_count();
    const int i0 = (int)rank * BW;  // first dh column of this CTA's band
    const uint32_t col_z = (uint32_t)BW, col_w = (uint32_t)BW + 2 * G;

    if (threadIdx.x == 0) {
        c.abort_flag = 0;
        for (int s = 0; s < S && s < kMaxS; ++s) {
            mbar_init(bar_addr(c.full[s]), kP * 32 + 1);
            mbar_init(bar_addr(c.empty[s]), 2);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_addr(c.zfull[i]), 1);
            mbar_init(bar_addr(c.zempty[i]), kBce * 32);
            mbar_init(bar_addr(c.dzwfull[i]), kBce * 32);
            mbar_init(bar_addr(c.dzwempty[i]), 1);
            mbar_init(bar_addr(c.dzhfull[i]), C > 1 ? 2 : 1);
            mbar_init(bar_addr(c.dzhdone[i]), 1);
            mbar_init(bar_addr(c.dzready[i]), C > 1 ? C - 1 : 1);
            mbar_init(bar_addr(c.dzcopied[i]), C > 1 ? C - 1 : 1);
            mbar_init(bar_addr(c.wsfull[i]), 1);
            mbar_init(bar_addr(c.wsempty[i]), 1);
        }
        mbar_init(bar_addr(c.wfull), 1);
        mbar_init(bar_addr(c.wempty), kDw * 32);
        mbar_init(bar_addr(c.drainA), 1);
        mbar_init(bar_addr(c.drainB), 1);
        fence_mbar_init();
    }
    if (warp == kWA) {
        tmem_alloc(smem_u32(&c.tmem), 512);
        tmem_relinquish();
    }
    // the Ws buffers start zeroed; the builders rewrite only the rows they use
    for (uint32_t o = threadIdx.x * 16u; o < 2 * a.ws_bytes; o += kThreads * 16u)
        *reinterpret_cast<uint4 *>(bp + a.off_ws + o) = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // every CTA's barriers exist before another CTA arrives on them
    tc_fence_after();
    const uint32_t tbase = c.tmem;
    volatile int *abort_flag = &c.abort_flag;

    if (warp < kP) {
        // ---------------------------------------------------------- producers
        // per step: W_k and I_k of every group of the step (TMA / bulk copies,
        // thread 0), and the own group's H_k by cp.async: producer warp pw
        // copies rows [pw RW, pw RW + RW) of H_k, two 256-byte hT rows per
        // instruction (16 lanes each; only the first chunk of 64 samples
        // when B <= 64)
        const int t = threadIdx.x;
        const int RW = F / kP;
        const int u = lane & 15, rsub = lane >> 4;
        const int ulim = a.nbc * 8;  // 16-byte units per row that are copied
        int it = 0;
        for (int64_t ps = cl; ps < a.NPS; ps += ncl, ++it) {
            const int s = it % S;
            const uint32_t ph = (uint32_t)(it / S) & 1u;
            const int64_t k0 = ps * C;
            const int ng = (int)(a.K - k0 < C ? a.K - k0 : C);
            const bool own = (int)rank < ng;
            uint32_t myrow = 0;
            if (own && lane < RW)
                myrow = __ldg(a.idx_s + (k0 + rank) * F + warp * RW + lane);
            if (!mbar_wait(bar_addr(c.empty[s]), ph ^ 1u, abort_flag, a.status))
                break;
            const uint32_t st = base + (uint32_t)s * a.stage_bytes;
            const uint32_t fb = bar_addr(c.full[s]);
            if (t == 0) {
                mbar_arrive_expect_tx(fb, (uint32_t)ng * (a.w_bytes + 2u * F));
                for (int g = 0; g < ng; ++g) {
                    const uint32_t wd = st + a.h_bytes + (uint32_t)g * a.w_bytes;
                    for (int ch = 0; ch * CW < F; ++ch)
                        tma_load_2d(wd + (uint32_t)ch * WCH, &tm_w, ch * CW, (int)((k0 + g) * G), fb);
                    bulk_load(st + a.h_bytes + (uint32_t)C * a.w_bytes + (uint32_t)g * a.i_bytes,
                              a.idx_s + (k0 + g) * F, 2u * F, fb);
                }
            }
            if (own) {  // warp-uniform: every lane takes part in the shuffles
                for (int r0 = 0; r0 < RW; r0 += 2) {
                    const int rr = r0 + rsub;
                    const uint32_t row = __shfl_sync(0xffffffffu, myrow, rr & 31);
                    const int f = warp * RW + rr;
                    if (u < ulim)
                        cp_async16(st + (uint32_t)(u >> 3) * F * 128 + (uint32_t)f * 128 +
                                       (uint32_t)(((u & 7) ^ (f & 7)) << 4),
                                   a.hT + (size_t)row * a.ldB + u * 8);
                }
            }
            cp_async_arrive_noinc(fb);
        }
        cp_async_wait_all();
        if (*abort_flag)
            for (int j = it - S < 0 ? 0 : it - S; j < it; ++j)
                mbar_wait_drain(bar_addr(c.full[j % S]), (uint32_t)(j / S) & 1u);
    } else if (warp == kWA) {
        // ---------------------------------------------------------- forward + dW MMA
        // the forward of a step's group is issued before the dW of the previous
        // one, so the BCE warps find the next Z ready when they finish a group
        const uint32_t idf = idesc_bf16(128, G, 1, 0);
        const uint32_t idw = idesc_bf16(128, 2 * G, 0, 1);
        const uint32_t wlay = layout_for_swizzle(2 * CW);
        const uint32_t zlay = layout_for_swizzle(ZSW);
        const int kb = a.nbc * 4;  // K steps of 16 samples of the dW MMA
        int it = 0, io = 0, prev_s = 0;
        bool ok = true;
        auto issue_dw = [&](int j, int s) -> bool {
            const int db = j & 1;
            if (!warp_wait(bar_addr(c.dzwfull[db]), (uint32_t)(j >> 1) & 1u, abort_flag, a.status))
                return false;
            if (!warp_wait(bar_addr(c.wempty), ((uint32_t)j & 1u) ^ 1u, abort_flag, a.status))
                return false;
            tc_fence_after();
            fence_proxy_async();
            if (lane == 0) {
                const uint32_t A = base + (uint32_t)s * a.stage_bytes;
                const uint32_t Zs = base + a.off_dzw + (uint32_t)db * a.dzw_bytes;
                for (int st = 0; st < kb; ++st) {
                    // A: H_k^T, K-major (rows f, K = samples): sample chunk st/4, 32 B per 16 samples
                    const uint64_t ad = sdesc(A + (uint32_t)(st >> 2) * F * 128 + (uint32_t)(st & 3) * 32, 16, 1024,
                                              kLayoutSW128);
                    // B: [hi | lo] dZ_k, MN-major (N = j, K = samples), the lo plane ZCH further on
                    const uint64_t bd = sdesc(Zs + (uint32_t)st * 16 * ZSW, ZCH, 8 * ZSW, zlay);
                    mma_bf16(tbase + col_w, ad, bd, idw, st > 0 ? 1u : 0u);
                }
                mma_commit(bar_addr(c.wfull));
                mma_commit(bar_addr(c.dzwempty[db]));
                mma_commit(bar_addr(c.empty[s]));  // last reader of H_k (and, earlier, of W_k)
            }
            __syncwarp();
            return true;
        };
        for (int64_t ps = cl; ps < a.NPS; ps += ncl, ++it) {
            const int s = it % S;
            const int ng = (int)(a.K - ps * C < C ? a.K - ps * C : C);
            if (!warp_wait(bar_addr(c.full[s]), (uint32_t)(it / S) & 1u, abort_flag, a.status)) {
                ok = false;
                break;
            }
            if ((int)rank >= ng) {  // no own group: the stage only carries the others' W_k
                if (lane == 0)
                    mbar_arrive(bar_addr(c.empty[s]));
                __syncwarp();
                continue;
            }
            const int zs = io & 1;
            if (!warp_wait(bar_addr(c.zempty[zs]), ((uint32_t)(io >> 1) & 1u) ^ 1u, abort_flag, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            fence_proxy_async();  // cp.async-written H_k -> the MMA (async proxy)
            if (lane == 0) {
                const uint32_t A = base + (uint32_t)s * a.stage_bytes;
                const uint32_t Wt = A + a.h_bytes + rank * a.w_bytes;
                for (int st = 0; st < F / 16; ++st) {
                    // A: H_k, MN-major (M = samples); 8 f rows per 1024-byte atom
                    const uint64_t ad = sdesc(A + (uint32_t)st * 2048, (uint32_t)F * 128, 1024, kLayoutSW128);
                    // B: W_k, K-major; box st*16/CW, 32 bytes per 16 f inside a 2 CW-byte row
                    const int f0 = st * 16;
                    const uint64_t bd = sdesc(Wt + (uint32_t)(f0 / CW) * WCH + (uint32_t)(f0 % CW) * 2, 16,
                                              8 * 2 * CW, wlay);
                    mma_bf16(tbase + col_z + (uint32_t)(zs * G), ad, bd, idf, st > 0 ? 1u : 0u);
                }
                mma_commit(bar_addr(c.zfull[zs]));
            }
            __syncwarp();
            if (io > 0 && !issue_dw(io - 1, prev_s)) {
                ok = false;
                break;
            }
            prev_s = s;
            ++io;
        }
        if (ok && io > 0)
            issue_dw(io - 1, prev_s);
        if (lane == 0)
            mma_commit(bar_addr(c.drainA));
        __syncwarp();
        mbar_wait_drain(bar_addr(c.drainA), 0);
    } else if (warp == kWB) {
        // ---------------------------------------------------------- dh MMA
        // A: a group's fp16 dZ tile (K-major, rows = samples); B: Ws (K-major,
        // rows = the band's dh columns); accumulated in TMEM over every group
        const uint64_t adesc0 = sdesc(0, 16, 8 * ZSW, layout_for_swizzle(ZSW));
        const uint64_t bdesc0 = sdesc(0, 16, 8 * RB, layout_for_swizzle(RB));
        const int n0 = BW > 256 ? 256 : BW, n1 = BW - n0;
        const uint32_t id0 = idesc_f16(128, n0, 0, 0);
        const uint32_t id1 = idesc_f16(128, n1 > 0 ? n1 : 16, 0, 0);
        int it = 0, gi = 0;
        uint32_t accf = 0;
        bool ok = true;
        for (int64_t ps = cl; ps < a.NPS && ok; ps += ncl, ++it) {
            const int db = it & 1;
            const int ng = (int)(a.K - ps * C < C ? a.K - ps * C : C);
            if (!warp_wait(bar_addr(c.dzhfull[db]), (uint32_t)(it >> 1) & 1u, abort_flag, a.status))
                break;
            for (int g = 0; g < ng; ++g, ++gi) {
                const int wb = gi & 1;
                if (!warp_wait(bar_addr(c.wsfull[wb]), (uint32_t)(gi >> 1) & 1u, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t au = adesc0 + (uint64_t)((base + a.off_dzh + (uint32_t)(db * C + g) * ZCH) >> 4);
                    const uint64_t bu = bdesc0 + (uint64_t)((base + a.off_ws + (uint32_t)wb * a.ws_bytes) >> 4);
                    for (int ks = 0; ks < G / 16; ++ks) {
                        mma_bf16(tbase, au + (uint64_t)((ks * 32) >> 4), bu + (uint64_t)((ks * 32) >> 4), id0, accf);
                        if (n1 > 0)
                            mma_bf16(tbase + (uint32_t)n0, au + (uint64_t)((ks * 32) >> 4),
                                     bu + (uint64_t)((ks * 32 + n0 * RB) >> 4), id1, accf);
                        accf = 1u;
                    }
                    mma_commit(bar_addr(c.wsempty[wb]));
                }
                __syncwarp();
            }
            if (!ok)
                break;
            if (lane == 0)
                mma_commit(bar_addr(c.dzhdone[db]));
            __syncwarp();
        }
        if (lane == 0)
            mma_commit(bar_addr(c.drainB));
        __syncwarp();
        mbar_wait_drain(bar_addr(c.drainB), 0);
    } else if (warp < kW0Dw) {
        // ---------------------------------------------------------- BCE
        const int q = warp & 3;
        const int sub = (warp - kW0Bce) >> 2;
        const int b = q * 32 + lane;  // sample row of this thread
        const int c0 = sub * CHB;     // first column of this warp
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        double lacc = 0.0;
        int it = 0, io = 0;
        for (int64_t ps = cl; ps < a.NPS; ps += ncl, ++it) {
            const int db = it & 1;
            const uint32_t dph = (uint32_t)(it >> 1) & 1u;
            const int64_t k = ps * C + rank;
            const bool own = k < a.K;
            bool ok = true;
            if (own) {
                const int zs = io & 1;
                const int e0 = __ldg(a.gptr + k), e1 = __ldg(a.gptr + k + 1);
                float v[CHB];
                ok = warp_wait(bar_addr(c.zfull[zs]), (uint32_t)(io >> 1) & 1u, abort_flag, a.status);
                if (ok) {
                    tc_fence_after();
                    tmem_ld_chunk<CHB>(tbase + lane_off + col_z + (uint32_t)(zs * G + c0), v);
                    tc_fence_before();
                    mbar_arrive(bar_addr(c.zempty[zs]));
                    if (b < a.B) {
                        const uint32_t y = e1 > e0 ? group_pos_mask(a.gent, e0, e1, b, c0, CHB) : 0u;
                        lacc += bce_chunk<CHB>(v, y);
                    } else {
#pragma unroll
                        for (int i = 0; i < CHB; ++i)
                            v[i] = 0.f;
                    }
                }
                const int dbw = io & 1;
                ok = ok && mbar_wait(bar_addr(c.dzwempty[dbw]), ((uint32_t)(io >> 1) & 1u) ^ 1u, abort_flag, a.status);
                if (ok) {
                    store_dz_tile<CHB>(bp + a.off_dzw + (size_t)dbw * a.dzw_bytes, b, c0, v, ZSW, 1, 128);
                    fence_proxy_async();
                    mbar_arrive(bar_addr(c.dzwfull[dbw]));
                }
                // the own fp16 tile: once the local dh MMAs and the other CTAs'
                // copies of this buffer's previous step are done
                ok = ok && mbar_wait(bar_addr(c.dzhdone[db]), dph ^ 1u, abort_flag, a.status);
                ok = ok && (C == 1 || mbar_wait_cluster(bar_addr(c.dzcopied[db]), dph ^ 1u, abort_flag, a.status));
                if (ok) {
                    store_dz_tile_f16<CHB>(bp + a.off_dzh + (size_t)(db * C + (int)rank) * ZCH, b, c0, v, ZSW, 128);
                    fence_proxy_async();
                }
                ++io;
            } else {
                // nothing to write; still wait for the buffer's previous step so
                // that the arrivals below count toward this step's phase
                ok = mbar_wait(bar_addr(c.dzhdone[db]), dph ^ 1u, abort_flag, a.status);
                ok = ok && (C == 1 || mbar_wait_cluster(bar_addr(c.dzcopied[db]), dph ^ 1u, abort_flag, a.status));
            }
            if (named_bar_any(kBarBce, kBce * 32, !ok))
                break;
            if (threadIdx.x == kW0Bce * 32) {
                fence_acq_rel_cluster();
                mbar_arrive(bar_addr(c.dzhfull[db]));
                for (int p = 0; p < C; ++p)
                    if (p != (int)rank)
                        mbar_arrive_remote(mapa(bar_addr(c.dzready[db]), (uint32_t)p));
            }
        }
        // loss partial of the CTA (fixed order)
        double v = lacc;
        for (int o = 16; o > 0; o >>= 1)
            v += __shfl_down_sync(0xffffffffu, v, o);
        if (lane == 0)
            c.red[warp - kW0Bce] = v;
        named_bar(kBarBce, kBce * 32);
        if (threadIdx.x == kW0Bce * 32) {
            double sum = 0.0;
            for (int i = 0; i < kBce; ++i)
                sum += c.red[i];
            a.loss_part[blockIdx.x] = sum;
        }
        // the band's partial of dh (lanes = samples, columns = dh columns
        // i0 ..) added into dh once, after the last dh MMA
        if (__all_sync(0xffffffffu, mbar_wait(bar_addr(c.drainB), 0, abort_flag, a.status) && !*abort_flag) &&
            it > 0) {
            tc_fence_after();
            const int half = BW / 2;
            const bool vec = (a.H & 3) == 0;
            float *drow = a.dh + (size_t)b * a.H;
            for (int cc = sub * half; cc < sub * half + half; cc += 32) {
                uint32_t rr[32];
                tmem_ld32(tbase + lane_off + (uint32_t)cc, rr);
                tmem_ld_wait();
                if (b >= a.B)
                    continue;
                const int ib = i0 + cc;
#pragma unroll
                for (int x = 0; x < 32; x += 4) {
                    const int i = ib + x;
                    if (vec && i + 3 < a.H) {
                        red_add_v4(drow + i, __uint_as_float(rr[x]), __uint_as_float(rr[x + 1]),
                                   __uint_as_float(rr[x + 2]), __uint_as_float(rr[x + 3]));
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (i + e < a.H)
                                atomicAdd(drow + i + e, __uint_as_float(rr[x + e]));
                    }
                }
            }
        }
    } else if (warp < kW0Bld) {
        // ---------------------------------------------------------- tile copies + dW
        const int q = warp & 3;
        const int f = q * 32 + lane;  // lane of the dW^T accumulator
        const int tt = threadIdx.x - kW0Dw * 32;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        int it = 0, io = 0;
        for (int64_t ps = cl; ps < a.NPS; ps += ncl, ++it) {
            const int db = it & 1;
            const uint32_t dph = (uint32_t)(it >> 1) & 1u;
            const int64_t k0 = ps * C;
            const int ng = (int)(a.K - k0 < C ? a.K - k0 : C);
            bool ok = true;
            if (C > 1) {
                // the other CTAs' fp16 tiles of this step into the local buffer
                ok = mbar_wait_cluster(bar_addr(c.dzready[db]), dph, abort_flag, a.status);
                ok = ok && mbar_wait(bar_addr(c.dzhdone[db]), dph ^ 1u, abort_flag, a.status);
                if (ok) {
                    for (int p = 0; p < ng; ++p) {
                        if (p == (int)rank)
                            continue;
                        const uint32_t off = a.off_dzh + (uint32_t)(db * C + p) * ZCH;
                        const uint32_t src = mapa(base + off, (uint32_t)p);
                        for (uint32_t o = (uint32_t)tt * 16u; o < ZCH; o += kDw * 32 * 16u)
                            *reinterpret_cast<uint4 *>(bp + off + o) = ld_dsmem16(src + o);
                    }
                    fence_proxy_async();
                }
                if (named_bar_any(kBarDw, kDw * 32, !ok))
                    break;
                if (tt == 0) {
                    mbar_arrive(bar_addr(c.dzhfull[db]));
                    for (int p = 0; p < C; ++p)
                        if (p != (int)rank)
                            mbar_arrive_remote(mapa(bar_addr(c.dzcopied[db]), (uint32_t)p));
                }
            }
            if ((int)rank < ng) {
                // dW_k^T accumulator [f][hi j | lo j] -> dW rows k G + j
                const int64_t k = k0 + rank;
                ok = mbar_wait(bar_addr(c.wfull), (uint32_t)io & 1u, abort_flag, a.status);
                if (named_bar_any(kBarDw, kDw * 32, !ok))
                    break;
                tc_fence_after();
#pragma unroll
                for (int cc = 0; cc < G; cc += DCH) {
                    float v[DCH], w[DCH];
                    tmem_ld_chunk2<DCH>(tbase + lane_off + col_w + (uint32_t)cc,
                                        tbase + lane_off + col_w + (uint32_t)(G + cc), v, w);
                    if (f < F) {
                        uint16_t *dst = a.dW + (k * G + cc) * F + f;
#pragma unroll
                        for (int i = 0; i < DCH; ++i)
                            dst[(int64_t)i * F] = bf16_rn(v[i] + w[i]);
                    }
                }
                tc_fence_before();
                mbar_arrive(bar_addr(c.wempty));
                ++io;
            }
        }
    } else {
        // ---------------------------------------------------------- Ws builders
        // thread f: if I_k[f] falls in the band, column f of W_k (fp16) becomes
        // row I_k[f] - i0 of the group's Ws buffer; the row it wrote there the
        // last time is zeroed first.  A group with |W| >= 2^15 in the band adds
        // its band's part of dh on CUDA cores instead (fp32, atomics).
        const int t = threadIdx.x - kW0Bld * 32;
        int prev[2] = {-1, -1};
        int it = 0, gi = 0;
        bool ok = true;
        for (int64_t ps = cl; ps < a.NPS && ok; ps += ncl, ++it) {
            const int s = it % S;
            const int db = it & 1;
            const uint32_t dph = (uint32_t)(it >> 1) & 1u;
            const int64_t k0 = ps * C;
            const int ng = (int)(a.K - k0 < C ? a.K - k0 : C);
            ok = mbar_wait(bar_addr(c.full[s]), (uint32_t)(it / S) & 1u, abort_flag, a.status);
            if (named_bar_any(kBarBld, kBld * 32, !ok))
                break;
            const uint8_t *st = bp + (size_t)s * a.stage_bytes;
            for (int g = 0; g < ng; ++g, ++gi) {
                const int wb = gi & 1;
                const uint8_t *Wg = st + a.h_bytes + (size_t)g * a.w_bytes;
                const uint16_t *Ig = reinterpret_cast<const uint16_t *>(st + a.h_bytes + (size_t)C * a.w_bytes +
                                                                         (size_t)g * a.i_bytes);
                int row = -1;
                bool big = false;
                uint32_t pk[G / 2];
                if (t < F) {
                    const int i = (int)Ig[t] - i0;
                    if (i >= 0 && i < BW) {
                        row = i;
                        // element (j, f) of the TMA box layout: box f / CW, row j,
                        // 16-byte unit ((f % CW) / 8) ^ swizzle(j), then f % 8
                        const int fc = t % CW;
                        const uint8_t *colp = Wg + (size_t)(t / CW) * WCH + (fc & 7) * 2;
#pragma unroll
                        for (int jj = 0; jj < G / 2; ++jj) {
                            const int j = 2 * jj;
                            const uint32_t lo = *reinterpret_cast<const uint16_t *>(
                                colp + (size_t)j * 2 * CW + ((((fc >> 3) ^ swz_of(j, 2 * CW))) << 4));
                            const uint32_t hi = *reinterpret_cast<const uint16_t *>(
                                colp + (size_t)(j + 1) * 2 * CW + ((((fc >> 3) ^ swz_of(j + 1, 2 * CW))) << 4));
                            big |= (lo & 0x7fffu) >= 0x4700u || (hi & 0x7fffu) >= 0x4700u;
                            pk[jj] = pack2_f16(__uint_as_float(lo << 16), __uint_as_float(hi << 16));
                        }
                    }
                }
                ok = mbar_wait(bar_addr(c.wsempty[wb]), ((uint32_t)(gi >> 1) & 1u) ^ 1u, abort_flag, a.status);
                if (named_bar_any(kBarBld, kBld * 32, !ok)) {
                    ok = false;
                    break;
                }
                uint8_t *Wb = bp + a.off_ws + (size_t)wb * a.ws_bytes;
                if (prev[wb] >= 0) {
#pragma unroll
                    for (int x = 0; x < RB / 16; ++x)
                        *reinterpret_cast<uint4 *>(Wb + (size_t)prev[wb] * RB + x * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                // zeroing before writing (rows move between threads); the vote
                // sends the whole group to the CUDA-core path
                const bool slow = named_bar_any(kBarBld, kBld * 32, big);
                prev[wb] = -1;
                if (!slow && row >= 0) {
                    uint8_t *d = Wb + (size_t)row * RB;
                    const int sw = swz_of(row, RB);
#pragma unroll
                    for (int x = 0; x < RB / 16; ++x)
                        *reinterpret_cast<uint4 *>(d + ((x ^ sw) << 4)) =
                            make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
                    prev[wb] = row;
                }
                fence_proxy_async();
                named_bar(kBarBld, kBld * 32);
                if (t == 0)
                    mbar_arrive(bar_addr(c.wsfull[wb]));
                if (slow) {
                    // dh[b][i0 + row] += sum_j dZ[b][j] W[j][f] from the step's fp16 tile
                    ok = mbar_wait(bar_addr(c.dzhfull[db]), dph, abort_flag, a.status);
                    if (ok && row >= 0) {
                        const uint8_t *tile = bp + a.off_dzh + (size_t)(db * C + g) * ZCH;
                        const int fc = t % CW;
                        const uint8_t *colp = Wg + (size_t)(t / CW) * WCH + (fc & 7) * 2;
                        for (int bb = 0; bb < a.B; ++bb) {
                            float acc = 0.f;
                            const int zsw_r = swz_of(bb, ZSW);
                            for (int j = 0; j < G; ++j) {
                                const uint32_t wbits = *reinterpret_cast<const uint16_t *>(
                                    colp + (size_t)j * 2 * CW + ((((fc >> 3) ^ swz_of(j, 2 * CW))) << 4));
                                const __half zh = *reinterpret_cast<const __half *>(
                                    tile + (size_t)bb * ZSW + ((((j * 2) >> 4) ^ zsw_r) << 4) + (j & 7) * 2);
                                acc = fmaf(__half2float(zh), __uint_as_float(wbits << 16), acc);
                            }
                            atomicAdd(a.dh + (size_t)bb * a.H + i0 + row, acc);
                        }
                    }
                    if (named_bar_any(kBarBld, kBld * 32, !ok)) {
                        ok = false;
                        break;
                    }
                }
            }
            if (!ok)
                break;
            named_bar(kBarBld, kBld * 32);
            if (t == 0)
                mbar_arrive(bar_addr(c.empty[s]));  // done with the stage's W_k and I_k
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no CTA leaves while another may still read its shared memory
    if (warp == kWA) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// ------------------------------------------------------------------ plan
struct StepPlan {
    bool ok = false;
    int C = 0, BW = 0, S = 0, CW = 0, nbc = 0;
    uint32_t h_bytes = 0, w_bytes = 0, i_bytes = 0, stage_bytes = 0, dzw_bytes = 0, ws_bytes = 0;
    uint32_t off_dzw = 0, off_dzh = 0, off_ws = 0;
    size_t smem = 0;
};

StepPlan plan_step(const sg_layout *lo, int B)
{
    StepPlan p;
    const int G = lo->G, F = lo->F, H = lo->H;
    if (B < 1 || B > 128 || (G != 16 && G != 32 && G != 64) || F % 16 != 0 || F > kMaxF ||
        lo->ldB < 128 || lo->K < 1)
        return p;
    const int bwmax = 512 - 4 * G;
    for (int C = 1; C <= kMaxC; ++C) {
        const int bw = (int)((ceil_div(H, C) + 63) / 64 * 64);
        if (bw <= bwmax) {
            p.C = C;
            p.BW = bw;
            break;
        }
    }
    if (p.C == 0)
        return p;
    p.CW = F % 64 == 0 ? 64 : F % 32 == 0 ? 32 : 16;
    p.nbc = B <= 64 ? 1 : 2;
    const uint32_t zsw = 2 * G >= 128 ? 128u : 2u * G;
    p.h_bytes = 128u * F * 2u;
    p.w_bytes = (uint32_t)G * F * 2u;
    p.i_bytes = (uint32_t)((2 * F + 127) / 128 * 128);
    p.stage_bytes = (p.h_bytes + p.C * (p.w_bytes + p.i_bytes) + 1023u) & ~1023u;
    p.dzw_bytes = 2u * 128u * zsw;
    p.ws_bytes = (uint32_t)p.BW * 2u * G;
    const long fixed = 2l * p.dzw_bytes + 2l * p.C * 128 * zsw + 2l * p.ws_bytes + 1024;
    long S = (kSmemBudget - fixed) / (long)p.stage_bytes;
    if (S > kMaxS)
        S = kMaxS;
    if (S < 2)
        return p;
    p.S = (int)S;
    p.off_dzw = (uint32_t)p.S * p.stage_bytes;
    p.off_dzh = p.off_dzw + 2u * p.dzw_bytes;
    p.off_ws = p.off_dzh + 2u * p.C * 128u * zsw;
    p.smem = (size_t)p.off_ws + 2u * p.ws_bytes + 1024;
    // more than half of an SM's shared memory: one CTA per SM, so that no two
    // CTAs ever wait for each other's 512 TMEM columns
    if (p.smem < 120 * 1024)
        p.smem = 120 * 1024;
    // the dW MMA reads up to 128 rows of 128 bytes from the start of the last
    // stage's second sample chunk: the buffers after the stages cover that
    if ((size_t)(p.S - 1) * p.stage_bytes + (size_t)F * 128 + 128 * 128 > p.smem - 1024)
        return p;
    p.ok = true;
    return p;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode_step = nullptr;

sg_status encode_w(CUtensorMap *m, const void *W, const sg_layout *lo, int CW)
{
    if (!g_encode_step) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn) {
            sg_set_error("cuTensorMapEncodeTiled is not available from the driver");
            return SG_ERR_CUDA;
        }
        g_encode_step = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    }
    if (((uintptr_t)W & 15) != 0) {
        sg_set_error("W: device pointer must be 16-byte aligned");
        return SG_ERR_INVALID;
    }
    cuuint64_t dims[2] = {(cuuint64_t)lo->F, (cuuint64_t)lo->L};
    cuuint64_t strides[1] = {(cuuint64_t)lo->F * 2};
    cuuint32_t box[2] = {(cuuint32_t)CW, (cuuint32_t)lo->G};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle sw = CW == 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : CW == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                             : CU_TENSOR_MAP_SWIZZLE_32B;
    CUresult r = g_encode_step(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(W), dims, strides, box,
                               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        sg_set_error("W: cuTensorMapEncodeTiled failed (%d)", (int)r);
        return SG_ERR_CUDA;
    }
    return SG_OK;
}

}  // namespace

bool tc_step_ok(const sg_layout *lo, int32_t B) { return plan_step(lo, B).ok; }

sg_status tc_step(sg_layout *lo, int32_t B, const uint16_t *W, uint16_t *dW, float *dh, double *loss,
                  cudaStream_t st)
{
    const StepPlan p = plan_step(lo, B);
    if (!p.ok) {
        sg_set_error("tc_step: shape not supported by the fused step kernel");
        return SG_ERR_UNSUPPORTED;
    }
    CUtensorMap tm_w;
    sg_status rc = encode_w(&tm_w, W, lo, p.CW);
    if (rc != SG_OK)
        return rc;
    void (*kern)(CUtensorMap, StepArgs) = lo->G == 16 ? k_tc_step<16> : lo->G == 32 ? k_tc_step<32> : k_tc_step<64>;
    SG_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem));
    if (p.C > 1)
        SG_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1));
    StepArgs a;
    a.idx_s = lo->idx_s;
    a.hT = lo->hT;
    a.dW = dW;
    a.dh = dh;
    a.gptr = lo->gptr;
    a.gent = lo->gent;
    a.loss_part = lo->loss_part;
    a.status = lo->status;
    a.K = lo->K;
    a.NPS = ceil_div(lo->K, p.C);
    a.B = B;
    a.F = lo->F;
    a.H = lo->H;
    a.ldB = lo->ldB;
    a.C = p.C;
    a.BW = p.BW;
    a.S = p.S;
    a.CW = p.CW;
    a.nbc = p.nbc;
    a.h_bytes = p.h_bytes;
    a.w_bytes = p.w_bytes;
    a.i_bytes = p.i_bytes;
    a.stage_bytes = p.stage_bytes;
    a.dzw_bytes = p.dzw_bytes;
    a.ws_bytes = p.ws_bytes;
    a.off_dzw = p.off_dzw;
    a.off_dzh = p.off_dzh;
    a.off_ws = p.off_ws;

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)p.C;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    // persistent: as many clusters as can be resident at once (cached per
    // layout and shape), never more than there are steps of C groups
    if (lo->step_ncl <= 0 || lo->step_ncl_key != (int64_t)p.C * 1000000 + (int64_t)p.smem) {
        cfg.gridDim = dim3((unsigned)p.C);
        int ncl = 0;
        SG_TRY_CUDA(cudaOccupancyMaxActiveClusters(&ncl, kern, &cfg));
        if (ncl < 1) {
            sg_set_error("tc_step: no cluster of %d CTAs with %zu bytes of shared memory fits", p.C, p.smem);
            return SG_ERR_UNSUPPORTED;
        }
        lo->step_ncl = ncl;
        lo->step_ncl_key = (int64_t)p.C * 1000000 + (int64_t)p.smem;
    }
    int64_t ncl = lo->step_ncl;
    if (ncl > a.NPS)
        ncl = a.NPS;
    cfg.gridDim = dim3((unsigned)(ncl * p.C));
    SG_TRY_CUDA(cudaMemsetAsync(dh, 0, sizeof(float) * (size_t)B * lo->H, st));
    SG_LAUNCH(lo, SG_KIND_STEP, st, rc = (cudaLaunchKernelEx(&cfg, kern, tm_w, a) == cudaSuccess) ? SG_OK : SG_ERR_CUDA);
    if (rc != SG_OK) {
        sg_set_error("tc_step: launch failed: %s", cudaGetErrorString(cudaGetLastError()));
        return rc;
    }
    return sg_loss_finalize(lo, (int32_t)(ncl * p.C), loss, st);
}
