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
//   [SH H slots: the own group's H_k (sample chunks of 64 x F rows x 128 B,
//                128-byte swizzle)]
//   [SW W slots: W of the C groups (TMA boxes of CW columns x G rows), then
//                I of the C groups]
//   [dZ bf16 value + residual planes (dW operand)]
//   [2 x C fp16 dZ tiles (dh operand): slot g holds group C*step + g]
//   [2 x Ws (band rows of 2G bytes)]
// TMEM: dh band [0, BW), Z slots [BW, BW + 2G), dW slot [BW + 2G, BW + 4G).
//
// Warp roles: producers (cp.async gather of H_k; TMA of the W and I rows),
// one MMA-issuing warp each for the forward, dW and dh, one warp that copies
// the other CTAs' dZ tiles, the BCE team, the dW-store team and the Ws
// builders (ldmatrix.trans of W_k's column blocks, fp16, one row per f).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "sg_internal.cuh"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

using namespace tc;

// Timeline hooks for profiling builds (-DSG_STEP_TRACE): every warp of the
// first cluster records clock64() at marked points of steps [kTrT0, kTrT0 +
// kTrN) into the buffer set with sg_step_trace_set.  Compiled out otherwise.
#ifdef SG_STEP_TRACE
__device__ unsigned long long *g_step_trace = nullptr;
constexpr int kTrT0 = 100, kTrN = 64, kTrW = 24, kTrS = 16;
#define STEP_TRACE(slot, itv)                                                                              \
    do {                                                                                                   \
        if (g_step_trace && blockIdx.x < 2 && (itv) >= kTrT0 && (itv) < kTrT0 + kTrN && (threadIdx.x & 31) == 0) \
            g_step_trace[((((size_t)blockIdx.x * kTrW + (threadIdx.x >> 5)) * kTrN + ((itv) - kTrT0)) * kTrS) + \
                         (slot)] = clock64();                                                              \
    } while (0)
extern "C" __attribute__((visibility("default"))) int sg_step_trace_set(void *p)
{
    return (int)cudaMemcpyToSymbol(g_step_trace, &p, sizeof(p));
}
#else
#define STEP_TRACE(slot, itv) \
    do {                      \
    } while (0)
#endif

namespace {

constexpr int kP = 4;     // producer warps
constexpr int kBce = 8;   // BCE warps: two per TMEM lane quarter
constexpr int kDw = 4;    // dW store warps: one per lane quarter
constexpr int kBld = 4;   // Ws builder warps
constexpr int kWF = kP;          // forward MMA warp
constexpr int kWD = kP + 1;      // dW MMA warp
constexpr int kWH = kP + 2;      // dh MMA warp
constexpr int kWC = kP + 3;      // copies the other CTAs' dZ tiles
constexpr int kW0Bce = kP + 4;
constexpr int kW0Dw = kW0Bce + kBce;
constexpr int kW0Bld = kW0Dw + kDw;
constexpr int kWarps = kW0Bld + kBld;
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxC = 4;
constexpr int kMaxSH = 4, kMaxSW = 4;
constexpr int kMaxF = 128;
constexpr int kMaxBlk = kMaxF / 8 / kBld;  // column blocks of W_k per builder warp
// dynamic shared memory the plan may use (the opt-in maximum is 227 KB,
// less the static control block)
constexpr int kSmemBudget = 227 * 1024 - 3072;
// named barriers
constexpr int kBarBce = 1, kBarBld = 3;

struct StepCtl {
    uint64_t hfull[kMaxSH], hempty[kMaxSH];  // H ring
    uint64_t wfull[kMaxSW], wempty[kMaxSW];  // W ring
    uint64_t zfull[2], zempty[2];            // Z slots
    uint64_t dzwfull, dzwempty;              // dZ bf16 planes (dW operand)
    uint64_t dwfull, dwempty;                // dW slot
    uint64_t dzhfull[2];                     // the step's fp16 tiles are all in place
    uint64_t dzhdone[2];                     // the local dh MMAs and builders are done with them
    uint64_t dzready[2];                     // the other CTAs wrote their tiles (cluster)
    uint64_t dzcopied[2];                    // the other CTAs copied this CTA's tile (cluster)
    uint64_t wsfull[2], wsempty[2];          // Ws buffers
    uint64_t drain[3];
    uint32_t tmem;
    int abort_flag;
    double red[kBce];
    // per builder lane and column block: the Ws row it wrote in buffer 0 / 1
    // (-1: none), zeroed the next time the buffer is used
    int16_t rowtab[2][kMaxBlk][kBld * 32];
};

struct StepArgs {
    const uint16_t *idx_s, *hT;
    uint16_t *dW;
    float *dh;
    const int32_t *gptr, *gent;
    double *loss_part;
    int32_t *status;
    int64_t K, NPS;  // groups; steps of C groups
    int32_t B, F, H, ldB, C, BW, SH, SW, nbc;
    uint32_t h_bytes, w_bytes, i_bytes, wslot_bytes, ws_bytes;
    uint32_t off_w, off_dzw, off_dzh, off_ws;
};

__device__ __forceinline__ uint32_t bar_addr(const uint64_t &b) { return smem_u32(&b); }

// a bounded wait whose outcome every lane of the warp shares (the warp then
// takes the same branch around .sync.aligned TMEM accesses and __syncwarp)
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag, int32_t *status)
{
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, status));
}

__device__ __forceinline__ int groups_in_step(const StepArgs &a, int64_t ps)
{
    return (int)(a.K - ps * a.C < a.C ? a.K - ps * a.C : a.C);
}

// The band's part of dh for a group whose W_k holds a magnitude >= 2^15 in
// the band (beyond fp16's exact range): dh[b][i0 + row] += sum_j dZ[b][j]
// W[j][f] in fp32 from the fp16 dZ tile (rows of zsw bytes, swizzle of that
// width) and the bf16 W_k box layout (rows of 2 CW bytes).  Out of line: it
// runs rarely and stays out of the instruction cache of the common path.
__device__ __noinline__ void dh_band_fp32(const uint8_t *tile, int zsw, const uint8_t *Wg, int G, int CW, int f,
                                          int row, int i0, int B, int H, float *dh)
{
    const int fc = f % CW;
    const uint32_t wrow = 2u * CW, wch = (uint32_t)G * wrow;
    const uint8_t *colp = Wg + (size_t)(f / CW) * wch + (fc & 7) * 2;
    for (int bb = 0; bb < B; ++bb) {
        float acc = 0.f;
        const int zr = swz_of(bb, zsw);
        for (int j = 0; j < G; ++j) {
            const uint32_t wbits = *reinterpret_cast<const uint16_t *>(
                colp + (size_t)j * wrow + ((((fc >> 3) ^ swz_of(j, (int)wrow))) << 4));
            const __half zh = *reinterpret_cast<const __half *>(tile + (size_t)bb * zsw +
                                                                 ((((j * 2) >> 4) ^ zr) << 4) + (j & 7) * 2);
            acc = fmaf(__half2float(zh), __uint_as_float(wbits << 16), acc);
        }
        atomicAdd(dh + (size_t)bb * H + i0 + row, acc);
    }
}

template <int G_, int CW>
__global__ void __launch_bounds__(kThreads, 1) k_tc_step(const __grid_constant__ CUtensorMap tm_w, const StepArgs a)
{
    constexpr int G = G_;
    constexpr int ZSW = 2 * G >= 128 ? 128 : 2 * G;  // bytes of a dZ row
    constexpr uint32_t ZCH = 128u * ZSW;              // one dZ plane (128 sample rows)
    constexpr int RB = 2 * G;                         // bytes of a Ws row
    constexpr int CHB = G / 2;                        // BCE columns per warp
    constexpr int DCH = G < 16 ? G : 16;              // dW columns per TMEM load
    constexpr int NI = G / 8;                         // 8-row blocks of W_k (one per Ws 16-byte unit)
    constexpr uint32_t WROW = 2u * CW;                // bytes of a row of one W box
    constexpr uint32_t WCH = (uint32_t)G * WROW;      // bytes of one W box
    __shared__ StepCtl c;
    extern __shared__ uint8_t dsm[];
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const uint32_t base = (smem_u32(dsm) + 1023u) & ~1023u;
    uint8_t *bp = dsm + (base - smem_u32(dsm));
    const int C = a.C, SH = a.SH, SW = a.SW, BW = a.BW, F = a.F;
    const uint32_t rank = cluster_rank();
    const int64_t cl = cluster_index(), ncl = cluster_count();
    const int i0 = (int)rank * BW;  // first dh column of this CTA's band
    const uint32_t col_z = (uint32_t)BW, col_w = (uint32_t)BW + 2 * G;

    if (threadIdx.x == 0) {
        c.abort_flag = 0;
        for (int s = 0; s < SH && s < kMaxSH; ++s) {
            mbar_init(bar_addr(c.hfull[s]), kP * 32);
            mbar_init(bar_addr(c.hempty[s]), 1);
        }
        for (int s = 0; s < SW && s < kMaxSW; ++s) {
            mbar_init(bar_addr(c.wfull[s]), 1);
            mbar_init(bar_addr(c.wempty[s]), 2);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_addr(c.zfull[i]), 1);
            mbar_init(bar_addr(c.zempty[i]), kBce * 32);
            mbar_init(bar_addr(c.dzhfull[i]), C > 1 ? 2 : 1);
            mbar_init(bar_addr(c.dzhdone[i]), 2);  // dh MMA commit + builders (fp32 path reads)
            mbar_init(bar_addr(c.dzready[i]), C > 1 ? C - 1 : 1);
            mbar_init(bar_addr(c.dzcopied[i]), C > 1 ? C - 1 : 1);
            mbar_init(bar_addr(c.wsfull[i]), 1);
            mbar_init(bar_addr(c.wsempty[i]), 1);
        }
        mbar_init(bar_addr(c.dzwfull), kBce * 32);
        mbar_init(bar_addr(c.dzwempty), 1);
        mbar_init(bar_addr(c.dwfull), 1);
        mbar_init(bar_addr(c.dwempty), kDw * 32);
        for (int i = 0; i < 3; ++i)
            mbar_init(bar_addr(c.drain[i]), 1);
        fence_mbar_init();
    }
    if (warp == kWF) {
        tmem_alloc(smem_u32(&c.tmem), 512);
        tmem_relinquish();
    }
    for (int i = threadIdx.x; i < 2 * kMaxBlk * kBld * 32; i += kThreads)
        (&c.rowtab[0][0][0])[i] = -1;
    // the Ws buffers start zeroed; the builders rewrite only the words they use
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
        // thread 0: W_k and I_k of every group of the step (TMA / bulk copy)
        // into the W ring.  Every producer thread: its share of the own group's
        // H_k by cp.async into the H ring -- warp pw copies rows
        // [pw RW, pw RW + RW), two 256-byte hT rows per instruction (16 lanes
        // each; only the first 64 samples when B <= 64).  The gather's index
        // rows are loaded one step ahead.
        const int t = threadIdx.x;
        const int RW = F / kP;
        const int u = lane & 15, rsub = lane >> 4;
        const int ulim = a.nbc * 8;
        uint32_t nrow = 0;
        if (cl < a.NPS && (int64_t)cl * C + rank < a.K && lane < RW)
            nrow = __ldg(a.idx_s + ((int64_t)cl * C + rank) * F + warp * RW + lane);
        int it = 0;
        bool ok = true;
        Ring rh, rw;
        for (int64_t ps = cl; ps < a.NPS; ps += ncl, ++it, rh.next(SH), rw.next(SW)) {
            const int sh = rh.i, sw = rw.i;
            const int64_t k0 = ps * C;
            const int ng = groups_in_step(a, ps);
            const bool own = (int)rank < ng;
            STEP_TRACE(0, it);
            const uint32_t myrow = nrow;
            const int64_t kn = (ps + ncl) * C + rank;
            if (ps + ncl < a.NPS && kn < a.K && lane < RW)
                nrow = __ldg(a.idx_s + kn * F + warp * RW + lane);
            if (t == 0 && ok) {
                ok = mbar_wait(bar_addr(c.wempty[sw]), rw.ph ^ 1u, abort_flag, a.status);
                if (ok) {
                    const uint32_t wfb = bar_addr(c.wfull[sw]);
                    const uint32_t ws = base + a.off_w + (uint32_t)sw * a.wslot_bytes;
                    mbar_arrive_expect_tx(wfb, (uint32_t)ng * (a.w_bytes + 2u * F));
                    for (int g = 0; g < ng; ++g) {
                        for (int ch = 0; ch * CW < F; ++ch)
                            tma_load_2d(ws + (uint32_t)g * a.w_bytes + (uint32_t)ch * WCH, &tm_w, ch * CW,
                                        (int)((k0 + g) * G), wfb);
                        bulk_load(ws + (uint32_t)C * a.w_bytes + (uint32_t)g * a.i_bytes, a.idx_s + (k0 + g) * F,
                                  2u * F, wfb);
                    }
                }
            }
            STEP_TRACE(1, it);
            if (!mbar_wait(bar_addr(c.hempty[sh]), rh.ph ^ 1u, abort_flag, a.status))
                break;
            STEP_TRACE(2, it);
            if (own) {  // warp-uniform: every lane takes part in the shuffles
                const uint32_t hs = base + (uint32_t)sh * a.h_bytes;
                for (int r0 = 0; r0 < RW; r0 += 2) {
                    const int rr = r0 + rsub;
                    const uint32_t row = __shfl_sync(0xffffffffu, myrow, rr & 31);
                    const int f = warp * RW + rr;
                    if (u < ulim)
                        cp_async16(hs + (uint32_t)(u >> 3) * F * 128 + (uint32_t)f * 128 +
                                       (uint32_t)(((u & 7) ^ (f & 7)) << 4),
                                   a.hT + (size_t)row * a.ldB + u * 8);
                }
            }
            STEP_TRACE(3, it);
            cp_async_arrive_noinc(bar_addr(c.hfull[sh]));
        }
        cp_async_wait_all();
        if (*abort_flag) {
            for (int j = it - SH < 0 ? 0 : it - SH; j < it; ++j)
                mbar_wait_drain(bar_addr(c.hfull[j % SH]), (uint32_t)(j / SH) & 1u);
            if (t == 0)
                for (int j = it - SW < 0 ? 0 : it - SW; j < it; ++j)
                    mbar_wait_drain(bar_addr(c.wfull[j % SW]), (uint32_t)(j / SW) & 1u);
        }
    } else if (warp == kWF) {
        // ---------------------------------------------------------- forward MMA
        const uint32_t idf = idesc_bf16(128, G, 1, 0);
        constexpr uint32_t wlay = CW == 64 ? kLayoutSW128 : CW == 32 ? kLayoutSW64 : kLayoutSW32;
        int it = 0, io = 0;
        Ring rh, rw;
        for (int64_t ps = cl; ps < a.NPS; ps += ncl, ++it, rh.next(SH), rw.next(SW)) {
            const int sh = rh.i, sw = rw.i;
            STEP_TRACE(0, it);
            if (!warp_wait(bar_addr(c.wfull[sw]), rw.ph, abort_flag, a.status))
                break;
            STEP_TRACE(1, it);
            if ((int)rank >= groups_in_step(a, ps)) {  // no own group this step
                if (lane == 0)
                    mbar_arrive(bar_addr(c.wempty[sw]));
                __syncwarp();
                continue;
            }
            const int zs = io & 1;
            if (!warp_wait(bar_addr(c.hfull[sh]), rh.ph, abort_flag, a.status))
                break;
            STEP_TRACE(2, it);
            if (!warp_wait(bar_addr(c.zempty[zs]), ((uint32_t)(io >> 1) & 1u) ^ 1u, abort_flag, a.status))
                break;
            STEP_TRACE(3, it);
            tc_fence_after();
            fence_proxy_async();  // cp.async-written H_k -> the MMA (async proxy)
            if (lane == 0) {
                const uint32_t A = base + (uint32_t)sh * a.h_bytes;
                const uint32_t Wt = base + a.off_w + (uint32_t)sw * a.wslot_bytes + rank * a.w_bytes;
                for (int st = 0; st < F / 16; ++st) {
                    // A: H_k, MN-major (M = samples); 8 f rows per 1024-byte atom
                    const uint64_t ad = sdesc(A + (uint32_t)st * 2048, (uint32_t)F * 128, 1024, kLayoutSW128);
                    // B: W_k, K-major; box st*16/CW, 32 bytes per 16 f inside a row
                    const int f0 = st * 16;
                    const uint64_t bd =
                        sdesc(Wt + (uint32_t)(f0 / CW) * WCH + (uint32_t)(f0 % CW) * 2, 16, 8 * WROW, wlay);
                    mma_bf16(tbase + col_z + (uint32_t)(zs * G), ad, bd, idf, st > 0 ? 1u : 0u);
                }
                mma_commit(bar_addr(c.zfull[zs]));
                mma_commit(bar_addr(c.wempty[sw]));  // done with the own W_k
            }
            __syncwarp();
            STEP_TRACE(4, it);
            ++io;
        }
        if (lane == 0)
            mma_commit(bar_addr(c.drain[0]));
        __syncwarp();
        mbar_wait_drain(bar_addr(c.drain[0]), 0);
    } else if (warp == kWD) {
        // ---------------------------------------------------------- dW MMA
        const uint32_t idw = idesc_bf16(128, 2 * G, 0, 1);
        constexpr uint32_t zlay = ZSW == 128 ? kLayoutSW128 : ZSW == 64 ? kLayoutSW64 : kLayoutSW32;
        const int kb = a.nbc * 4;  // K steps of 16 samples
        int it = 0, io = 0;
        Ring rh;
        for (int64_t ps = cl; ps < a.NPS; ps += ncl, ++it, rh.next(SH)) {
            const int sh = rh.i;
            // this warp sees the H barrier itself before its MMAs read the cp.async data
            if (!warp_wait(bar_addr(c.hfull[sh]), rh.ph, abort_flag, a.status))
                break;
            if ((int)rank >= groups_in_step(a, ps)) {
                if (lane == 0)
                    mbar_arrive(bar_addr(c.hempty[sh]));
                __syncwarp();
                continue;
            }
            STEP_TRACE(0, it);
            if (!warp_wait(bar_addr(c.dzwfull), (uint32_t)io & 1u, abort_flag, a.status))
                break;
            STEP_TRACE(1, it);
            if (!warp_wait(bar_addr(c.dwempty), ((uint32_t)io & 1u) ^ 1u, abort_flag, a.status))
                break;
            STEP_TRACE(2, it);
            tc_fence_after();
            fence_proxy_async();
            if (lane == 0) {
                const uint32_t A = base + (uint32_t)sh * a.h_bytes;
                const uint32_t Zs = base + a.off_dzw;
                for (int st = 0; st < kb; ++st) {
                    // A: H_k^T, K-major (rows f, K = samples): sample chunk st/4, 32 B per 16 samples
                    const uint64_t ad =
                        sdesc(A + (uint32_t)(st >> 2) * F * 128 + (uint32_t)(st & 3) * 32, 16, 1024, kLayoutSW128);
                    // B: [hi | lo] dZ_k, MN-major (N = j, K = samples), the lo plane ZCH further on
                    const uint64_t bd = sdesc(Zs + (uint32_t)st * 16 * ZSW, ZCH, 8 * ZSW, zlay);
                    mma_bf16(tbase + col_w, ad, bd, idw, st > 0 ? 1u : 0u);
                }
                mma_commit(bar_addr(c.dwfull));
                mma_commit(bar_addr(c.dzwempty));
                mma_commit(bar_addr(c.hempty[sh]));  // last reader of H_k
            }
            __syncwarp();
            ++io;
        }
        if (lane == 0)
            mma_commit(bar_addr(c.drain[1]));
        __syncwarp();
        mbar_wait_drain(bar_addr(c.drain[1]), 0);
    } else if (warp == kWH) {
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
            const int ng = groups_in_step(a, ps);
            STEP_TRACE(0, it);
            if (!warp_wait(bar_addr(c.dzhfull[db]), (uint32_t)(it >> 1) & 1u, abort_flag, a.status))
                break;
            STEP_TRACE(1, it);
            for (int g = 0; g < ng; ++g, ++gi) {
                const int wb = gi & 1;
                if (!warp_wait(bar_addr(c.wsfull[wb]), (uint32_t)(gi >> 1) & 1u, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                STEP_TRACE(2 + g, it);
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t au = adesc0 + (uint64_t)((base + a.off_dzh + (uint32_t)(db * C + g) * ZCH) >> 4);
                    const uint64_t bu = bdesc0 + (uint64_t)((base + a.off_ws + (uint32_t)wb * a.ws_bytes) >> 4);
#pragma unroll
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
            mma_commit(bar_addr(c.drain[2]));
        __syncwarp();
        mbar_wait_drain(bar_addr(c.drain[2]), 0);
    } else if (warp == kWC) {
        // ---------------------------------------------------------- tile copies
        // the other CTAs' fp16 dZ tiles of a step, by distributed-shared-memory
        // loads, into this CTA's buffer for the step
        constexpr int NV = (int)(ZCH / (32 * 16));  // 16-byte loads per lane per tile
        constexpr int NB = NV > 8 ? 8 : NV;          // loads in flight per lane
        int it = 0;
        for (int64_t ps = cl; ps < a.NPS && C > 1; ps += ncl, ++it) {
            const int db = it & 1;
            const uint32_t dph = (uint32_t)(it >> 1) & 1u;
            const int ng = groups_in_step(a, ps);
            STEP_TRACE(0, it);
            if (!__all_sync(0xffffffffu, mbar_wait_cluster(bar_addr(c.dzready[db]), dph, abort_flag, a.status)))
                break;
            STEP_TRACE(1, it);
            if (!warp_wait(bar_addr(c.dzhdone[db]), dph ^ 1u, abort_flag, a.status))
                break;
            STEP_TRACE(2, it);
            for (int p = 0; p < ng; ++p) {
                if (p == (int)rank)
                    continue;
                const uint32_t off = a.off_dzh + (uint32_t)(db * C + p) * ZCH;
                const uint32_t src = mapa(base + off, (uint32_t)p);
#pragma unroll
                for (int x0 = 0; x0 < NV; x0 += NB) {
                    uint4 v[NB];
#pragma unroll
                    for (int x = 0; x < NB; ++x)
                        v[x] = ld_dsmem16(src + (uint32_t)(lane + (x0 + x) * 32) * 16u);
#pragma unroll
                    for (int x = 0; x < NB; ++x)
                        *reinterpret_cast<uint4 *>(bp + off + (uint32_t)(lane + (x0 + x) * 32) * 16u) = v[x];
                }
            }
            fence_proxy_async();
            __syncwarp();
            STEP_TRACE(3, it);
            if (lane == 0) {
                mbar_arrive(bar_addr(c.dzhfull[db]));
                // the copied values are in use already: nothing to publish
                for (int p = 0; p < C; ++p)
                    if (p != (int)rank)
                        mbar_arrive_remote_relaxed(mapa(bar_addr(c.dzcopied[db]), (uint32_t)p));
            }
            __syncwarp();
        }
    } else if (warp < kW0Dw) {
        // ---------------------------------------------------------- BCE
        const int q = warp & 3;
        const int sub = (warp - kW0Bce) >> 2;
        const int b = q * 32 + lane;  // sample row of this thread
        const int c0 = sub * CHB;     // first column of this warp
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        double lacc = 0.0;  // folded in from lf every 32 groups (fp64 is slow on this part)
        float lf = 0.f;
        int it = 0, io = 0;
        // positive-list bounds of the own group, loaded one step ahead
        int e0n = 0, e1n = 0;
        if (cl < a.NPS && (int64_t)cl * C + rank < a.K) {
            e0n = __ldg(a.gptr + (int64_t)cl * C + rank);
            e1n = __ldg(a.gptr + (int64_t)cl * C + rank + 1);
        }
        for (int64_t ps = cl; ps < a.NPS; ps += ncl, ++it) {
            const int db = it & 1;
            const uint32_t dph = (uint32_t)(it >> 1) & 1u;
            const int64_t k = ps * C + rank;
            const bool own = k < a.K;
            const int e0 = e0n, e1 = e1n;
            const int64_t kn = k + ncl * C;
            if (kn < a.K) {
                e0n = __ldg(a.gptr + kn);
                e1n = __ldg(a.gptr + kn + 1);
            }
            bool ok = true;
            STEP_TRACE(0, it);
            if (own) {
                const int zs = io & 1;
                float v[CHB];
                ok = warp_wait(bar_addr(c.zfull[zs]), (uint32_t)(io >> 1) & 1u, abort_flag, a.status);
                STEP_TRACE(1, it);
                if (ok) {
                    tc_fence_after();
                    tmem_ld_chunk<CHB>(tbase + lane_off + col_z + (uint32_t)(zs * G + c0), v);
                    STEP_TRACE(2, it);
                    tc_fence_before();
                    mbar_arrive(bar_addr(c.zempty[zs]));
                    if (b < a.B) {
                        const uint32_t y = e1 > e0 ? group_pos_mask(a.gent, e0, e1, b, c0, CHB) : 0u;
                        lf += bce_chunk_ftz<CHB>(v, y);
                        if ((io & 31) == 31) {
                            lacc += (double)lf;
                            lf = 0.f;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < CHB; ++i)
                            v[i] = 0.f;
                    }
                }
                STEP_TRACE(3, it);
                ok = ok && mbar_wait(bar_addr(c.dzwempty), ((uint32_t)io & 1u) ^ 1u, abort_flag, a.status);
                STEP_TRACE(4, it);
                if (ok) {
                    store_dz_tile<CHB>(bp + a.off_dzw, b, c0, v, ZSW, 1, 128);
                    fence_proxy_async();
                    mbar_arrive(bar_addr(c.dzwfull));
                }
                STEP_TRACE(5, it);
                // the own fp16 tile: once the local dh MMAs and the other CTAs'
                // copies of this buffer's previous step are done
                ok = ok && mbar_wait(bar_addr(c.dzhdone[db]), dph ^ 1u, abort_flag, a.status);
                STEP_TRACE(6, it);
                ok = ok && (C == 1 || mbar_wait_cluster(bar_addr(c.dzcopied[db]), dph ^ 1u, abort_flag, a.status));
                STEP_TRACE(7, it);
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
            STEP_TRACE(8, it);
            if (named_bar_any(kBarBce, kBce * 32, !ok))
                break;
            STEP_TRACE(9, it);
            if (threadIdx.x == kW0Bce * 32) {
                // the team's tile writes precede this release (bar.sync orders them)
                mbar_arrive(bar_addr(c.dzhfull[db]));
                for (int p = 0; p < C; ++p)
                    if (p != (int)rank)
                        mbar_arrive_remote(mapa(bar_addr(c.dzready[db]), (uint32_t)p));
            }
        }
        // loss partial of the CTA (fixed order)
        double v = lacc + (double)lf;
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
        if (__all_sync(0xffffffffu, mbar_wait(bar_addr(c.drain[2]), 0, abort_flag, a.status) && !*abort_flag) &&
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
        // ---------------------------------------------------------- dW stores
        const int q = warp & 3;
        const int f = q * 32 + lane;  // lane of the dW^T accumulator
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        int io = 0;
        for (int64_t ps = cl; ps < a.NPS; ps += ncl) {
            const int64_t k = ps * C + rank;
            if (k >= a.K)
                break;  // the own groups are a prefix of the steps
            // dW_k^T accumulator [f][hi j | lo j] -> dW rows k G + j
            STEP_TRACE(0, io);
            if (!warp_wait(bar_addr(c.dwfull), (uint32_t)io & 1u, abort_flag, a.status))
                break;
            STEP_TRACE(1, io);
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < G; cc += DCH) {
                float v[DCH], w[DCH];
                tmem_ld_chunk2<DCH>(tbase + lane_off + col_w + (uint32_t)cc,
                                    tbase + lane_off + col_w + (uint32_t)(G + cc), v, w);
                if (cc + DCH >= G) {
                    tc_fence_before();
                    mbar_arrive(bar_addr(c.dwempty));  // the slot is in registers
                }
                if (f < F) {
                    uint16_t *dst = a.dW + (k * G + cc) * F + f;
#pragma unroll
                    for (int i = 0; i < DCH; ++i)
                        dst[(int64_t)i * F] = bf16_rn(v[i] + w[i]);
                }
            }
            STEP_TRACE(2, io);
            ++io;
        }
    } else {
        // ---------------------------------------------------------- Ws builders
        // Column block x of W_k (8 columns f, all G rows) comes in with
        // ldmatrix.trans: lane l holds rows j = 8i + 2(l%4), +1 of column
        // f = 8x + l/4 (i = 0 .. G/8-1), which is word l%4 of 16-byte unit i
        // of Ws row I_k[f] - i0.  Blocks whose columns all fall outside the
        // band are skipped (I_k is sorted).  The words a lane wrote in a
        // buffer are zeroed the next time the lane uses that buffer.  A group
        // with |W| >= 2^15 in the band adds its band's part of dh on CUDA
        // cores instead (fp32, atomics).
        const int bw = warp - kW0Bld;
        const int qd = lane & 3;
        const int tb = threadIdx.x - kW0Bld * 32;  // lane of the team
        const int nblk = F / 8;
        int it = 0, gi = 0;
        bool ok = true;
        Ring rw;
        for (int64_t ps = cl; ps < a.NPS && ok; ps += ncl, ++it, rw.next(SW)) {
            const int sw = rw.i;
            const int db = it & 1;
            const uint32_t dph = (uint32_t)(it >> 1) & 1u;
            const int ng = groups_in_step(a, ps);
            STEP_TRACE(0, it);
            ok = mbar_wait(bar_addr(c.wfull[sw]), rw.ph, abort_flag, a.status);
            STEP_TRACE(1, it);
            if (named_bar_any(kBarBld, kBld * 32, !ok))
                break;
            STEP_TRACE(2, it);
            const uint32_t wslot = base + a.off_w + (uint32_t)sw * a.wslot_bytes;
            for (int g = 0; g < ng; ++g, ++gi) {
                const int wb = gi & 1;
                const uint32_t Wg = wslot + (uint32_t)g * a.w_bytes;
                const uint16_t *Ig =
                    reinterpret_cast<const uint16_t *>(bp + a.off_w + (size_t)sw * a.wslot_bytes +
                                                       (size_t)C * a.w_bytes + (size_t)g * a.i_bytes);
                // the band's columns [fa, fe) of the sorted I_k: one ballot per
                // 32 columns, no per-block loads
                int fa = 0, fe = 0;
                for (int f0 = 0; f0 < F; f0 += 32) {
                    const int iv = f0 + lane < F ? (int)Ig[f0 + lane] : 0x7fffffff;
                    fa += __popc(__ballot_sync(0xffffffffu, iv < i0));
                    fe += __popc(__ballot_sync(0xffffffffu, iv < i0 + BW));
                }
                ok = mbar_wait(bar_addr(c.wsempty[wb]), ((uint32_t)(gi >> 1) & 1u) ^ 1u, abort_flag, a.status);
                STEP_TRACE(3 + 4 * g, it);
                if (named_bar_any(kBarBld, kBld * 32, !ok)) {
                    ok = false;
                    break;
                }
                uint8_t *Wb = bp + a.off_ws + (size_t)wb * a.ws_bytes;
                // the words this lane wrote the last time it used the buffer
#pragma unroll 1
                for (int x = 0; x < kMaxBlk; ++x) {
                    const int pr = c.rowtab[wb][x][tb];
                    if (pr >= 0) {
                        const int sw2 = swz_of(pr, RB);
#pragma unroll
                        for (int i2 = 0; i2 < NI; ++i2)
                            *reinterpret_cast<uint32_t *>(Wb + (size_t)pr * RB + ((i2 ^ sw2) << 4) + qd * 4) = 0u;
                    }
                }
                named_bar(kBarBld, kBld * 32);  // zeroing before writing: rows move between lanes
                STEP_TRACE(4 + 4 * g, it);
                uint32_t mx = 0;
#pragma unroll 1
                for (int x = 0; x < kMaxBlk; ++x) {
                    int row = -1;
                    const int blk = bw + x * kBld;
                    const int fb = blk * 8;
                    if (blk < nblk && fb + 8 > fa && fb < fe) {  // warp-uniform: some column is in the band
                        // row address of lane l: W_k row j, 16-byte unit of columns fb..fb+7
                        const uint32_t ubox = (uint32_t)(fb / CW) * WCH;
                        const int un = (fb % CW) >> 3;
                        uint32_t pk[NI];
#pragma unroll
                        for (int h = 0; h < (NI + 3) / 4; ++h) {
                            const int j = h * 32 + lane;
                            const int jj = j < G ? j : 0;
                            const uint32_t addr =
                                Wg + ubox + (uint32_t)jj * WROW + (uint32_t)((un ^ swz_of(jj, (int)WROW)) << 4);
                            if constexpr (NI >= 4) {
                                uint32_t r4[4];
                                ldsm_x4_trans(addr, r4);
#pragma unroll
                                for (int i = 0; i < 4; ++i)
                                    pk[h * 4 + i] = r4[i];
                            } else {
                                uint32_t r2[2];
                                ldsm_x2_trans(addr, r2);
                                pk[0] = r2[0];
                                pk[1] = r2[1];
                            }
                        }
                        const int f = fb + (lane >> 2);
                        if (f >= fa && f < fe)
                            row = (int)Ig[f] - i0;
                        if (row >= 0) {
                            const int sw2 = swz_of(row, RB);
#pragma unroll
                            for (int i2 = 0; i2 < NI; ++i2) {
                                const uint32_t r = pk[i2];
                                mx = __vmaxu2(mx, r & 0x7fff7fffu);
                                *reinterpret_cast<uint32_t *>(Wb + (size_t)row * RB + ((i2 ^ sw2) << 4) + qd * 4) =
                                    pack2_f16(__uint_as_float(r << 16), __uint_as_float(r & 0xffff0000u));
                            }
                        }
                    }
                    c.rowtab[wb][x][tb] = (int16_t)row;
                }
                const bool big = (mx & 0xffffu) >= 0x4700u || (mx >> 16) >= 0x4700u;
                STEP_TRACE(5 + 4 * g, it);
                // a group with |W| >= 2^15 in the band takes the CUDA-core path:
                // its rows go back to zero (the rare case pays for it)
                const bool slow = named_bar_any(kBarBld, kBld * 32, big);
                if (slow) {
#pragma unroll 1
                    for (int x = 0; x < kMaxBlk; ++x) {
                        const int pr = c.rowtab[wb][x][tb];
                        if (pr >= 0) {
                            const int sw2 = swz_of(pr, RB);
#pragma unroll
                            for (int i2 = 0; i2 < NI; ++i2)
                                *reinterpret_cast<uint32_t *>(Wb + (size_t)pr * RB + ((i2 ^ sw2) << 4) + qd * 4) = 0u;
                        }
                    }
                }
                fence_proxy_async();
                named_bar(kBarBld, kBld * 32);
                STEP_TRACE(6 + 4 * g, it);
                if (warp == kW0Bld && lane == 0)
                    mbar_arrive(bar_addr(c.wsfull[wb]));
                if (slow) {
                    // one lane per column of the band (lanes with l%4 == 0),
                    // from the step's fp16 tile of the group
                    ok = mbar_wait(bar_addr(c.dzhfull[db]), dph, abort_flag, a.status);
                    const uint8_t *tile = bp + a.off_dzh + (size_t)(db * C + g) * ZCH;
#pragma unroll 1
                    for (int x = 0; x < kMaxBlk; ++x) {
                        const int pr = c.rowtab[wb][x][tb];
                        if (ok && qd == 0 && pr >= 0)
                            dh_band_fp32(tile, ZSW, bp + (Wg - base), G, CW, (bw + x * kBld) * 8 + (lane >> 2), pr,
                                         i0, a.B, a.H, a.dh);
                        c.rowtab[wb][x][tb] = -1;  // nothing to zero next time
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
            if (warp == kW0Bld && lane == 0) {
                mbar_arrive(bar_addr(c.wempty[sw]));  // done with the slot's W_k and I_k
                mbar_arrive(bar_addr(c.dzhdone[db]));  // and with the step's dZ tiles (fp32 path)
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no CTA leaves while another may still read its shared memory
    if (warp == kWF) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

// ------------------------------------------------------------------ plan
struct StepPlan {
    bool ok = false;
    int C = 0, BW = 0, SH = 0, SW = 0, CW = 0, nbc = 0;
    uint32_t h_bytes = 0, w_bytes = 0, i_bytes = 0, wslot_bytes = 0, ws_bytes = 0;
    uint32_t off_w = 0, off_dzw = 0, off_dzh = 0, off_ws = 0;
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
    // one H slot: the sample chunks that are gathered (the forward MMA reads
    // a second chunk's worth past the first; with one chunk that is the next
    // buffer's bytes, in bounds, multiplied into accumulator rows >= 64 that
    // are never used)
    p.h_bytes = (uint32_t)p.nbc * 64u * F * 2u;
    p.w_bytes = (uint32_t)G * F * 2u;
    p.i_bytes = (uint32_t)((2 * F + 127) / 128 * 128);
    p.wslot_bytes = (p.C * (p.w_bytes + p.i_bytes) + 1023u) & ~1023u;
    p.ws_bytes = (uint32_t)p.BW * 2u * G;
    const long fixed = 2l * 128 * zsw + 2l * p.C * 128 * zsw + 2l * p.ws_bytes + 1024;
    // deepest H ring first (the gather is the longest latency), then W
    p.SH = 0;
    for (int sh = kMaxSH; sh >= 2 && p.SH == 0; --sh)
        for (int sw = kMaxSW; sw >= 2; --sw)
            if (fixed + (long)sh * p.h_bytes + (long)sw * p.wslot_bytes <= kSmemBudget) {
                p.SH = sh;
                p.SW = sw;
                break;
            }
    if (p.SH == 0)
        return p;
    p.off_w = (uint32_t)p.SH * p.h_bytes;
    p.off_dzw = p.off_w + (uint32_t)p.SW * p.wslot_bytes;
    p.off_dzh = p.off_dzw + 2u * 128u * zsw;
    p.off_ws = p.off_dzh + 2u * p.C * 128u * zsw;
    p.smem = (size_t)p.off_ws + 2u * p.ws_bytes + 1024;
    // the MMAs read past the last H slot (the dW MMA up to 128 rows of 128
    // bytes from a sample chunk, the forward a second chunk): the buffers after
    // the ring cover that
    if ((size_t)p.off_w + 2 * (size_t)F * 128 + 128 * 128 > p.smem - 1024)
        return p;
    // more than half of an SM's shared memory: one CTA per SM, so that no two
    // CTAs ever wait for each other's 512 TMEM columns
    if (p.smem < 120 * 1024)
        p.smem = 120 * 1024;
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
    void (*kern)(CUtensorMap, StepArgs) = nullptr;
#define SG_STEP_PICK(GG, CC)                  \
    if (lo->G == GG && p.CW == CC)            \
        kern = k_tc_step<GG, CC>;
    SG_STEP_PICK(16, 16) SG_STEP_PICK(16, 32) SG_STEP_PICK(16, 64)
    SG_STEP_PICK(32, 16) SG_STEP_PICK(32, 32) SG_STEP_PICK(32, 64)
    SG_STEP_PICK(64, 16) SG_STEP_PICK(64, 32) SG_STEP_PICK(64, 64)
#undef SG_STEP_PICK
    if (!kern) {
        sg_set_error("tc_step: no kernel for G = %d", lo->G);
        return SG_ERR_UNSUPPORTED;
    }
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
    a.SH = p.SH;
    a.SW = p.SW;
    a.nbc = p.nbc;
    a.h_bytes = p.h_bytes;
    a.w_bytes = p.w_bytes;
    a.i_bytes = p.i_bytes;
    a.wslot_bytes = p.wslot_bytes;
    a.ws_bytes = p.ws_bytes;
    a.off_w = p.off_w;
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
