// Tensor-core engine (sm_103a): tcgen05 MMA with TMEM accumulators, operands
// staged in shared memory by TMA (tile loads for W_k and dZ_k, bulk copies of
// the step's tiles, a cp.async gather for H_k).  HASTE, key design
// "gather-once + dense MMA kernel":
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
//          K-major B (N = j, K = f) of the forward.  The feature gradient
//          copies W_k row-major ([G][F]) and scatters its columns.
//   dZ_k : rows b of min(G,64) j (one chunk per 64 j), swizzle = row width:
//          MN-major B (N = j, K = b) of the weight gradient, K-major A
//          (M = b, K = j) of the feature gradient.  From a caller's row-major
//          [B][L] dZ it is a TMA box; inside the training step dZ lives in a
//          group-tiled workspace whose tiles already hold these bytes, so one
//          bulk copy brings a group's tile in.
//
// Group-tiled dZ workspace (training step only).  Tile k holds, for plane p,
// chunk cj of 64 columns and row r < Bp = 128 ceil(B/128) (rows >= B are
// zero), the 16-byte unit u of columns 8u .. 8u+7 of that chunk at byte
//     ((p * nzc + cj) * Bp + r) * zsw + ((u ^ swz(r)) * 16),
// zsw = min(2G, 128) the row width and swz the TMA swizzle of that width.  The
// fused step writes one fp16 plane (the feature gradient's operand); the
// unfused step writes p = 0: bf16(dZ), p = 1: the residual dZ - bf16(dZ).  A
// tile is contiguous, so writing it touches one or two pages instead of one
// page per sample row.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sg_internal.cuh"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

using namespace tc;

// Timeline hooks for profiling builds (-DSG_FW_TRACE): every warp of CTA 0
// of the fused forward kernel records clock64() at marked points of its
// groups [kFwT0, kFwT0 + kFwN) into the buffer set with sg_fw_trace_set.
// Compiled out otherwise.
#ifdef SG_FW_TRACE
__device__ unsigned long long *g_fw_trace = nullptr;
constexpr int kFwT0 = 100, kFwN = 64, kFwW = 22, kFwS = 8;
#define TRACE_REC(slot, itv)                                                                                 \
    do {                                                                                                     \
        if (g_fw_trace && blockIdx.x == 0 && (itv) >= kFwT0 && (itv) < kFwT0 + kFwN && (threadIdx.x & 31) == 0) \
            g_fw_trace[(((size_t)(threadIdx.x >> 5) * kFwN + ((itv) - kFwT0)) * kFwS) + (slot)] = clock64();   \
    } while (0)
extern "C" __attribute__((visibility("default"))) int sg_fw_trace_set(void *p)
{
    return (int)cudaMemcpyToSymbol(g_fw_trace, &p, sizeof(p));
}
#else
#define TRACE_REC(slot, itv) \
    do {                     \
    } while (0)
#endif
// the forward kernel's hooks, or (-DSG_DH_TRACE) the dh kernel's instead
#ifdef SG_DH_TRACE
#define FW_TRACE(slot, itv) \
    do {                    \
    } while (0)
#define DH_TRACE(slot, itv) TRACE_REC(slot, itv)
#else
#define FW_TRACE(slot, itv) TRACE_REC(slot, itv)
#define DH_TRACE(slot, itv) \
    do {                    \
    } while (0)
#endif

namespace {

constexpr int kMaxStages = 8;
constexpr int kSmemBudget = 220 * 1024;  // dynamic shared memory we plan with
constexpr int kEpiWarps = 8;   // two per TMEM lane quarter
constexpr int kProdWarps = 8;  // cp.async gather + TMA issue (8: measured ~2x the copy rate of 4)
// forward / dW: producers, two MMA-issuing warps, epilogue
constexpr int kFwdThreads = 32 * (kProdWarps + 2 + kEpiWarps);
constexpr int kFirstEpi = kProdWarps + 2;
// dh: one load warp, one MMA warp, sixteen builder warps in two teams of
// eight (a team thread per (group, feature) slot of a unit: 2 x 128 at the
// 3M shape, so the slots spread evenly; teams of six measured slower)
constexpr int kDhBuilders = 16;
constexpr int kDhMaxBuf = 3;  // scattered-W buffers in shared memory (one per builder team)
// groups per pipeline unit (one stage, one scattered-W buffer): a unit's
// fixed costs (barrier round trips, the builders' team barriers, the MMA
// commits) outweigh deeper pipelining, so a unit carries as many groups as two
// scattered-W buffers of 384 columns allow: 64 labels (four groups at G = 16:
// 14 % faster than two at B = 256; two at G = 32), else one group (one group
// per unit measured 4-40 % slower than two at G <= 32)
__host__ __device__ constexpr int dh_units(int G) { return G <= 16 ? 4 : G <= 32 ? 2 : 1; }
// threads of the dh kernel with `iss` MMA-issuing warps: one load warp, the
// issuers, the builders
__host__ __device__ constexpr int dh_threads(int iss) { return 32 * (1 + iss + kDhBuilders); }

// ------------------------------------------------------------------ plans
struct FwdPlan {
    bool ok = false;
    int MT = 0, nk = 0, cw = 0, S = 0, issuers = 0;  // nk TMA boxes of cw columns of W_k
    uint32_t a_bytes = 0, w_bytes = 0, stage_bytes = 0, tmem_cols = 0;
};

struct DWPlan {
    bool ok = false;
    int MT = 0, FT = 0, S = 0, nzc = 0, zsw = 0, issuers = 0;
    int planes = 0;   // dZ planes in smem (2 with the lo residual)
    int ncat = 0;     // 1: the planes are concatenated along N in one pass
    int Nacc = 0;     // accumulator columns per (f tile, group)
    uint32_t a_bytes = 0, z_bytes = 0, stage_bytes = 0, tmem_cols = 0;
    uint32_t pad_bytes = 0;  // the last f tile's MMA reads this far past the last stage
    int stream_t = 0;        // 1: a stage holds one 128-sample tile, a group takes MT stages
};

struct DhPlan {
    bool ok = false;
    int MT = 0, S = 0, zsw = 0, nbands = 0, band_w = 0, bwt = 0, nbuf = 0;
    int gs = 0, sub = 1;  // subgroup size (<= 64) and subgroups per dZ tile
    int idiv = 1;         // subgroups per index row (per group)
    uint32_t z_bytes = 0, w_bytes = 0, i_bytes = 0, stage_bytes = 0, ws_bytes = 0, tmem_cols = 0;
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

// the stage kernels (forward, dW, dh) take any F that is a multiple of 16
bool shape_ok16(const sg_layout *lo)
{
    return lo->G % 16 == 0 && lo->G <= 256 && lo->F % 16 == 0 && lo->F <= 256 &&
           lo->L % 8 == 0 && lo->ldB % 128 == 0;
}

// width (columns) of the TMA boxes W_k is loaded in: 64 (128-byte rows,
// 128-byte swizzle) when it divides F, else 32 (64-byte swizzle), else 16
int w_box_cols(int F) { return F % 64 == 0 ? 64 : F % 32 == 0 ? 32 : 16; }

// dZ rows of a group must fill whole swizzle rows: 16 or 32 columns, or
// whole chunks of 64
bool dz_ok(int G) { return G == 16 || G == 32 || G % 64 == 0; }


int stages_for(uint32_t stage_bytes)
{
    int S = (int)(kSmemBudget / stage_bytes);
    return S > 6 ? 6 : S;
}

FwdPlan plan_fwd(const sg_layout *lo, int B)
{
    FwdPlan p;
    if (!shape_ok16(lo) || B < 1 || B > 256)
        return p;
    p.MT = (B + 127) / 128;
    if (p.MT * 128 > lo->ldB)
        return p;
    p.cw = w_box_cols(lo->F);
    p.nk = lo->F / p.cw;
    p.a_bytes = (uint32_t)p.MT * 2 * lo->F * 128;
    p.w_bytes = (uint32_t)lo->G * lo->F * 2;
    p.stage_bytes = p.a_bytes + p.w_bytes;
    p.S = stages_for(p.stage_bytes);
    if (p.S < 2)  // two stages still overlap loads with MMAs (G = 64, B = 256 has only room for two)
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

// log2 of a power of two, else -1
int log2_exact(int v)
{
    if (v < 1 || (v & (v - 1)))
        return -1;
    int l = 0;
    while ((1 << l) < v)
        ++l;
    return l;
}

DWPlan plan_dW(const sg_layout *lo, int B, bool split)
{
    DWPlan p;
    if (!shape_ok16(lo) || !dz_ok(lo->G) || B < 1 || B > 256)
        return p;
    p.MT = (B + 127) / 128;
    if (p.MT * 128 > lo->ldB)
        return p;
    // tiles of M = 128 rows of f; with F % 128 != 0 the last tile's upper
    // accumulator lanes read rows past F (the next sample chunk, or the pad
    // after the last stage) and are never stored
    p.FT = (lo->F + 127) / 128;
    p.pad_bytes = (uint32_t)(p.FT * 128 - lo->F) * 128u;
    p.zsw = dz_swizzle(lo->G);
    p.nzc = lo->G * 2 > 128 ? lo->G / 64 : 1;
    p.planes = split ? 2 : 1;
    // hi and lo side by side along N when that fits the MMA's N and, double
    // buffered, TMEM; else the lo pass accumulates onto the hi pass
    p.ncat = (split && 2 * lo->G <= 256 && 2 * p.FT * 2 * lo->G <= 512) ? 1 : 0;
    p.Nacc = p.ncat ? 2 * lo->G : lo->G;
    p.a_bytes = (uint32_t)p.MT * 2 * lo->F * 128;
    p.z_bytes = (uint32_t)p.planes * p.nzc * p.MT * 128 * p.zsw;
    p.stage_bytes = p.a_bytes + p.z_bytes;
    p.S = stages_for(p.stage_bytes);
    // the last f tile's pad sits after the last stage
    while (p.S > 0 && (long)p.S * p.stage_bytes + p.pad_bytes > (long)kSmemBudget)
        --p.S;
    if (p.S < 2 && p.MT > 1) {
        // both sample tiles of a group do not fit twice: stream the tiles
        // through the stages, accumulating over them in TMEM
        p.stream_t = 1;
        p.a_bytes = 2u * (uint32_t)lo->F * 128;
        p.z_bytes = (uint32_t)p.planes * p.nzc * 128 * p.zsw;
        p.stage_bytes = p.a_bytes + p.z_bytes;
        p.S = stages_for(p.stage_bytes);
        while (p.S > 0 && (long)p.S * p.stage_bytes + p.pad_bytes > (long)kSmemBudget)
            --p.S;
    }
    if (p.S < 2)
        return p;
    const int per = p.FT * p.Nacc;
    p.issuers = 4 * per <= 512 ? 2 : 1;
    if (2 * p.issuers * per > 512)
        return p;
    p.tmem_cols = pow2_cols(2 * p.issuers * per);
    p.ok = true;
    return p;
}

// tile_g: labels per dZ workspace tile (G, or the fused forward kernel's
// subgroup size when it ran the groups as subgroups)
DhPlan plan_dh(const sg_layout *lo, int B, bool split, int tile_g = 0)
{
    DhPlan p;
    if (tile_g <= 0)
        tile_g = lo->G;
    if (!shape_ok16(lo) || !dz_ok(lo->G) || !dz_ok(tile_g) || lo->G > 256 || lo->G % tile_g != 0 || B < 1 ||
        B > 256)
        return p;
    p.MT = (B + 127) / 128;
    if (p.MT * 128 > lo->ldB)
        return p;
    // groups of more than 64 labels run as subgroups of 64 that share the
    // group's I_k (dh = sum over the subgroups of dZ_sub Ws_sub)
    const int Gs = tile_g > 64 ? 64 : tile_g;
    p.gs = Gs;
    p.sub = tile_g / Gs;      // subgroups per workspace tile
    p.idiv = lo->G / Gs;      // subgroups per index row
    p.zsw = dz_swizzle(Gs);
    p.z_bytes = (uint32_t)(split ? 2 : 1) * 128 * p.zsw;
    p.w_bytes = (uint32_t)Gs * lo->F * 2;
    // the group's sorted index row I_k (u16)
    p.i_bytes = (uint32_t)((lo->F * 2 + 127) / 128 * 128);
    // one unit = P groups: [dZ x P][W^T x P][I_k x P]
    // (whole KB, so that every stage's dZ tiles sit on swizzle-atom boundaries)
    const uint32_t P = (uint32_t)dh_units(Gs);
    p.stage_bytes = (P * (p.z_bytes + p.w_bytes + p.i_bytes) + 1023u) & ~1023u;
    // two builder teams, one buffer each (a third team and buffer cost a
    // stage, and measured slower)
    p.nbuf = 2;
    // bands of at most 384 dh columns (TMEM accumulator: 128 samples x band),
    // narrower where two Ws buffers of that width leave no room for two stages
    for (int maxw = 3; maxw >= 1; --maxw) {
        p.nbands = (lo->H + 128 * maxw - 1) / (128 * maxw);
        p.bwt = ((lo->H + p.nbands - 1) / p.nbands + 127) / 128;
        p.band_w = p.bwt * 128;
        p.ws_bytes = P * (uint32_t)p.band_w * 2 * Gs;  // one row of Gs values per dh column
        const long room = (long)kSmemBudget - (long)p.nbuf * p.ws_bytes;
        p.S = room > 0 ? (int)(room / p.stage_bytes) : 0;
        if (p.S >= 2)
            break;
    }
    p.tmem_cols = pow2_cols(p.band_w);
    if (p.S > kMaxStages)
        p.S = kMaxStages;
    // the flush transposes through kDhBuilders x 33 x 32 floats of shared memory
    p.ok = p.S >= 2 && (long)p.nbuf * p.ws_bytes + (long)p.S * p.stage_bytes >= (long)kDhBuilders * 33 * 32 * 4;
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

// sum of one double per thread over the nwarps (<= kEpiWarps) epilogue warps
// first_epi ..; every thread of those warps calls it
__device__ __forceinline__ void epi_sum_to(double v, Ctl &c, double *dst, int first_epi,
                                           int nwarps = kEpiWarps)
{
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_down_sync(0xffffffffu, v, o);
    const int ew = threadIdx.x / 32 - first_epi;
    if ((threadIdx.x & 31) == 0)
        c.red[ew] = v;
    named_bar(1, nwarps * 32);
    if (ew == 0 && (threadIdx.x & 31) == 0) {
        double s = 0.0;
        for (int i = 0; i < nwarps; ++i)
            s += c.red[i];
        *dst = s;
    }
}

// ------------------------------------------------------------------ gather
// H_k = rows I_k[f] of hT, copied with 16-byte cp.async by the producer
// warps into the 128-byte-swizzled layout [b-chunk of 64][f][64 b]: unit u
// (16 B) of row f lands at chunk(u/8) * F*128 + f*128 + ((u%8) ^ (f%8))*16.
// Producer warp pw copies rows f in [pw*RW, pw*RW + RW), RW = F/kProdWarps.  The lanes
// of one cp.async instruction cover whole rows (16 lanes per 256-byte row when
// B <= 128, all 32 when B <= 256), so every 32-byte sector fetched from L2 is
// used in full.  A lane holds the hT row index of rows pw*RW + lane (+ 32),
// loaded one group ahead; the copy loop broadcasts them with shuffles.
struct GatherIdx {
    uint32_t i[2];
};

template <int NPW = kProdWarps>
__device__ __forceinline__ GatherIdx gather_idx_of(const uint16_t *idx_s, int64_t k, int F, int lane)
{
    const int RW = F / NPW;
    const int pw = threadIdx.x / 32;
    const uint16_t *I = idx_s + k * F + pw * RW;
    GatherIdx g;
    g.i[0] = lane < RW ? __ldg(I + lane) : 0u;
    g.i[1] = lane + 32 < RW ? __ldg(I + lane + 32) : 0u;
    return g;
}

__device__ __forceinline__ void issue_gather(const uint16_t *hT, int ldB, uint32_t A, int F,
                                             int units, const GatherIdx &g, int lane)
{
    const int RW = F / kProdWarps;
    const int pw = threadIdx.x / 32;
    const int lpr = units < 32 ? units : 32;  // lanes per row
    const int rpi = 32 / lpr;                 // rows per instruction
    const int u = lane % lpr, rsub = lane / lpr;
    for (int r0 = 0; r0 < RW; r0 += rpi) {
        const int r = r0 + rsub;
        const uint32_t row = __shfl_sync(0xffffffffu, r0 < 32 ? g.i[0] : g.i[1], r & 31);
        if (r < RW) {
            const int f = pw * RW + r;
            cp_async16(A + (uint32_t)(u >> 3) * F * 128 + (uint32_t)f * 128 + (uint32_t)(((u & 7) ^ (f & 7)) << 4),
                       hT + (size_t)row * ldB + u * 8);
        }
    }
}

// The same copy with the shape known at compile time (F rows, U 16-byte units
// per row): the loop unrolls, the per-lane offsets are computed once, and an
// instruction costs a shuffle, a 32-bit multiply-add and the copy.
//
// PAIR (U_ = 16): the second 64-sample chunk holds samples 0 .. 63 of the
// rows I_k2[f] of a second group instead of samples 64 .. 127 of I_k[f].
template <int F_, int U_, bool PAIR = false, int NPW = kProdWarps>
__device__ __forceinline__ void issue_gather_t(const uint16_t *hT, int ldB, uint32_t A, const GatherIdx &g,
                                               int lane, const GatherIdx &g2 = GatherIdx{{0u, 0u}})
{
    constexpr int RW = F_ / NPW;
    constexpr int LPR = U_ < 32 ? U_ : 32;  // lanes per row
    constexpr int RPI = 32 / LPR;           // rows per instruction
    static_assert(RW % RPI == 0 && RW <= 64, "rows per producer warp");
    static_assert(!PAIR || U_ == 16, "pairs take the two chunks of one 128-sample tile");
    const int pw = threadIdx.x / 32;
    const int u = lane % LPR, rsub = lane / LPR;
    const uint32_t dst0 = A + (uint32_t)(u >> 3) * F_ * 128 + (uint32_t)(pw * RW + rsub) * 128;
    const uint16_t *src0 = hT + (PAIR ? (u & 7) : u) * 8;
#pragma unroll
    for (int t = 0; t < RW / RPI; ++t) {
        const int r = t * RPI + rsub;  // row within the warp's RW rows (RW is a multiple of 8)
        uint32_t row = __shfl_sync(0xffffffffu, t * RPI < 32 ? g.i[0] : g.i[1], r & 31);
        if (PAIR) {
            const uint32_t row2 = __shfl_sync(0xffffffffu, t * RPI < 32 ? g2.i[0] : g2.i[1], r & 31);
            row = u < 8 ? row : row2;
        }
        cp_async16(dst0 + (uint32_t)(t * RPI) * 128 + (uint32_t)(((u & 7) ^ (r & 7)) << 4),
                   src0 + row * (uint32_t)ldB);
    }
}

// The items a persistent CTA works through: its groups k = blockIdx.x,
// blockIdx.x + gridDim.x, ..., each as TI consecutive items (its sample tiles
// when TI > 1).
template <int TI>
struct Items {
    int64_t k;
    int ti = 0;
    __device__ explicit Items(int64_t k0) : k(k0) {}
    __device__ void next()
    {
        if (++ti == TI) {
            ti = 0;
            k += gridDim.x;
        }
    }
};

// nothing to do after a group's copies are issued
struct NoAfterIssue {
    __device__ bool operator()(int, uint32_t) const { return true; }
};

// Producer loop shared by the forward and the weight gradient: per group, one
// thread arms the stage barrier with the TMA bytes (`tma_bytes`, issued by
// `issue_tma`), every producer thread copies its share of H_k and has the
// copy hardware arrive on the stage barrier once its copies land, so the
// producers run ahead as far as free stages allow.  The cp.async writes are
// generic-proxy writes: every MMA warp fences (proxy.async) after it has seen
// the stage barrier and before its MMAs read the stage.  `after(s, ph)` runs
// once per group, with the group's stage and phase, right after the copies of
// the next group are issued (the last group's after the loop); it returns
// false if a wait in it gave up.  TI > 1: each group is TI items, item ti
// gathering samples 128 ti .. 128 ti + 127 (and the TMA copies again).
template <int F_ = 0, int U_ = 0, bool PAIR = false, int TI = 1, int NPW = kProdWarps, typename IssueTma,
          typename AfterIssue = NoAfterIssue>
__device__ __forceinline__ void producer_loop(Ctl &c, uint32_t stage0, uint32_t stage_bytes, int S,
                                              int64_t K, const uint16_t *idx_s, const uint16_t *hT,
                                              int ldB, int F, int MT, uint32_t tma_bytes,
                                              volatile int *abort_flag, int32_t *status,
                                              IssueTma issue_tma, int ishift = 0,
                                              AfterIssue after = AfterIssue())
{
    static_assert(TI == 1 || !PAIR, "pairs hold one sample tile");
    const int t = threadIdx.x;  // producer threads are 0 .. NPW*32-1
    const int lane = t & 31;
    const int units = MT * 16;
    int it = 0;
    // PAIR: kernel group k is the layout groups 2k (first chunk) and 2k + 1
    GatherIdx cur = {{0u, 0u}}, cur2 = {{0u, 0u}};
    if (blockIdx.x < K) {
        cur = gather_idx_of<NPW>(idx_s, PAIR ? 2 * (int64_t)blockIdx.x : (int64_t)blockIdx.x >> ishift, F, lane);
        if (PAIR)
            cur2 = gather_idx_of<NPW>(idx_s, 2 * (int64_t)blockIdx.x + 1, F, lane);
    }
    Ring r;
    int prev_s = 0;
    uint32_t prev_ph = 0;
    for (Items<TI> itm(blockIdx.x); itm.k < K; itm.next(), ++it, r.next(S)) {
        const int64_t k = itm.k;
        const int s = r.i;
        const uint32_t ph = r.ph;
        GatherIdx nxt = cur, nxt2 = cur2;
        if (itm.ti == TI - 1 && k + gridDim.x < K) {
            nxt = gather_idx_of<NPW>(idx_s, PAIR ? 2 * (k + gridDim.x) : (k + gridDim.x) >> ishift, F, lane);
            if (PAIR)
                nxt2 = gather_idx_of<NPW>(idx_s, 2 * (k + gridDim.x) + 1, F, lane);
        }
        FW_TRACE(0, it);
        if (!mbar_wait(bar_addr(c.empty[s]), ph ^ 1u, abort_flag, status))
            break;
        FW_TRACE(1, it);
        const uint32_t A = stage0 + (uint32_t)s * stage_bytes;
        if (t == 0) {
            mbar_arrive_expect_tx(bar_addr(c.full[s]), tma_bytes);
            issue_tma(k, A, bar_addr(c.full[s]));
        }
        const uint16_t *hTi = TI > 1 ? hT + itm.ti * 128 : hT;
        if constexpr (F_ > 0)
            issue_gather_t<F_, U_, PAIR, NPW>(hTi, ldB, A, cur, lane, cur2);
        else
            issue_gather(hTi, ldB, A, F, units, cur, lane);
        cp_async_arrive_noinc(bar_addr(c.full[s]));
        FW_TRACE(2, it);
        cur = nxt;
        cur2 = nxt2;
        if (it > 0 && !after(prev_s, prev_ph)) {
            ++it;
            break;
        }
        prev_s = s;
        prev_ph = ph;
    }
    if (it > 0 && !*abort_flag)
        after(prev_s, prev_ph);
    cp_async_wait_all();
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
    uint8_t *dZt;          // group-tiled dZ output (instead of dZ / dZ_lo)
    uint64_t tile_bytes;
    int32_t zsw, nzc, Bp;
    const int32_t *gptr, *gent;
    double *loss_part;
    int32_t *status;
    int64_t K, L;
    int32_t B, G, F, MT, nk, cw, S, issuers, ldB;
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
        // W_k: nk boxes of cw columns (rows of 2 cw bytes, swizzle of that width)
        producer_loop(c, stage0, a.stage_bytes, S, a.K, a.idx_s, a.hT, a.ldB, F, a.MT, a.w_bytes,
                      abort_flag, a.status, [&](int64_t k, uint32_t A, uint32_t fb) {
                          const uint32_t Wt = A + a.a_bytes;
                          for (int kc = 0; kc < a.nk; ++kc)
                              tma_load_2d(Wt + (uint32_t)kc * G * 2 * a.cw, &tm_w, kc * a.cw, (int)(k * G), fb);
                      });
    } else if (warp < kFirstEpi) {
        // ---------------------------------------------------------- MMA issue
        const int me = warp - kProdWarps;
        const uint32_t idesc = idesc_bf16(128, G, 1, 0);
        const uint32_t wlay = layout_for_swizzle(2 * a.cw);
        const int cw_shift = a.cw == 64 ? 6 : a.cw == 32 ? 5 : 4;  // cw is 16, 32 or 64
        int it = 0;
        Ring rs;
        for (int64_t k = blockIdx.x; k < a.K; k += gridDim.x, ++it, rs.next(S)) {
            if ((a.issuers == 2 ? (it & 1) : 0) != me)
                continue;
            const int s = rs.i;
            const uint32_t ph = rs.ph;
            const int acc = acc_slot(it, a.issuers);
            if (!mbar_wait(bar_addr(c.tempty[acc]), acc_phase(it, a.issuers) ^ 1u, abort_flag, a.status))
                break;
            tc_fence_after();
            if (!mbar_wait(bar_addr(c.full[s]), ph, abort_flag, a.status))
                break;
            tc_fence_after();
            fence_proxy_async();  // cp.async-written H_k -> the MMA (async proxy)
            if (lane == 0) {
                const uint32_t A = stage0 + (uint32_t)s * a.stage_bytes;
                const uint32_t Wt = A + a.a_bytes;
                for (int t = 0; t < a.MT; ++t) {
                    const uint32_t d = tbase + (uint32_t)(acc * per + t * G);
                    for (int st = 0; st < F / 16; ++st) {
                        // A: H_k, MN-major; 8 f-rows per 1024-byte atom, b chunks F*128 apart
                        const uint64_t ad = sdesc(A + (uint32_t)t * 2 * F * 128 + (uint32_t)st * 2048,
                                                  (uint32_t)F * 128, 1024, kLayoutSW128);
                        // B: W_k, K-major; box 16 st / cw, 32 bytes per 16 f inside a 2 cw-byte row
                        const int f0 = st * 16;
                        const uint64_t bd = sdesc(Wt + (uint32_t)(f0 >> cw_shift) * G * 2 * a.cw +
                                                      (uint32_t)(f0 & (a.cw - 1)) * 2,
                                                  16, 16 * a.cw, wlay);
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
        double lacc = 0.0;  // folded in from lf every 32 groups (fp64 is slow on this part)
        float lf = 0.f;
        int it = 0;
        // positive-list bounds of the group, loaded one group ahead
        int e0n = 0, e1n = 0;
        if (BCE && blockIdx.x < a.K) {
            e0n = __ldg(a.gptr + blockIdx.x);
            e1n = __ldg(a.gptr + blockIdx.x + 1);
        }
        for (int64_t k = blockIdx.x; k < a.K; k += gridDim.x, ++it) {
            const int acc = acc_slot(it, a.issuers);
            const int e0 = e0n, e1 = e1n;
            if (BCE && k + gridDim.x < a.K) {
                e0n = __ldg(a.gptr + k + gridDim.x);
                e1n = __ldg(a.gptr + k + gridDim.x + 1);
            }
            if (!mbar_wait(bar_addr(c.tfull[acc]), acc_phase(it, a.issuers), abort_flag, a.status))
                break;
            tc_fence_after();
            // unit u = (tile t, columns c0 ..): t = u / (G / CH), c0 = (u % (G / CH)) CH,
            // stepped without dividing by the run-time G
            int t = 0, c0 = sub * CH;
            auto next_unit = [&]() {
                for (; c0 >= G; c0 -= G)
                    ++t;
            };
            next_unit();
            for (int u = sub; u < units; u += 2, c0 += 2 * CH, next_unit()) {
                const int b = t * 128 + q * 32 + lane;
                float v[CH];
                tmem_ld_chunk<CH>(tbase + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * per + t * G + c0), v);
                if (BCE && a.dZt) {
                    // every row of the tile is written; rows >= B hold zeros
                    if (b < a.B) {
                        const uint32_t y = e1 > e0 ? group_pos_mask(a.gent, e0, e1, b, c0, CH) : 0u;
                        lf += bce_chunk_ftz<CH>(v, y);
                    } else {
#pragma unroll
                        for (int i = 0; i < CH; ++i)
                            v[i] = 0.f;
                    }
                    store_dz_tile<CH>(a.dZt + (size_t)k * a.tile_bytes, b, c0, v, a.zsw, a.nzc, a.Bp);
                    continue;
                }
                if (b >= a.B)
                    continue;
                const int64_t off = (int64_t)b * a.L + k * G + c0;
                if (a.Z)
                    store_bf16_row<CH>(a.Z + off, nullptr, v);
                if (BCE) {
                    const uint32_t y = e1 > e0 ? group_pos_mask(a.gent, e0, e1, b, c0, CH) : 0u;
                    lf += bce_chunk_ftz<CH>(v, y);
                    store_bf16_row<CH>(a.dZ + off, a.dZ_lo ? a.dZ_lo + off : nullptr, v);
                }
            }
            tc_fence_before();
            mbar_arrive(bar_addr(c.tempty[acc]));
            if ((it & 31) == 31) {
                lacc += (double)lf;
                lf = 0.f;
            }
        }
        if (BCE)
            epi_sum_to(lacc + (double)lf, c, a.loss_part + blockIdx.x, kFirstEpi);
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
    const uint8_t *dZt;    // group-tiled dZ input (else the tensor maps)
    uint64_t tile_bytes;
    uint16_t *dW;
    int32_t *status;
    int64_t K, L;
    int32_t B, G, F, MT, FT, S, nzc, zsw, planes, ncat, Nacc, issuers, ldB;
    int32_t stream_t;  // 1: one 128-sample tile per stage, MT stages per group
    uint32_t a_bytes, z_bytes, stage_bytes, tmem_cols;
};

// The producers of the dW stage when a group's sample tiles stream through
// the stages one at a time: group k, tile t fills stage (k's position) * MT + t
// with the tile's H_k rows and dZ rows.
template <typename IssueTma>
__device__ __forceinline__ void producer_loop_tiles(Ctl &c, uint32_t stage0, uint32_t stage_bytes, int S,
                                                    int64_t K, int MT, const uint16_t *idx_s,
                                                    const uint16_t *hT, int ldB, int F, uint32_t tma_bytes,
                                                    volatile int *abort_flag, int32_t *status,
                                                    IssueTma issue_tma)
{
    const int t0 = threadIdx.x;
    const int lane = t0 & 31;
    int it = 0;
    bool live = true;
    Ring r;
    for (int64_t k = blockIdx.x; k < K && live; k += gridDim.x) {
        const GatherIdx cur = gather_idx_of(idx_s, k, F, lane);
        for (int t = 0; t < MT; ++t, ++it, r.next(S)) {
            const int s = r.i;
            const uint32_t ph = r.ph;
            if (!mbar_wait(bar_addr(c.empty[s]), ph ^ 1u, abort_flag, status)) {
                live = false;
                break;
            }
            const uint32_t A = stage0 + (uint32_t)s * stage_bytes;
            if (t0 == 0) {
                mbar_arrive_expect_tx(bar_addr(c.full[s]), tma_bytes);
                issue_tma(k, t, A, bar_addr(c.full[s]));
            }
            issue_gather(hT + (size_t)t * 128, ldB, A, F, 16, cur, lane);
            cp_async_arrive_noinc(bar_addr(c.full[s]));
        }
    }
    cp_async_wait_all();
    if (*abort_flag) {
        for (int j = it - S < 0 ? 0 : it - S; j < it; ++j)
            mbar_wait_drain(bar_addr(c.full[j % S]), (uint32_t)(j / S) & 1u);
    }
}

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
    const int MTs = a.stream_t ? 1 : a.MT;  // sample tiles held by one stage
    const int T = a.stream_t ? a.MT : 1;    // stages per group
    const uint32_t zrows = (uint32_t)MTs * 128;
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

    if (warp < kProdWarps && T > 1) {
        producer_loop_tiles(c, stage0, a.stage_bytes, S, a.K, T, a.idx_s, a.hT, a.ldB, F, a.z_bytes, abort_flag,
                            a.status, [&](int64_t k, int t, uint32_t A, uint32_t fb) {
                                const uint32_t Zs = A + a.a_bytes;
                                for (int pc = 0; pc < a.planes * a.nzc; ++pc) {
                                    const int pl = pc / a.nzc, cj = pc % a.nzc;
                                    if (a.dZt) {
                                        // rows [128 t, 128 t + 128) of chunk cj of plane pl
                                        const size_t src = (size_t)k * a.tile_bytes +
                                                           ((size_t)pc * a.MT * 128 + (size_t)t * 128) * a.zsw;
                                        bulk_load(Zs + (uint32_t)pc * zchunk, a.dZt + src, zchunk, fb);
                                    } else {
                                        tma_load_2d(Zs + (uint32_t)pc * zchunk, pl ? &tm_zl : &tm_z,
                                                    (int)(k * G + cj * 64), t * 128, fb);
                                    }
                                }
                            });
    } else if (warp < kProdWarps) {
        producer_loop(c, stage0, a.stage_bytes, S, a.K, a.idx_s, a.hT, a.ldB, F, a.MT, a.z_bytes,
                      abort_flag, a.status, [&](int64_t k, uint32_t A, uint32_t fb) {
                          const uint32_t Zs = A + a.a_bytes;
                          if (a.dZt) {  // the tile is the stage image of both planes
                              bulk_load(Zs, a.dZt + (size_t)k * a.tile_bytes, a.z_bytes, fb);
                              return;
                          }
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
        bool live = true;
        Ring rs;  // stage of sequence number it * T + t
        for (int64_t k = blockIdx.x; k < a.K && live; k += gridDim.x, ++it) {
            if ((a.issuers == 2 ? (it & 1) : 0) != me) {
                for (int t = 0; t < T; ++t)
                    rs.next(S);
                continue;
            }
            const int acc = acc_slot(it, a.issuers);
            if (!mbar_wait(bar_addr(c.tempty[acc]), acc_phase(it, a.issuers) ^ 1u, abort_flag, a.status))
                break;
            tc_fence_after();
          for (int t = 0; t < T; ++t, rs.next(S)) {
            const int s = rs.i;
            const uint32_t ph = rs.ph;
            if (!mbar_wait(bar_addr(c.full[s]), ph, abort_flag, a.status)) {
                live = false;
                break;
            }
            tc_fence_after();
            fence_proxy_async();  // cp.async-written H_k -> the MMA (async proxy)
            if (lane == 0) {
                const uint32_t A = stage0 + (uint32_t)s * a.stage_bytes;
                const uint32_t Zs = A + a.a_bytes;
                for (int tf = 0; tf < a.FT; ++tf) {
                    const uint32_t d = tbase + (uint32_t)(acc * per + tf * a.Nacc);
                    for (int ps = 0; ps < passes; ++ps) {
                        for (int st = 0; st < MTs * 8; ++st) {
                            // A: H_k^T, K-major (rows f, K = b): b chunk st/4, 32 B per 16 b
                            const uint64_t ad = sdesc(A + (uint32_t)(st / 4) * F * 128 +
                                                          (uint32_t)tf * 128 * 128 + (uint32_t)(st % 4) * 32,
                                                      16, 1024, kLayoutSW128);
                            // B: dZ_k, MN-major (N = j, K = b): 16 b rows per step
                            const uint64_t bd = sdesc(Zs + (uint32_t)ps * zplane + (uint32_t)st * 16 * a.zsw,
                                                      zchunk, 8 * a.zsw, zlayout);
                            mma_bf16(d, ad, bd, idesc, (t > 0 || ps > 0 || st > 0) ? 1u : 0u);
                        }
                    }
                }
                mma_commit(bar_addr(c.empty[s]));
                if (t == T - 1)
                    mma_commit(bar_addr(c.tfull[acc]));
            }
            __syncwarp();
          }
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
            // unit u = (f tile tf, columns c0 ..), stepped as in the forward stage
            int tf = 0, c0 = sub * CH;
            auto next_unit = [&]() {
                for (; c0 >= G; c0 -= G)
                    ++tf;
            };
            next_unit();
            for (int u = sub; u < units; u += 2, c0 += 2 * CH, next_unit()) {
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
                if (f < F) {  // lanes past F (last f tile) hold nothing to store
                    uint16_t *dst = a.dW + (k * G + c0) * F + f;
#pragma unroll
                    for (int i = 0; i < CH; ++i)
                        dst[(int64_t)i * F] = bf16_rn(v[i]);
                }
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

// ================================================================== fused forward + BCE + dW
// One pass over the groups for the training step: per group the producers
// gather H_k and load W_k, one MMA warp computes Z_k = H_k W_k^T, the epilogue
// turns it into dZ_k (BCE), writes it to the group-tiled workspace as one fp16
// plane (for dh) and into shared memory as bf16 value + residual planes, and a
// second MMA warp computes dW_k^T = H_k^T [dZ_hi | dZ_lo] from the same
// shared-memory H_k, so H_k is gathered once and dZ_k is never read back for
// dW.  The dW warps store dW_k (or, in the SGD instance, apply the momentum
// update to it and store the new W_k); the producers record max |W| for
// dh's fp16 scale.
// Warps: the producers, one forward MMA warp, one dW MMA warp, eight BCE
// warps and four dW warps.
// BCE warps, a multiple of the four TMEM lane quarters: eight in the plain
// instance; four in the momentum-SGD one, whose dW warps (the update's loads
// and stores of m and W) set its pace and gain the issue slots (SGD step
// 1.886 -> 1.800 ms at 3M; the plain instance measured 16 % slower with four)
__host__ __device__ constexpr int fw_bce(bool sgd) { return sgd ? 4 : 8; }
// dW store warps, a multiple of the four TMEM lane quarters: four, or
// sixteen in the momentum-SGD instance, where they carry the update (four
// per lane quarter on 8-column units; SGD step at 3M 1.798 ms with four,
// 1.677 with eight, then 1.576 -> 1.551 ms from eight to sixteen)
__host__ __device__ constexpr int fw_dw(bool sgd) { return sgd ? 16 : 4; }
// Producer warps: four where a stage holds one 128-sample tile (eight
// measured up to 4 % slower there: each producer warp's per-group costs of
// waits, index loads, the max |W| pass and arrivals took issue slots from the
// rest; two, 10 % slower), eight where it holds two (four: 2.4 % slower;
// twice the gather per group); two in the momentum-SGD instance at F <= 128
// (its update-bound dW warps gain the issue slots: SGD step 1.677 -> 1.590
// ms at 3M).
__host__ __device__ constexpr int fw_prod(int MT, int FK, bool sgd)
{
    return MT > 1 ? 8 : (sgd && FK <= 8) ? 2 : 4;
}
__host__ __device__ constexpr int fw_threads(int MT, bool sgd, int FK)
{
    return 32 * (fw_prod(MT, FK, sgd) + 2 + fw_bce(sgd) + fw_dw(sgd));
}
// dynamic shared memory the fused plan may use (the opt-in maximum is 227 KB)
constexpr int kFWBudget = 224 * 1024;

struct FWPlan {
    bool ok = false;
    int MT = 0, FT = 0, nk = 0, S = 0, zsw = 0, nzc = 0, nslot = 0;
    int TI = 1;  // sample tiles of a group streamed through the stages as separate items (MT = 1)
    int gs = 0, sub = 1;  // labels per kernel group (a subgroup sharing I_k) and subgroups per group
    uint32_t a_bytes = 0, w_bytes = 0, stage_bytes = 0, dz_bytes = 0, stg_bytes = 0, zcols = 0, wcols = 0,
             tmem_cols = 0, pad_bytes = 0;
    // the fp16 dZ tile staged in shared memory (two buffers) and bulk-stored,
    // where that costs no stage; 0: the epilogue stores it to global memory
    uint32_t f16_bytes = 0;
};

// the plan for groups of Gv labels (Gv = G, or a subgroup size).  `stream`
// (B > 128): a group's two sample tiles pass through the stages as two items
// of one tile each, the dW MMA accumulating over both, so a stage, the dZ
// buffers and the fp16 staging hold one tile's rows.
FWPlan plan_fwdw_g(const sg_layout *lo, int B, int Gv, bool stream = false)
{
    FWPlan p;
    if (!shape_ok(lo) || !dz_ok(Gv) || (lo->F != 64 && lo->F != 128 && lo->F != 256) ||
        2 * Gv > 256 || B < 1 || B > 256)
        return p;
    p.MT = (B + 127) / 128;
    if (p.MT * 128 > lo->ldB)
        return p;
    if (stream) {
        // the items' rows are contiguous in the workspace tile only with one
        // 64-column chunk
        if (p.MT < 2 || Gv > 64)
            return p;
        p.TI = p.MT;
        p.MT = 1;
    }
    // dW tiles of M = 128 rows of f; with F = 64 the upper 64 accumulator
    // lanes read the next 64 rows of shared memory and are never stored
    p.FT = (lo->F + 127) / 128;
    p.nk = lo->F / 64;
    p.zsw = dz_swizzle(Gv);
    p.nzc = Gv * 2 > 128 ? Gv / 64 : 1;
    p.a_bytes = (uint32_t)p.MT * 2 * lo->F * 128;
    p.w_bytes = (uint32_t)p.nk * Gv * 128;
    p.stage_bytes = p.a_bytes + p.w_bytes;
    p.dz_bytes = 2u * (uint32_t)p.nzc * p.MT * 128 * p.zsw;  // both planes, all rows
    p.stg_bytes = (uint32_t)Gv * lo->F * 2;                 // dW_k staged for its store
    p.zcols = (uint32_t)p.MT * Gv;
    p.wcols = (uint32_t)p.FT * 2 * Gv;
    p.nslot = 4 * (p.zcols + p.wcols) <= 512 ? 4 : 2;
    if (p.nslot * (p.zcols + p.wcols) > 512)
        return p;
    p.tmem_cols = pow2_cols(p.nslot * (p.zcols + p.wcols));
    // F = 64: the last stage's dW MMA reads up to 8 KB past it
    p.pad_bytes = lo->F < 128 ? 8192u : 0u;
    // two dW_k staging buffers
    const long room = (long)kFWBudget - 2l * p.dz_bytes - 2l * p.stg_bytes - (long)p.pad_bytes;
    p.S = room > 0 ? (int)(room / p.stage_bytes) : 0;
    if (p.S > 6)
        p.S = 6;
    p.ok = p.S >= 2;
    // two staging buffers for the fp16 tile when the stages still fit: the
    // epilogue's 16-byte global stores of the tile measured ~10 % of the
    // kernel's time at B <= 128, F >= 128 (3M shape: 4.5 % faster with one
    // bulk store per group); with F = 64 or two sample tiles the groups are
    // shorter and the dW MMA warp's wait for the store's reads measured 1-3 %
    // slower, so those keep the direct stores
    const uint32_t f16 = (uint32_t)p.nzc * p.MT * 128 * p.zsw;
    const long room2 = room - 2l * f16;
    const int S2 = room2 > 0 ? (int)(room2 / p.stage_bytes) : 0;
    if (p.ok && p.MT == 1 && lo->F >= 128 && S2 >= 2 && S2 >= (p.S < 4 ? p.S : 4)) {
        p.f16_bytes = f16;
        p.S = S2 > 6 ? 6 : S2;
    }
    return p;
}

// With B > 128 a group's two sample tiles stream through the stages as
// separate items (at B = 256, F = 128 the forward kernel measured 4-5 %
// faster than with both tiles in one stage at G = 16 and 32, and it is the
// only way G = 64 fits); both tiles in one stage remain the fallback.
// Groups that fit neither way run as subgroups of half the labels sharing
// the group's I_k: the kernel then sees K * sub groups of G / sub labels,
// each with its own workspace tile.
FWPlan plan_fwdw(const sg_layout *lo, int B)
{
    // subgroups of G, G / 2 or G / 4 labels
    for (int gs = lo->G; gs >= 16 && lo->G % gs == 0 && 4 * gs >= lo->G; gs /= 2) {
        FWPlan p = plan_fwdw_g(lo, B, gs, true);
        if (!p.ok)
            p = plan_fwdw_g(lo, B, gs);
        if (p.ok) {
            p.gs = gs;
            p.sub = lo->G / gs;
            return p;
        }
        if (gs % 2)
            break;
    }
    return FWPlan();
}

struct FWArgs {
    const uint16_t *idx_s, *hT;
    uint8_t *dZt;
    uint64_t tile_bytes;
    uint16_t *dW;     // dW, or the updated weights when `mom` is set
    uint32_t *wmax;   // max |W| (bf16 magnitude bits) over the step, for dh (zero at entry)
    uint32_t *wmax_next;  // the other slot, cleared by CTA 0 for the next launch
    float *dh_zero;       // dh to clear (dh_n floats) for the dh kernel, or nullptr
    int32_t dh_n;
    // momentum SGD in the dW epilogue (mom != nullptr): m <- mu m + dW,
    // W_out <- bf16(W - lr m), W_out written where dW would be
    const uint16_t *W;
    float *mom;
    float lr, mu;
    const int32_t *gptr, *gent;
    double *loss_part;
    // the step's loss: the CTA that takes the last ticket sums the partials
    // in block order (no separate launch); the ticket starts at zero
    double *loss;
    uint32_t *ticket;
    int32_t *status;
    int64_t K, L;
    int32_t B, G, F, MT, FT, nk, S, zsw, nzc, nslot, Bp, ldB;
    int32_t sub_shift;  // log2 of the kernel groups per layout group (they share its I_k and positives)
    uint32_t a_bytes, w_bytes, stage_bytes, dz_bytes, stg_bytes, zcols, wcols, tmem_cols;
    uint32_t f16_bytes;  // fp16 tile staging buffer (0: stored from registers)
};

// the common control block (stages; tfull/tempty = Z accumulators; drain of
// the forward MMA warps) plus the barriers of the dW half
struct CtlFW {
    Ctl c;
    uint64_t wfull[4], wempty[4];    // dW accumulators
    uint64_t dzfull[2], dzempty[2];  // dZ_k in shared memory
    uint64_t wdrain[2];              // drain of the dW MMA warps
};

// The MMA issue loops have compile-time trip counts (FK = F/16 K steps, MT
// sample tiles): tcgen05.mma issued from a loop with a run-time trip count
// measured about 2x slower per instruction than the same MMAs unrolled.
//
// SGD: the dW epilogue applies the momentum-SGD update instead of storing dW
// (its own instance, so the plain step's kernel carries none of that code).
//
// PAIR (B <= 64, one 128-row sample tile): kernel group k is the layout
// groups 2k and 2k + 1 of GL = G_ / 2 labels each.  The stage's two 64-sample
// chunks hold their H rows (the first group's samples as rows 0 .. 63, the
// second's as rows 64 .. 127) and W_k their 2 GL consecutive weight rows, so
// one forward MMA of N = 2 GL computes both groups' logits (plus two unused
// off-diagonal blocks) and one dW MMA set over the 128 rows both weight
// gradients, with dZ block-diagonal in shared memory (the off-diagonal
// blocks are cleared once and never written).  Each layout group's fp16 dZ
// tile is written as without pairing.
//
// TI = 2 (B > 128, one 64-column dZ chunk): a group's two sample tiles are two
// items, each with its own stage (H rows of its 128 samples and W_k), forward
// MMA, BCE and dZ buffer; the dW MMA accumulates over both items and the dW
// warps see the group once.  A group of 64 labels then needs the shared
// memory of one tile instead of two, and runs as one group with N = 64 MMAs
// instead of two subgroups of 32 with twice as many.
// The loss ticket of the fused kernel, out of line (its SGD instance): the
// warp of the CTA that takes the last ticket sums the partials, lane l the
// partials l, l + 32, ..., then a fixed shuffle tree, and resets the ticket.
static __device__ __noinline__ void fw_loss_ticket(const double *part, double *loss, uint32_t *ticket, int lane)
{
    uint32_t last = 0;
    if (lane == 0) {
        __threadfence();  // this CTA's partial before its ticket
        last = atomicAdd(ticket, 1u) == gridDim.x - 1 ? 1u : 0u;
    }
    if (__shfl_sync(0xffffffffu, last, 0)) {
        __threadfence();
        double sum = 0.0;
        for (unsigned i = lane; i < gridDim.x; i += 32)
            sum += __ldcg(part + i);
        for (int o = 16; o > 0; o >>= 1)
            sum += __shfl_down_sync(0xffffffffu, sum, o);
        if (lane == 0) {
            *loss = sum;
            *ticket = 0u;  // for the next launch
        }
    }
}

template <int G_, int FK, int MT, bool SGD, bool PAIR = false, int TI = 1>
__global__ void __launch_bounds__(fw_threads(MT, SGD, FK), 1)
    k_tc_fwdw(const __grid_constant__ CUtensorMap tm_w, const FWArgs a)
{
    constexpr int NPW = fw_prod(MT, FK, SGD), NTHR = fw_threads(MT, SGD, FK), FIRST_EPI = NPW + 2;
    constexpr int NBCE = fw_bce(SGD), kBcePerQ = NBCE / 4;
    constexpr int NDW = fw_dw(SGD), kDwPerQ = NDW / 4;
    static_assert(NBCE % 4 == 0 && NBCE <= kEpiWarps, "whole lane quarters");
    static_assert(!PAIR || MT == 1, "pairs share one 128-row sample tile");
    // compile-time group width: column chunk of the epilogue (with pairs,
    // half a layout group's columns, so that both BCE warps of a lane quarter
    // work on its diagonal block), dZ row width (swizzle) and 64-column chunks
    // of the dZ tile
    constexpr int CH = PAIR ? G_ / 4 : G_ >= 64 && TI == 1 ? 32 : 16;
    constexpr int ZSW = G_ * 2 >= 128 ? 128 : G_ * 2;
    constexpr int NZC = G_ * 2 > 128 ? G_ / 64 : 1;
    static_assert(TI == 1 || (MT == 1 && !PAIR && NZC == 1), "streamed tiles: one tile per item, one dZ chunk");
    __shared__ CtlFW cf;
    Ctl &c = cf.c;
    extern __shared__ uint8_t dsm[];
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const uint32_t base = (smem_u32(dsm) + 1023u) & ~1023u;
    uint8_t *base_ptr = dsm + (base - smem_u32(dsm));
    // [dZ_k buffer 0][dZ_k buffer 1][dW_k staging 0, 1][fp16 tile staging 0, 1][stages]
    const uint32_t stg0 = base + 2 * a.dz_bytes;
    const uint32_t f160 = stg0 + 2 * a.stg_bytes;  // fp16 tile staging (two buffers, or none)
    const uint32_t stage0 = f160 + 2 * a.f16_bytes;
    constexpr int G = G_;
    const int F = a.F, S = a.S, NS = a.nslot;
    constexpr uint32_t zrows = (uint32_t)MT * 128;
    constexpr uint32_t zchunk = zrows * (uint32_t)ZSW;
    // the stage geometry follows from the shape: H_k (MT sample tiles of
    // 2 x 64 samples x F rows) then W_k (F/64 chunks of G rows x 128 bytes)
    constexpr uint32_t kABytes = (uint32_t)MT * 2 * FK * 16 * 128;
    constexpr uint32_t kWBytes = (uint32_t)((FK + 3) / 4) * G_ * 128;
    constexpr uint32_t kDzBytes = 2u * NZC * MT * 128 * ZSW;
    const uint32_t wbase = (uint32_t)NS * a.zcols;  // first dW accumulator column

    // the epilogue is two teams: the BCE warps turn Z_k into dZ_k, the dW
    // warps store dW of the group.  A stage is freed by the dW MMA (last
    // reader of H_k) and by the producer warps, which take max |W_k| from it
    // one group after they issued its copies.
    if (threadIdx.x == 0) {
        setup_ctl(c, S, 0, NPW * 32 + 1, NPW + 1);
        for (int i = 0; i < NS && i < 4; ++i) {
            mbar_init(bar_addr(c.tfull[i]), 1);
            mbar_init(bar_addr(c.tempty[i]), NBCE * 32);
            mbar_init(bar_addr(cf.wfull[i]), 1);
            mbar_init(bar_addr(cf.wempty[i]), NDW * 32);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_addr(cf.dzfull[i]), NBCE * 32);
            // freed by the dW MMA (commit)
            mbar_init(bar_addr(cf.dzempty[i]), 1);
            mbar_init(bar_addr(cf.wdrain[i]), 1);
        }
        fence_mbar_init();
    }
    if (warp == NPW) {
        tmem_alloc(smem_u32(&c.tmem), a.tmem_cols);
        tmem_relinquish();
    }
    if (PAIR) {
        // both dZ buffers start zero: the BCE writes only the diagonal blocks
        for (uint32_t o = threadIdx.x * 16u; o < 2 * a.dz_bytes; o += NTHR * 16u)
            *reinterpret_cast<uint4 *>(base_ptr + o) = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async();  // generic writes -> the dW MMA (async proxy)
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = c.tmem;
    volatile int *abort_flag = &c.abort_flag;
    // the other max |W| slot for the next launch (read by no one until then),
    // and this CTA's share of dh for the dh kernel that follows: by every
    // thread here, or (SGD) by the dW warps before their first group.  Where
    // these few instructions and the loss ticket below sit in the code moved
    // the SGD instance's time by up to 5 % either way (1.422 ms with this
    // arrangement, 1.501 ms with the plain instance's), and the plain one's
    // by 1 % the other way, so each keeps the arrangement it measured
    // fastest with.
    if (!SGD) {
        if (blockIdx.x == 0 && threadIdx.x == 0)
            *a.wmax_next = 0u;
        for (int i = blockIdx.x * NTHR + threadIdx.x; i < a.dh_n; i += gridDim.x * NTHR)
            a.dh_zero[i] = 0.f;
    }

    if (warp < NPW) {
        // ---------------------------------------------------------- producers
        // After issuing a group's copies the producers take max |W| over the
        // previous group's W_k (the scale of the feature gradient's fp16
        // operands; that group's copies have landed by then) and release its
        // stage, so no epilogue warp holds a stage.
        uint32_t wmag = 0;  // running max of |W| bits, two bf16 lanes
        const int t = threadIdx.x;
        producer_loop<FK * 16, MT * 16, PAIR, TI, NPW>(
            c, stage0, a.stage_bytes, S, a.K, a.idx_s, a.hT, a.ldB, F, a.MT, a.w_bytes, abort_flag, a.status,
            [&](int64_t k, uint32_t A, uint32_t fb) {
                const uint32_t Wt = A + a.a_bytes;
                for (int kc = 0; kc < a.nk; ++kc)
                    tma_load_2d(Wt + (uint32_t)kc * G * 128, &tm_w, kc * 64, (int)(k * G), fb);
            },
            a.sub_shift,
            [&](int sj, uint32_t phj) -> bool {
                if (!mbar_wait(bar_addr(c.full[sj]), phj, abort_flag, a.status))
                    return false;
                const uint4 *Wsm = reinterpret_cast<const uint4 *>(base_ptr + (stage0 - base) +
                                                                   (size_t)sj * a.stage_bytes + kABytes);
#pragma unroll
                for (int x = t; x < (int)(kWBytes / 16); x += NPW * 32) {
                    const uint4 v = Wsm[x];
                    wmag = __vmaxu2(wmag, v.x & 0x7fff7fffu);
                    wmag = __vmaxu2(wmag, v.y & 0x7fff7fffu);
                    wmag = __vmaxu2(wmag, v.z & 0x7fff7fffu);
                    wmag = __vmaxu2(wmag, v.w & 0x7fff7fffu);
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar_addr(c.empty[sj]));  // done with the stage's W_k
                return true;
            });
        wmag = max(wmag & 0xffffu, wmag >> 16);
        for (int o = 16; o > 0; o >>= 1)
            wmag = max(wmag, __shfl_xor_sync(0xffffffffu, wmag, o));
        if (lane == 0)
            atomicMax(a.wmax, wmag);
    } else if (warp == NPW) {
        // ---------------------------------------------------------- forward MMA
        const uint32_t idesc = idesc_bf16(128, G, 1, 0);
        int it = 0;
        Ring rs, rz;
        for (Items<TI> itm(blockIdx.x); itm.k < a.K; itm.next(), ++it, rs.next(S), rz.next(NS)) {
            const int s = rs.i;
            const int zs = rz.i;
            FW_TRACE(0, it);
            if (!mbar_wait(bar_addr(c.tempty[zs]), rz.ph ^ 1u, abort_flag, a.status))
                break;
            FW_TRACE(1, it);
            tc_fence_after();
            if (!mbar_wait(bar_addr(c.full[s]), rs.ph, abort_flag, a.status))
                break;
            FW_TRACE(2, it);
            tc_fence_after();
            fence_proxy_async();  // cp.async-written H_k -> the MMA (async proxy)
            if (lane == 0) {
                // one thread issues an MMA about every 100 cycles at best, and
                // address arithmetic between the MMAs adds to that: the
                // descriptors are the stage's base descriptor plus constants.
                // A descriptor's address field is addr >> 4 (below 2^14 for
                // any shared address), so an offset adds to the whole word.
                const uint32_t A = stage0 + (uint32_t)s * (kABytes + kWBytes);
                const uint64_t ad0 = sdesc(A, (uint32_t)FK * 2048, 1024, kLayoutSW128);
                const uint64_t bd0 = sdesc(A + kABytes, 16, 1024, kLayoutSW128);
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    const uint32_t d = tbase + (uint32_t)(zs * a.zcols + t * G);
#pragma unroll
                    for (int st = 0; st < FK; ++st)
                        mma_bf16(d, ad0 + (uint64_t)(((uint32_t)t * 2 * FK * 2048 + (uint32_t)st * 2048) >> 4),
                                 bd0 + (uint64_t)(((uint32_t)(st / 4) * G * 128 + (uint32_t)(st % 4) * 32) >> 4),
                                 idesc, st > 0 ? 1u : 0u);
                }
                mma_commit(bar_addr(c.tfull[zs]));
            }
            __syncwarp();
        }
        if (lane == 0)
            mma_commit(bar_addr(c.drain[0]));
        __syncwarp();
        mbar_wait_drain(bar_addr(c.drain[0]), 0);
    } else if (warp < FIRST_EPI) {
        // ---------------------------------------------------------- dW MMA
        const uint32_t zlayout = layout_for_swizzle(ZSW);
        const uint32_t idesc = idesc_bf16(128, 2 * G, 0, 1);  // N = [hi | lo] along j
        int it = 0;
        Ring rs, rw;  // rs per item, rw per group
        for (Items<TI> itm(blockIdx.x); itm.k < a.K; itm.next(), ++it, rs.next(S)) {
            const int64_t k = itm.k;
            const int s = rs.i;
            const int ws = rw.i;
            const int db = it & 1;
            FW_TRACE(0, it);
            if (itm.ti == 0 && !mbar_wait(bar_addr(cf.wempty[ws]), rw.ph ^ 1u, abort_flag, a.status))
                break;
            FW_TRACE(1, it);
            tc_fence_after();
            if (!mbar_wait(bar_addr(cf.dzfull[db]), (uint32_t)(it >> 1) & 1u, abort_flag, a.status))
                break;
            FW_TRACE(2, it);
            // H_k of this stage landed long ago (the forward MMA used it); this
            // warp sees the barrier itself before its MMAs read the cp.async data
            if (!mbar_wait(bar_addr(c.full[s]), rs.ph, abort_flag, a.status))
                break;
            tc_fence_after();
            fence_proxy_async();
            if (lane == 0 && a.f16_bytes) {
                // the staged fp16 tile to the workspace; its shared-memory
                // reads are waited for before the buffer is released (dzempty)
                bulk_store(a.dZt + (size_t)k * a.tile_bytes + (size_t)itm.ti * a.f16_bytes,
                           f160 + (uint32_t)db * a.f16_bytes, a.f16_bytes);
                bulk_commit();
            }
            if (lane == 0) {
                // base descriptors plus constants (as above)
                constexpr int NT = (FK + 7) / 8, NKS = MT * 8;
                const uint32_t A = stage0 + (uint32_t)s * (kABytes + kWBytes);
                const uint64_t ad0 = sdesc(A, 16, 1024, kLayoutSW128);
                const uint64_t bd0 = sdesc(base + (uint32_t)db * kDzBytes, zchunk, 8 * ZSW, zlayout);
#pragma unroll
                // the second and later items of a group add to its accumulator
                const uint32_t acc0 = TI > 1 && itm.ti > 0 ? 1u : 0u;
#pragma unroll
                for (int tf = 0; tf < NT; ++tf) {
                    const uint32_t d = tbase + wbase + (uint32_t)(ws * a.wcols + tf * 2 * G);
#pragma unroll
                    for (int st = 0; st < NKS; ++st)
                        mma_bf16(d,
                                 ad0 + (uint64_t)(((uint32_t)(st / 4) * FK * 2048 + (uint32_t)tf * 128 * 128 +
                                                   (uint32_t)(st % 4) * 32) >> 4),
                                 bd0 + (uint64_t)(((uint32_t)st * 16 * ZSW) >> 4), idesc, st > 0 ? 1u : acc0);
                }
                if (itm.ti == TI - 1)
                    mma_commit(bar_addr(cf.wfull[ws]));
                if (a.f16_bytes)
                    bulk_wait_read<0>();  // the fp16 tile store has read the buffer
                mma_commit(bar_addr(cf.dzempty[db]));
                mma_commit(bar_addr(c.empty[s]));  // last reader of the stage's H_k
            }
            __syncwarp();
            if (itm.ti == TI - 1)
                rw.next(NS);
        }
        if (lane == 0) {
            if (a.f16_bytes)
                bulk_wait<0>();  // every fp16 tile store has landed
            mma_commit(bar_addr(cf.wdrain[0]));
        }
        __syncwarp();
        mbar_wait_drain(bar_addr(cf.wdrain[0]), 0);
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int ew = warp - FIRST_EPI;  // BCE warps 0 .. NBCE-1, then the dW warps
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        if (ew < NBCE) {
            double lacc = 0.0;  // folded in from lf every 32 groups (fp64 is slow on this part)
            float lf = 0.f;
            const int sub = ew / 4;  // the kBcePerQ warps of a lane quarter split the column units
            // Z_k -> BCE -> dZ_k (workspace tile and shared memory for the dW MMA)
            constexpr int zunits = MT * (G / CH);
            // positive-list bounds of the group, loaded one group ahead (with
            // pairs, of both groups: entries e0 .. e1 and e1 .. e2)
            int e0n = 0, e1n = 0, e2n = 0;
            if (blockIdx.x < a.K) {
                const int64_t kl = PAIR ? 2 * (int64_t)blockIdx.x : (int64_t)blockIdx.x >> a.sub_shift;
                e0n = __ldg(a.gptr + kl);
                e1n = __ldg(a.gptr + kl + 1);
                if (PAIR)
                    e2n = __ldg(a.gptr + kl + 2);
            }
            int it = 0;
            Ring rz;
            int e0 = 0, e1 = 0, e2 = 0;
            for (Items<TI> itm(blockIdx.x); itm.k < a.K; itm.next(), ++it, rz.next(NS)) {
                const int64_t k = itm.k;
                const int zs = rz.i;
                const int db = it & 1;
                if (itm.ti == 0) {
                    e0 = e0n;
                    e1 = e1n;
                    e2 = e2n;
                    if (k + gridDim.x < a.K) {
                        const int64_t kl = PAIR ? 2 * (k + gridDim.x) : (k + gridDim.x) >> a.sub_shift;
                        e0n = __ldg(a.gptr + kl);
                        e1n = __ldg(a.gptr + kl + 1);
                        if (PAIR)
                            e2n = __ldg(a.gptr + kl + 2);
                    }
                }
                // columns of the layout group this kernel group starts at
                const int coff = (int)(k & ((1 << a.sub_shift) - 1)) * G;
                FW_TRACE(0, it);
                if (!mbar_wait(bar_addr(c.tfull[zs]), rz.ph, abort_flag, a.status))
                    break;
                FW_TRACE(1, it);
                // the dZ buffer of two groups ago must have been consumed by its dW MMA
                if (!mbar_wait(bar_addr(cf.dzempty[db]), ((uint32_t)(it >> 1) & 1u) ^ 1u, abort_flag, a.status))
                    break;
                FW_TRACE(2, it);
                tc_fence_after();
                uint8_t *zs_smem = base_ptr + (size_t)db * a.dz_bytes;
                if constexpr (PAIR) {
                    // lane quarters 0, 1: the first group's samples (rows
                    // 0 .. 63), columns 0 .. GL - 1; quarters 2, 3: the second
                    // group's, columns GL .. 2 GL - 1
                    constexpr int GL = G / 2;
                    constexpr int ZSW_L = GL * 2 >= 128 ? 128 : GL * 2;  // the layout group's tile rows
                    const int grp = q >> 1;
                    const int ga = grp ? e1 : e0, gb = grp ? e2 : e1;
                    const int64_t kl = 2 * k + grp;
                    const int bz = q * 32 + lane, b = bz & 63;
#pragma unroll
                    for (int hc = sub; hc < 2; hc += kBcePerQ) {  // the two CH-column halves
                    const int cl = hc * CH, c0 = grp * GL + cl;
                    float v[CH];
                    tmem_ld_chunk<CH>(tbase + lane_off + (uint32_t)(zs * a.zcols + c0), v);
                    if (b < a.B) {
                        const uint32_t y = gb > ga ? group_pos_mask(a.gent, ga, gb, b, cl, CH) : 0u;
                        lf += bce_chunk_ftz<CH>(v, y);
                    } else {
#pragma unroll
                        for (int i = 0; i < CH; ++i)
                            v[i] = 0.f;
                    }
                    store_dz_tile<CH>(zs_smem, bz, c0, v, ZSW, NZC, 128);
                    store_dz_tile_f16<CH>(a.dZt + (size_t)kl * a.tile_bytes, b, cl, v, ZSW_L, 128);
                    }
                } else {
#pragma unroll
                for (int u = sub; u < zunits; u += kBcePerQ) {
                    const int t = u / (G / CH), c0 = (u % (G / CH)) * CH;
                    const int b = t * 128 + q * 32 + lane;  // row of the item's tiles
                    const int bg = TI > 1 ? itm.ti * 128 + b : b;  // sample
                    float v[CH];
                    tmem_ld_chunk<CH>(tbase + lane_off + (uint32_t)(zs * a.zcols + t * G + c0), v);
                    if (bg < a.B) {
                        const uint32_t y = e1 > e0 ? group_pos_mask(a.gent, e0, e1, bg, coff + c0, CH) : 0u;
                        lf += bce_chunk_ftz<CH>(v, y);
                    } else {
#pragma unroll
                        for (int i = 0; i < CH; ++i)
                            v[i] = 0.f;
                    }
                    // bf16 value + residual planes for the dW MMA; the fp16
                    // tile for the feature gradient straight to the workspace
                    store_dz_tile<CH>(zs_smem, b, c0, v, ZSW, NZC, MT * 128);
                    if (a.f16_bytes)  // bulk-stored by the dW MMA warp
                        store_dz_tile_f16<CH>(base_ptr + (f160 - base) + (size_t)db * a.f16_bytes, b, c0, v, ZSW,
                                              MT * 128);
                    else
                        store_dz_tile_f16<CH>(a.dZt + (size_t)k * a.tile_bytes, bg, c0, v, ZSW, TI * MT * 128);
                }
                }
                FW_TRACE(3, it);
                tc_fence_before();
                mbar_arrive(bar_addr(c.tempty[zs]));
                fence_proxy_async();  // dZ_k in shared memory -> the dW MMA (async proxy)
                mbar_arrive(bar_addr(cf.dzfull[db]));
                if ((it & 31) == 31) {
                    lacc += (double)lf;
                    lf = 0.f;
                }
            }
            epi_sum_to(lacc + (double)lf, c, a.loss_part + blockIdx.x, FIRST_EPI, NBCE);
            if (SGD) {
                if (ew == 0 && a.loss)
                    fw_loss_ticket(a.loss_part, a.loss, a.ticket, lane);
            } else if (ew == 0 && a.loss) {
                // the warp of the CTA that takes the last ticket sums the
                // partials: lane l the partials l, l + 32, ..., then a fixed
                // shuffle tree (one thread summing them serially at the end of
                // the kernel cost 8-15 us)
                uint32_t last = 0;
                if (lane == 0) {
                    __threadfence();  // this CTA's partial before its ticket
                    last = atomicAdd(a.ticket, 1u) == gridDim.x - 1 ? 1u : 0u;
                }
                if (__shfl_sync(0xffffffffu, last, 0)) {
                    __threadfence();
                    double sum = 0.0;
                    for (unsigned i = lane; i < gridDim.x; i += 32)
                        sum += __ldcg(a.loss_part + i);
                    for (int o = 16; o > 0; o >>= 1)
                        sum += __shfl_down_sync(0xffffffffu, sum, o);
                    if (lane == 0) {
                        *a.loss = sum;
                        *a.ticket = 0u;  // for the next launch
                    }
                }
            }
        } else {
            // dW_k^T accumulator [f lanes][hi j | lo j] -> dW rows k*G + j,
            // staged in shared memory as [j][f] and stored with one bulk copy.
            // The team leaves together: every named barrier below is then
            // reached by all of its warps or by none.
            const int dw = ew - NBCE;  // 0 .. NDW-1
            const int dsub = dw / 4;   // the kDwPerQ warps of a lane quarter split the column units
            if (SGD) {
                if (blockIdx.x == 0 && dw == 0 && lane == 0)
                    *a.wmax_next = 0u;
                for (int i = blockIdx.x * (NDW * 32) + dw * 32 + lane; i < a.dh_n; i += gridDim.x * (NDW * 32))
                    a.dh_zero[i] = 0.f;
            }
            // columns of a dW epilogue unit: CH, or 8 where four dW warps share
            // a lane quarter
            constexpr int CHW = kDwPerQ > 2 ? 8 : CH;
            constexpr int wunits = ((FK + 7) / 8) * (G / CHW);
            int it = 0;
            Ring rw;
            for (int64_t k = blockIdx.x; k < a.K; k += gridDim.x, ++it, rw.next(NS)) {
                const int ws = rw.i;
                const int wb = it & 1;
                uint16_t *stg = reinterpret_cast<uint16_t *>(base_ptr + 2 * (size_t)a.dz_bytes + (size_t)wb * a.stg_bytes);
                FW_TRACE(0, it);
                // ---- dW_k
                if (SGD) {
                    // the optimiser step's rows of m and W into L2 while the
                    // dW MMA runs (lane r: row k G + r, this warp's 32 f)
                    for (int r = lane; r < G; r += 32) {
#pragma unroll
                        for (int tf = 0; tf < (FK + 7) / 8; ++tf) {
                            if ((tf * (G / CHW) + r / CHW) % kDwPerQ != dsub)
                                continue;  // another warp's column unit
                            const int64_t e = (k * G + r) * (int64_t)F + tf * 128 + q * 32;
                            prefetch_l2(a.mom + e);
                            prefetch_l2(a.W + e);
                        }
                    }
                }
                FW_TRACE(1, it);
                if (named_bar_any(2, NDW * 32,
                                  !mbar_wait(bar_addr(cf.wfull[ws]), rw.ph, abort_flag, a.status)))
                    break;
                FW_TRACE(2, it);
                tc_fence_after();
                // the staging buffer's store of two groups ago has read it
                if (dw == 0 && lane == 0)
                    bulk_wait_read<1>();
                named_bar(2, NDW * 32);
#pragma unroll 1
                for (int u = dsub; u < wunits; u += kDwPerQ) {
                    const int tf = u / (G / CHW), c0 = (u % (G / CHW)) * CHW;
                    const int f = tf * 128 + q * 32 + lane;
                    const uint32_t col = tbase + lane_off + wbase + (uint32_t)(ws * a.wcols + tf * 2 * G + c0);
                    float v[CHW], w[CHW];
                    tmem_ld_chunk2<CHW>(col, col + (uint32_t)G, v, w);
                    if (SGD && f < F) {
                        // the optimiser step on dW while it is in registers
                        // (lanes run along f: coalesced rows of m and W)
                        const int64_t e0 = (k * G + c0) * (int64_t)F + f;
                        float mv[CHW];
                        uint16_t wv[CHW];
#pragma unroll
                        for (int i = 0; i < CHW; ++i) {
                            mv[i] = a.mom[e0 + (int64_t)i * F];
                            wv[i] = __ldg(a.W + e0 + (int64_t)i * F);
                        }
#pragma unroll
                        for (int i = 0; i < CHW; ++i) {
                            const float m = fmaf(a.mu, mv[i], v[i] + w[i]);
                            a.mom[e0 + (int64_t)i * F] = m;
                            stg[(c0 + i) * F + f] = bf16_rn(__uint_as_float((uint32_t)wv[i] << 16) - a.lr * m);
                        }
                    } else if (f < F) {
#pragma unroll
                        for (int i = 0; i < CHW; ++i)
                            stg[(c0 + i) * F + f] = bf16_rn(v[i] + w[i]);
                    }
                }
                FW_TRACE(3, it);
                tc_fence_before();
                mbar_arrive(bar_addr(cf.wempty[ws]));
                fence_proxy_async();  // staged dW_k -> the bulk store (async proxy)
                named_bar(2, NDW * 32);
                if (dw == 0 && lane == 0) {
                    bulk_store(a.dW + k * G * F, stg0 + (uint32_t)wb * a.stg_bytes, a.stg_bytes);
                    bulk_commit();
                }
            }
            if (dw == 0 && lane == 0)
                bulk_wait<0>();  // every dW store has landed
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == NPW) {
        tc_fence_after();
        tmem_dealloc(tbase, a.tmem_cols);
    }
}

// ================================================================== dh
struct DhArgs {
    const uint16_t *idx_s;  // [K][F] sorted index rows I_k
    const uint16_t *W;     // [L][F] in slot order
    const uint32_t *wmax;  // max |W| bits of the step (fp16 operands only)
    const uint8_t *dZt;    // group-tiled dZ input (else the tensor maps)
    uint64_t tile_bytes;
    float *dh;
    int32_t *status;
    int64_t K, L, Kc;      // K: subgroups; Kc: subgroups per CTA (a contiguous range)
    int32_t B, G, F, H, MT, S, zsw, nbands, band_w, parts, npass, Bp, nbuf;
    int32_t sub;           // subgroups (<= 64 labels) per dZ workspace tile
    int32_t idiv;          // subgroups per group (they share its index row)
    int32_t sub_shift, idiv_shift;  // log2 of sub and idiv where they are powers of two, else -1
    uint32_t z_bytes, w_bytes, i_bytes, stage_bytes, ws_bytes, tmem_cols;
};


struct CtlDh {
    Ctl c;                                           // stages, drain
    uint64_t wfull[kDhMaxBuf], wempty[kDhMaxBuf];    // scattered-W buffers
};

// CTA (band, mtile, part): dh columns [i0, i0 + BW) of the band (BW = 128 BWT),
// samples [128 mt, 128 mt + 128), the contiguous groups [Kc part, Kc part + Kc).
//
// The scatter-add of dH_k = dZ_k W_k into the columns I_k of dh is itself a
// product:
//     dh[:, band] += dZ_k Ws_k,   Ws_k[j][i - i0] = W_k[j][f] where I_k[f] = i
// (zero columns elsewhere).  The accumulator (M = 128 samples, N = BW dh
// columns: one MMA of N = 256 and one of N = 128 per K step at BW = 384) stays
// in TMEM over all the CTA's groups and is added to dh once at the end.  A is
// the group's dZ tile (K-major, rows = samples) as it arrives in shared
// memory; B = Ws_k^T (K-major, one 2G-byte row per dh column) lives in
// shared memory, zero except for the rows of the band's I_k: builder thread
// (g, f) copies column f of the staged W_k to row I_k[f] - i0 when that falls
// in the band, after zeroing the row it wrote the last time the buffer was
// used (the buffers start zeroed).  Loads, builders and MMAs move in
// units of P groups: one stage and one Ws buffer per unit.
//
// Compile-time shape: NPASS dZ planes, NKS = G/16 K steps per plane, BWT
// 128-column blocks per band.  F16: dZ is one fp16 plane (the training step's
// workspace) and the builders write W_k as fp16, scaled by 2^-s so that the
// step's largest |W| stays finite (s = 0 unless |W| >= 2^15); the flush
// scales the sums back by 2^s.
// Column f of a staged W_k ([G][F] row-major, bf16) as NCW 16-byte units (8
// labels each) of its Ws row, kept as bf16 or converted to fp16 as below
template <int NCW, bool F16, bool SCALED>
__device__ __forceinline__ void read_w_column(const uint16_t *Wk, int F, float down, uint4 (&row)[NCW])
{
#pragma unroll
    for (int u = 0; u < NCW; ++u) {
        uint32_t w[4];
#pragma unroll
        for (int c2 = 0; c2 < 4; ++c2) {
            const uint32_t lo = Wk[(8 * u + 2 * c2) * F], hi = Wk[(8 * u + 2 * c2 + 1) * F];
            if (F16)
                w[c2] = SCALED ? pack2_f16(__uint_as_float(lo << 16) * down, __uint_as_float(hi << 16) * down)
                               : pack2_f16(__uint_as_float(lo << 16), __uint_as_float(hi << 16));
            else
                w[c2] = lo | (hi << 16);
        }
        row[u] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Columns f and f + 1 of a staged W_k ([G][F] row-major, bf16) as the same
// NCWH 16-byte units (8 labels each) of their two Ws rows, from one 4-byte
// load per label: `Wp` points at the word (first label, f), F2 = F / 2 words
// per W_k row.  The values are kept as bf16, or converted to fp16 (times
// `down` when SCALED; unscaled when the step's largest |W| is below 2^15,
// which spares a multiply per value).
template <int NCWH, bool F16, bool SCALED>
__device__ __forceinline__ void read_w_pair(const uint32_t *Wp, int F2, float down, uint4 (&ra)[NCWH],
                                            uint4 (&rb)[NCWH])
{
#pragma unroll
    for (int u = 0; u < NCWH; ++u) {
        uint32_t wa[4], wb[4];
#pragma unroll
        for (int c2 = 0; c2 < 4; ++c2) {
            const uint32_t w0 = Wp[(8 * u + 2 * c2) * F2], w1 = Wp[(8 * u + 2 * c2 + 1) * F2];
            if (F16) {
                const float a0 = __uint_as_float(w0 << 16), a1 = __uint_as_float(w1 << 16);
                const float b0 = __uint_as_float(w0 & 0xffff0000u), b1 = __uint_as_float(w1 & 0xffff0000u);
                wa[c2] = SCALED ? pack2_f16(a0 * down, a1 * down) : pack2_f16(a0, a1);
                wb[c2] = SCALED ? pack2_f16(b0 * down, b1 * down) : pack2_f16(b0, b1);
            } else {
                wa[c2] = __byte_perm(w0, w1, 0x5410);  // the low halves: column f
                wb[c2] = __byte_perm(w0, w1, 0x7632);  // the high halves: column f + 1
            }
        }
        ra[u] = make_uint4(wa[0], wa[1], wa[2], wa[3]);
        rb[u] = make_uint4(wb[0], wb[1], wb[2], wb[3]);
    }
}

template <int NPASS, int NKS, int BWT, bool F16, int ISS = 1, int FMX = 256>
__global__ void __launch_bounds__(dh_threads(ISS), 1)
    k_tc_dh(const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_zl,
            const DhArgs a)
{
    static_assert(!F16 || NPASS == 1, "the fp16 dZ workspace has one plane");
    static_assert(ISS == 1 || ISS == 2, "one or two MMA-issuing warps");
    constexpr int FIRST_B = 1 + ISS;  // warp 0: loads, warps 1 .. ISS: MMA, then the builders
    constexpr int G = NKS * 16;
    constexpr int RB = 2 * G;         // bytes of one Ws row (one dh column)
    constexpr int BW = BWT * 128;     // dh columns of the band
    constexpr int N0 = BW > 256 ? 256 : BW;
    constexpr int N1 = BW - N0;       // 0 or 128
    constexpr int NCW = G / 8;        // 16-byte units of a row
    constexpr int P = dh_units(G);
    __shared__ CtlDh cd;
    Ctl &c = cd.c;
    extern __shared__ uint8_t dsm[];
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const uint32_t base = (smem_u32(dsm) + 1023u) & ~1023u;
    uint8_t *base_ptr = dsm + (base - smem_u32(dsm));
    // [Ws buffers][stages]; a stage: [dZ x P][W_k x P][I_k x P]
    const uint32_t stage0 = base + (uint32_t)a.nbuf * a.ws_bytes;
    uint8_t *stage0_ptr = base_ptr + (size_t)a.nbuf * a.ws_bytes;
    const int F = a.F, S = a.S, NB = a.nbuf;
    const uint32_t zoff = 0, woff = P * a.z_bytes, ioff = P * (a.z_bytes + a.w_bytes);
    const int band = blockIdx.x % a.nbands;
    const int mt = (blockIdx.x / a.nbands) % a.MT;
    const int part_id = blockIdx.x / (a.nbands * a.MT);
    const int i0 = band * BW;
    const uint32_t zchunk = 128u * (uint32_t)a.zsw;  // one plane of one group (G <= 64)
    const int64_t kbeg = (int64_t)part_id * a.Kc;
    const int64_t kend = kbeg + a.Kc < a.K ? kbeg + a.Kc : a.K;

    // stages: full = loads landed; empty = the MMAs (and builders) are done
    // with them.  wfull/wempty: Ws buffer written / consumed.
    if (threadIdx.x == 0) {
        setup_ctl(c, S, 0, 1, ISS);  // every issuer releases stages and buffers
        for (int i = 0; i < NB && i < kDhMaxBuf; ++i) {
            mbar_init(bar_addr(cd.wfull[i]), kDhBuilders / NB);  // one arrival per warp of its team
            mbar_init(bar_addr(cd.wempty[i]), ISS);
        }
        fence_mbar_init();
    }
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
        // ---------------------------------------------------------- producer
        int it = 0;
        Ring rs;
        for (int64_t k0 = kbeg; k0 < kend; k0 += P, ++it, rs.next(S)) {
            const int s = rs.i;
            const int np = kend - k0 < P ? (int)(kend - k0) : P;
            DH_TRACE(0, it);
            if (!mbar_wait(bar_addr(c.empty[s]), rs.ph ^ 1u, abort_flag, a.status))
                break;
            DH_TRACE(1, it);
            const uint32_t st = stage0 + (uint32_t)s * a.stage_bytes;
            const uint32_t fb = bar_addr(c.full[s]);
            if (lane == 0)
                mbar_arrive_expect_tx(fb, (uint32_t)np * (a.z_bytes + a.w_bytes + (uint32_t)(2 * F)));
            __syncwarp();
            if (lane < np) {
                // lane g loads group k0 + g
                const int64_t k = k0 + lane;
                const uint32_t Zs = st + zoff + (uint32_t)lane * a.z_bytes;
                if (a.dZt) {
                    // rows [128 mt, 128 mt + 128) of the subgroup's chunk of
                    // each plane of its group's tile
                    const int64_t kg = a.sub_shift >= 0 ? (k >> a.sub_shift) : (int64_t)((uint32_t)k / (uint32_t)a.sub);
                    const int cj = (int)(k - kg * a.sub);
                    const uint8_t *tz = a.dZt + (size_t)kg * a.tile_bytes +
                                        ((size_t)cj * a.Bp + (size_t)mt * 128) * a.zsw;
                    for (int pl = 0; pl < NPASS; ++pl)
                        bulk_load(Zs + (uint32_t)pl * zchunk, tz + (size_t)pl * a.sub * a.Bp * a.zsw, zchunk, fb);
                } else {
                    tma_load_2d(Zs, &tm_z, (int)(k * G), mt * 128, fb);
                    if (NPASS > 1)
                        tma_load_2d(Zs + zchunk, &tm_zl, (int)(k * G), mt * 128, fb);
                }
                // W_k: G contiguous rows of F
                bulk_load(st + woff + (uint32_t)lane * a.w_bytes, a.W + k * G * F, a.w_bytes, fb);
                // I_k: the dh column of each f (shared by the group's subgroups)
                const int64_t ki = a.idiv_shift >= 0 ? (k >> a.idiv_shift) : (int64_t)((uint32_t)k / (uint32_t)a.idiv);
                bulk_load(st + ioff + (uint32_t)lane * a.i_bytes, a.idx_s + ki * F, (uint32_t)(2 * F), fb);
            }
            __syncwarp();
        }
        drain_loads(c, it, S);
    } else if (warp <= ISS) {
        // ---------------------------------------------------------- MMA issue
        // One warp issues an N = 256 and an N = 128 MMA per K step (a band of
        // 384 columns), or, with ISS = 2, two warps each one MMA over half of
        // the band's columns into their half of the accumulator: one thread
        // issues a tcgen05.mma about every 100 cycles (N <= 128) to 128 (N =
        // 256), which sets the pace where the builders have little to do.
        // Descriptors: everything but the start address is fixed, and within
        // a unit the start addresses differ by compile-time offsets.
        constexpr int ZSW = 2 * G >= 128 ? 128 : 2 * G;  // dZ row bytes (= a.zsw)
        constexpr uint32_t ZCH = 128u * ZSW;             // one plane of one group
        constexpr uint32_t ZB = NPASS * ZCH;             // one group's dZ (= a.z_bytes)
        constexpr int NH = BW / ISS;                     // columns of this warp's accumulator
        constexpr int NA = ISS == 1 ? N0 : NH, NB1 = ISS == 1 ? N1 : 0;
        const int mh = warp - 1;
        const uint32_t dcol = tbase + (uint32_t)(mh * NH);
        const uint32_t boff = (uint32_t)(mh * NH * RB);
        const uint64_t adesc0 = sdesc(0, 16, 8 * ZSW, layout_for_swizzle(ZSW));
        const uint64_t bdesc0 = sdesc(0, 16, 8 * RB, layout_for_swizzle(RB));
        constexpr uint32_t id0 = F16 ? idesc_f16(128, NA, 0, 0) : idesc_bf16(128, NA, 0, 0);
        constexpr uint32_t id1 = NB1 == 0 ? 0u : F16 ? idesc_f16(128, NB1 > 0 ? NB1 : 16, 0, 0)
                                                      : idesc_bf16(128, NB1 > 0 ? NB1 : 16, 0, 0);
        int it = 0, buf = 0;
        uint32_t wph = 0;
        Ring rs;
        for (int64_t k0 = kbeg; k0 < kend; k0 += P, ++it, rs.next(S)) {
            const int s = rs.i;
            const int np = kend - k0 < P ? (int)(kend - k0) : P;
            DH_TRACE(0, it);
            if (!mbar_wait(bar_addr(c.full[s]), rs.ph, abort_flag, a.status))
                break;
            DH_TRACE(1, it);
            if (!mbar_wait(bar_addr(cd.wfull[buf]), wph, abort_flag, a.status))
                break;
            DH_TRACE(2, it);
            tc_fence_after();
            if (lane == 0) {
                // A: dZ (rows = samples), B: Ws rows (dh columns); 16 j per K step
                const uint64_t au = adesc0 + (uint64_t)((stage0 + (uint32_t)s * a.stage_bytes + zoff) >> 4);
                const uint64_t bu = bdesc0 + (uint64_t)((base + (uint32_t)buf * a.ws_bytes + boff) >> 4);
#pragma unroll
                for (int g = 0; g < P; ++g) {
                    if (g < np) {
#pragma unroll
                        for (int ks2 = 0; ks2 < NPASS * NKS; ++ks2) {
                            const int ks = ks2 % NKS;
                            const uint32_t acc = (it > 0 || g > 0 || ks2 > 0) ? 1u : 0u;
                            const uint64_t ad = au + ((g * ZB + (ks2 / NKS) * ZCH + ks * 32) >> 4);
                            const uint64_t bd = bu + ((g * BW * RB + ks * 32) >> 4);
                            mma_bf16(dcol, ad, bd, id0, acc);
                            if (NB1 > 0)
                                mma_bf16(dcol + (uint32_t)NA, ad, bd + ((NA * RB) >> 4), id1, acc);
                        }
                    }
                }
                mma_commit(bar_addr(cd.wempty[buf]));
                mma_commit(bar_addr(c.empty[s]));
            }
            __syncwarp();
            if (++buf == NB) {
                buf = 0;
                wph ^= 1u;
            }
        }
        if (lane == 0)
            mma_commit(bar_addr(c.drain[mh]));
        __syncwarp();
        mbar_wait_drain(bar_addr(c.drain[mh]), 0);  // no MMA in flight at the dealloc
    } else {
        // ---------------------------------------------------------- builders
        // NB = 2 teams of kDhBuilders / 2 warps take turns at the units (team
        // t: units t, t + 2, ..., always Ws buffer t), so the teams build
        // concurrently while the MMAs consume.  A slot is FP consecutive
        // features of one group and one span of NCWH 16-byte units (8 labels
        // each) of their Ws rows; a unit has P x HS x F/FP slots (HS spans per
        // row), and team thread tt handles slots e = tt, tt + NT, ... (group
        // g = e / (HS F/FP), then the span h, then the feature block fq).
        //   G = 16: FP = 2, one 4-byte load per label gives both features, so
        //     a warp's load moves 128 contiguous bytes instead of 64 (dh at
        //     G = 16: 5 % faster; at G = 32 pairs measured 2 % slower);
        //   G = 32: one feature, whole rows of 32 labels;
        //   G = 64: one feature, half rows: one slot per (g, f) left half the
        //     team idle at F = 128 and gave the other half twice the chain of
        //     dependent loads (1-2 % slower).
        const int NT = kDhBuilders * 32 / NB;  // threads of a team
        constexpr int NT_MIN = kDhBuilders * 32 / 2;
        constexpr int FP = G == 16 ? 2 : 1;                    // features per slot
        // G = 64: half rows; G = 32: whole rows, or half rows in the F <= 64
        // instance (FMX = 64), whose F = 64 features left half the team idle
        constexpr int NCWH = FP == 2 ? 2 : G == 64 ? 4 : FMX <= 64 ? 2 : NCW;  // 16-byte units of a span
        constexpr int HS = NCW / NCWH;                         // spans per Ws row
        constexpr int NSLOT = (P * HS * (FMX / FP) + NT_MIN - 1) / NT_MIN;  // the host keeps F <= FMX
        static_assert(NCW % NCWH == 0, "rows of whole spans");
        const int FW = F / FP;  // feature blocks per row of W_k
        const int tb = threadIdx.x - FIRST_B * 32;  // 0 .. kDhBuilders * 32 - 1
        const int team = tb / NT, tt = tb - team * NT;
        const int q = warp & 3, sub = (warp - FIRST_B) / 4;
        float down = 1.f, up = 1.f;  // 2^-s, 2^s (fp16 operands)
        if (F16) {
            const uint32_t m = __ldg(a.wmax);
            const int e = (int)(m >> 7) - 127;  // exponent of the largest |W|
            const int sh = (m < 0x7f80u && e > 14) ? e - 14 : 0;
            down = __uint_as_float((uint32_t)(127 - sh) << 23);
            up = __uint_as_float((uint32_t)(127 + sh) << 23);
        }
        const bool scaled = down != 1.f;  // the same for every thread of the grid
        // the team's buffer starts zeroed; prev[x][c]: the row that feature
        // FP fq + c of slot x wrote in it
        uint8_t *Wb = base_ptr + (size_t)team * a.ws_bytes;
        for (uint32_t o = (uint32_t)tt * 16; o < a.ws_bytes; o += NT * 16)
            *reinterpret_cast<uint4 *>(Wb + o) = make_uint4(0u, 0u, 0u, 0u);
        int prev[NSLOT][FP];
#pragma unroll
        for (int x = 0; x < NSLOT; ++x)
#pragma unroll
            for (int c = 0; c < FP; ++c)
                prev[x][c] = -1;
        // (group, span, feature block) of each slot: fixed per thread
        int gsl[NSLOT], psl[NSLOT], hsl[NSLOT];
#pragma unroll
        for (int x = 0; x < NSLOT; ++x) {
            const int e = tt + x * NT;
            gsl[x] = e / (HS * FW);
            const int r = e - gsl[x] * HS * FW;
            hsl[x] = HS > 1 ? r / FW : 0;
            psl[x] = r - hsl[x] * FW;
        }
        int it = team;
        uint32_t wph = 0;
        // stage and phase of unit `it`, advanced by NB units per turn
        int s = team % S;
        uint32_t sph = (uint32_t)(team / S) & 1u;
        for (int64_t k0 = kbeg + (int64_t)team * P; k0 < kend; k0 += (int64_t)NB * P, it += NB) {
            const int np = kend - k0 < P ? (int)(kend - k0) : P;
            DH_TRACE(0, it);
            bool ok = mbar_wait(bar_addr(c.full[s]), sph, abort_flag, a.status);
            DH_TRACE(1, it);
            const uint8_t *st = stage0_ptr + (size_t)s * a.stage_bytes;
            // this thread's rows, read from the stage before waiting for the buffer
            uint4 row[NSLOT][FP][NCWH];
            int dst[NSLOT][FP];
#pragma unroll
            for (int x = 0; x < NSLOT; ++x) {
                bool any = false;
                const int g = gsl[x], fq = psl[x];
#pragma unroll
                for (int c = 0; c < FP; ++c)
                    dst[x][c] = -1;
                if (ok && g < np && x * NT < P * HS * FW) {
                    const uint8_t *Ig = st + ioff + (size_t)g * a.i_bytes;
                    // I_k of the slot's features: one 4-byte load for a pair
                    // (F even, rows 4-byte aligned)
                    const uint32_t ii = FP == 2 ? reinterpret_cast<const uint32_t *>(Ig)[fq]
                                                : (uint32_t)reinterpret_cast<const uint16_t *>(Ig)[fq];
#pragma unroll
                    for (int c = 0; c < FP; ++c) {
                        const int i = (int)((ii >> (16 * c)) & 0xffffu) - i0;
                        if (i >= 0 && i < BW) {
                            dst[x][c] = g * BW + i;
                            any = true;
                        }
                    }
                    if (any) {
                        // consecutive threads read consecutive features of a W_k row
                        const uint8_t *Wg = st + woff + (size_t)g * a.w_bytes;
                        if constexpr (FP == 2) {
                            const uint32_t *Wp = reinterpret_cast<const uint32_t *>(Wg) + fq +
                                                 (size_t)hsl[x] * NCWH * 8 * FW;
                            if (F16 && scaled)
                                read_w_pair<NCWH, true, true>(Wp, FW, down, row[x][0], row[x][FP - 1]);
                            else
                                read_w_pair<NCWH, F16, false>(Wp, FW, down, row[x][0], row[x][FP - 1]);
                        } else {
                            const uint16_t *Wk = reinterpret_cast<const uint16_t *>(Wg) + fq +
                                                 (size_t)hsl[x] * NCWH * 8 * F;
                            if (F16 && scaled)
                                read_w_column<NCWH, true, true>(Wk, F, down, row[x][0]);
                            else
                                read_w_column<NCWH, F16, false>(Wk, F, down, row[x][0]);
                        }
                    }
                }
            }
            DH_TRACE(2, it);
            // the buffer's last unit must be through its MMAs before it is rewritten
            ok = ok && mbar_wait(bar_addr(cd.wempty[team]), wph ^ 1u, abort_flag, a.status);
            DH_TRACE(3, it);
            if (named_bar_any(1 + team, NT, !ok))
                break;  // the whole team leaves together
            DH_TRACE(4, it);
            // zero the rows of the buffer's last unit, then write this unit's.
            // Each slot clears the 16-byte units it wrote there (the slots of
            // one row share its (g, f), hence its row, and together cover it),
            // at their swizzled places: unswizzled, every thread of a warp
            // stored unit u of its row into the same banks (a warp's 32 random
            // rows, one wavefront each)
#pragma unroll
            for (int x = 0; x < NSLOT; ++x) {
#pragma unroll
                for (int c2 = 0; c2 < FP; ++c2) {
                    if (prev[x][c2] >= 0) {
                        uint8_t *d = Wb + (size_t)prev[x][c2] * RB;
                        const int sw = swz_of(prev[x][c2], RB);
#pragma unroll
                        for (int u = 0; u < NCWH; ++u)
                            *reinterpret_cast<uint4 *>(d + (((hsl[x] * NCWH + u) ^ sw) << 4)) =
                                make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
            named_bar(1 + team, NT);
            DH_TRACE(5, it);
#pragma unroll
            for (int x = 0; x < NSLOT; ++x) {
#pragma unroll
                for (int c2 = 0; c2 < FP; ++c2) {
                    if (dst[x][c2] >= 0) {
                        uint8_t *d = Wb + (size_t)dst[x][c2] * RB;
                        const int sw = swz_of(dst[x][c2], RB);
#pragma unroll
                        for (int u = 0; u < NCWH; ++u)
                            *reinterpret_cast<uint4 *>(d + (((hsl[x] * NCWH + u) ^ sw) << 4)) = row[x][c2][u];
                    }
                    prev[x][c2] = dst[x][c2];
                }
            }
            fence_proxy_async();  // Ws rows (generic writes) -> the MMA (async proxy)
            __syncwarp();
            DH_TRACE(6, it);
            if (lane == 0)
                mbar_arrive(bar_addr(cd.wfull[team]));
            wph ^= 1u;
            for (s += NB; s >= S; s -= S)
                sph ^= 1u;
        }
        // the accumulator (lanes = samples, columns = the band's dh columns)
        // holds this CTA's partial: add it in, transposed through shared memory
        // (free once every MMA is done) so that the atomics run along dh rows
        if (mbar_wait(bar_addr(c.drain[0]), 0, abort_flag, a.status) &&
            (ISS < 2 || mbar_wait(bar_addr(c.drain[1]), 0, abort_flag, a.status)) && !*abort_flag && it > 0) {
            tc_fence_after();
            float *tr = reinterpret_cast<float *>(base_ptr) + (size_t)(warp - FIRST_B) * 33 * 32;
            const uint32_t lane_off = (uint32_t)(q * 32) << 16;
            for (int cs = sub; cs < BWT; cs += kDhBuilders / 4) {
                for (int c0 = 0; c0 < 128; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tbase + lane_off + (uint32_t)(cs * 128 + c0), r);
                    tmem_ld_wait();
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        tr[lane * 33 + x] = __uint_as_float(r[x]);
                    __syncwarp();
                    const int i = i0 + cs * 128 + c0 + lane;  // this lane's dh column
                    if (i < a.H) {
                        for (int y = 0; y < 32; ++y) {
                            const int b = mt * 128 + q * 32 + y;
                            if (b < a.B)
                                atomicAdd(a.dh + (int64_t)b * a.H + i, F16 ? tr[y * 33 + lane] * up
                                                                           : tr[y * 33 + lane]);
                        }
                    }
                    __syncwarp();
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
// some phase of a step of up to max_B samples fits the tensor cores
bool tc_supported(const sg_layout *lo)
{
    return plan_fwd(lo, lo->max_B).ok || plan_dW(lo, lo->max_B, true).ok || plan_dh(lo, lo->max_B, true).ok;
}

bool tc_stage_ok(const sg_layout *lo, int stage, int B)
{
    switch (stage) {
    case SG_KIND_FWD: return plan_fwd(lo, B).ok;
    case SG_KIND_DW: return plan_dW(lo, B, true).ok;
    case SG_KIND_DH: return plan_dh(lo, B, true).ok;
    default: return false;
    }
}

uint64_t tc_dz_tile_bytes(const sg_layout *lo, int32_t B)
{
    const int Bp = (B + 127) / 128 * 128;
    return 2ull * (uint64_t)Bp * (uint64_t)lo->G * 2ull;
}

bool tc_tiled_ok(const sg_layout *lo, int32_t B)
{
    return dz_ok(lo->G) && plan_fwd(lo, B).ok && plan_dW(lo, B, true).ok && plan_dh(lo, B, true).ok;
}

sg_status tc_fwd(sg_layout *lo, int32_t B, const uint16_t *W, uint16_t *Z, uint16_t *dZ,
                 uint16_t *dZ_lo, uint8_t *dZt, double *loss, cudaStream_t st)
{
    const FwdPlan p = plan_fwd(lo, B);
    if (dZt && !dz_ok(lo->G)) {
        sg_set_error("tc_fwd: group size %d has no tiled dZ layout", lo->G);
        return SG_ERR_UNSUPPORTED;
    }
    if (!p.ok) {
        sg_set_error("tc_fwd: shape not supported by the tensor-core engine");
        return SG_ERR_UNSUPPORTED;
    }
    CUtensorMap tm_w;
    sg_status rc = make_map_2d(&tm_w, W, (uint64_t)lo->F, (uint64_t)lo->L, (uint32_t)p.cw, (uint32_t)lo->G,
                               2 * p.cw, "W");
    if (rc != SG_OK)
        return rc;
    FwdArgs a;
    a.idx_s = lo->idx_s;
    a.hT = lo->hT;
    a.Z = Z;
    a.dZ = dZ;
    a.dZ_lo = dZ_lo;
    a.dZt = dZt;
    a.tile_bytes = tc_dz_tile_bytes(lo, B);
    a.zsw = dz_swizzle(lo->G);
    a.nzc = lo->G * 2 > 128 ? lo->G / 64 : 1;
    a.Bp = p.MT * 128;
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
    a.cw = p.cw;
    a.S = p.S;
    a.issuers = p.issuers;
    a.ldB = lo->ldB;
    a.a_bytes = p.a_bytes;
    a.w_bytes = p.w_bytes;
    a.stage_bytes = p.stage_bytes;
    a.tmem_cols = p.tmem_cols;
    const size_t smem = (size_t)p.S * p.stage_bytes + 1024;
    const int grid = persistent_grid(lo, lo->K);
    const bool bce = dZ != nullptr || dZt != nullptr;
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


// Pairs of groups (the kernel's PAIR form) when one 64-sample chunk holds a
// group's samples: B <= 64, G of 16 or 32 (pairs of 32 or 64 columns), an
// even number of groups, and the plan for 2G-label kernel groups fits.
FWPlan plan_fwdw_pair(const sg_layout *lo, int B)
{
    if (B > 64 || (lo->G != 16 && lo->G != 32) || lo->K % 2 != 0)
        return FWPlan();
    FWPlan p = plan_fwdw_g(lo, B, 2 * lo->G);
    if (!p.ok || p.MT != 1)
        return FWPlan();
    p.gs = 2 * lo->G;
    p.sub = 1;
    p.f16_bytes = 0;  // each layout group's tile is stored from registers
    return p;
}

using FwdwKernel = void (*)(CUtensorMap, FWArgs);

// The instance for a plan (nullptr: none).  Only the instances some plan
// reaches are built: with B > 128 every group streams its sample tiles, and
// G = 64, F = 256 runs as subgroups of 32.
FwdwKernel fwdw_kernel(const FWPlan &p, int F, bool pair, bool sgd)
{
    FwdwKernel kern = nullptr;
#define SG_FW_PICK(GG, KK, MM)                                           \
    if (!pair && p.TI == 1 && p.gs == GG && F == KK * 16 && p.MT == MM)  \
        kern = sgd ? k_tc_fwdw<GG, KK, MM, true> : k_tc_fwdw<GG, KK, MM, false>;
#define SG_FW_STREAM(GG, KK)                                             \
    if (!pair && p.TI == 2 && p.gs == GG && F == KK * 16)               \
        kern = sgd ? k_tc_fwdw<GG, KK, 1, true, false, 2> : k_tc_fwdw<GG, KK, 1, false, false, 2>;
#define SG_FW_PAIR(GG, KK)                                               \
    if (pair && p.gs == GG && F == KK * 16)                             \
        kern = sgd ? k_tc_fwdw<GG, KK, 1, true, true> : k_tc_fwdw<GG, KK, 1, false, true>;
    SG_FW_PICK(16, 4, 1) SG_FW_PICK(16, 8, 1) SG_FW_PICK(16, 16, 1)
    SG_FW_PICK(32, 4, 1) SG_FW_PICK(32, 8, 1) SG_FW_PICK(32, 16, 1)
    SG_FW_PICK(64, 4, 1) SG_FW_PICK(64, 8, 1)
    SG_FW_STREAM(16, 4) SG_FW_STREAM(16, 8) SG_FW_STREAM(16, 16) SG_FW_STREAM(32, 4) SG_FW_STREAM(32, 8) SG_FW_STREAM(32, 16) SG_FW_STREAM(64, 4)
    SG_FW_STREAM(64, 8)
    SG_FW_PAIR(32, 4) SG_FW_PAIR(32, 8) SG_FW_PAIR(32, 16) SG_FW_PAIR(64, 4) SG_FW_PAIR(64, 8) SG_FW_PAIR(64, 16)
#undef SG_FW_PICK
#undef SG_FW_STREAM
#undef SG_FW_PAIR
    return kern;
}

// the step's fused kernel for a plan: pairs of groups where they apply
static FWPlan fwdw_plan_of(const sg_layout *lo, int32_t B, bool *pair)
{
    const FWPlan pp = plan_fwdw_pair(lo, B);
    *pair = pp.ok;
    return pp.ok ? pp : plan_fwdw(lo, B);
}

bool tc_fwdw_ok(const sg_layout *lo, int32_t B)
{
    bool pair = false;
    const FWPlan p = fwdw_plan_of(lo, B, &pair);
    return p.ok && fwdw_kernel(p, lo->F, pair, false) != nullptr;
}

sg_status tc_fwdw(sg_layout *lo, int32_t B, const uint16_t *W, uint8_t *dZt, uint16_t *dW,
                  const sg_sgd *sgd, double *loss, float *dh_zero, cudaStream_t st)
{
    bool pair = false;
    const FWPlan p = fwdw_plan_of(lo, B, &pair);
    if (!p.ok) {
        sg_set_error("tc_fwdw: shape not supported by the fused forward + dW kernel");
        return SG_ERR_UNSUPPORTED;
    }
    // the kernel derives its stage and dZ buffer sizes from its template shape
    if (p.stage_bytes != (uint32_t)p.MT * 2 * lo->F * 128 + (uint32_t)(lo->F / 64) * p.gs * 128 ||
        p.dz_bytes != 2u * (uint32_t)p.nzc * p.MT * 128 * p.zsw || p.zsw != dz_swizzle(p.gs)) {
        sg_set_error("tc_fwdw: internal error: plan and kernel disagree on the stage layout");
        return SG_ERR_UNSUPPORTED;
    }
    CUtensorMap tm_w;
    sg_status rc = make_map_2d(&tm_w, W, (uint64_t)lo->F, (uint64_t)lo->L, 64, (uint32_t)p.gs, 128, "W");
    if (rc != SG_OK)
        return rc;
    FWArgs a;
    a.idx_s = lo->idx_s;
    a.hT = lo->hT;
    rc = tc_ensure_wmax(lo);
    if (rc != SG_OK)
        return rc;
    a.dZt = dZt;
    // one fp16 plane of a kernel group's tile (with pairs: of a layout group's)
    a.tile_bytes = tc_dz_tile_bytes(lo, B) / 2 / p.sub;
    a.dW = dW;
    const int wslot = lo->wmax_slot ^ 1;  // the slot the previous launch cleared
    a.wmax = lo->wmax + wslot;
    a.wmax_next = lo->wmax + (wslot ^ 1);
    a.dh_zero = dh_zero;
    a.dh_n = dh_zero ? B * lo->H : 0;
    a.W = W;
    a.mom = sgd ? sgd->mom : nullptr;
    a.lr = sgd ? sgd->lr : 0.f;
    a.mu = sgd ? sgd->mu : 0.f;
    a.gptr = lo->gptr;
    a.gent = lo->gent;
    a.loss_part = lo->loss_part;
    a.loss = loss;
    a.ticket = lo->wmax + 2;
    a.status = lo->status;
    a.K = pair ? lo->K / 2 : lo->K * p.sub;
    a.sub_shift = log2_exact(p.sub);  // 0, 1 or 2
    a.L = lo->L;
    a.B = B;
    a.G = p.gs;
    a.F = lo->F;
    a.MT = p.MT;
    a.FT = p.FT;
    a.nk = p.nk;
    a.S = p.S;
    a.zsw = p.zsw;
    a.nzc = p.nzc;
    a.nslot = p.nslot;
    a.Bp = p.TI * p.MT * 128;
    a.ldB = lo->ldB;
    a.a_bytes = p.a_bytes;
    a.w_bytes = p.w_bytes;
    a.stage_bytes = p.stage_bytes;
    a.dz_bytes = p.dz_bytes;
    a.stg_bytes = p.stg_bytes;
    a.zcols = p.zcols;
    a.wcols = p.wcols;
    a.tmem_cols = p.tmem_cols;
    // the staged rows are the kernel group's whole workspace tile (with
    // streamed tiles, the item's share of it)
    a.f16_bytes = (uint64_t)p.f16_bytes * p.TI == a.tile_bytes ? p.f16_bytes : 0u;
    const size_t smem = 2 * (size_t)p.dz_bytes + 2 * (size_t)p.stg_bytes + 2 * (size_t)p.f16_bytes +
                        (size_t)p.S * p.stage_bytes + p.pad_bytes + 1024;
    const int grid = persistent_grid(lo, a.K);
    void (*kern)(CUtensorMap, FWArgs) = fwdw_kernel(p, lo->F, pair, sgd != nullptr);
    if (!kern) {
        sg_set_error("tc_fwdw: G = %d, F = %d has no fused kernel", lo->G, lo->F);
        return SG_ERR_UNSUPPORTED;
    }
    rc = set_smem(kern, smem);
    if (rc != SG_OK)
        return rc;
    SG_LAUNCH(lo, SG_KIND_FWD, st,
              kern<<<grid, fw_threads(p.MT, sgd != nullptr, lo->F / 16), smem, st>>>(tm_w, a));
    SG_TRY_CUDA(cudaGetLastError());
    lo->wmax_slot = wslot;  // the slot the dh kernel reads
    return SG_OK;           // the kernel wrote the loss
}

sg_status tc_dW(sg_layout *lo, const uint16_t *dZ, const uint16_t *dZ_lo, const uint8_t *dZt,
                int32_t B, uint16_t *dW, cudaStream_t st)
{
    const DWPlan p = plan_dW(lo, B, dZ_lo != nullptr || dZt != nullptr);
    if (!p.ok) {
        sg_set_error("tc_dW: shape not supported by the tensor-core engine");
        return SG_ERR_UNSUPPORTED;
    }
    CUtensorMap tm_z, tm_zl;
    const int zbox = lo->G < 64 ? lo->G : 64;
    sg_status rc = SG_OK;
    memset(&tm_z, 0, sizeof(tm_z));
    if (!dZt) {
        rc = make_map_2d(&tm_z, dZ, (uint64_t)lo->L, (uint64_t)B, (uint32_t)zbox,
                         (uint32_t)(p.stream_t ? 128 : p.MT * 128), p.zsw, "dZ");
        if (rc != SG_OK)
            return rc;
    }
    tm_zl = tm_z;
    if (dZ_lo && !dZt) {
        rc = make_map_2d(&tm_zl, dZ_lo, (uint64_t)lo->L, (uint64_t)B, (uint32_t)zbox,
                         (uint32_t)(p.stream_t ? 128 : p.MT * 128), p.zsw, "dZ_lo");
        if (rc != SG_OK)
            return rc;
    }
    DWArgs a;
    a.idx_s = lo->idx_s;
    a.hT = lo->hT;
    a.dZt = dZt;
    a.tile_bytes = tc_dz_tile_bytes(lo, B);
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
    a.stream_t = p.stream_t;
    a.a_bytes = p.a_bytes;
    a.z_bytes = p.z_bytes;
    a.stage_bytes = p.stage_bytes;
    a.tmem_cols = p.tmem_cols;
    const size_t smem = (size_t)p.S * p.stage_bytes + p.pad_bytes + 1024;
    const int grid = persistent_grid(lo, lo->K);
    void (*kern)(CUtensorMap, CUtensorMap, DWArgs) = lo->G >= 64 ? k_tc_dW<32> : k_tc_dW<16>;
    rc = set_smem(kern, smem);
    if (rc != SG_OK)
        return rc;
    SG_LAUNCH(lo, SG_KIND_DW, st, kern<<<grid, kFwdThreads, smem, st>>>(tm_z, tm_zl, a));
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}

sg_status tc_ensure_wmax(sg_layout *lo)
{
    if (lo->wmax)
        return SG_OK;
    if (cudaMalloc((void **)&lo->wmax, 16) != cudaSuccess) {
        cudaGetLastError();
        lo->wmax = nullptr;
        sg_set_error("cudaMalloc of 16 bytes for the step's max |W| failed");
        return SG_ERR_OOM;
    }
    SG_TRY_CUDA(cudaMemset(lo->wmax, 0, 16));
    lo->wmax_slot = 0;
    return SG_OK;
}

sg_status tc_dh(sg_layout *lo, const uint16_t *dZ, const uint16_t *dZ_lo, const uint8_t *dZt,
                bool dzt_f16, int32_t B, const uint16_t *W, float *dh, cudaStream_t st)
{
    if (dzt_f16 && (!dZt || !lo->wmax)) {
        sg_set_error("tc_dh: the fp16 dZ workspace comes with the step's max |W|");
        return SG_ERR_INVALID;
    }
    const bool split = dZ_lo != nullptr || (dZt != nullptr && !dzt_f16);
    // the fp16 workspace comes from the fused forward kernel, whose tiles may
    // hold subgroups of the layout's groups
    const DhPlan p = plan_dh(lo, B, split, dzt_f16 ? plan_fwdw(lo, B).gs : 0);
    if (!p.ok) {
        sg_set_error("tc_dh: shape not supported by the tensor-core engine");
        return SG_ERR_UNSUPPORTED;
    }
    CUtensorMap tm_z, tm_zl;
    sg_status rc = SG_OK;
    memset(&tm_z, 0, sizeof(tm_z));
    if (!dZt) {
        rc = make_map_2d(&tm_z, dZ, (uint64_t)lo->L, (uint64_t)B, (uint32_t)p.gs, 128, p.zsw, "dZ");
        if (rc != SG_OK)
            return rc;
    }
    tm_zl = tm_z;
    if (dZ_lo && !dZt) {
        rc = make_map_2d(&tm_zl, dZ_lo, (uint64_t)lo->L, (uint64_t)B, (uint32_t)p.gs, 128, p.zsw,
                         "dZ_lo");
        if (rc != SG_OK)
            return rc;
    }
    if (((uintptr_t)W & 15) != 0) {
        sg_set_error("W: device pointer must be 16-byte aligned");
        return SG_ERR_INVALID;
    }
    DhArgs a;
    a.idx_s = lo->idx_s;
    a.W = W;
    a.wmax = lo->wmax ? lo->wmax + lo->wmax_slot : nullptr;
    a.dZt = dZt;
    // one tile holds sub subgroups of gs labels (a whole group, or the fused
    // forward kernel's subgroup)
    a.tile_bytes = (dzt_f16 ? tc_dz_tile_bytes(lo, B) / 2 : tc_dz_tile_bytes(lo, B)) / (uint64_t)(lo->G / (p.gs * p.sub));
    a.dh = dh;
    a.status = lo->status;
    a.K = lo->K * p.idiv;  // subgroups
    a.sub = p.sub;
    a.idiv = p.idiv;
    a.sub_shift = log2_exact(p.sub);
    a.idiv_shift = log2_exact(p.idiv);
    a.L = lo->L;
    a.B = B;
    a.G = p.gs;
    a.F = lo->F;
    a.H = lo->H;
    a.MT = p.MT;
    a.S = p.S;
    a.zsw = p.zsw;  // = min(2 Gs, 128), which the kernel also derives from Gs
    a.nbands = p.nbands;
    a.band_w = p.band_w;
    a.npass = split ? 2 : 1;
    a.Bp = p.MT * 128;
    int parts = lo->num_sms / (p.nbands * p.MT);
    if (parts < 1)
        parts = 1;
    // contiguous ranges of whole units of subgroups
    int64_t kc = (a.K + parts - 1) / parts;
    kc = (kc + dh_units(p.gs) - 1) / dh_units(p.gs) * dh_units(p.gs);
    parts = (int)((a.K + kc - 1) / kc);
    a.parts = parts;
    a.Kc = kc;
    a.z_bytes = p.z_bytes;
    a.w_bytes = p.w_bytes;
    a.i_bytes = p.i_bytes;
    a.stage_bytes = p.stage_bytes;
    a.ws_bytes = p.ws_bytes;
    a.nbuf = p.nbuf;
    a.tmem_cols = p.tmem_cols;
    // kernel instance for (planes, K steps per plane, 128-column blocks per band)
    void (*kern)(CUtensorMap, CUtensorMap, DhArgs) = nullptr;
    const int nks = p.gs / 16;
#define SG_DH_PICK(P, K, N, H16)                                          \
    if (a.npass == P && nks == K && p.bwt == N && dzt_f16 == H16)         \
        kern = k_tc_dh<P, K, N, H16>;
    SG_DH_PICK(1, 1, 1, false) SG_DH_PICK(1, 1, 2, false) SG_DH_PICK(1, 1, 3, false)
    SG_DH_PICK(1, 2, 1, false) SG_DH_PICK(1, 2, 2, false) SG_DH_PICK(1, 2, 3, false)
    SG_DH_PICK(1, 4, 1, false) SG_DH_PICK(1, 4, 2, false) SG_DH_PICK(1, 4, 3, false)
    SG_DH_PICK(2, 1, 1, false) SG_DH_PICK(2, 1, 2, false) SG_DH_PICK(2, 1, 3, false)
    SG_DH_PICK(2, 2, 1, false) SG_DH_PICK(2, 2, 2, false) SG_DH_PICK(2, 2, 3, false)
    SG_DH_PICK(2, 4, 1, false) SG_DH_PICK(2, 4, 2, false) SG_DH_PICK(2, 4, 3, false)
    SG_DH_PICK(1, 1, 1, true) SG_DH_PICK(1, 1, 2, true) SG_DH_PICK(1, 1, 3, true)
    SG_DH_PICK(1, 2, 1, true) SG_DH_PICK(1, 2, 2, true) SG_DH_PICK(1, 2, 3, true)
    SG_DH_PICK(1, 4, 1, true) SG_DH_PICK(1, 4, 2, true) SG_DH_PICK(1, 4, 3, true)
#undef SG_DH_PICK
    // two MMA-issuing warps where a unit's builders have little to do: the
    // fp16 workspace at G = 32 with F <= 64 and 384-column bands (the LF-8.6M
    // shape: dh 1.011 -> 0.944 ms together with the half-row builders of
    // FMX = 64; at F = 128 the second issuer measured 1-3 % slower, also
    // after the builders got cheaper)
    const int iss = (dzt_f16 && lo->F <= 64 && nks == 2 && p.bwt == 3) ? 2 : 1;
    if (iss == 2)
        kern = k_tc_dh<1, 2, 3, true, 2, 64>;  // FMX = 64: rows in halves, slots for F <= 64
    if (!kern) {
        sg_set_error("tc_dh: no kernel for G = %d (subgroups of %d), band of %d columns", lo->G, p.gs, p.band_w);
        return SG_ERR_UNSUPPORTED;
    }
    const size_t smem = (size_t)p.nbuf * p.ws_bytes + (size_t)p.S * p.stage_bytes + 1024;
    rc = set_smem(kern, smem);
    if (rc != SG_OK)
        return rc;
    if (!dzt_f16)  // the fused kernel that wrote the fp16 workspace cleared dh
        SG_TRY_CUDA(cudaMemsetAsync(dh, 0, sizeof(float) * B * lo->H, st));
    SG_LAUNCH(lo, SG_KIND_DH, st,
              kern<<<p.nbands * p.MT * parts, dh_threads(iss), smem, st>>>(tm_z, tm_zl, a));
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}
