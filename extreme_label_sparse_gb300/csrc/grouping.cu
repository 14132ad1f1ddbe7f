// Semantic grouping of the labels (HASTE, "Key designs / group-shared fixed
// fan-in sparsity"): label embeddings from the encoder outputs of each label's
// positive samples, mini-batch spherical k-means into coarse clusters on the
// tensor cores, then greedy groups of a seed and its G - 1 nearest remaining
// neighbours inside each cluster.  The groups feed sg_layout_build.
//
// Decisions taken here (the page leaves them open):
//  * e_l = bf16(Normalize(sum of h_i over the distinct samples i with l
//    positive)); a label without a positive (or with a zero sum) has no
//    embedding, takes part in neither stage and is grouped last.
//  * Similarity = dot product of bf16 vectors (embeddings, and centroids
//    rounded to bf16 for scoring), fp32 accumulation.
//  * k-means: per-centre learning rate 1/n_c over a batch assigned with the
//    centroids of the batch start (ties to the smaller centroid), which in
//    closed form is mu_c <- Normalize((n_c mu_c + S_c) / (n_c + m_c)), S_c and
//    m_c the sum and count of the batch's members of c.
//  * Greedy: clusters in index order, seed = the remaining member most similar
//    to the centroid, then the G - 1 remaining members most similar to the
//    seed (ties to the smaller label id); groups numbered as formed.  Members a
//    cluster leaves over (in cluster order, ascending id), then the labels
//    without embedding (ascending id), are cut into consecutive groups of G.
//
// Sums that decide outputs are order-independent: embedding and centroid sums
// accumulate in 64-bit fixed point (h x 2^24, e x 2^40), so the atomics give
// the same bits every run.
#include <climits>
#include <cstring>
#include <vector>

#include "sg_internal.cuh"

sg_status gemm_argmax_bf16(const uint16_t *A, int64_t lda, int M, const uint16_t *B, int64_t ldb, int N, int K,
                           int32_t *best_idx, float *best_val, int32_t *status, cudaStream_t st);

struct sg_grouping {
    int64_t L = 0;
    int32_t D = 0, G = 0, C = 0;
    int32_t device = 0;
    int64_t A = 0;      // labels with at least one positive (after embed)
    int64_t A_cap = 0;  // rows allocated for the compact arrays
    bool embedded = false, centred = false;

    int32_t *status = nullptr;     // sticky device status word
    int32_t *cnt = nullptr;        // [L] distinct positive samples per label
    int32_t *aidx = nullptr;       // [L] exclusive scan of (cnt > 0): compact row of an active label
    int32_t *noemb = nullptr;      // [L] 1 where the label has no embedding
    int32_t *noemb_rank = nullptr; // [L] exclusive scan of noemb
    int32_t *scan_part = nullptr;  // scan tile sums
    int32_t *scan_tot = nullptr;   // [4] scan totals
    int32_t *act_label = nullptr;  // [A_cap] label of a compact row
    uint8_t *has = nullptr;        // [A_cap] the row has an embedding
    uint16_t *E = nullptr;         // [A_cap][D] bf16 embeddings (zero rows without one)
    long long *acc = nullptr;      // [A_cap][D] fixed-point sums of h (embed only)

    float *cent = nullptr;         // [C][D]
    uint16_t *cent_b = nullptr;    // [C][D] bf16 copy for scoring
    long long *ncount = nullptr;   // [C] running counts
    int32_t *mcount = nullptr;     // [C] a batch's counts
    long long *csum = nullptr;     // [C][D] a batch's fixed-point sums
    uint16_t *rows = nullptr;      // [rows_cap][D] gathered batch rows
    int64_t rows_cap = 0;
    int32_t *assign = nullptr;     // [max(A_cap, rows_cap)] argmax results

    // greedy stage
    int32_t *ccount = nullptr;     // [C] members per cluster
    int32_t *cstart = nullptr;     // [C] exclusive scan of ccount
    int32_t *ccur = nullptr;       // [C] placement cursors
    int32_t *gbase = nullptr;      // [C] first greedy group of the cluster
    int32_t *pbase = nullptr;      // [C] first pool position of the cluster's leftovers
    int32_t *members = nullptr;    // [A_cap] compact rows by cluster
    int32_t *mlab = nullptr;       // [A_cap] label of each member slot
    float *to_mu = nullptr;        // [A_cap] similarity to the cluster's centroid
    float *to_seed = nullptr;      // [A_cap] similarity to the current seed
    uint8_t *state = nullptr;      // [A_cap] 0 = remaining, 1 = grouped
};

namespace {

constexpr int kT = 256;
constexpr int kScanItems = 4096;  // items per scan tile (1024 threads x 4)
constexpr double kHScale = 16777216.0;           // 2^24
constexpr double kEScale = 1099511627776.0;      // 2^40
constexpr float kHMax = 16384.f;                 // |h| < 2^14 keeps the sums in 63 bits
constexpr int32_t kMaxSamples = 1 << 22;
constexpr int32_t kMaxBatch = 1 << 22;

#define GR_FAIL(code, ...)         \
    do {                           \
        sg_set_error(__VA_ARGS__); \
        return code;               \
    } while (0)

#define GR_TRY(expr)            \
    do {                        \
        sg_status rc_ = (expr); \
        if (rc_ != SG_OK)       \
            return rc_;         \
    } while (0)

__device__ __forceinline__ float bf2f(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }

__device__ __forceinline__ uint16_t f2bf_rn(float x)
{
    uint32_t u = __float_as_uint(x);
    if ((u & 0x7f800000u) == 0x7f800000u)  // inf / nan: keep (quiet the nan)
        return (uint16_t)((u >> 16) | ((u & 0xffffu) ? 0x40u : 0u));
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

__device__ __forceinline__ void flag(int32_t *status, int32_t code) { atomicCAS(status, 0, code); }

// entry j of a row is the first occurrence of its label in the row
__device__ __forceinline__ bool first_in_row(const int32_t *labels, int64_t r0, int64_t j, int32_t l)
{
    for (int64_t k = r0; k < j; ++k)
        if (__ldg(labels + k) == l)
            return false;
    return true;
}

// a row [r0, r1) is well formed
__device__ __forceinline__ bool row_ok(int64_t r0, int64_t r1, int64_t nnz) { return 0 <= r0 && r0 <= r1 && r1 <= nnz; }

// ---------------------------------------------------------------- scan
// exclusive scan of in[] (mode 0: the values, mode 1: in > 0) into out[],
// the total into *total
__global__ void __launch_bounds__(1024) k_scan_tiles(const int32_t *in, int64_t n, int mode, int32_t *out,
                                                     int32_t *part)
{
    __shared__ int32_t ws[32];
    const int64_t i0 = (int64_t)blockIdx.x * kScanItems + threadIdx.x * 4;
    int32_t v[4], s = 0;
    for (int u = 0; u < 4; ++u) {
        const int64_t i = i0 + u;
        int32_t x = i < n ? in[i] : 0;
        if (mode == 1)
            x = x > 0 ? 1 : 0;
        v[u] = s;
        s += x;
    }
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int32_t incl = s;
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += y;
    }
    if (lane == 31)
        ws[w] = incl;
    __syncthreads();
    if (w == 0) {
        int32_t t = ws[lane];
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o)
                t += y;
        }
        ws[lane] = t;  // inclusive over warps
    }
    __syncthreads();
    const int32_t base = (w > 0 ? ws[w - 1] : 0) + incl - s;
    for (int u = 0; u < 4; ++u) {
        const int64_t i = i0 + u;
        if (i < n)
            out[i] = base + v[u];
    }
    if (threadIdx.x == 1023)
        part[blockIdx.x] = ws[31];
}

// one block: exclusive scan of the tile sums (in chunks of 1024), total last
__global__ void __launch_bounds__(1024) k_scan_parts(int32_t *part, int64_t ntiles, int32_t *total)
{
    __shared__ int32_t ws[32];
    __shared__ int32_t carry;
    if (threadIdx.x == 0)
        carry = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (int64_t c0 = 0; c0 < ntiles; c0 += 1024) {
        const int64_t i = c0 + threadIdx.x;
        const int32_t x = i < ntiles ? part[i] : 0;
        int32_t incl = x;
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += y;
        }
        if (lane == 31)
            ws[w] = incl;
        __syncthreads();
        if (w == 0) {
            int32_t t = ws[lane];
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, t, o);
                if (lane >= o)
                    t += y;
            }
            ws[lane] = t;
        }
        __syncthreads();
        const int32_t excl = carry + (w > 0 ? ws[w - 1] : 0) + incl - x;
        if (i < ntiles)
            part[i] = excl;
        __syncthreads();
        if (threadIdx.x == 0)
            carry += ws[31];
        __syncthreads();
    }
    if (threadIdx.x == 0)
        *total = carry;
}

__global__ void k_scan_add(int32_t *out, int64_t n, const int32_t *part)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n)
        out[i] += part[i / kScanItems];
}

sg_status scan_excl(const int32_t *in, int64_t n, int mode, int32_t *out, int32_t *part, int32_t *total,
                    cudaStream_t st)
{
    if (n <= 0) {
        SG_TRY_CUDA(cudaMemsetAsync(total, 0, sizeof(int32_t), st));
        return SG_OK;
    }
    const int64_t tiles = (n + kScanItems - 1) / kScanItems;
    k_scan_tiles<<<(unsigned)tiles, 1024, 0, st>>>(in, n, mode, out, part);
    k_scan_parts<<<1, 1024, 0, st>>>(part, tiles, total);
    k_scan_add<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(out, n, part);
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}

// ---------------------------------------------------------------- embeddings
// distinct positive samples per label (one warp per sample row)
__global__ void k_emb_count(int32_t N, const int32_t *rowptr, const int32_t *labels, int64_t nnz, int64_t L,
                            int32_t *cnt, int32_t *status)
{
    const int lane = threadIdx.x & 31;
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
    if (i >= N)
        return;
    const int64_t r0 = rowptr[i], r1 = rowptr[i + 1];
    if (!row_ok(r0, r1, nnz)) {
        if (lane == 0)
            flag(status, SG_ERR_DATA);
        return;
    }
    for (int64_t j = r0 + lane; j < r1; j += 32) {
        const int32_t l = __ldg(labels + j);
        if (l < 0 || l >= L) {
            flag(status, SG_ERR_DATA);
            continue;
        }
        if (first_in_row(labels, r0, j, l))
            atomicAdd(cnt + l, 1);
    }
}

__global__ void k_emb_rows(int64_t L, const int32_t *cnt, const int32_t *aidx, int32_t *act_label)
{
    const int64_t l = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (l < L && cnt[l] > 0)
        act_label[aidx[l]] = (int32_t)l;
}

// fixed-point sums of h over each label's distinct positive samples (one warp
// per sample row; lanes over the features)
__global__ void k_emb_accum(int32_t N, int32_t D, const uint16_t *h, const int32_t *rowptr, const int32_t *labels,
                            int64_t nnz, int64_t L, const int32_t *aidx, long long *acc, int32_t *status)
{
    const int lane = threadIdx.x & 31;
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
    if (i >= N)
        return;
    const int64_t r0 = rowptr[i], r1 = rowptr[i + 1];
    if (!row_ok(r0, r1, nnz))
        return;
    const uint16_t *hi = h + (int64_t)i * D;
    for (int64_t j = r0; j < r1; ++j) {
        const int32_t l = __ldg(labels + j);
        if (l < 0 || l >= L || !first_in_row(labels, r0, j, l))
            continue;
        long long *a = acc + (int64_t)aidx[l] * D;
        for (int d = lane; d < D; d += 32) {
            const float x = bf2f(hi[d]);
            if (!(fabsf(x) < kHMax)) {
                flag(status, SG_ERR_DATA);
                continue;
            }
            atomicAdd(reinterpret_cast<unsigned long long *>(a + d),
                      (unsigned long long)__double2ll_rn((double)x * kHScale));
        }
    }
}

// e = bf16(x / |x|) per compact row (one warp per row); has = |x| > 0
__global__ void k_emb_norm(int64_t A, int32_t D, const long long *acc, uint16_t *E, uint8_t *has)
{
    const int lane = threadIdx.x & 31;
    const int64_t a = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
    if (a >= A)
        return;
    const long long *x = acc + a * D;
    double s = 0.0;
    for (int d = lane; d < D; d += 32) {
        const double v = (double)x[d] / kHScale;
        s = fma(v, v, s);
    }
    for (int o = 16; o > 0; o >>= 1)
        s += __shfl_xor_sync(0xffffffffu, s, o);
    const bool ok = s > 0.0;
    const double inv = ok ? 1.0 / sqrt(s) : 0.0;
    for (int d = lane; d < D; d += 32)
        E[a * D + d] = ok ? f2bf_rn((float)(((double)x[d] / kHScale) * inv)) : (uint16_t)0;
    if (lane == 0)
        has[a] = ok ? 1 : 0;
}

// noemb[l] = 1 where label l has no embedding
__global__ void k_noemb(int64_t L, const int32_t *cnt, const int32_t *aidx, const uint8_t *has, int32_t *noemb)
{
    const int64_t l = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (l < L)
        noemb[l] = (cnt[l] > 0 && has[aidx[l]]) ? 0 : 1;
}

// ---------------------------------------------------------------- k-means
// compact row of label l if it has an embedding, else -1
__device__ __forceinline__ int64_t row_of(int64_t L, const int32_t *cnt, const int32_t *aidx, const uint8_t *has,
                                          int32_t l)
{
    if (l < 0 || l >= L || cnt[l] <= 0)
        return -1;
    const int64_t a = aidx[l];
    return has[a] ? a : -1;
}

// centroid c = Normalize(e of init label c) (one warp per centroid)
__global__ void k_cent_init(int32_t C, int32_t D, int64_t L, const int32_t *init, const int32_t *cnt,
                            const int32_t *aidx, const uint8_t *has, const uint16_t *E, float *cent,
                            uint16_t *cent_b, long long *ncount, int32_t *mcount, int32_t *status)
{
    const int lane = threadIdx.x & 31;
    const int64_t c = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
    if (c >= C)
        return;
    const int64_t a = row_of(L, cnt, aidx, has, init[c]);
    if (a < 0) {
        if (lane == 0)
            flag(status, SG_ERR_DATA);
        return;
    }
    double s = 0.0;
    for (int d = lane; d < D; d += 32) {
        const double v = bf2f(E[a * D + d]);
        s = fma(v, v, s);
    }
    for (int o = 16; o > 0; o >>= 1)
        s += __shfl_xor_sync(0xffffffffu, s, o);
    const double inv = 1.0 / sqrt(s);
    for (int d = lane; d < D; d += 32) {
        const float v = (float)((double)bf2f(E[a * D + d]) * inv);
        cent[c * D + d] = v;
        cent_b[c * D + d] = f2bf_rn(v);
    }
    if (lane == 0) {
        ncount[c] = 0;
        mcount[c] = 0;
    }
}

// rows[m] = E of batch label m (zero and a data error where it has none)
__global__ void k_gather_rows(int32_t M, int32_t D, int64_t L, const int32_t *batch, const int32_t *cnt,
                              const int32_t *aidx, const uint8_t *has, const uint16_t *E, uint16_t *rows,
                              int32_t *status)
{
    const int lane = threadIdx.x & 31;
    const int64_t m = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
    if (m >= M)
        return;
    const int64_t a = row_of(L, cnt, aidx, has, batch[m]);
    if (a < 0 && lane == 0)
        flag(status, SG_ERR_DATA);
    for (int d = lane; d < D; d += 32)
        rows[m * D + d] = a >= 0 ? E[a * D + d] : (uint16_t)0;
}

// batch sums and counts per assigned centroid (one warp per batch member)
__global__ void k_cent_accum(int32_t M, int32_t D, const int32_t *assign, const uint16_t *rows, long long *csum,
                             int32_t *mcount)
{
    const int lane = threadIdx.x & 31;
    const int64_t m = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
    if (m >= M)
        return;
    const int32_t c = assign[m];
    if (c < 0)
        return;
    if (lane == 0)
        atomicAdd(mcount + c, 1);
    for (int d = lane; d < D; d += 32)
        atomicAdd(reinterpret_cast<unsigned long long *>(csum + (int64_t)c * D + d),
                  (unsigned long long)__double2ll_rn((double)bf2f(rows[m * D + d]) * kEScale));
}

// mu_c <- Normalize((n_c mu_c + S_c) / (n_c + m_c)) for every centroid the
// batch moved; the batch's sums and counts are cleared
__global__ void k_cent_update(int32_t C, int32_t D, float *cent, uint16_t *cent_b, long long *ncount,
                              int32_t *mcount, long long *csum)
{
    const int lane = threadIdx.x & 31;
    const int64_t c = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
    if (c >= C)
        return;
    const int32_t m = mcount[c];
    if (m == 0)
        return;
    const double n = (double)ncount[c];
    const double inv_tot = 1.0 / (n + (double)m);
    double s = 0.0;
    for (int d = lane; d < D; d += 32) {
        const double v = (n * (double)cent[c * D + d] + (double)csum[c * D + d] / kEScale) * inv_tot;
        s = fma(v, v, s);
    }
    for (int o = 16; o > 0; o >>= 1)
        s += __shfl_xor_sync(0xffffffffu, s, o);
    const double inv = s > 0.0 ? 1.0 / sqrt(s) : 0.0;
    for (int d = lane; d < D; d += 32) {
        const double v = (n * (double)cent[c * D + d] + (double)csum[c * D + d] / kEScale) * inv_tot;
        const float u = s > 0.0 ? (float)(v * inv) : cent[c * D + d];
        cent[c * D + d] = u;
        cent_b[c * D + d] = f2bf_rn(u);
        csum[c * D + d] = 0;
    }
    __syncwarp();
    if (lane == 0) {
        ncount[c] += m;
        mcount[c] = 0;
    }
}

// ---------------------------------------------------------------- greedy
__global__ void k_cluster_count(int64_t A, const uint8_t *has, const int32_t *assign, int32_t *ccount)
{
    const int64_t a = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (a < A && has[a])
        atomicAdd(ccount + assign[a], 1);
}

__global__ void k_cluster_place(int64_t A, const uint8_t *has, const int32_t *assign, const int32_t *cstart,
                                int32_t *ccur, int32_t *members)
{
    const int64_t a = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (a < A && has[a]) {
        const int32_t c = assign[a];
        members[cstart[c] + atomicAdd(ccur + c, 1)] = (int32_t)a;
    }
}

// groups and leftovers per cluster: gsz[c] = n_c / G, rsz[c] = n_c % G
__global__ void k_cluster_sizes(int32_t C, int32_t G, const int32_t *ccount, int32_t *gsz, int32_t *rsz)
{
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c < C) {
        gsz[c] = ccount[c] / G;
        rsz[c] = ccount[c] % G;
    }
}

// dot product of two bf16 rows in fp32, ascending features (one thread)
__device__ __forceinline__ float dot_bf16(const uint16_t *x, const uint16_t *y, int D)
{
    float s = 0.f;
    for (int d = 0; d < D; d += 2) {
        const uint32_t a = *reinterpret_cast<const uint32_t *>(x + d);
        const uint32_t b = *reinterpret_cast<const uint32_t *>(y + d);
        s = fmaf(__uint_as_float(a << 16), __uint_as_float(b << 16), s);
        s = fmaf(__uint_as_float(a & 0xffff0000u), __uint_as_float(b & 0xffff0000u), s);
    }
    return s;
}

// the better of two candidates: larger value, then smaller label
__device__ __forceinline__ bool better(float v, int32_t l, float bv, int32_t bl)
{
    return v > bv || (v == bv && l < bl);
}

struct Cand {
    float v;
    int32_t l, i;
};

// block-wide best remaining member by (val, -label); every thread gets it
__device__ Cand block_best(const float *val, const int32_t *lab, const uint8_t *state, int n, Cand *ws)
{
    Cand b{-INFINITY, INT_MAX, -1};
    for (int i = threadIdx.x; i < n; i += blockDim.x)
        if (!state[i] && (b.i < 0 || better(val[i], lab[i], b.v, b.l)))
            b = Cand{val[i], lab[i], i};
    for (int o = 16; o > 0; o >>= 1) {
        Cand y;
        y.v = __shfl_xor_sync(0xffffffffu, b.v, o);
        y.l = __shfl_xor_sync(0xffffffffu, b.l, o);
        y.i = __shfl_xor_sync(0xffffffffu, b.i, o);
        if (y.i >= 0 && (b.i < 0 || better(y.v, y.l, b.v, b.l)))
            b = y;
    }
    const int w = threadIdx.x / 32, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0)
        ws[w] = b;
    __syncthreads();
    if (w == 0) {
        b = lane < (int)(blockDim.x / 32) ? ws[lane] : Cand{-INFINITY, INT_MAX, -1};
        for (int o = 16; o > 0; o >>= 1) {
            Cand y;
            y.v = __shfl_xor_sync(0xffffffffu, b.v, o);
            y.l = __shfl_xor_sync(0xffffffffu, b.l, o);
            y.i = __shfl_xor_sync(0xffffffffu, b.i, o);
            if (y.i >= 0 && (b.i < 0 || better(y.v, y.l, b.v, b.l)))
                b = y;
        }
        if (lane == 0)
            ws[32] = b;
    }
    __syncthreads();
    return ws[32];
}

struct GreedyArgs {
    int32_t D, G;
    const uint16_t *E, *cent_b;
    const int32_t *act_label, *ccount, *cstart, *gbase, *pbase;
    int32_t *members, *groups;
    const int32_t *ng_total;  // greedy groups over all clusters
    float *to_mu, *to_seed;
    uint8_t *state;
    int32_t *lab;             // [A_cap] label of each member slot
};

// one CTA per cluster
__global__ void __launch_bounds__(kT) k_greedy(GreedyArgs a)
{
    __shared__ Cand ws[33];
    extern __shared__ uint16_t seedrow[];
    const int c = blockIdx.x;
    const int n = a.ccount[c];
    if (n == 0)
        return;
    const int64_t o = a.cstart[c];
    int32_t *mem = a.members + o;
    int32_t *lab = a.lab + o;
    float *tm = a.to_mu + o, *ts = a.to_seed + o;
    uint8_t *stt = a.state + o;
    const uint16_t *mu = a.cent_b + (int64_t)c * a.D;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int32_t r = mem[i];
        lab[i] = a.act_label[r];
        tm[i] = dot_bf16(a.E + (int64_t)r * a.D, mu, a.D);
        stt[i] = 0;
    }
    __syncthreads();
    const int ng = n / a.G;
    for (int s = 0; s < ng; ++s) {
        const int32_t gid = a.gbase[c] + s;
        const Cand seed = block_best(tm, lab, stt, n, ws);
        if (threadIdx.x == 0) {
            stt[seed.i] = 1;
            a.groups[seed.l] = gid;
        }
        const uint16_t *srow = a.E + (int64_t)mem[seed.i] * a.D;
        for (int d = threadIdx.x; d < a.D; d += blockDim.x)
            seedrow[d] = srow[d];
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += blockDim.x)
            if (!stt[i])
                ts[i] = dot_bf16(a.E + (int64_t)mem[i] * a.D, seedrow, a.D);
        __syncthreads();
        for (int g = 1; g < a.G; ++g) {
            const Cand b = block_best(ts, lab, stt, n, ws);
            if (threadIdx.x == 0) {
                stt[b.i] = 1;
                a.groups[b.l] = gid;
            }
            __syncthreads();
        }
    }
    // leftovers: pool position = the cluster's base + rank by label
    const int32_t NG = *a.ng_total;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        if (stt[i])
            continue;
        int rank = 0;
        for (int j = 0; j < n; ++j)
            rank += (!stt[j] && lab[j] < lab[i]) ? 1 : 0;
        a.groups[lab[i]] = NG + (a.pbase[c] + rank) / a.G;
    }
}

__global__ void k_cluster_out(int64_t A, const uint8_t *has, const int32_t *assign, const int32_t *act_label,
                              int32_t *cluster_out)
{
    const int64_t a = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (a < A && has[a])
        cluster_out[act_label[a]] = assign[a];
}

// embeddings per label (zero rows without one), one warp per label
__global__ void k_expand_E(int64_t L, int32_t D, const int32_t *cnt, const int32_t *aidx, const uint8_t *has,
                           const uint16_t *E, uint16_t *out, uint8_t *out_has)
{
    const int lane = threadIdx.x & 31;
    const int64_t l = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
    if (l >= L)
        return;
    const int64_t a = (cnt[l] > 0 && has[aidx[l]]) ? aidx[l] : -1;
    for (int d = lane; d < D; d += 32)
        out[l * D + d] = a >= 0 ? E[a * D + d] : (uint16_t)0;
    if (lane == 0 && out_has)
        out_has[l] = a >= 0 ? 1 : 0;
}

// labels without embedding: after every leftover, ascending id
__global__ void k_pool_noemb(int64_t L, int32_t G, const int32_t *noemb_rank, const int32_t *cnt,
                             const int32_t *aidx, const uint8_t *has, const int32_t *ng_total,
                             const int32_t *np_total, int32_t *groups)
{
    const int64_t l = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (l >= L)
        return;
    if (cnt[l] > 0 && has[aidx[l]])
        return;
    groups[l] = *ng_total + (*np_total + noemb_rank[l]) / G;
}

template <typename T>
sg_status dev_alloc(T **p, size_t n, const char *what)
{
    if (*p)
        cudaFree(*p);
    *p = nullptr;
    if (n == 0)
        n = 1;
    if (cudaMalloc((void **)p, n * sizeof(T)) != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        sg_set_error("cudaMalloc of %zu bytes for %s failed", n * sizeof(T), what);
        return SG_ERR_OOM;
    }
    return SG_OK;
}

unsigned warp_grid(int64_t items) { return (unsigned)((items * 32 + kT - 1) / kT); }
unsigned thread_grid(int64_t items) { return (unsigned)((items + kT - 1) / kT); }

struct DevScope {
    int prev = -1;
    explicit DevScope(int dev)
    {
        if (cudaGetDevice(&prev) == cudaSuccess && prev != dev)
            cudaSetDevice(dev);
    }
    ~DevScope()
    {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev)
            cudaSetDevice(prev);
    }
};

void free_all(sg_grouping *g)
{
    void *ptrs[] = {g->status, g->cnt, g->aidx, g->noemb, g->noemb_rank, g->mlab, g->scan_part, g->scan_tot, g->act_label, g->has, g->E,
                    g->acc, g->cent, g->cent_b, g->ncount, g->mcount, g->csum, g->rows, g->assign, g->ccount,
                    g->cstart, g->ccur, g->gbase, g->pbase, g->members, g->to_mu, g->to_seed, g->state};
    for (void *p : ptrs)
        if (p)
            cudaFree(p);
}

}  // namespace

extern "C" {

sg_status sg_grouping_create(int64_t L, int32_t D, int32_t G, int32_t C, sg_grouping **out)
{
    const char *fn = "sg_grouping_create";
    if (!out)
        GR_FAIL(SG_ERR_INVALID, "%s: out is NULL", fn);
    *out = nullptr;
    if (L < 1 || G < 1 || L % G != 0 || L > INT32_MAX)
        GR_FAIL(SG_ERR_INVALID, "%s: need 1 <= L < 2^31 with L %% G == 0 (L=%lld G=%d)", fn, (long long)L, G);
    if (D < 16 || D % 16 != 0 || D > 4096)
        GR_FAIL(SG_ERR_INVALID, "%s: need D a multiple of 16 in [16, 4096] (D=%d)", fn, D);
    if (C < 1 || (int64_t)C > L)
        GR_FAIL(SG_ERR_INVALID, "%s: need 1 <= C <= L (C=%d)", fn, C);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        GR_FAIL(SG_ERR_CUDA, "%s: no usable CUDA device", fn);
    }
    sg_grouping *g = new sg_grouping();
    g->L = L;
    g->D = D;
    g->G = G;
    g->C = C;
    g->device = dev;
    const int64_t tiles = (L + kScanItems - 1) / kScanItems + (C + kScanItems - 1) / kScanItems + 8;
    sg_status rc = SG_OK;
    if ((rc = dev_alloc(&g->status, 1, "status")) != SG_OK || (rc = dev_alloc(&g->cnt, L, "counts")) != SG_OK ||
        (rc = dev_alloc(&g->aidx, L, "rows")) != SG_OK || (rc = dev_alloc(&g->noemb, L, "flags")) != SG_OK ||
        (rc = dev_alloc(&g->noemb_rank, L, "flags")) != SG_OK ||
        (rc = dev_alloc(&g->scan_part, tiles, "scan")) != SG_OK ||
        (rc = dev_alloc(&g->scan_tot, 4, "scan")) != SG_OK ||
        (rc = dev_alloc(&g->cent, (size_t)C * D, "centroids")) != SG_OK ||
        (rc = dev_alloc(&g->cent_b, (size_t)C * D, "centroids")) != SG_OK ||
        (rc = dev_alloc(&g->ncount, C, "counts")) != SG_OK || (rc = dev_alloc(&g->mcount, C, "counts")) != SG_OK ||
        (rc = dev_alloc(&g->csum, (size_t)C * D, "sums")) != SG_OK ||
        (rc = dev_alloc(&g->ccount, C, "clusters")) != SG_OK || (rc = dev_alloc(&g->cstart, C, "clusters")) != SG_OK ||
        (rc = dev_alloc(&g->ccur, C, "clusters")) != SG_OK || (rc = dev_alloc(&g->gbase, C, "clusters")) != SG_OK ||
        (rc = dev_alloc(&g->pbase, C, "clusters")) != SG_OK) {
        free_all(g);
        delete g;
        return rc;
    }
    if (cudaMemset(g->status, 0, 4) != cudaSuccess || cudaMemset(g->csum, 0, sizeof(long long) * C * D) != cudaSuccess ||
        cudaMemset(g->mcount, 0, 4 * (size_t)C) != cudaSuccess) {
        cudaGetLastError();
        free_all(g);
        delete g;
        GR_FAIL(SG_ERR_CUDA, "%s: cudaMemset failed", fn);
    }
    *out = g;
    return SG_OK;
}

void sg_grouping_free(sg_grouping *g)
{
    if (!g)
        return;
    DevScope ds(g->device);
    cudaDeviceSynchronize();
    free_all(g);
    delete g;
}

sg_status sg_grouping_status(sg_grouping *g, int32_t *code)
{
    if (!g || !code)
        GR_FAIL(SG_ERR_INVALID, "sg_grouping_status: NULL argument");
    DevScope ds(g->device);
    SG_TRY_CUDA(cudaMemcpy(code, g->status, 4, cudaMemcpyDeviceToHost));
    SG_TRY_CUDA(cudaMemset(g->status, 0, 4));
    return SG_OK;
}

// compact arrays for A labels (rows_cap for batches allocated separately)
static sg_status alloc_compact(sg_grouping *g, int64_t A)
{
    if (A <= g->A_cap && g->E)
        return SG_OK;
    const int64_t cap = A > 0 ? A : 1;
    GR_TRY(dev_alloc(&g->act_label, cap, "labels"));
    GR_TRY(dev_alloc(&g->has, cap, "flags"));
    GR_TRY(dev_alloc(&g->E, (size_t)cap * g->D, "embeddings"));
    GR_TRY(dev_alloc(&g->members, cap, "members"));
    GR_TRY(dev_alloc(&g->mlab, cap, "member labels"));
    GR_TRY(dev_alloc(&g->to_mu, cap, "similarities"));
    GR_TRY(dev_alloc(&g->to_seed, cap, "similarities"));
    GR_TRY(dev_alloc(&g->state, cap, "state"));
    GR_TRY(dev_alloc(&g->assign, cap > g->rows_cap ? cap : g->rows_cap, "assignment"));
    g->A_cap = cap;
    return SG_OK;
}

sg_status sg_grouping_embed(sg_grouping *g, const sg_bf16 *h, int32_t N, const int32_t *rowptr,
                            const int32_t *labels, int64_t nnz, int64_t *n_embedded, void *stream)
{
    const char *fn = "sg_grouping_embed";
    NvtxRange nvtx_(fn);
    if (!g || !h || !rowptr || (nnz > 0 && !labels))
        GR_FAIL(SG_ERR_INVALID, "%s: a required pointer is NULL", fn);
    if (N < 1 || N > kMaxSamples || nnz < 0)
        GR_FAIL(SG_ERR_INVALID, "%s: need 1 <= N <= %d and nnz >= 0 (N=%d)", fn, kMaxSamples, N);
    DevScope ds(g->device);
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t L = g->L;
    const int D = g->D;
    SG_TRY_CUDA(cudaMemsetAsync(g->cnt, 0, sizeof(int32_t) * L, st));
    k_emb_count<<<warp_grid(N), kT, 0, st>>>(N, rowptr, labels, nnz, L, g->cnt, g->status);
    SG_TRY_CUDA(cudaGetLastError());
    GR_TRY(scan_excl(g->cnt, L, 1, g->aidx, g->scan_part, g->scan_tot, st));
    int32_t A = 0;
    SG_TRY_CUDA(cudaMemcpyAsync(&A, g->scan_tot, 4, cudaMemcpyDeviceToHost, st));
    SG_TRY_CUDA(cudaStreamSynchronize(st));
    GR_TRY(alloc_compact(g, A));
    GR_TRY(dev_alloc(&g->acc, (size_t)(A > 0 ? A : 1) * D, "embedding sums"));
    SG_TRY_CUDA(cudaMemsetAsync(g->acc, 0, sizeof(long long) * (size_t)(A > 0 ? A : 1) * D, st));
    k_emb_rows<<<thread_grid(L), kT, 0, st>>>(L, g->cnt, g->aidx, g->act_label);
    k_emb_accum<<<warp_grid(N), kT, 0, st>>>(N, D, h, rowptr, labels, nnz, L, g->aidx, g->acc, g->status);
    if (A > 0)
        k_emb_norm<<<warp_grid(A), kT, 0, st>>>(A, D, g->acc, g->E, g->has);
    k_noemb<<<thread_grid(L), kT, 0, st>>>(L, g->cnt, g->aidx, g->has, g->noemb);
    SG_TRY_CUDA(cudaGetLastError());
    GR_TRY(scan_excl(g->noemb, L, 0, g->noemb_rank, g->scan_part, g->scan_tot + 1, st));
    int32_t none = 0;
    SG_TRY_CUDA(cudaMemcpyAsync(&none, g->scan_tot + 1, 4, cudaMemcpyDeviceToHost, st));
    SG_TRY_CUDA(cudaStreamSynchronize(st));
    cudaFree(g->acc);  // the sums are not needed after normalising
    g->acc = nullptr;
    g->A = A;
    g->embedded = true;
    g->centred = false;
    if (n_embedded)
        *n_embedded = L - none;
    return SG_OK;
}

sg_status sg_grouping_set_embeddings(sg_grouping *g, const sg_bf16 *E, const uint8_t *has, void *stream)
{
    const char *fn = "sg_grouping_set_embeddings";
    if (!g || !E || !has)
        GR_FAIL(SG_ERR_INVALID, "%s: a required pointer is NULL", fn);
    DevScope ds(g->device);
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t L = g->L;
    // every label gets a compact row (A = L); cnt = 1 marks them all present
    GR_TRY(alloc_compact(g, L));
    SG_TRY_CUDA(cudaMemcpyAsync(g->E, E, sizeof(uint16_t) * (size_t)L * g->D, cudaMemcpyDeviceToDevice, st));
    SG_TRY_CUDA(cudaMemcpyAsync(g->has, has, (size_t)L, cudaMemcpyDeviceToDevice, st));
    SG_TRY_CUDA(cudaMemsetAsync(g->cnt, 0, sizeof(int32_t) * L, st));
    // cnt[l] = 1, aidx[l] = l, act_label[l] = l
    std::vector<int32_t> ones(L, 1), iota(L);
    for (int64_t l = 0; l < L; ++l)
        iota[l] = (int32_t)l;
    SG_TRY_CUDA(cudaMemcpyAsync(g->cnt, ones.data(), sizeof(int32_t) * L, cudaMemcpyHostToDevice, st));
    SG_TRY_CUDA(cudaMemcpyAsync(g->aidx, iota.data(), sizeof(int32_t) * L, cudaMemcpyHostToDevice, st));
    SG_TRY_CUDA(cudaMemcpyAsync(g->act_label, iota.data(), sizeof(int32_t) * L, cudaMemcpyHostToDevice, st));
    k_noemb<<<thread_grid(L), kT, 0, st>>>(L, g->cnt, g->aidx, g->has, g->noemb);
    SG_TRY_CUDA(cudaGetLastError());
    GR_TRY(scan_excl(g->noemb, L, 0, g->noemb_rank, g->scan_part, g->scan_tot + 1, st));
    SG_TRY_CUDA(cudaStreamSynchronize(st));
    g->A = L;
    g->embedded = true;
    g->centred = false;
    return SG_OK;
}

sg_status sg_grouping_kmeans_init(sg_grouping *g, const int32_t *init_labels, void *stream)
{
    const char *fn = "sg_grouping_kmeans_init";
    NvtxRange nvtx_(fn);
    if (!g || !init_labels)
        GR_FAIL(SG_ERR_INVALID, "%s: a required pointer is NULL", fn);
    if (!g->embedded)
        GR_FAIL(SG_ERR_INVALID, "%s: no embeddings yet", fn);
    DevScope ds(g->device);
    cudaStream_t st = (cudaStream_t)stream;
    k_cent_init<<<warp_grid(g->C), kT, 0, st>>>(g->C, g->D, g->L, init_labels, g->cnt, g->aidx, g->has, g->E,
                                               g->cent, g->cent_b, g->ncount, g->mcount, g->status);
    SG_TRY_CUDA(cudaGetLastError());
    g->centred = true;
    return SG_OK;
}

sg_status sg_grouping_set_centroids(sg_grouping *g, const float *centroids, const int64_t *counts, void *stream)
{
    const char *fn = "sg_grouping_set_centroids";
    if (!g || !centroids)
        GR_FAIL(SG_ERR_INVALID, "%s: a required pointer is NULL", fn);
    DevScope ds(g->device);
    cudaStream_t st = (cudaStream_t)stream;
    const size_t n = (size_t)g->C * g->D;
    SG_TRY_CUDA(cudaMemcpyAsync(g->cent, centroids, sizeof(float) * n, cudaMemcpyDeviceToDevice, st));
    std::vector<float> hc(n);
    std::vector<uint16_t> hb(n);
    SG_TRY_CUDA(cudaMemcpyAsync(hc.data(), centroids, sizeof(float) * n, cudaMemcpyDeviceToHost, st));
    SG_TRY_CUDA(cudaStreamSynchronize(st));
    for (size_t i = 0; i < n; ++i) {
        uint32_t u;
        memcpy(&u, &hc[i], 4);
        if ((u & 0x7f800000u) == 0x7f800000u)
            GR_FAIL(SG_ERR_INVALID, "%s: centroid %zu is not finite", fn, i / g->D);
        u += 0x7fffu + ((u >> 16) & 1u);
        hb[i] = (uint16_t)(u >> 16);
    }
    SG_TRY_CUDA(cudaMemcpyAsync(g->cent_b, hb.data(), sizeof(uint16_t) * n, cudaMemcpyHostToDevice, st));
    if (counts)
        SG_TRY_CUDA(cudaMemcpyAsync(g->ncount, counts, sizeof(long long) * g->C, cudaMemcpyDeviceToDevice, st));
    else
        SG_TRY_CUDA(cudaMemsetAsync(g->ncount, 0, sizeof(long long) * g->C, st));
    SG_TRY_CUDA(cudaStreamSynchronize(st));
    g->centred = true;
    return SG_OK;
}

sg_status sg_grouping_kmeans_batch(sg_grouping *g, const int32_t *batch, int32_t M, int32_t *assign_out,
                                   void *stream)
{
    const char *fn = "sg_grouping_kmeans_batch";
    NvtxRange nvtx_(fn);
    if (!g || !batch)
        GR_FAIL(SG_ERR_INVALID, "%s: a required pointer is NULL", fn);
    if (!g->centred)
        GR_FAIL(SG_ERR_INVALID, "%s: centroids not initialised", fn);
    if (M < 1 || M > kMaxBatch)
        GR_FAIL(SG_ERR_INVALID, "%s: need 1 <= M <= %d (M=%d)", fn, kMaxBatch, M);
    DevScope ds(g->device);
    cudaStream_t st = (cudaStream_t)stream;
    const int D = g->D;
    if (M > g->rows_cap) {
        GR_TRY(dev_alloc(&g->rows, (size_t)M * D, "batch rows"));
        g->rows_cap = M;
        if (M > g->A_cap)
            GR_TRY(dev_alloc(&g->assign, (size_t)M, "assignment"));
    }
    k_gather_rows<<<warp_grid(M), kT, 0, st>>>(M, D, g->L, batch, g->cnt, g->aidx, g->has, g->E, g->rows,
                                              g->status);
    SG_TRY_CUDA(cudaGetLastError());
    GR_TRY(gemm_argmax_bf16(g->rows, D, M, g->cent_b, D, g->C, D, g->assign, nullptr, g->status, st));
    if (assign_out)
        SG_TRY_CUDA(cudaMemcpyAsync(assign_out, g->assign, sizeof(int32_t) * M, cudaMemcpyDeviceToDevice, st));
    k_cent_accum<<<warp_grid(M), kT, 0, st>>>(M, D, g->assign, g->rows, g->csum, g->mcount);
    k_cent_update<<<warp_grid(g->C), kT, 0, st>>>(g->C, D, g->cent, g->cent_b, g->ncount, g->mcount, g->csum);
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}

sg_status sg_grouping_groups(sg_grouping *g, int32_t *groups, int32_t *cluster_out, void *stream)
{
    const char *fn = "sg_grouping_groups";
    NvtxRange nvtx_(fn);
    if (!g || !groups)
        GR_FAIL(SG_ERR_INVALID, "%s: a required pointer is NULL", fn);
    if (!g->centred)
        GR_FAIL(SG_ERR_INVALID, "%s: centroids not initialised", fn);
    DevScope ds(g->device);
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t L = g->L, A = g->A;
    const int C = g->C, D = g->D, G = g->G;
    // final assignment of every compact row (rows without embedding are
    // assigned too, and ignored)
    if (A > 0)
        GR_TRY(gemm_argmax_bf16(g->E, D, (int)A, g->cent_b, D, C, D, g->assign, nullptr, g->status, st));
    SG_TRY_CUDA(cudaMemsetAsync(g->ccount, 0, sizeof(int32_t) * C, st));
    SG_TRY_CUDA(cudaMemsetAsync(g->ccur, 0, sizeof(int32_t) * C, st));
    k_cluster_count<<<thread_grid(A), kT, 0, st>>>(A, g->has, g->assign, g->ccount);
    SG_TRY_CUDA(cudaGetLastError());
    int32_t *tot = g->scan_tot;  // [0]: members, [1]: greedy groups, [2]: leftovers, [3]: labels without
    GR_TRY(scan_excl(g->ccount, C, 0, g->cstart, g->scan_part, tot + 0, st));
    k_cluster_place<<<thread_grid(A), kT, 0, st>>>(A, g->has, g->assign, g->cstart, g->ccur, g->members);
    // per cluster: groups n / G and leftovers n % G, scanned into bases
    k_cluster_sizes<<<thread_grid(C), kT, 0, st>>>(C, G, g->ccount, g->gbase, g->pbase);
    SG_TRY_CUDA(cudaGetLastError());
    GR_TRY(scan_excl(g->gbase, C, 0, g->gbase, g->scan_part, tot + 1, st));
    GR_TRY(scan_excl(g->pbase, C, 0, g->pbase, g->scan_part, tot + 2, st));
    GreedyArgs ga;
    ga.D = D;
    ga.G = G;
    ga.E = g->E;
    ga.cent_b = g->cent_b;
    ga.act_label = g->act_label;
    ga.ccount = g->ccount;
    ga.cstart = g->cstart;
    ga.gbase = g->gbase;
    ga.pbase = g->pbase;
    ga.members = g->members;
    ga.groups = groups;
    ga.ng_total = tot + 1;
    ga.to_mu = g->to_mu;
    ga.to_seed = g->to_seed;
    ga.state = g->state;
    ga.lab = g->mlab;
    k_greedy<<<C, kT, sizeof(uint16_t) * D, st>>>(ga);
    SG_TRY_CUDA(cudaGetLastError());
    // the pool's tail: labels without embedding in ascending id
    k_pool_noemb<<<thread_grid(L), kT, 0, st>>>(L, G, g->noemb_rank, g->cnt, g->aidx, g->has, tot + 1, tot + 2,
                                                groups);
    if (cluster_out) {
        SG_TRY_CUDA(cudaMemsetAsync(cluster_out, 0xff, sizeof(int32_t) * L, st));
        k_cluster_out<<<thread_grid(A), kT, 0, st>>>(A, g->has, g->assign, g->act_label, cluster_out);
    }
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}

sg_status sg_grouping_export(sg_grouping *g, sg_bf16 *E, uint8_t *has, float *centroids, int64_t *counts,
                             void *stream)
{
    const char *fn = "sg_grouping_export";
    if (!g)
        GR_FAIL(SG_ERR_INVALID, "%s: grouping is NULL", fn);
    if ((E || has) && !g->embedded)
        GR_FAIL(SG_ERR_INVALID, "%s: no embeddings yet", fn);
    if ((centroids || counts) && !g->centred)
        GR_FAIL(SG_ERR_INVALID, "%s: centroids not initialised", fn);
    DevScope ds(g->device);
    cudaStream_t st = (cudaStream_t)stream;
    if (E)
        k_expand_E<<<warp_grid(g->L), kT, 0, st>>>(g->L, g->D, g->cnt, g->aidx, g->has, g->E, E, has);
    else if (has)
        GR_FAIL(SG_ERR_INVALID, "%s: has is exported with E", fn);
    SG_TRY_CUDA(cudaGetLastError());
    if (centroids)
        SG_TRY_CUDA(cudaMemcpyAsync(centroids, g->cent, sizeof(float) * (size_t)g->C * g->D,
                                    cudaMemcpyDeviceToDevice, st));
    if (counts)
        SG_TRY_CUDA(cudaMemcpyAsync(counts, g->ncount, sizeof(long long) * (size_t)g->C, cudaMemcpyDeviceToDevice,
                                    st));
    SG_TRY_CUDA(cudaStreamSynchronize(st));
    return SG_OK;
}

}  // extern "C"
