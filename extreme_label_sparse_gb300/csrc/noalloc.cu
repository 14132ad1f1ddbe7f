// sg_bce_grad_noalloc: the BCE step from a stored Z (dZ = sigmoid(Z) - Y and
// the summed loss) for callers that cannot allocate device memory: processes
// embedded in a framework whose caching allocator already owns the device's
// memory, or deployments that forbid any allocation after start-up.  It takes
// no layout handle and calls no allocator; its working memory is one
// file-scope device array, reserved when the library is loaded.
//
// Working memory (fixed maximum sizes, see kNa* below): per-group positive
// counters, pointers and entries, per-sample sorted slot lists, per-block loss
// partials.  Every call reuses the same array, so calls that overlap on the
// GPU (two streams, or two host threads) race and must be serialized by the
// caller.  The counters are cleared at the start of every call.
#include <atomic>
#include <climits>

#include "sg_internal.cuh"

namespace {

constexpr int64_t kNaMaxK = 300000;   // groups (L / G)
constexpr int64_t kNaMaxNnz = 65536;  // positives per call
constexpr int32_t kNaMaxB = 256;      // samples
constexpr int kNaParts = 1024;        // loss partials (blocks of the BCE kernel)
constexpr int kThreads = 256;

struct NaScratch {
    int32_t gcount[kNaMaxK + 1];
    int32_t gptr[kNaMaxK + 1];
    int32_t gent[kNaMaxNnz];
    int32_t tsorted[kNaMaxNnz];
    int32_t tslots[kNaMaxNnz];
    int32_t rowcnt[kNaMaxB];
    double loss_part[kNaParts];
};

// about 3.2 MB, held by every GPU that loads the library until the process exits
static __device__ __align__(256) NaScratch g_na_scratch;

// Host-side device addresses of g_na_scratch, looked up once per device (the
// symbol's host name is only a stand-in, never a device address).  Two host
// threads may race on the first lookup: both find the same address, and the
// atomic store keeps the race benign.  cudaDeviceReset ends the context the
// address belongs to; this cache does not follow a reset.
constexpr int kNaMaxDevices = 64;
std::atomic<NaScratch *> g_na_addr[kNaMaxDevices];

// Row b of the positives is well formed when 0 <= rowptr[b] <= rowptr[b+1]
// <= nnz and rowptr[b] is at least every earlier row's start: well-formed rows
// then never overlap (each starts at or after the end of every earlier one),
// so their sorted copies below never share scratch entries.
__device__ __forceinline__ bool na_row_ok(const int32_t *__restrict__ rowptr, int b, int64_t nnz, int lane)
{
    const int64_t r0 = rowptr[b], r1 = rowptr[b + 1];
    int32_t mx = INT32_MIN;
    for (int c = lane; c < b; c += 32)
        mx = max(mx, rowptr[c]);
    for (int o = 16; o > 0; o >>= 1)
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    return r0 >= 0 && r1 >= r0 && r1 <= nnz && r0 >= mx;
}

// one warp per sample: validate, sort and deduplicate the sample's slots,
// count them per group; out-of-range slots and malformed rows are dropped
__global__ void k_na_rows(int32_t B, const int32_t *__restrict__ rowptr,
                          const int32_t *__restrict__ slots, int64_t nnz, int64_t L,
                          int32_t G, NaScratch *sc)
{
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (b >= B)
        return;
    const int64_t r0 = rowptr[b], r1 = rowptr[b + 1];
    if (!na_row_ok(rowptr, b, nnz, lane)) {
        if (lane == 0)
            sc->rowcnt[b] = 0;
        return;
    }
    const int n = (int)(r1 - r0);
    for (int i = lane; i < n; i += 32) {
        int32_t v = slots[r0 + i];
        if (v < 0 || v >= L)
            v = -1;
        int rank = 0;
        for (int q = 0; q < n; ++q) {
            int32_t u = slots[r0 + q];
            if (u < 0 || u >= L)
                u = -1;
            rank += (u < v) | ((u == v) & (q < i));
        }
        sc->tsorted[r0 + rank] = v;
    }
    __syncwarp();
    __threadfence_block();
    int kept = 0;
    for (int base = 0; base < n; base += 32) {
        const int p = base + lane;
        const int32_t v = p < n ? sc->tsorted[r0 + p] : -1;
        const int32_t prev = (p > 0 && p <= n) ? sc->tsorted[r0 + p - 1] : -1;
        const bool keep = p < n && v >= 0 && (p == 0 || v != prev);
        const unsigned m = __ballot_sync(0xffffffffu, keep);
        if (keep) {
            sc->tslots[r0 + kept + __popc(m & ((1u << lane) - 1u))] = v;
            atomicAdd(&sc->gcount[v / G], 1);
        }
        kept += __popc(m);
    }
    if (lane == 0)
        sc->rowcnt[b] = kept;
}

// single block: gptr = exclusive scan of gcount[0..K), gptr[K] = total
__global__ void __launch_bounds__(1024) k_na_scan(int64_t K, NaScratch *sc)
{
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t carry_s;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0)
        carry_s = 0;
    __syncthreads();
    for (int64_t base = 0; base < K; base += 1024) {
        const int64_t i = base + tid;
        const int32_t v = i < K ? sc->gcount[i] : 0;
        int32_t x = v;
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o)
                x += y;
        }
        if (lane == 31)
            warp_sums[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int32_t w = warp_sums[lane];
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o)
                    w += y;
            }
            warp_sums[lane] = w;
        }
        __syncthreads();
        const int32_t excl = carry_s + (wid ? warp_sums[wid - 1] : 0) + x - v;
        if (i < K)
            sc->gptr[i] = excl;
        __syncthreads();
        if (tid == 1023)
            carry_s = excl + v;
        __syncthreads();
    }
    if (tid == 0)
        sc->gptr[K] = carry_s;
}

// bucket the kept entries by group: (b << 16) | j
__global__ void k_na_place(int32_t B, const int32_t *__restrict__ rowptr, int32_t G, NaScratch *sc)
{
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (b >= B)
        return;
    const int64_t r0 = rowptr[b];
    const int n = sc->rowcnt[b];
    for (int c = lane; c < n; c += 32) {
        const int32_t v = sc->tslots[r0 + c];
        const int32_t k = v / G;
        const int32_t pos = atomicSub(&sc->gcount[k], 1) - 1;
        sc->gent[sc->gptr[k] + pos] = (b << 16) | (v - k * G);
    }
}

__device__ __forceinline__ int na_is_positive(const NaScratch *sc, int64_t k, int b, int j)
{
    const int e1 = sc->gptr[k + 1];
    const int want = (b << 16) | j;
    for (int e = sc->gptr[k]; e < e1; ++e)
        if (sc->gent[e] == want)
            return 1;
    return 0;
}

// dZ = sigmoid(Z) - Y over all B x L entries; one loss partial per block
__global__ void __launch_bounds__(kThreads)
    k_na_bce(const uint16_t *__restrict__ Z, int B, int64_t L, int G,
             uint16_t *__restrict__ dZ, NaScratch *sc)
{
    const int64_t total = (int64_t)B * L;
    double lacc = 0.0;
    for (int64_t e = blockIdx.x * (int64_t)kThreads + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * kThreads) {
        const int b = (int)(e / L);
        const int64_t s = e - (int64_t)b * L;
        const int64_t k = s / G;
        const int y = na_is_positive(sc, k, b, (int)(s - k * G));
        float lt;
        const float d = bce_grad_loss(bf2f(Z[e]), y, &lt);
        dZ[e] = f2bf(d);
        lacc += lt;
    }
    __shared__ double red[kThreads / 32];
    for (int o = 16; o > 0; o >>= 1)
        lacc += __shfl_down_sync(0xffffffffu, lacc, o);
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = lacc;
    __syncthreads();
    if (threadIdx.x == 0) {
        double s = 0.0;
        for (int w = 0; w < kThreads / 32; ++w)
            s += red[w];
        sc->loss_part[blockIdx.x] = s;
    }
}

__global__ void __launch_bounds__(1024) k_na_loss(int n, const NaScratch *sc, double *loss)
{
    __shared__ double s[1024];
    double acc = 0.0;
    for (int i = threadIdx.x; i < n; i += 1024)
        acc += sc->loss_part[i];
    s[threadIdx.x] = acc;
    __syncthreads();
    for (int w = 512; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w)
            s[threadIdx.x] += s[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0)
        *loss = s[0];
}

#define NA_FAIL(code, ...)          \
    do {                            \
        sg_set_error(__VA_ARGS__);  \
        return code;                \
    } while (0)

}  // namespace

extern "C" sg_status sg_bce_grad_noalloc(const sg_bf16 *Z, int32_t B, int64_t L, int32_t G,
                                         const int32_t *pos_rowptr, const int32_t *pos_slot,
                                         int64_t nnz, sg_bf16 *dZ, double *loss, void *stream)
{
    const char *fn = "sg_bce_grad_noalloc";
    if (!Z || !dZ || !loss || !pos_rowptr || (nnz > 0 && !pos_slot))
        NA_FAIL(SG_ERR_INVALID, "%s: a required pointer is NULL", fn);
    if (B < 1 || L < 1 || G < 1 || nnz < 0 || L % G != 0)
        NA_FAIL(SG_ERR_INVALID, "%s: bad sizes (B=%d L=%lld G=%d nnz=%lld)", fn, B,
                (long long)L, G, (long long)nnz);
    if (B > kNaMaxB || L / G > kNaMaxK || nnz > kNaMaxNnz || G > 65535)
        NA_FAIL(SG_ERR_UNSUPPORTED, "%s: above the fixed working-memory limits "
                "(B <= %d, L/G <= %lld, nnz <= %lld, G <= 65535)", fn, kNaMaxB,
                (long long)kNaMaxK, (long long)kNaMaxNnz);
    int dev = 0;
    SG_TRY_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kNaMaxDevices)
        NA_FAIL(SG_ERR_UNSUPPORTED, "%s: device ordinal %d above %d", fn, dev, kNaMaxDevices);
    NaScratch *sc = g_na_addr[dev].load(std::memory_order_acquire);
    if (!sc) {
        // first call on this device (its device current): resolve the array's
        // device address, a runtime lookup that allocates nothing
        void *p = nullptr;
        SG_TRY_CUDA(cudaGetSymbolAddress(&p, g_na_scratch));
        sc = static_cast<NaScratch *>(p);
        g_na_addr[dev].store(sc, std::memory_order_release);
    }
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t K = L / G;
    SG_TRY_CUDA(cudaMemsetAsync(sc->gcount, 0, sizeof(int32_t) * (K + 1), st));
    const int wpb = kThreads / 32;
    const int rows_grid = (int)ceil_div(B, wpb);
    k_na_rows<<<rows_grid, kThreads, 0, st>>>(B, pos_rowptr, pos_slot, nnz, L, G, sc);
    k_na_scan<<<1, 1024, 0, st>>>(K, sc);
    k_na_place<<<rows_grid, kThreads, 0, st>>>(B, pos_rowptr, G, sc);
    int64_t blocks = ceil_div((int64_t)B * L, kThreads);
    if (blocks > kNaParts)
        blocks = kNaParts;
    k_na_bce<<<(int)blocks, kThreads, 0, st>>>(Z, B, L, G, dZ, sc);
    k_na_loss<<<1, 1024, 0, st>>>((int)blocks, sc, loss);
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}
