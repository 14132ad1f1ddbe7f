// Positive-label preparation for one call: Y of the BCE objective (HASTE, key
// design "head-tail split": sum of per-label BCE terms) as per-group lists, so
// the forward epilogue of group k can read its few positives directly.
//
//   1. k_pos_rows  : one warp per sample: labels -> slots, sort, drop
//                    duplicates (Y is binary), count positives per group.
//   2. k_scan_*    : exclusive scan of the per-group counts -> gptr[K+1].
//   3. k_pos_place : bucket the entries by group: gent[] = (b << 16) | j.
//                    Placement counts the group counters back down to zero,
//                    so they are ready for the next call without a memset.
#include "sg_internal.cuh"

namespace {

constexpr int kThreads = 256;

// sample row b, by one warp
__device__ __forceinline__ void pos_row(int b, int32_t B, const int32_t *__restrict__ rowptr,
                                        const int32_t *__restrict__ labels, int64_t nnz, int64_t L, int32_t G,
                                        const int32_t *__restrict__ slot_of_label, int32_t *tsorted,
                                        int32_t *tslots, int32_t *rowcnt, int32_t *gcount, int32_t *status)
{
    const int lane = threadIdx.x & 31;
    if (b == 0 && lane == 0 && (rowptr[0] != 0 || (int64_t)rowptr[B] != nnz))
        sg_flag(status, SG_ERR_DATA);
    const int64_t r0 = rowptr[b], r1 = rowptr[b + 1];
    if (r0 < 0 || r1 < r0 || r1 > nnz) {
        if (lane == 0) {
            sg_flag(status, SG_ERR_DATA);
            rowcnt[b] = 0;
        }
        return;
    }
    const int n = (int)(r1 - r0);
    // pass 1: stable rank sort of the row's slots (invalid labels -> -1 first)
    for (int i = lane; i < n; i += 32) {
        int32_t lab = labels[r0 + i];
        int32_t v;
        if (lab < 0 || lab >= L) {
            sg_flag(status, SG_ERR_DATA);
            v = -1;
        } else {
            v = slot_of_label[lab];
        }
        int rank = 0;
        for (int q = 0; q < n; ++q) {
            int32_t lq = labels[r0 + q];
            int32_t u = (lq < 0 || lq >= L) ? -1 : slot_of_label[lq];
            rank += (u < v) | ((u == v) & (q < i));
        }
        tsorted[r0 + rank] = v;
    }
    __syncwarp();
    __threadfence_block();
    // pass 2: keep the first of each run of equal values, compact in order
    int kept = 0;
    for (int base = 0; base < n; base += 32) {
        int p = base + lane;
        int32_t v = p < n ? tsorted[r0 + p] : -1;
        int32_t prev = (p > 0 && p <= n) ? tsorted[r0 + p - 1] : -1;
        bool keep = p < n && v >= 0 && (p == 0 || v != prev);
        unsigned m = __ballot_sync(0xffffffffu, keep);
        if (keep) {
            int at = kept + __popc(m & ((1u << lane) - 1u));
            tslots[r0 + at] = v;
            atomicAdd(&gcount[v / G], 1);
        }
        kept += __popc(m);
    }
    if (lane == 0)
        rowcnt[b] = kept;
}

__global__ void k_pos_rows(int32_t B, const int32_t *__restrict__ rowptr,
                           const int32_t *__restrict__ labels, int64_t nnz,
                           int64_t L, int32_t G,
                           const int32_t *__restrict__ slot_of_label,
                           int32_t *tsorted, int32_t *tslots, int32_t *rowcnt,
                           int32_t *gcount, int32_t *status)
{
    const int b = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (b < B)
        pos_row(b, B, rowptr, labels, nnz, L, G, slot_of_label, tsorted, tslots, rowcnt, gcount, status);
}

// The step's first launch: blocks [0, rows_blocks) take the positive rows
// (a warp per sample), the others one 32 x 32 tile of h^T each (tiles_x tiles
// along H), so the two independent parts run side by side.
__global__ void __launch_bounds__(kThreads) k_prep_step(int rows_blocks, int tiles_x, int32_t B,
                                                        const int32_t *__restrict__ rowptr,
                                                        const int32_t *__restrict__ labels, int64_t nnz,
                                                        int64_t L, int32_t G,
                                                        const int32_t *__restrict__ slot_of_label,
                                                        int32_t *tsorted, int32_t *tslots, int32_t *rowcnt,
                                                        int32_t *gcount, int32_t *status,
                                                        const uint16_t *__restrict__ h, int32_t H, int32_t ldB,
                                                        uint16_t *__restrict__ hT)
{
    __shared__ uint16_t tile[32][34];
    if ((int)blockIdx.x >= rows_blocks) {
        const int t = (int)blockIdx.x - rows_blocks;
        transpose_h_tile(h, B, H, ldB, hT, (t % tiles_x) * 32, (t / tiles_x) * 32, threadIdx.x & 31,
                         threadIdx.x >> 5, tile);
        return;
    }
    const int b = blockIdx.x * (kThreads / 32) + threadIdx.x / 32;
    if (b < B)
        pos_row(b, B, rowptr, labels, nnz, L, G, slot_of_label, tsorted, tslots, rowcnt, gcount, status);
}

// Exclusive scan out[i] = sum_{j<i} in[j], out[n] = total, in two passes over
// tiles of kScanTile entries: k_scan_tiles scans each tile on its own and
// records the tile's total; k_scan_add adds the totals of the tiles before it.
constexpr int kScanTile = 4096;  // 1024 threads x 4 entries

__global__ void __launch_bounds__(1024) k_scan_tiles(const int32_t *__restrict__ in, int64_t n,
                                                     int32_t *out, int32_t *tile_sum)
{
    __shared__ int32_t warp_sums[32];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int64_t base = (int64_t)blockIdx.x * kScanTile + (int64_t)tid * 4;
    int32_t v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
        v[e] = base + e < n ? in[base + e] : 0;
    const int32_t own = v[0] + v[1] + v[2] + v[3];
    int32_t x = own;
#pragma unroll
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
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o)
                w += y;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    int32_t run = (wid ? warp_sums[wid - 1] : 0) + x - own;  // exclusive prefix in the tile
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        if (base + e < n)
            out[base + e] = run;
        run += v[e];
    }
    if (tid == 1023)
        tile_sum[blockIdx.x] = warp_sums[31];
}

__global__ void __launch_bounds__(1024) k_scan_add(int64_t n, int32_t *out, const int32_t *tile_sum)
{
    __shared__ int32_t off_s;
    if (threadIdx.x < 32) {
        int32_t s = 0;
        for (int t = threadIdx.x; t < (int)blockIdx.x; t += 32)
            s += tile_sum[t];
        for (int o = 16; o > 0; o >>= 1)
            s += __shfl_down_sync(0xffffffffu, s, o);
        if (threadIdx.x == 0)
            off_s = s;
    }
    __syncthreads();
    const int32_t off = off_s;
    const int64_t base = (int64_t)blockIdx.x * kScanTile + (int64_t)threadIdx.x * 4;
    if (off)
        for (int e = 0; e < 4; ++e)
            if (base + e < n)
                out[base + e] += off;
    if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0)
        out[n] = off + tile_sum[blockIdx.x];
}

__global__ void k_pos_place(int32_t B, const int32_t *__restrict__ rowptr,
                            const int32_t *__restrict__ tslots,
                            const int32_t *__restrict__ rowcnt, int32_t G,
                            const int32_t *__restrict__ gptr, int32_t *gcount,
                            int32_t *gent)
{
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (b >= B)
        return;
    const int64_t r0 = rowptr[b];
    const int n = rowcnt[b];
    for (int c = lane; c < n; c += 32) {
        int32_t v = tslots[r0 + c];
        int32_t k = v / G;
        int32_t pos = atomicSub(&gcount[k], 1) - 1;
        gent[gptr[k] + pos] = (b << 16) | (v - k * G);
    }
}

// canonical slot-CSR: compacted rows
__global__ void k_pos_compact(int32_t B, const int32_t *__restrict__ rowptr,
                              const int32_t *__restrict__ tslots,
                              const int32_t *__restrict__ rowcnt,
                              const int32_t *__restrict__ out_rowptr,
                              int32_t *out_slots)
{
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (b >= B)
        return;
    const int64_t r0 = rowptr[b];
    const int n = rowcnt[b];
    for (int c = lane; c < n; c += 32)
        out_slots[out_rowptr[b] + c] = tslots[r0 + c];
}

__global__ void __launch_bounds__(1024) k_loss_finalize(const double *__restrict__ part,
                                                        int n, double *loss)
{
    __shared__ double s[1024];
    double acc = 0.0;
    for (int i = threadIdx.x; i < n; i += 1024)
        acc += part[i];
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

}  // namespace

sg_status sg_pos_prepare(sg_layout *lo, int32_t B, const int32_t *rowptr,
                         const int32_t *labels, int64_t nnz, cudaStream_t st)
{
    const int wpb = kThreads / 32;
    const int rows_grid = (int)ceil_div(B, wpb);
    SG_LAUNCH(lo, SG_KIND_PREP, st, k_pos_rows<<<rows_grid, kThreads, 0, st>>>(B, rowptr, labels, nnz, lo->L,
                                               lo->G, lo->slot_of_label,
                                               lo->tsorted, lo->tslots,
                                               lo->rowcnt, lo->gcount,
                                               lo->status));
    const int tiles = (int)((lo->K + kScanTile - 1) / kScanTile);
    SG_LAUNCH(lo, SG_KIND_PREP, st,
              k_scan_tiles<<<tiles, 1024, 0, st>>>(lo->gcount, lo->K, lo->gptr, lo->scan_part));
    SG_LAUNCH(lo, SG_KIND_PREP, st, k_scan_add<<<tiles, 1024, 0, st>>>(lo->K, lo->gptr, lo->scan_part));
    SG_LAUNCH(lo, SG_KIND_PREP, st, k_pos_place<<<rows_grid, kThreads, 0, st>>>(B, rowptr, lo->tslots,
                                                lo->rowcnt, lo->G, lo->gptr,
                                                lo->gcount, lo->gent));
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}

sg_status sg_step_prepare(sg_layout *lo, const uint16_t *h, int32_t B, const int32_t *rowptr,
                          const int32_t *labels, int64_t nnz, cudaStream_t st)
{
    const int wpb = kThreads / 32;
    const int rows_grid = (int)ceil_div(B, wpb);
    const int tiles_x = (int)ceil_div(lo->H, 32), tiles_y = (int)ceil_div(lo->ldB, 32);
    SG_LAUNCH(lo, SG_KIND_PREP, st,
              k_prep_step<<<rows_grid + tiles_x * tiles_y, kThreads, 0, st>>>(
                  rows_grid, tiles_x, B, rowptr, labels, nnz, lo->L, lo->G, lo->slot_of_label, lo->tsorted,
                  lo->tslots, lo->rowcnt, lo->gcount, lo->status, h, lo->H, lo->ldB, lo->hT));
    const int tiles = (int)((lo->K + kScanTile - 1) / kScanTile);
    SG_LAUNCH(lo, SG_KIND_PREP, st,
              k_scan_tiles<<<tiles, 1024, 0, st>>>(lo->gcount, lo->K, lo->gptr, lo->scan_part));
    SG_LAUNCH(lo, SG_KIND_PREP, st, k_scan_add<<<tiles, 1024, 0, st>>>(lo->K, lo->gptr, lo->scan_part));
    SG_LAUNCH(lo, SG_KIND_PREP, st, k_pos_place<<<rows_grid, kThreads, 0, st>>>(B, rowptr, lo->tslots,
                                                lo->rowcnt, lo->G, lo->gptr,
                                                lo->gcount, lo->gent));
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}

sg_status sg_pos_compact(sg_layout *lo, int32_t B, const int32_t *rowptr,
                         int32_t *out_rowptr, int32_t *out_slots,
                         cudaStream_t st)
{
    SG_LAUNCH(lo, SG_KIND_PREP, st, k_scan_tiles<<<1, 1024, 0, st>>>(lo->rowcnt, B, out_rowptr, lo->scan_part));
    SG_LAUNCH(lo, SG_KIND_PREP, st, k_scan_add<<<1, 1024, 0, st>>>(B, out_rowptr, lo->scan_part));
    if (out_slots) {
        const int wpb = kThreads / 32;
        SG_LAUNCH(lo, SG_KIND_PREP, st,
                  k_pos_compact<<<(int)ceil_div(B, wpb), kThreads, 0, st>>>(
                      B, rowptr, lo->tslots, lo->rowcnt, out_rowptr, out_slots));
    }
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}

sg_status sg_loss_finalize(sg_layout *lo, int32_t nparts, double *loss,
                           cudaStream_t st)
{
    SG_LAUNCH(lo, SG_KIND_PREP, st, k_loss_finalize<<<1, 1024, 0, st>>>(lo->loss_part, nparts, loss));
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}
