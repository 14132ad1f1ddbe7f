// Layout builder: groups the labels into slots and fixes each group's sorted
// fan-in set (HASTE, key design "group-shared fixed fan-in sparsity": K groups
// of exactly G labels, one shared I_k of F dims per group, index memory
// (L/G)*F stored as uint16).
#include "sg_internal.cuh"

namespace {

constexpr int kThreads = 256;

// Count the labels of every group and drop each label into a free position
// of its group (unordered for now).
__global__ void k_group_count(const int32_t *__restrict__ groups, int64_t L,
                              int64_t K, int32_t G, int32_t *cnt, int32_t *tmp,
                              int32_t *status)
{
    for (int64_t l = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; l < L;
         l += (int64_t)gridDim.x * blockDim.x) {
        int32_t g = groups[l];
        if (g < 0 || g >= K) {
            sg_flag(status, SG_ERR_DATA);
            continue;
        }
        int32_t pos = atomicAdd(&cnt[g], 1);
        if (pos < G)
            tmp[(int64_t)g * G + pos] = (int32_t)l;
    }
}

__global__ void k_group_check(const int32_t *__restrict__ cnt, int64_t K,
                              int32_t G, int32_t *status)
{
    for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < K;
         k += (int64_t)gridDim.x * blockDim.x)
        if (cnt[k] != G)
            sg_flag(status, SG_ERR_DATA);
}

// One warp per group: rank the group's G (distinct) label ids; the label of
// rank r takes slot k*G + r.
__global__ void k_group_slots(const int32_t *__restrict__ tmp, int64_t K,
                              int32_t G, int32_t *label_of_slot,
                              int32_t *slot_of_label)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t k = blockIdx.x * (int64_t)(blockDim.x / 32) + threadIdx.x / 32;
         k < K; k += warps) {
        const int32_t *grp = tmp + k * G;
        for (int j = lane; j < G; j += 32) {
            int32_t v = grp[j];
            int r = 0;
            for (int i = 0; i < G; ++i)
                r += grp[i] < v;
            int64_t s = k * G + r;
            label_of_slot[s] = v;
            slot_of_label[v] = (int32_t)s;
        }
    }
}

// One warp per group: validate and sort I_k ascending, store as uint16.
__global__ void k_idx_sort(const int32_t *__restrict__ idx, int64_t K,
                           int32_t F, int32_t H, uint16_t *idx_s,
                           int32_t *status)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t k = blockIdx.x * (int64_t)(blockDim.x / 32) + threadIdx.x / 32;
         k < K; k += warps) {
        const int32_t *row = idx + k * F;
        for (int f = lane; f < F; f += 32) {
            int32_t v = row[f];
            if (v < 0 || v >= H) {
                sg_flag(status, SG_ERR_DATA);
                continue;
            }
            int less = 0, same_before = 0, same = 0;
            for (int i = 0; i < F; ++i) {
                int32_t u = row[i];
                less += u < v;
                same += u == v;
                same_before += (u == v) & (i < f);
            }
            if (same > 1)
                sg_flag(status, SG_ERR_DATA);
            idx_s[k * F + less + same_before] = (uint16_t)v;
        }
    }
}

int grid_for(int64_t n, int threads, int cap)
{
    int64_t g = ceil_div(n, threads);
    if (g < 1)
        g = 1;
    return (int)(g < cap ? g : cap);
}

}  // namespace

sg_status sg_layout_kernels(sg_layout *lo, const int32_t *groups,
                            const int32_t *idx, cudaStream_t st)
{
    const int64_t L = lo->L, K = lo->K;
    const int32_t G = lo->G;
    const int cap = lo->num_sms * 16;
    int32_t *cnt = nullptr, *tmp = nullptr;
    sg_status rc = SG_OK;
    int32_t code = 0;

    if (cudaMallocAsync((void **)&cnt, sizeof(int32_t) * K, st) != cudaSuccess ||
        cudaMallocAsync((void **)&tmp, sizeof(int32_t) * L, st) != cudaSuccess) {
        sg_set_error("sg_layout_build: device allocation of %lld bytes failed",
                     (long long)(4 * (K + L)));
        rc = SG_ERR_OOM;
        goto done;
    }
    if (cudaMemsetAsync(cnt, 0, sizeof(int32_t) * K, st) != cudaSuccess ||
        cudaMemsetAsync(tmp, 0xff, sizeof(int32_t) * L, st) != cudaSuccess) {
        rc = SG_ERR_CUDA;
        goto done;
    }
    k_group_count<<<grid_for(L, kThreads, cap), kThreads, 0, st>>>(
        groups, L, K, G, cnt, tmp, lo->status);
    k_group_check<<<grid_for(K, kThreads, cap), kThreads, 0, st>>>(cnt, K, G,
                                                                 lo->status);
    k_idx_sort<<<grid_for(K * 32, kThreads, cap), kThreads, 0, st>>>(
        idx, K, lo->F, lo->H, lo->idx_s, lo->status);
    if (cudaMemcpyAsync(&code, lo->status, sizeof code, cudaMemcpyDeviceToHost,
                        st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        sg_set_error("sg_layout_build: %s", cudaGetErrorString(cudaGetLastError()));
        rc = SG_ERR_CUDA;
        goto done;
    }
    if (code != 0) {
        sg_set_error("sg_layout_build: bad groups or idx (a group id outside "
                     "[0,K), a group without exactly G labels, or an index "
                     "duplicated / outside [0,H))");
        rc = (sg_status)code;
        goto done;
    }
    // every group now holds exactly G distinct labels: rank them into slots
    k_group_slots<<<grid_for(K * 32, kThreads, cap), kThreads, 0, st>>>(
        tmp, K, G, lo->label_of_slot, lo->slot_of_label);
    if (cudaStreamSynchronize(st) != cudaSuccess) {
        sg_set_error("sg_layout_build: %s", cudaGetErrorString(cudaGetLastError()));
        rc = SG_ERR_CUDA;
    }
done:
    if (cnt)
        cudaFreeAsync(cnt, st);
    if (tmp)
        cudaFreeAsync(tmp, st);
    cudaStreamSynchronize(st);
    return rc;
}
