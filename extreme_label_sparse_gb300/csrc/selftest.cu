// Self-test of the library's failure detection: a kernel whose bounded
// waits run out.  Every wait of the tensor-core kernels goes through
// mbar_wait (tc_ptx.cuh), which gives up after a limit of %globaltimer time,
// records SG_ERR_TIMEOUT and makes the kernel wind down: it releases its TMEM
// and returns, so the context stays usable.  Here two warps wait on an
// mbarrier that nothing arrives on, while the CTA holds TMEM columns, exactly
// as a stalled pipeline would; the recorded status goes back to the host.
#include "sg_internal.cuh"
#include "tc_ptx.cuh"

using namespace tc;

namespace {

__global__ void __launch_bounds__(64, 1) k_wait_timeout(int32_t *status)
{
    __shared__ uint64_t bar;
    __shared__ uint32_t holder;
    __shared__ int abort_flag;
    const int warp = threadIdx.x / 32;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bar), 1);  // one arrival expected; none comes
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&holder), 32);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = holder;
    volatile int *ab = &abort_flag;
    // both warps wait; the first to reach the limit flags the timeout, the
    // other sees the abort flag (or its own limit) and gives up too
    const bool ok = mbar_wait(smem_u32(&bar), 0, ab, status);
    if (ok)  // cannot happen: nothing arrives
        sg_flag(status, SG_ERR_INVALID);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tbase, 32);
    }
}

}  // namespace

extern "C" sg_status sg_selftest_wait_timeout(int32_t *code)
{
    if (!code) {
        sg_set_error("sg_selftest_wait_timeout: code is NULL");
        return SG_ERR_INVALID;
    }
    int32_t *d = nullptr;
    if (cudaMalloc((void **)&d, sizeof(int32_t)) != cudaSuccess) {
        cudaGetLastError();
        sg_set_error("sg_selftest_wait_timeout: cudaMalloc of 4 bytes failed");
        return SG_ERR_OOM;
    }
    sg_status rc = SG_OK;
    if (cudaMemset(d, 0, sizeof(int32_t)) != cudaSuccess) {
        rc = SG_ERR_CUDA;
    } else {
        k_wait_timeout<<<1, 64>>>(d);
        if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess ||
            cudaMemcpy(code, d, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
            rc = SG_ERR_CUDA;
    }
    if (rc != SG_OK)
        sg_set_error("sg_selftest_wait_timeout: %s", cudaGetErrorString(cudaGetLastError()));
    cudaFree(d);
    return rc;
}
