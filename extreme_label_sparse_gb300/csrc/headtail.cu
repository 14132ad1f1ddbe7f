// The head-tail split of the output layer (HASTE, "Method / overall
// framework" and key design "head-tail split"): the encoder output h (B x E)
// feeds a dense head and the group-shared sparse tail through two light
// projections, and the objective is the sum of both branches' BCE terms.
//
//   h_head = h P_head^T,  h_tail = h P_tail^T                (tcgen05 GEMMs)
//   head: the layer itself with every group's index set [0, Dh) -- the
//         dense logits h_head W_head^T, their BCE, dW_head and dh_head
//   tail: the layer on h_tail -- dW_tail, dh_tail
//   dP_head = dh_head^T h, dP_tail = dh_tail^T h, dh = dh_head P_head +
//   dh_tail P_tail                                           (tcgen05 GEMMs)
//
// The fp32 gradients dh_head, dh_tail enter the backward GEMMs as two bf16
// planes (value and rounding residual), so they keep about 16 bits.
#include "sg_internal.cuh"

sg_status gemm_bf16(const uint16_t *A, int a_mn, int64_t lda, const uint16_t *B, int b_mn, int64_t ldb, int M,
                    int N, int K, void *C, int c_bf16, int64_t ldc, int accumulate, int32_t *status, cudaStream_t st);
sg_status split_hilo(const float *x, int64_t n, uint16_t *hi, uint16_t *lo, cudaStream_t st);

namespace {

#define HT_FAIL(code, ...)         \
    do {                           \
        sg_set_error(__VA_ARGS__); \
        return code;               \
    } while (0)

#define HT_TRY(expr)            \
    do {                        \
        sg_status rc_ = (expr); \
        if (rc_ != SG_OK)       \
            return rc_;         \
    } while (0)

__global__ void k_add_loss(const double *a, const double *b, double *out)
{
    if (threadIdx.x == 0 && blockIdx.x == 0)
        *out = *a + *b;
}

// dP (D x E) = g^T h and dh (B x E) (+)= g P from g = dL/d(h P^T) (B x D, fp32),
// g split into the bf16 planes gh, gl (B x D each)
sg_status proj_bwd(const uint16_t *h, int B, int E, const uint16_t *P, int D, const float *g, uint16_t *gh,
                   uint16_t *gl, float *dP, float *dh, int accumulate_dh, int32_t *status, cudaStream_t st)
{
    HT_TRY(split_hilo(g, (int64_t)B * D, gh, gl, st));
    // dP[d][e] = sum_b g[b][d] h[b][e]: A = g^T (MN-major, M = D), B = h^T (MN-major, N = E)
    HT_TRY(gemm_bf16(gh, 1, D, h, 1, E, D, E, B, dP, 0, E, 0, status, st));
    HT_TRY(gemm_bf16(gl, 1, D, h, 1, E, D, E, B, dP, 0, E, 1, status, st));
    // dh[b][e] (+)= sum_d g[b][d] P[d][e]: A = g (K-major), B = P^T (MN-major, N = E)
    HT_TRY(gemm_bf16(gh, 0, D, P, 1, E, B, E, D, dh, 0, E, accumulate_dh, status, st));
    HT_TRY(gemm_bf16(gl, 0, D, P, 1, E, B, E, D, dh, 0, E, 1, status, st));
    return SG_OK;
}

bool sizes_ok(int32_t B, int32_t E, int32_t D) { return B >= 1 && E >= 8 && D >= 8 && E % 8 == 0 && D % 8 == 0; }

// makes `dev` current for the duration of a call
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

}  // namespace

extern "C" {

sg_status sg_proj_fwd(const sg_bf16 *h, int32_t B, int32_t E, const sg_bf16 *P, int32_t D, sg_bf16 *out,
                      void *stream)
{
    const char *fn = "sg_proj_fwd";
    NvtxRange nvtx_(fn);
    if (!h || !P || !out)
        HT_FAIL(SG_ERR_INVALID, "%s: a required pointer is NULL", fn);
    if (!sizes_ok(B, E, D))
        HT_FAIL(SG_ERR_INVALID, "%s: need B >= 1 and E, D multiples of 8 (B=%d E=%d D=%d)", fn, B, E, D);
    // out[b][d] = sum_e h[b][e] P[d][e]: A = h (K-major), B = P (K-major)
    return gemm_bf16(h, 0, E, P, 0, E, B, D, E, out, 1, D, 0, nullptr, (cudaStream_t)stream);
}

sg_status sg_proj_bwd(const sg_bf16 *h, int32_t B, int32_t E, const sg_bf16 *P, int32_t D, const float *g,
                      sg_bf16 *work, float *dP, float *dh, int32_t accumulate_dh, void *stream)
{
    const char *fn = "sg_proj_bwd";
    NvtxRange nvtx_(fn);
    if (!h || !P || !g || !work || !dP || !dh)
        HT_FAIL(SG_ERR_INVALID, "%s: a required pointer is NULL", fn);
    if (!sizes_ok(B, E, D))
        HT_FAIL(SG_ERR_INVALID, "%s: need B >= 1 and E, D multiples of 8 (B=%d E=%d D=%d)", fn, B, E, D);
    return proj_bwd(h, B, E, P, D, g, work, work + (size_t)B * D, dP, dh, accumulate_dh, nullptr,
                    (cudaStream_t)stream);
}

sg_status sg_headtail_step(sg_layout *head, sg_layout *tail, const sg_bf16 *h, int32_t B, int32_t E,
                           const sg_bf16 *P_head, const sg_bf16 *P_tail, const sg_bf16 *W_head,
                           const int32_t *head_rowptr, const int32_t *head_label, int64_t head_nnz,
                           const sg_bf16 *W_tail, const int32_t *tail_rowptr, const int32_t *tail_label,
                           int64_t tail_nnz, sg_bf16 *dW_head, sg_bf16 *dW_tail, float *dP_head, float *dP_tail,
                           float *dh, double *loss, void *stream)
{
    const char *fn = "sg_headtail_step";
    NvtxRange nvtx_(fn);
    if (!head || !tail)
        HT_FAIL(SG_ERR_INVALID, "%s: layout is NULL", fn);
    if (!h || !P_head || !P_tail || !W_head || !W_tail || !dW_head || !dW_tail || !dP_head || !dP_tail || !dh ||
        !loss)
        HT_FAIL(SG_ERR_INVALID, "%s: a required pointer is NULL", fn);
    if (head->device != tail->device)
        HT_FAIL(SG_ERR_INVALID, "%s: the head and tail layouts live on different devices", fn);
    const int32_t Dh = head->H, H = tail->H;
    if (!sizes_ok(B, E, Dh) || !sizes_ok(B, E, H))
        HT_FAIL(SG_ERR_INVALID, "%s: need B >= 1 and E, Dh, H multiples of 8 (B=%d E=%d Dh=%d H=%d)", fn, B, E,
                Dh, H);
    if (B > head->max_B || B > tail->max_B)
        HT_FAIL(SG_ERR_INVALID, "%s: B=%d exceeds a layout's max_B", fn, B);
    DevScope ds(tail->device);
    cudaStream_t st = (cudaStream_t)stream;
    // scratch in the tail layout: the projected activations (bf16), both
    // branches' dh (fp32), the bf16 planes of one of them, two losses
    const size_t need = (size_t)B * (Dh + H) * 2 + (size_t)B * (Dh + H) * 4 + (size_t)B * (Dh > H ? Dh : H) * 4 + 64;
    if (tail->ht_ws_bytes < need) {
        if (tail->ht_ws)
            cudaFree(tail->ht_ws);
        tail->ht_ws = nullptr;
        tail->ht_ws_bytes = 0;
        if (cudaMalloc(&tail->ht_ws, need) != cudaSuccess) {
            cudaGetLastError();
            HT_FAIL(SG_ERR_OOM, "%s: cudaMalloc of %zu bytes of scratch failed", fn, need);
        }
        tail->ht_ws_bytes = need;
    }
    uint8_t *w8 = static_cast<uint8_t *>(tail->ht_ws);
    double *losses = reinterpret_cast<double *>(w8);
    uint16_t *h_head = reinterpret_cast<uint16_t *>(w8 + 64);
    uint16_t *h_tail = h_head + (size_t)B * Dh;
    float *dh_head = reinterpret_cast<float *>(h_tail + (size_t)B * H);
    float *dh_tail = dh_head + (size_t)B * Dh;
    uint16_t *gh = reinterpret_cast<uint16_t *>(dh_tail + (size_t)B * H);
    uint16_t *gl = gh + (size_t)B * (Dh > H ? Dh : H);
    HT_TRY(gemm_bf16(h, 0, E, P_head, 0, E, B, Dh, E, h_head, 1, Dh, 0, tail->status, st));
    HT_TRY(gemm_bf16(h, 0, E, P_tail, 0, E, B, H, E, h_tail, 1, H, 0, tail->status, st));
    HT_TRY(sg_step(head, h_head, B, W_head, head_rowptr, head_label, head_nnz, dW_head, dh_head, losses, stream));
    HT_TRY(sg_step(tail, h_tail, B, W_tail, tail_rowptr, tail_label, tail_nnz, dW_tail, dh_tail, losses + 1,
                   stream));
    HT_TRY(proj_bwd(h, B, E, P_head, Dh, dh_head, gh, gl, dP_head, dh, 0, tail->status, st));
    HT_TRY(proj_bwd(h, B, E, P_tail, H, dh_tail, gh, gl, dP_tail, dh, 1, tail->status, st));
    k_add_loss<<<1, 32, 0, st>>>(losses, losses + 1, loss);
    SG_TRY_CUDA(cudaGetLastError());
    return SG_OK;
}

}  // extern "C"
