/*
 * sg.h -- C ABI of the group-shared fixed fan-in sparse output layer, one
 * training step, on one GB300 (sm_103a).
 *
 * The layer (HASTE: Hardware-Aware Dynamic Sparse Training for Large Output
 * Spaces -- "Method / overall framework" and key design "group-shared fixed
 * fan-in sparsity"): L labels are split into K = L/G groups of G labels.  All
 * labels of group k share one fan-in index set I_k of F feature dims; every
 * label keeps its own F weights.  The logit of label l in group k is
 *     z_l = < w_l , h[I_k] >                       (no bias)
 * Per group this is the dense product Z_k = H_k W_k^T with H_k = h[:, I_k]
 * (key design "gather-once + dense MMA kernel"), trained with BCE
 * (key design "head-tail split"; section "loss / training strategy").
 *
 * Conventions used by every call
 *   - bf16 tensors are passed as sg_bf16 (the raw bit pattern, RNE-rounded).
 *   - A "slot" is a label's position after grouping: slot s = k*G + j is the
 *     j-th smallest label id of group k.  W, dW are [L][F] row-major in slot
 *     order; Z, dZ are [B][L] row-major in slot order; h is [B][H] row-major;
 *     dh is [B][H] row-major fp32.
 *   - Positives are given per sample as CSR over LABEL ids:
 *     pos_rowptr[B+1] (pos_rowptr[0] = 0, non-decreasing, pos_rowptr[B] = nnz)
 *     and pos_label[nnz] in [0, L), any order, duplicates allowed (a sample's
 *     label is positive once: Y is binary).
 *   - The loss written is the SUM over all (sample, label) of
 *     max(z,0) - y z + log(1 + exp(-|z|)); dZ = sigmoid(Z) - Y is its exact
 *     gradient.  The page's per-sample mean is that sum divided by B.
 *   - All pointers to tensors are DEVICE pointers to caller-owned memory; the
 *     library never frees or keeps them.  Outputs are overwritten, never
 *     accumulated into.  `stream` is a cudaStream_t (NULL = legacy default).
 *   - Every call except sg_layout_build, sg_layout_export and
 *     sg_layout_status is asynchronous on `stream`.  Argument/shape errors are
 *     returned before anything is launched.  Data errors found on the device
 *     (a label id out of range, a malformed CSR, a bounded wait that gave up)
 *     set the layout's sticky status word, read with sg_layout_status.
 *   - A layout holds scratch memory, so one layout must not be used by two
 *     streams at the same time.
 *   - Thread safety: calls on different layouts may run from different host
 *     threads; sg_last_error is per host thread.
 *
 * Supported range (anything else returns SG_ERR_UNSUPPORTED)
 *   1 <= B <= 256, 1 <= F <= 256, F <= H <= 65535 (idx is u16), 1 <= G <=
 *   256, L = K*G < 2^31.
 *   Tensor-core engine (used when the shape fits it): G in {16, 32} or a
 *   multiple of 64, F % 16 == 0, and a group's tiles within one CTA's shared
 *   memory and TMEM.  All three phases (forward + BCE, dW, dh) run on the
 *   tensor cores for F % 16 == 0 up to
 *                      G = 16, 32   G = 64   G = 128   G = 192   G = 256
 *       B <= 128          256         256       160        32      (dh only)
 *       B <= 256          192         176       144     (dh only)  (dh only)
 *   and also, through the fused forward + BCE + dW kernel (F = 64, 128 or
 *   256), at F = 256 for every G up to 128 and at G = 256 with F = 64 or
 *   128.  dh runs on them for every such G and F.  A phase outside that runs
 *   on CUDA cores (SG_ENGINE_TC makes it an error instead).  With B > 128 the
 *   fused kernel takes a group's two sample tiles one after the other;
 *   groups that still do not fit run there as
 *   subgroups of G/2 or G/4 labels sharing I_k, and groups of more than 64
 *   labels enter dh as subgroups of at most 64.  Every other G
 *   (including G = 1, per-label fixed fan-in) runs on the CUDA-core engine.
 *   sg_step_plan reports which kernels and engines a step will use.
 */
#ifndef SG_H
#define SG_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* exported symbols keep default visibility even when the library is built
 * with -fvisibility=hidden */
#if defined(__GNUC__)
#define SG_API __attribute__((visibility("default")))
#else
#define SG_API
#endif

typedef uint16_t sg_bf16;

typedef enum sg_status {
    SG_OK = 0,
    SG_ERR_INVALID = -1,     /* bad argument (null pointer, negative size, ...) */
    SG_ERR_UNSUPPORTED = -2, /* outside the supported range above */
    SG_ERR_CUDA = -3,        /* a CUDA runtime call failed */
    SG_ERR_OOM = -4,         /* device allocation failed */
    SG_ERR_TIMEOUT = -5,     /* a bounded device wait gave up */
    SG_ERR_DATA = -6         /* the data breaks the layer's rules */
} sg_status;

typedef enum sg_engine {
    SG_ENGINE_AUTO = 0,  /* tensor-core engine where supported, else CUDA cores */
    SG_ENGINE_SIMT = 1,  /* CUDA-core engine for every call */
    SG_ENGINE_TC = 2,    /* tensor-core engine; calls it cannot run fail */
    SG_ENGINE_FUSED = 3  /* as SG_ENGINE_TC, and sg_step runs the whole step in
                            one kernel on clusters of CTAs wherever that kernel
                            fits (B <= 128, G in {16, 32, 64}, F % 16 == 0,
                            F <= 128): W is read once and dZ never leaves the
                            chip.  SG_ENGINE_AUTO takes that kernel only for
                            shapes the two-kernel tensor-core step cannot run. */
} sg_engine;

/* Opaque, library-owned: the canonical layout plus per-layout scratch. */
typedef struct sg_layout sg_layout;

/* ---------------------------------------------------------------- layout
 * sg_layout_build -- group the labels and fix each group's fan-in set
 * (key design "group-shared fixed fan-in sparsity": K groups of exactly G
 * labels, shared I_k with |I_k| = F, index memory (L/G)*F).
 *   groups[L]   device int32, group id of every label, each id in [0, K) used
 *               by exactly G labels.
 *   idx[K*F]    device int32, row k = I_k in any order; entries distinct and
 *               in [0, H).
 *   max_B       largest batch the layout's scratch will serve (<= 256).
 *   max_nnz     largest positive count (nnz) a call will pass.
 * Result: slots in ascending label id within each group, I_k sorted ascending
 * and stored as uint16.  Synchronous (waits for `stream`) because data errors
 * are returned: SG_ERR_DATA for a bad group id, a group of size != G, a
 * duplicate or out-of-range index.  On success *out owns about
 * 2*K*F + 8*L + 2*H*max_B + 8*K + 12*max_nnz bytes of device memory; free
 * it with sg_layout_free.  On error *out is set to NULL.                    */
SG_API sg_status sg_layout_build(const int32_t *groups, int64_t L, int32_t G,
                          const int32_t *idx, int32_t F, int32_t H,
                          int32_t max_B, int64_t max_nnz, void *stream,
                          sg_layout **out);

/* Copy the canonical layout out (device outputs, any may be NULL):
 * slot_of_label[L], label_of_slot[L], idx_sorted[K*F] (uint16). Synchronous. */
SG_API sg_status sg_layout_export(const sg_layout *layout, int32_t *slot_of_label,
                           int32_t *label_of_slot, uint16_t *idx_sorted,
                           void *stream);

/* Release the layout and its scratch (NULL is a no-op).  Waits for the
 * device to finish work that uses it. */
SG_API void sg_layout_free(sg_layout *layout);

/* Pick the engine for later calls on this layout (sg_engine value).
 * SG_ENGINE_TC on a layout the tensor-core engine cannot run returns
 * SG_ERR_UNSUPPORTED and leaves the engine unchanged. */
SG_API sg_status sg_layout_set_engine(sg_layout *layout, int32_t engine);

/* The kernels a step (sg_step, or sg_step_sgd when sgd != 0) of B samples
 * will run on this layout with its current engine: plan[0] is one of
 * sg_step_path, plan[1..3] are 1 where the forward (+BCE), dW and dh run on
 * the tensor cores and 0 where they run on CUDA cores.  plan holds 4 int32
 * (host memory).  Synchronous, launches nothing; SG_ERR_UNSUPPORTED where the
 * step itself would fail (a layout pinned to the tensor cores outside their
 * range). */
typedef enum sg_step_path {
    SG_PLAN_PER_PHASE = 0,   /* one kernel per phase, dZ through HBM */
    SG_PLAN_FUSED_FWDW = 1,  /* fused forward + BCE + dW kernel, then dh */
    SG_PLAN_ONE_KERNEL = 2   /* the whole step in one kernel on CTA clusters */
} sg_step_path;
SG_API sg_status sg_step_plan(const sg_layout *layout, int32_t B, int32_t sgd, int32_t *plan);

/* Sizes of a layout (any pointer may be NULL). */
SG_API sg_status sg_layout_info(const sg_layout *layout, int64_t *L, int32_t *G,
                         int32_t *F, int32_t *H, int64_t *K);

/* Read (and if `clear`, reset) the layout's sticky device status word.
 * Synchronous (waits for the device).  *code is an sg_status value. */
SG_API sg_status sg_layout_status(sg_layout *layout, int32_t *code, int32_t clear);

/* The device-wide view of the same words: waits for the current device, then
 * sets *code to the first non-zero status word among the live layouts built on
 * that device (in the order they were built), or SG_OK.  Clears nothing: a
 * layout's word is reset with sg_layout_status(..., clear = 1).  Returns
 * SG_ERR_INVALID for a NULL `code` and SG_ERR_CUDA if the device reports an
 * error.  Thread-safe against concurrent build and free. */
SG_API sg_status sg_device_status(int32_t *code);

/* ---------------------------------------------------------------- positives
 * sg_pos_export -- the positive lists as the step uses them (Y of the BCE in
 * key design "head-tail split"): labels mapped to slots, sorted ascending and
 * deduplicated per sample (out_rowptr[B+1], out_slots[<= nnz]); and the same
 * entries bucketed by group (out_gptr[K+1]; out_gentry[] = (b << 16) | j for
 * slot k*G + j; order inside one group unspecified).  Any output may be NULL.
 * Asynchronous; a label id out of range sets the status word (SG_ERR_DATA)
 * and that entry is dropped. */
SG_API sg_status sg_pos_export(sg_layout *layout, int32_t B, const int32_t *pos_rowptr,
                        const int32_t *pos_label, int64_t nnz,
                        int32_t *out_rowptr, int32_t *out_slots,
                        int32_t *out_gptr, int32_t *out_gentry, void *stream);

/* ---------------------------------------------------------------- forward
 * sg_fwd -- Z_k = H_k W_k^T for every group (key design "gather-once + dense
 * MMA kernel"), i.e. Z[b][s] = sum_f W[s][f] h[b][I_k[f]], k = s / G.
 * FP32 accumulation, Z rounded to bf16 (RNE).
 *   h[B][H] bf16, W[L][F] bf16 (slot order), Z[B][L] bf16 (slot order).     */
SG_API sg_status sg_fwd(sg_layout *layout, const sg_bf16 *h, int32_t B,
                 const sg_bf16 *W, sg_bf16 *Z, void *stream);

/* sg_bce_grad -- dZ = sigmoid(Z) - Y (bf16) and loss = sum of the BCE terms
 * (double, device scalar), from a stored Z[B][L].                         */
SG_API sg_status sg_bce_grad(sg_layout *layout, const sg_bf16 *Z, int32_t B,
                      const int32_t *pos_rowptr, const int32_t *pos_label,
                      int64_t nnz, sg_bf16 *dZ, double *loss, void *stream);

/* sg_fwd_bce -- sg_fwd with the BCE step fused into its epilogue: Z stays in
 * FP32 on chip; writes dZ (bf16), the loss, and Z (bf16) only if Z_or_null is
 * not NULL.                                                              */
SG_API sg_status sg_fwd_bce(sg_layout *layout, const sg_bf16 *h, int32_t B,
                     const sg_bf16 *W, const int32_t *pos_rowptr,
                     const int32_t *pos_label, int64_t nnz, sg_bf16 *dZ,
                     double *loss, sg_bf16 *Z_or_null, void *stream);

/* ---------------------------------------------------------------- backward
 * sg_bwd_dW -- dW_k = dZ_k^T H_k (key design "gather-once + dense MMA
 * kernel": the weight gradient is the symmetric dense GEMM), i.e.
 * dW[s][f] = sum_b dZ[b][s] h[b][I_k[f]].  FP32 accumulation, bf16 output.
 *   dZ[B][L] bf16, h[B][H] bf16, dW[L][F] bf16.                            */
SG_API sg_status sg_bwd_dW(sg_layout *layout, const sg_bf16 *dZ, const sg_bf16 *h,
                    int32_t B, sg_bf16 *dW, void *stream);

/* sg_bwd_dh -- the feature gradient, summed over groups whose I_k overlap
 * (same key design: Split-K along the label dimension), i.e.
 * dh[b][i] = sum_s sum_f [I_k(s)[f] = i] dZ[b][s] W[s][f].  FP32 output;
 * partial sums are added with atomics, so the last bits are not reproducible
 * run to run.   dZ[B][L] bf16, W[L][F] bf16, dh[B][H] fp32.                */
SG_API sg_status sg_bwd_dh(sg_layout *layout, const sg_bf16 *dZ, int32_t B,
                    const sg_bf16 *W, float *dh, void *stream);

/* sg_bwd -- sg_bwd_dW and sg_bwd_dh in one call. */
SG_API sg_status sg_bwd(sg_layout *layout, const sg_bf16 *dZ, const sg_bf16 *h,
                 int32_t B, const sg_bf16 *W, sg_bf16 *dW, float *dh,
                 void *stream);

/* ---------------------------------------------------------------- step
 * sg_step -- the whole training step of the layer: forward, BCE gradient,
 * dW and dh, from h, W and the positives.  Writes dW[L][F] bf16, dh[B][H]
 * fp32 and the loss (double).  dZ is never returned.                       */
SG_API sg_status sg_step(sg_layout *layout, const sg_bf16 *h, int32_t B,
                  const sg_bf16 *W, const int32_t *pos_rowptr,
                  const int32_t *pos_label, int64_t nnz, sg_bf16 *dW,
                  float *dh, double *loss, void *stream);

/* sg_step_sgd -- the training step followed by the output layer's optimiser
 * step (HASTE, Loss and training strategy: the output layer trains with
 * momentum SGD; the heavy-ball rule without dampening or weight decay is the
 * reading taken).  The gradients are those of sg_step at W_in; then, for
 * every weight,
 *     m <- mu m + dW,      W_out <- bf16(W_in - lr m)    (fp32 arithmetic)
 * When the step takes the fused forward + BCE + dW kernel the update is
 * applied to dW while it is still on chip, and dW is never written.
 *   W_in[L][F] bf16 (read), W_out[L][F] bf16 (written; must not overlap W_in,
 *   since dh is taken at W_in), mom[L][F] fp32 (read and written), dh[B][H]
 *   fp32 and the loss as in sg_step.
 * Errors: as sg_step; SG_ERR_INVALID for NULL mom / W_out, overlapping W_in and
 * W_out, or a non-finite lr or mu.                                          */
SG_API sg_status sg_step_sgd(sg_layout *layout, const sg_bf16 *h, int32_t B,
                      const sg_bf16 *W_in, const int32_t *pos_rowptr,
                      const int32_t *pos_label, int64_t nnz, float lr, float mu,
                      float *mom, sg_bf16 *W_out, float *dh, double *loss,
                      void *stream);

/* ---------------------------------------------------------------- head-tail split
 * The output layer's head-tail split (HASTE, "Method / overall framework" and
 * key design "head-tail split"): the encoder output h (B x E) reaches a dense
 * head and the sparse tail through two light projections, and the objective
 * is the sum of both branches' BCE terms.  All matrices are row-major; bf16
 * inputs, fp32 accumulation on the tensor cores.  E, D, Dh and H must be
 * multiples of 8; pointers 16-byte aligned.
 *
 * sg_proj_fwd -- out[B][D] = bf16(h[B][E] P[D][E]^T).                      */
SG_API sg_status sg_proj_fwd(const sg_bf16 *h, int32_t B, int32_t E, const sg_bf16 *P, int32_t D,
                             sg_bf16 *out, void *stream);

/* sg_proj_bwd -- the projection's backward from g = dL/d out (fp32 [B][D]):
 * dP[D][E] = g^T h (fp32, overwritten) and dh[B][E] = g P (fp32; added to dh
 * when accumulate_dh is nonzero, else overwritten).  g enters the products as
 * two bf16 planes (value and rounding residual, about 16 bits), written to
 * work (caller-owned device memory of 2*B*D bf16).                         */
SG_API sg_status sg_proj_bwd(const sg_bf16 *h, int32_t B, int32_t E, const sg_bf16 *P, int32_t D,
                             const float *g, sg_bf16 *work, float *dP, float *dh, int32_t accumulate_dh,
                             void *stream);

/* sg_headtail_step -- the whole step of the split layer:
 *   h_head = bf16(h P_head^T) (B x Dh),  h_tail = bf16(h P_tail^T) (B x H);
 *   the head is the layer of `head` (built with every group's index set
 *   [0, Dh), Dh = head's H: the dense logits h_head W_head^T) stepped on
 *   h_head with the head positives; the tail is the layer of `tail` stepped
 *   on h_tail with the tail positives (each as sg_step, same conventions);
 *   dP_head[Dh][E] = dh_head^T h, dP_tail[H][E] = dh_tail^T h (fp32),
 *   dh[B][E] = dh_head P_head + dh_tail P_tail (fp32), loss = head + tail.
 * dW_head[Lh][Dh] and dW_tail[L][F] are bf16 in each layout's slot order.
 * Scratch for the activations and branch gradients lives in `tail` (about
 * 10 B (Dh + H) bytes, allocated on first use).                            */
SG_API sg_status sg_headtail_step(sg_layout *head, sg_layout *tail, const sg_bf16 *h, int32_t B, int32_t E,
                                  const sg_bf16 *P_head, const sg_bf16 *P_tail, const sg_bf16 *W_head,
                                  const int32_t *head_rowptr, const int32_t *head_label, int64_t head_nnz,
                                  const sg_bf16 *W_tail, const int32_t *tail_rowptr, const int32_t *tail_label,
                                  int64_t tail_nnz, sg_bf16 *dW_head, sg_bf16 *dW_tail, float *dP_head,
                                  float *dP_tail, float *dh, double *loss, void *stream);

/* ---------------------------------------------------------------- rewiring
 * sg_rewire -- one discrete phase of the training (HASTE, "Method / overall
 * framework" and "Loss and training strategy": each group's fan-in set is
 * re-selected periodically by the RigL protocol, |I_k| = F).  The pages do not
 * give the rule; this is the RigL reading for group-shared fan-in:
 *   prune score of an active index f of group k: sum over the group's labels
 *     of |W[l][f]|;  grow score of a feature j: sum over the group's labels of
 *     |sum_b dZ[b][l] h[b][j]| (the dense gradient a weight at (l, j) would get);
 *   per group, drop the n_drop smallest prune scores and grow the n_drop
 *   largest grow scores among the features outside the old I_k (ties: the
 *   smaller feature index first); kept columns keep their weights, grown ones
 *   start at zero; the new I_k is sorted ascending.
 *   h[B][H] bf16 (the samples the gradient is taken on), dZ[B][L] bf16 in
 *   slot order (e.g. from sg_fwd_bce), W[L][F] in slot order (columns follow
 *   the layout's sorted I_k).  Outputs: idx_out[K][F] int32 (sorted rows; pass
 *   it with the same groups to sg_layout_build for the next phase) and
 *   W_out[L][F] bf16 (columns follow idx_out), which must not overlap W.
 * Needs G a power of two <= 128, F <= 256, L and H multiples of 8, 0 <=
 * n_drop <= min(F, H - F).  The grow scores are one tcgen05 GEMM (dZ^T h with
 * the group |.|-sum in its epilogue) into K*H floats of scratch the layout
 * keeps (allocated on first use).  Asynchronous on `stream`.               */
SG_API sg_status sg_rewire(sg_layout *layout, const sg_bf16 *h, int32_t B, const sg_bf16 *dZ, const sg_bf16 *W,
                           int32_t n_drop, int32_t *idx_out, sg_bf16 *W_out, void *stream);

/* ---------------------------------------------------------------- semantic grouping
 * Grouping of the labels before training (HASTE, key design "group-shared
 * fixed fan-in sparsity": group members close in embedding space, label
 * embeddings from the encoder outputs of each label's positives, two stages:
 * mini-batch spherical k-means into about L / (beta G) coarse clusters, then
 * greedy groups of a seed and its G - 1 nearest remaining neighbours inside
 * each cluster).  The groups[] it writes feed sg_layout_build.
 *   * e_l = bf16(Normalize(sum of h_i over the distinct samples i with l
 *     positive)); labels without a positive (or with a zero sum) have no
 *     embedding and are grouped last.
 *   * Similarity = dot product of bf16 vectors; centroids are kept in fp32
 *     and rounded to bf16 for scoring (tcgen05 argmax GEMM).
 *   * A k-means batch is assigned with the centroids of its start (ties to the
 *     smaller centroid); then mu_c <- Normalize((n_c mu_c + S_c) / (n_c + m_c))
 *     (per-centre learning rate 1/n_c), n_c += m_c.
 *   * Greedy: clusters in index order; seed = the remaining member most
 *     similar to the centroid; its group = the seed and the G - 1 remaining
 *     members most similar to it (ties to the smaller label id); groups are
 *     numbered as formed.  What a cluster leaves over (in cluster order,
 *     ascending id), then the labels without embedding (ascending id), are cut
 *     into consecutive groups of G, numbered after the greedy ones.
 * Sums accumulate in 64-bit fixed point, so results do not depend on the
 * order of atomics.  The handle owns its device memory (about
 * L * (16 + 2 D) + C * 14 D bytes after embedding); calls on one handle must
 * not overlap.  Data errors (a malformed row, a label outside [0, L), |h| >=
 * 2^14, a k-means label without embedding) set the handle's status word,
 * read and cleared with sg_grouping_status.                                 */
typedef struct sg_grouping sg_grouping;

/* L labels (L % G == 0), embeddings of D features (D % 16 == 0, <= 4096),
 * C clusters (1 <= C <= L).  The current device is the handle's. */
SG_API sg_status sg_grouping_create(int64_t L, int32_t D, int32_t G, int32_t C, sg_grouping **out);
SG_API void sg_grouping_free(sg_grouping *g);
SG_API sg_status sg_grouping_status(sg_grouping *g, int32_t *code);

/* Embeddings from N samples h[N][D] (bf16, row-major) and their positive
 * labels (CSR: rowptr[N+1], labels[nnz], device).  N <= 2^22.  Synchronous;
 * *n_embedded (host, may be NULL) = labels that got an embedding. */
SG_API sg_status sg_grouping_embed(sg_grouping *g, const sg_bf16 *h, int32_t N, const int32_t *rowptr,
                                   const int32_t *labels, int64_t nnz, int64_t *n_embedded, void *stream);

/* Embeddings given directly: E[L][D] bf16 and has[L] (0/1), device.
 * Synchronous. */
SG_API sg_status sg_grouping_set_embeddings(sg_grouping *g, const sg_bf16 *E, const uint8_t *has, void *stream);

/* Centroid c = Normalize(e of init_labels[c]) (device int32[C]; each label
 * must have an embedding), counts 0. */
SG_API sg_status sg_grouping_kmeans_init(sg_grouping *g, const int32_t *init_labels, void *stream);

/* Centroids given directly: centroids[C][D] fp32 (unit rows), counts[C]
 * int64 (NULL: zeros), device.  Synchronous. */
SG_API sg_status sg_grouping_set_centroids(sg_grouping *g, const float *centroids, const int64_t *counts,
                                           void *stream);

/* One k-means batch of M label ids (device int32[M], each with an
 * embedding, M <= 2^22); assign_out (device int32[M], may be NULL) receives
 * the batch's assignment. */
SG_API sg_status sg_grouping_kmeans_batch(sg_grouping *g, const int32_t *batch, int32_t M, int32_t *assign_out,
                                          void *stream);

/* Final assignment of every label with an embedding to its nearest centroid,
 * then the greedy stage and the pool: groups[L] (device int32, ids in
 * [0, L / G)); cluster_out[L] (device int32, may be NULL): the cluster of
 * each label, -1 without embedding. */
SG_API sg_status sg_grouping_groups(sg_grouping *g, int32_t *groups, int32_t *cluster_out, void *stream);

/* Copy out (device outputs, each may be NULL): E[L][D] and has[L] (has only
 * with E), centroids[C][D], counts[C].  Synchronous. */
SG_API sg_status sg_grouping_export(sg_grouping *g, sg_bf16 *E, uint8_t *has, float *centroids, int64_t *counts,
                                    void *stream);

/* ---------------------------------------------------------------- timing
 * Per-kernel device timing for benchmarks: while enabled, every kernel the
 * library launches for this layout is bracketed by a pair of CUDA events
 * recorded on the stream of the call, tagged by its kind (sg_kernel_kind).
 * sg_timing_start(capacity) clears the record and keeps room for `capacity`
 * launches (later ones are counted but not timed); sg_timing_stop waits for
 * the device, writes per-kind total milliseconds and launch counts
 * (arrays of SG_KIND_COUNT), and disables the record.                       */
typedef enum sg_kernel_kind {
    SG_KIND_PREP = 0,    /* h transpose, positive lists, loss reduction */
    SG_KIND_FWD = 1,     /* forward (with or without the fused BCE)     */
    SG_KIND_BCE = 2,     /* BCE from a stored Z                          */
    SG_KIND_DW = 3,      /* weight gradient                              */
    SG_KIND_DH = 4,      /* feature gradient                             */
    SG_KIND_STEP = 5,    /* the whole step in one kernel (fwd+BCE+dW+dh) */
    SG_KIND_COUNT = 6
} sg_kernel_kind;

SG_API sg_status sg_timing_start(sg_layout *layout, int32_t capacity);
SG_API sg_status sg_timing_stop(sg_layout *layout, double *ms_per_kind,
                                int32_t *launches_per_kind);

/* ---------------------------------------------------------------- no allocation
 * sg_bce_grad_noalloc -- the same BCE step as sg_bce_grad (dZ = sigmoid(Z) - Y,
 * bf16, and the summed loss, double), for callers that cannot allocate device
 * memory: processes whose framework's caching allocator already holds the
 * device memory, or deployments that allow no allocation after start-up.  It
 * needs no layout and calls no allocator (cudaMalloc, cudaFree or any library
 * routine that allocates).  The paper has no counterpart: this is a service
 * of the library, not part of the method.
 *   Z[B][L], dZ[B][L] bf16, slot order; L = K*G.
 *   pos_rowptr[B+1], pos_slot[nnz]: each sample's positives as SLOT ids in
 *   [0, L) (any order, duplicates count once); out-of-range slots and
 *   malformed rows are dropped, since there is no layout status word.  Row b
 *   is well formed when 0 <= pos_rowptr[b] <= pos_rowptr[b+1] <= nnz and
 *   pos_rowptr[b] is at least every earlier row's start (pos_rowptr[0] may be
 *   non-zero).
 * Working memory is one device array built into the library (about 3.2 MB,
 * held by every GPU that loads the library until the process exits), so the
 * sizes are capped: B <= 256, L/G <= 300000, nnz <= 65536; larger calls
 * return SG_ERR_UNSUPPORTED before launching anything.  Every call uses that
 * same array (it clears what must start at zero), so calls that overlap on
 * the GPU -- from two streams or two host threads -- race; serialize them.
 * The first call on a device looks up the array's device address (a runtime
 * query, no allocation) and keeps it for the life of the process; make that
 * first call before any stream capture.  A cudaDeviceReset invalidates the
 * kept address: do not call this entry point after resetting the device.
 * Asynchronous on `stream` otherwise.                                       */
SG_API sg_status sg_bce_grad_noalloc(const sg_bf16 *Z, int32_t B, int64_t L, int32_t G,
                                     const int32_t *pos_rowptr, const int32_t *pos_slot,
                                     int64_t nnz, sg_bf16 *dZ, double *loss, void *stream);

/* ---------------------------------------------------------------- self-test
 * sg_selftest_wait_timeout -- exercises the library's failure detection on
 * the current device: a one-CTA kernel that holds TMEM columns waits, through
 * the same bounded wait every tensor-core kernel uses, on an mbarrier that
 * nothing ever arrives on.  After the wait limit (about 2 s of %globaltimer
 * time) the kernel records SG_ERR_TIMEOUT, releases its TMEM and returns, so
 * the CUDA context stays usable.  *code receives the status the kernel
 * recorded (SG_ERR_TIMEOUT when the mechanism works).  Synchronous; allocates
 * and frees 4 bytes of device memory.                                      */
SG_API sg_status sg_selftest_wait_timeout(int32_t *code);

/* ---------------------------------------------------------------- misc */
/* Message of the last failing call on this host thread ("" if none). */
SG_API const char *sg_last_error(void);
/* Constant name of a status value. */
SG_API const char *sg_status_string(int32_t status);
/* ABI version of this header (bumped on incompatible change). */
SG_API int32_t sg_abi_version(void);

#define SG_ABI_VERSION 1

#ifdef __cplusplus
}
#endif

#endif /* SG_H */
