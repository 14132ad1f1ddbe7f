/*
 * sg_oracle.c -- plain, slow, double-precision CPU oracle for one training step
 * of the group-shared fixed fan-in sparse output layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file: only the tests, the package's smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code with the CUDA library.
 *
 * Source: "HASTE: Hardware-Aware Dynamic Sparse Training for Large Output
 * Spaces" (review notes), sections
 *   - Method / overall framework: the logit z_l(x) = <w_l, h_{I_g(l)}>, w_l in
 *     R^F private to label l, I_k a shared index set of size F, no bias.
 *   - Key design "group-shared fixed fan-in sparsity": labels split into K
 *     groups of size G, each group sharing one index set I_k.
 *   - Key design "gather-once + dense MMA kernel": Z_k = H_k W_k^T with
 *     H_k = h[:, I_k]; grad W_k = (grad Z_k)^T H_k; the feature gradient sums
 *     over groups whose I_k overlap.
 *   - Key design "head-tail split": the objective is a sum of per-label BCE
 *     terms.
 *
 * Readings taken where the page is silent (each is also listed in the design
 * notes of the repository):
 *   - exactly G labels per group; a group's labels take slots kG..kG+G-1 in
 *     ascending label id; I_k is stored ascending; duplicate or out-of-range
 *     indices are data errors;
 *   - Y is binary: duplicate positives of a sample count once;
 *   - the loss returned is the SUM of per-(sample, label) BCE terms, so dZ,
 *     dW and dh are exact gradients of it (the page's 1/n mean is that sum / B);
 *   - inputs are bf16 values widened exactly to double; nothing is rounded
 *     in between.
 *
 * Every input array may be given as double or as bf16 bit patterns (the
 * `*_bf16` flag): the value is the same either way, the double form only exists
 * so finite-difference checks can perturb entries.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_OK 0
#define OR_ERR_INVALID (-1)
#define OR_ERR_DATA (-6)

/* ------------------------------------------------------------------ threads */

int or_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int or_thread_id(void)
{
#ifdef _OPENMP
    return omp_get_thread_num();
#else
    return 0;
#endif
}

/* ------------------------------------------------------------------ inputs */

static double bf16_value(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* element i of an input given either as double or as bf16 bits */
static double in_at(const void *p, int is_bf16, int64_t i)
{
    if (is_bf16)
        return bf16_value(((const uint16_t *)p)[i]);
    return ((const double *)p)[i];
}

double or_bf16_value(uint16_t bits) { return bf16_value(bits); }

/* ------------------------------------------------------- O1: the layout
 * Group-shared fixed fan-in sparsity: L labels in K = L/G groups of exactly G;
 * index memory (L/G)*F.  Slot s = k*G + j is the j-th smallest label id of
 * group k; idx_sorted[k*F + f] is the f-th smallest element of I_k.          */
int or_layout_build(int64_t L, int32_t G, const int32_t *groups,
                    const int32_t *idx, int32_t F, int32_t H,
                    int32_t *slot_of_label, int32_t *label_of_slot,
                    uint16_t *idx_sorted)
{
    if (L < 1 || G < 1 || F < 1 || H < 1 || H > 65535 || F > H || L % G != 0)
        return OR_ERR_INVALID;
    int64_t K = L / G;

    int64_t *count = calloc((size_t)K, sizeof *count);
    if (!count)
        return OR_ERR_INVALID;
    for (int64_t l = 0; l < L; ++l) {
        int32_t g = groups[l];
        if (g < 0 || g >= K) {
            free(count);
            return OR_ERR_DATA;
        }
        count[g] += 1;
    }
    for (int64_t k = 0; k < K; ++k) {
        if (count[k] != G) {
            free(count);
            return OR_ERR_DATA;
        }
    }
    /* next free slot of each group; labels visited in ascending id */
    for (int64_t k = 0; k < K; ++k)
        count[k] = k * (int64_t)G;
    for (int64_t l = 0; l < L; ++l) {
        int64_t s = count[groups[l]]++;
        slot_of_label[l] = (int32_t)s;
        label_of_slot[s] = (int32_t)l;
    }
    free(count);

    /* I_k ascending; entries must be distinct and inside [0, H) */
    for (int64_t k = 0; k < K; ++k) {
        const int32_t *src = idx + k * (int64_t)F;
        uint16_t *dst = idx_sorted + k * (int64_t)F;
        for (int32_t f = 0; f < F; ++f) {
            int32_t v = src[f];
            if (v < 0 || v >= H)
                return OR_ERR_DATA;
            /* insertion sort */
            int32_t p = f;
            while (p > 0 && dst[p - 1] > v) {
                dst[p] = dst[p - 1];
                --p;
            }
            dst[p] = (uint16_t)v;
        }
        for (int32_t f = 1; f < F; ++f)
            if (dst[f] == dst[f - 1])
                return OR_ERR_DATA;
    }
    return OR_OK;
}

/* ------------------------------------------------------- O2: positives
 * Y[b, s] = 1 iff slot s is a positive of sample b.  Input: per-sample label
 * lists (CSR, label ids, any order, duplicates allowed).  Output: canonical
 * slot lists, ascending and without duplicates, compacted (out_rowptr).     */
int or_pos_slots(int32_t B, const int32_t *rowptr, const int32_t *labels,
                 int64_t L, const int32_t *slot_of_label,
                 int32_t *out_rowptr, int32_t *out_slots)
{
    if (B < 0 || rowptr[0] != 0)
        return OR_ERR_DATA;
    for (int32_t b = 0; b < B; ++b)
        if (rowptr[b + 1] < rowptr[b])
            return OR_ERR_DATA;
    int64_t nnz = rowptr[B];
    for (int64_t e = 0; e < nnz; ++e)
        if (labels[e] < 0 || labels[e] >= L)
            return OR_ERR_DATA;

    int32_t out = 0;
    out_rowptr[0] = 0;
    for (int32_t b = 0; b < B; ++b) {
        int32_t start = out;
        for (int32_t e = rowptr[b]; e < rowptr[b + 1]; ++e) {
            int32_t s = slot_of_label[labels[e]];
            /* insert s into out_slots[start..out) keeping it ascending, once */
            int32_t p = out;
            int dup = 0;
            for (int32_t q = start; q < out; ++q)
                if (out_slots[q] == s)
                    dup = 1;
            if (dup)
                continue;
            while (p > start && out_slots[p - 1] > s) {
                out_slots[p] = out_slots[p - 1];
                --p;
            }
            out_slots[p] = s;
            ++out;
        }
        out_rowptr[b + 1] = out;
    }
    return OR_OK;
}

/* is slot s a positive of sample b?  (plain scan of the sample's slot list) */
static int is_positive(const int32_t *srowptr, const int32_t *sslots,
                       int32_t b, int64_t s)
{
    for (int32_t e = srowptr[b]; e < srowptr[b + 1]; ++e)
        if (sslots[e] == s)
            return 1;
    return 0;
}

/* ------------------------------------------------------- O3: the logit
 * z[b, s] = sum_f W[s, f] * h[b, I_k[f]],  k = s div G, f ascending.        */
static double logit(int32_t H, int32_t G, int32_t F,
                    const void *h, int h_bf16, const void *W, int W_bf16,
                    const uint16_t *idx_sorted, int32_t b, int64_t s)
{
    int64_t k = s / G;
    const uint16_t *I = idx_sorted + k * (int64_t)F;
    double z = 0.0;
    for (int32_t f = 0; f < F; ++f)
        z += in_at(W, W_bf16, s * (int64_t)F + f) *
             in_at(h, h_bf16, (int64_t)b * H + I[f]);
    return z;
}

void or_forward(int32_t B, int32_t H, int64_t L, int32_t G, int32_t F,
                const void *h, int h_bf16, const void *W, int W_bf16,
                const uint16_t *idx_sorted, double *Z)
{
#pragma omp parallel for schedule(static)
    for (int32_t b = 0; b < B; ++b)
        for (int64_t s = 0; s < L; ++s)
            Z[(int64_t)b * L + s] = logit(H, G, F, h, h_bf16, W, W_bf16,
                                          idx_sorted, b, s);
}

void or_forward_at(int32_t H, int32_t G, int32_t F,
                   const void *h, int h_bf16, const void *W, int W_bf16,
                   const uint16_t *idx_sorted, int64_t n, const int32_t *bs,
                   const int64_t *ss, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = logit(H, G, F, h, h_bf16, W, W_bf16, idx_sorted, bs[i], ss[i]);
}

/* ------------------------------------------------------- O4: BCE
 * l(z, y) = -[y log sigma(z) + (1-y) log(1 - sigma(z))]
 *         = max(z, 0) - y z + log(1 + exp(-|z|))     (overflow-free form)
 * dl/dz   = sigma(z) - y.                                                    */
double or_sigmoid(double z)
{
    if (z >= 0.0)
        return 1.0 / (1.0 + exp(-z));
    double e = exp(z);
    return e / (1.0 + e);
}

double or_bce_term(double z, int y)
{
    return fmax(z, 0.0) - (y ? z : 0.0) + log1p(exp(-fabs(z)));
}

void or_bce(int32_t B, int64_t L, const void *Z, int Z_bf16,
            const int32_t *srowptr, const int32_t *sslots, double *dZ,
            double *loss)
{
    double total = 0.0;
    unsigned char *y = malloc((size_t)L);
    for (int32_t b = 0; b < B; ++b) {
        /* Y[b, :] as a 0/1 mask over slots */
        memset(y, 0, (size_t)L);
        for (int32_t e = srowptr[b]; e < srowptr[b + 1]; ++e)
            y[sslots[e]] = 1;
        for (int64_t s = 0; s < L; ++s) {
            double z = in_at(Z, Z_bf16, (int64_t)b * L + s);
            total += or_bce_term(z, y[s]);
            if (dZ)
                dZ[(int64_t)b * L + s] = or_sigmoid(z) - (double)y[s];
        }
    }
    free(y);
    *loss = total;
}

/* ------------------------------------------------------- O5: weight gradient
 * dW[s, f] = sum_b dZ[b, s] * h[b, I_k[f]]        (grad W_k = dZ_k^T H_k)    */
void or_weight_grad(int32_t B, int32_t H, int64_t L, int32_t G, int32_t F,
                    const void *h, int h_bf16, const void *dZ, int dZ_bf16,
                    const uint16_t *idx_sorted, double *dW)
{
#pragma omp parallel for schedule(static)
    for (int64_t s = 0; s < L; ++s) {
        const uint16_t *I = idx_sorted + (s / G) * (int64_t)F;
        for (int32_t f = 0; f < F; ++f) {
            double acc = 0.0;
            for (int32_t b = 0; b < B; ++b)
                acc += in_at(dZ, dZ_bf16, (int64_t)b * L + s) *
                       in_at(h, h_bf16, (int64_t)b * H + I[f]);
            dW[s * (int64_t)F + f] = acc;
        }
    }
}

/* ------------------------------------------------------- O6: feature gradient
 * dh[b, i] = sum_s sum_f [I_k(s)[f] = i] * dZ[b, s] * W[s, f]
 * i.e. every group scatters dZ_k W_k into the columns I_k; groups whose I_k
 * overlap add into the same column.                                          */
void or_feature_grad(int32_t B, int32_t H, int64_t L, int32_t G, int32_t F,
                     const void *W, int W_bf16, const void *dZ, int dZ_bf16,
                     const uint16_t *idx_sorted, double *dh)
{
#pragma omp parallel for schedule(static)
    for (int32_t b = 0; b < B; ++b) {
        double *row = dh + (int64_t)b * H;
        for (int32_t i = 0; i < H; ++i)
            row[i] = 0.0;
        for (int64_t s = 0; s < L; ++s) {
            const uint16_t *I = idx_sorted + (s / G) * (int64_t)F;
            double d = in_at(dZ, dZ_bf16, (int64_t)b * L + s);
            for (int32_t f = 0; f < F; ++f)
                row[I[f]] += d * in_at(W, W_bf16, s * (int64_t)F + f);
        }
    }
}

/* ------------------------------------------------------- O7: momentum SGD
 * The output layer's optimiser ("Loss and training strategy": the output
 * layer trains with momentum SGD; the pages give no formula, the plain
 * heavy-ball rule without dampening or weight decay is the reading taken):
 *     m <- mu * m + dW,        W <- bf16(W - lr * m)
 * m is kept in double here; the new W is rounded to the layer's bf16 storage
 * (double -> fp32 -> bf16, both round-to-nearest-even, as the inputs are
 * made).                                                                     */
static uint16_t bf16_round(double x)
{
    const float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

void or_sgd_momentum(int64_t n, const uint16_t *W, const double *dW, double *m, double lr, double mu,
                     uint16_t *W_out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        m[i] = mu * m[i] + dW[i];
        W_out[i] = bf16_round(bf16_value(W[i]) - lr * m[i]);
    }
}

/* ---------------------------------------------- sampled outputs (full size)
 * The same definitions evaluated only at chosen outputs, from h and W, so a
 * multi-GB problem can be checked without materialising Z.                   */

/* dW rows of the chosen slots: needs dZ[:, s] = sigma(z[:, s]) - Y[:, s]    */
void or_weight_grad_rows(int32_t B, int32_t H, int64_t L, int32_t G, int32_t F,
                         const void *h, int h_bf16, const void *W, int W_bf16,
                         const uint16_t *idx_sorted, const int32_t *srowptr,
                         const int32_t *sslots, int64_t n, const int64_t *slots,
                         double *out)
{
    (void)L;
#pragma omp parallel for schedule(dynamic)
    for (int64_t r = 0; r < n; ++r) {
        int64_t s = slots[r];
        const uint16_t *I = idx_sorted + (s / G) * (int64_t)F;
        double *dst = out + r * F;
        for (int32_t f = 0; f < F; ++f)
            dst[f] = 0.0;
        for (int32_t b = 0; b < B; ++b) {
            double z = logit(H, G, F, h, h_bf16, W, W_bf16, idx_sorted, b, s);
            double d = or_sigmoid(z) - (double)is_positive(srowptr, sslots, b, s);
            for (int32_t f = 0; f < F; ++f)
                dst[f] += d * in_at(h, h_bf16, (int64_t)b * H + I[f]);
        }
    }
}

/* dh rows and per-row loss of the chosen samples: needs the whole row
 * dZ[b, :], i.e. every logit of sample b.                                   */
void or_feature_grad_rows(int32_t B, int32_t H, int64_t L, int32_t G, int32_t F,
                          const void *h, int h_bf16, const void *W, int W_bf16,
                          const uint16_t *idx_sorted, const int32_t *srowptr,
                          const int32_t *sslots, int64_t n, const int32_t *rows,
                          double *out_dh, double *out_row_loss)
{
    (void)B;
    for (int64_t r = 0; r < n; ++r) {
        int32_t b = rows[r];
        double *dst = out_dh ? out_dh + r * H : NULL;
        double row_loss = 0.0;
        if (dst)
            for (int32_t i = 0; i < H; ++i)
                dst[i] = 0.0;
        /* positives of this row as a dense 0/1 mask over slots */
        unsigned char *y = calloc((size_t)L, 1);
        for (int32_t e = srowptr[b]; e < srowptr[b + 1]; ++e)
            y[sslots[e]] = 1;
        int nt = or_num_threads();
        double *part_all = dst ? calloc((size_t)nt * H, sizeof(double)) : NULL;
        double *loss_all = calloc((size_t)nt, sizeof(double));
#pragma omp parallel num_threads(nt)
        {
            int t = or_thread_id();
            double *part = part_all ? part_all + (int64_t)t * H : NULL;
            double part_loss = 0.0;
#pragma omp for schedule(static)
            for (int64_t s = 0; s < L; ++s) {
                double z = logit(H, G, F, h, h_bf16, W, W_bf16, idx_sorted, b, s);
                part_loss += or_bce_term(z, y[s]);
                if (part) {
                    double d = or_sigmoid(z) - (double)y[s];
                    const uint16_t *I = idx_sorted + (s / G) * (int64_t)F;
                    for (int32_t f = 0; f < F; ++f)
                        part[I[f]] += d * in_at(W, W_bf16, s * (int64_t)F + f);
                }
            }
            loss_all[t] = part_loss;
        }
        /* fixed-order merge of the per-thread partial sums */
        for (int t = 0; t < nt; ++t) {
            row_loss += loss_all[t];
            if (dst)
                for (int32_t i = 0; i < H; ++i)
                    dst[i] += part_all[(int64_t)t * H + i];
        }
        free(part_all);
        free(loss_all);
        free(y);
        if (out_row_loss)
            out_row_loss[r] = row_loss;
    }
}

