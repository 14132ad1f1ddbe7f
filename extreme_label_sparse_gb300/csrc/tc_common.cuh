// Device helpers shared by the tensor-core kernels (sm_103a): bf16 / fp16
// packing, the swizzled dZ tile stores, TMEM chunk loads, the positive-label
// mask of a group and the BCE of a chunk of logits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tc_ptx.cuh"

namespace tc {

// two floats -> packed bf16x2 (a in the low half), round to nearest even
__device__ __forceinline__ uint32_t pack2(float a, float b)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack2_f16(float a, float b)
{
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float lo_half(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_half(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// store N (multiple of 8) floats as bf16 to 16-byte aligned global memory;
// with `lo`, also store the rounding residual v - bf16(v) as a second plane
template <int N>
__device__ __forceinline__ void store_bf16_row(uint16_t *dst, uint16_t *lo, const float (&v)[N])
{
#pragma unroll
    for (int i = 0; i < N; i += 8) {
        uint4 q;
        q.x = pack2(v[i + 0], v[i + 1]);
        q.y = pack2(v[i + 2], v[i + 3]);
        q.z = pack2(v[i + 4], v[i + 5]);
        q.w = pack2(v[i + 6], v[i + 7]);
        *reinterpret_cast<uint4 *>(dst + i) = q;
        if (lo) {
            uint4 r;
            r.x = pack2(v[i + 0] - lo_half(q.x), v[i + 1] - hi_half(q.x));
            r.y = pack2(v[i + 2] - lo_half(q.y), v[i + 3] - hi_half(q.y));
            r.z = pack2(v[i + 4] - lo_half(q.z), v[i + 5] - hi_half(q.z));
            r.w = pack2(v[i + 6] - lo_half(q.w), v[i + 7] - hi_half(q.w));
            *reinterpret_cast<uint4 *>(lo + i) = r;
        }
    }
}

// 16-byte unit that unit u of row r lands on under the TMA swizzle of a
// zsw-byte row (the XOR of the unit index with address bits 7.. of the row)
__device__ __forceinline__ int swz_of(int r, int zsw)
{
    return zsw == 128 ? (r & 7) : zsw == 64 ? ((r >> 1) & 3) : ((r >> 2) & 1);
}

// CH values (columns c0 .. c0+CH-1, sample row r) into a group's fp16 dZ
// tile in global memory (one plane, same unit layout as the bf16 plane 0)
template <int CH>
__device__ __forceinline__ void store_dz_tile_f16(uint8_t *tile, int r, int c0, const float (&v)[CH],
                                                  int zsw, int Bp)
{
    const int sw = swz_of(r, zsw);
    const int u0 = (c0 & 63) >> 3;
    uint8_t *row = tile + ((size_t)(c0 >> 6) * Bp + r) * zsw;
#pragma unroll
    for (int i = 0; i < CH / 8; ++i) {
        const float *x = v + 8 * i;
        uint4 q;
        q.x = pack2_f16(x[0], x[1]);
        q.y = pack2_f16(x[2], x[3]);
        q.z = pack2_f16(x[4], x[5]);
        q.w = pack2_f16(x[6], x[7]);
        *reinterpret_cast<uint4 *>(row + (((u0 + i) ^ sw) << 4)) = q;
    }
}

// CH values (columns c0 .. c0+CH-1, sample row r) into a group's dZ tile:
// bf16 values into plane 0, their rounding residuals into plane 1
template <int CH>
__device__ __forceinline__ void store_dz_tile(uint8_t *tile, int r, int c0, const float (&v)[CH],
                                              int zsw, int nzc, int Bp, uint8_t *tile2 = nullptr)
{
    const int sw = swz_of(r, zsw);
    const int u0 = (c0 & 63) >> 3;
    const size_t row = ((size_t)(c0 >> 6) * Bp + r) * zsw;
    const size_t plane = (size_t)nzc * Bp * zsw;
    uint8_t *hi = tile + row;
    uint8_t *lo = hi + plane;
#pragma unroll
    for (int i = 0; i < CH / 8; ++i) {
        const float *x = v + 8 * i;
        uint4 q, e;
        q.x = pack2(x[0], x[1]);
        q.y = pack2(x[2], x[3]);
        q.z = pack2(x[4], x[5]);
        q.w = pack2(x[6], x[7]);
        e.x = pack2(x[0] - lo_half(q.x), x[1] - hi_half(q.x));
        e.y = pack2(x[2] - lo_half(q.y), x[3] - hi_half(q.y));
        e.z = pack2(x[4] - lo_half(q.z), x[5] - hi_half(q.z));
        e.w = pack2(x[6] - lo_half(q.w), x[7] - hi_half(q.w));
        const int off = ((u0 + i) ^ sw) << 4;
        *reinterpret_cast<uint4 *>(hi + off) = q;
        *reinterpret_cast<uint4 *>(lo + off) = e;
        if (tile2) {  // the same bytes into a second copy of the tile
            *reinterpret_cast<uint4 *>(tile2 + row + off) = q;
            *reinterpret_cast<uint4 *>(tile2 + row + plane + off) = e;
        }
    }
}

template <int CH>
__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, float (&v)[CH])
{
    static_assert(CH == 8 || CH == 16 || CH == 32, "TMEM chunk of 8, 16 or 32 columns");
    uint32_t r[CH];
    if constexpr (CH == 32)
        tmem_ld32(taddr, r);
    else if constexpr (CH == 16)
        tmem_ld16(taddr, r);
    else
        tmem_ld8(taddr, r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < CH; ++i)
        v[i] = __uint_as_float(r[i]);
}

// two chunks (e.g. the hi and lo halves of an accumulator) with one wait
template <int CH>
__device__ __forceinline__ void tmem_ld_chunk2(uint32_t ta, uint32_t tb, float (&v)[CH], float (&w)[CH])
{
    static_assert(CH == 8 || CH == 16 || CH == 32, "TMEM chunk of 8, 16 or 32 columns");
    uint32_t r[CH], u[CH];
    if constexpr (CH == 32) {
        tmem_ld32(ta, r);
        tmem_ld32(tb, u);
    } else if constexpr (CH == 16) {
        tmem_ld16(ta, r);
        tmem_ld16(tb, u);
    } else {
        tmem_ld8(ta, r);
        tmem_ld8(tb, u);
    }
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < CH; ++i) {
        v[i] = __uint_as_float(r[i]);
        w[i] = __uint_as_float(u[i]);
    }
}

// positives of sample b among columns c0 .. c0+n-1 of a group whose entries
// are gent[e0 .. e1)
__device__ __forceinline__ uint32_t group_pos_mask(const int32_t *__restrict__ gent, int e0,
                                                   int e1, int b, int c0, int n)
{
    uint32_t y = 0;
    for (int e = e0; e < e1; ++e) {
        const int v = __ldg(gent + e);
        const int jj = (v & 0xffff) - c0;
        if ((v >> 16) == b && jj >= 0 && jj < n)
            y |= 1u << jj;
    }
    return y;
}

// BCE on a chunk of logits in place: v[i] <- sigmoid(v[i]) - y_i; returns the
// chunk's loss sum(max(z,0) - y z + log(1 + e^-|z|)).  The log of the product
// of the (1 + e^-|z|) factors (each in (1, 2], so at most 2^32 for 32 of
// them) replaces one log per element.
template <int CH>
__device__ __forceinline__ float bce_chunk(float (&v)[CH], uint32_t y)
{
    float prod = 1.f, lin = 0.f, zpos = 0.f;
    if (y) {  // positives are rare: their terms are applied separately
#pragma unroll
        for (int i = 0; i < CH; ++i)
            if ((y >> i) & 1u)
                zpos += v[i];
    }
#pragma unroll
    for (int i = 0; i < CH; ++i) {
        const float z = v[i];
        const float e = __expf(-fabsf(z));
        const float one_e = 1.f + e;
        const float r = __fdividef(1.f, one_e);
        v[i] = z >= 0.f ? r : e * r;
        lin += fmaxf(z, 0.f);
        prod *= one_e;
    }
    if (y) {
#pragma unroll
        for (int i = 0; i < CH; ++i)
            if ((y >> i) & 1u)
                v[i] -= 1.f;
    }
    return lin - zpos + __logf(prod);
}

// 2^x and 1/x on the special-function unit, subnormal inputs and results
// flushed to zero (no fix-up instructions around the approximation)
__device__ __forceinline__ float ex2_ftz(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_ftz(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2_ftz(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// bce_chunk with the flushing approximations: e = 2^(-|z| log2 e) is 0 for
// |z| > 87 (where sigma(-|z|) and log(1 + e^-|z|) are below fp32's normal
// range), the product of the (1 + e) factors stays in [1, 2^CH]
template <int CH>
__device__ __forceinline__ float bce_chunk_ftz(float (&v)[CH], uint32_t y)
{
    constexpr float kLog2e = 1.4426950408889634f, kLn2 = 0.6931471805599453f;
    float prod = 1.f, lin = 0.f, zpos = 0.f;
    if (y) {
#pragma unroll
        for (int i = 0; i < CH; ++i)
            if ((y >> i) & 1u)
                zpos += v[i];
    }
#pragma unroll
    for (int i = 0; i < CH; ++i) {
        const float z = v[i];
        const float e = ex2_ftz(-fabsf(z) * kLog2e);
        const float one_e = 1.f + e;
        const float r = rcp_ftz(one_e);
        v[i] = z >= 0.f ? r : e * r;
        lin += fmaxf(z, 0.f);
        prod *= one_e;
    }
    if (y) {
#pragma unroll
        for (int i = 0; i < CH; ++i)
            if ((y >> i) & 1u)
                v[i] -= 1.f;
    }
    return lin - zpos + lg2_ftz(prod) * kLn2;
}

// fp32 -> bf16 bits, round to nearest even (the hardware conversion)
__device__ __forceinline__ uint16_t bf16_rn(float x)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

}  // namespace tc
