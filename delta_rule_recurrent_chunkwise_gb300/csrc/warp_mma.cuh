// warp_mma.cuh -- warp-level bf16 tensor-core products (mma.sync m16n8k16,
// fp32 accumulation) on shared-memory operands, for the backward kernels.
//
// Operands are read through "views": PadView is a row-major bf16 matrix
// with a padded row stride; RsView is a row-swizzled record tile (the
// tcgen05 operand format of the forward pass, copied into shared memory
// byte for byte).  ldmatrix hands every lane its fragment: lanes 8j .. 8j + 7
// address the eight 16-byte rows of 8 x 8 block j, transposed on the way for
// operands stored the other way round.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "tc_tile.cuh"

namespace la {
namespace wmma16 {

using bf16 = __nv_bfloat16;

__device__ __forceinline__ uint32_t saddr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldsm(uint32_t (&r)[4], const bf16 *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(saddr(p)));
}

__device__ __forceinline__ void ldsm_t(uint32_t (&r)[4], const bf16 *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(saddr(p)));
}

// A pure function of its registers (not volatile), so the compiler may issue
// the next step's fragment loads ahead of it.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Row-major bf16 matrix, row stride ld elements (a multiple of 8).
struct PadView {
    const bf16 *p;
    int ld;
    __device__ __forceinline__ const bf16 *at(int r, int c) const { return p + r * ld + c; }
};

// Row-swizzled tile of `rows` rows (tile::rs_off), seen from row row0 on.
struct RsView {
    const uint8_t *p;
    int rows, row0;
    __device__ __forceinline__ const bf16 *at(int r, int c) const {
        return reinterpret_cast<const bf16 *>(p + tile::rs_off(rows, row0 + r, c));
    }
};

// Fragments of one 16-deep step (m16n8k16): A for rows m0 .. m0+15, B for
// columns n0 .. n0+15 (two n8 tiles).  op(A) = A (stored [m][k], TA = false)
// or A^T (stored [k][m]); op(B) = B (stored [k][n], TB = false) or B^T
// (stored [n][k]).  m0, n0 multiples of 8, k of 16.
template <bool TA, class VA>
__device__ __forceinline__ void frag_a(uint32_t (&a)[4], const VA &A, int m0, int k) {
    const int lane = threadIdx.x & 31, li = lane & 7, lj = lane >> 3;
    if constexpr (!TA) ldsm(a, A.at(m0 + (lane & 15), k + (lane >> 4) * 8));
    else ldsm_t(a, A.at(k + li + 8 * (lj >> 1), m0 + 8 * (lj & 1)));
}

template <bool TB, class VB>
__device__ __forceinline__ void frag_b(uint32_t (&b)[4], const VB &B, int n0, int k) {
    const int lane = threadIdx.x & 31, li = lane & 7, lj = lane >> 3;
    if constexpr (TB) ldsm(b, B.at(n0 + li + 8 * (lj >> 1), k + 8 * (lj & 1)));
    else ldsm_t(b, B.at(k + li + 8 * (lj & 1), n0 + 8 * (lj >> 1)));
}

// One 16-deep step of a warp's 16 x 16 output block (two n8 tiles):
//   d += op(A)[m0 .. m0+15][k .. k+15] op(B)[k .. k+15][n0 .. n0+15]
// Accumulator element e of tile j sits at row m0 + g + 8 (e/2), column
// n0 + 8j + 2t + e%2 (g = lane / 4, t = lane % 4).
template <bool TA, bool TB, class VA, class VB>
__device__ __forceinline__ void mma_step(float (&d)[2][4], const VA &A, const VB &B, int m0,
                                         int n0, int k) {
    uint32_t a[4], b[4];
    frag_a<TA>(a, A, m0, k);
    frag_b<TB>(b, B, n0, k);
    mma16816(d[0], a, b[0], b[1]);
    mma16816(d[1], a, b[2], b[3]);
}

// One 16-deep step of NT n8 tiles from column n0 (NT even): the A fragment
// is loaded once for all of them.
template <int NT, bool TA, bool TB, class VA, class VB>
__device__ __forceinline__ void mma_kstep(float (&d)[NT][4], const VA &A, const VB &B, int m0,
                                          int n0, int k) {
    uint32_t a[4];
    frag_a<TA>(a, A, m0, k);
#pragma unroll
    for (int j = 0; j < NT; j += 2) {
        uint32_t b[4];
        frag_b<TB>(b, B, n0 + 8 * j, k);
        mma16816(d[j], a, b[0], b[1]);
        mma16816(d[j + 1], a, b[2], b[3]);
    }
}

// d (NT n8 tiles from column n0, NT even) += op(A) op(B) over k in [k0, k1).
template <int NT, bool TA, bool TB, class VA, class VB>
__device__ __forceinline__ void mma_rows(float (&d)[NT][4], const VA &A, const VB &B, int m0,
                                         int n0, int k0, int k1) {
#pragma unroll 2
    for (int k = k0; k < k1; k += 16) mma_kstep<NT, TA, TB>(d, A, B, m0, n0, k);
}

// The same over a compile-time range [K0, K1), fully unrolled.
template <int K0, int K1, int NT, bool TA, bool TB, class VA, class VB>
__device__ __forceinline__ void mma_rows_c(float (&d)[NT][4], const VA &A, const VB &B, int m0,
                                           int n0) {
#pragma unroll
    for (int k = K0; k < K1; k += 16) mma_kstep<NT, TA, TB>(d, A, B, m0, n0, k);
}

template <int NT>
__device__ __forceinline__ void zero(float (&d)[NT][4]) {
#pragma unroll
    for (int j = 0; j < NT; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.0f;
}

__device__ __forceinline__ void st2(bf16 *p, float a, float b) {
    *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(a, b);
}

__device__ __forceinline__ float2 ld2(const bf16 *p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
}

}  // namespace wmma16
}  // namespace la
