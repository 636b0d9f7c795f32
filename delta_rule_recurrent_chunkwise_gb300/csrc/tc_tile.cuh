// tc_tile.cuh -- operand tiles shared by the two tensor-core delta-rule
// kernels (intra-chunk and inter-chunk): the row-swizzled bf16 tile format,
// its tcgen05 descriptors, TMEM readback helpers and the layout of the
// per-chunk record the intra-chunk kernel hands to the inter-chunk kernel.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "tc.cuh"

namespace la {
namespace tile {

using namespace tc;

constexpr int C = 64;  // tokens per chunk

// A "row-swizzled" (RS) tile holds `rows` rows of D bf16 as D/64 column
// blocks of rows x 128 bytes, 128-byte swizzled in 1024-byte atoms.  The
// same bytes serve as a K-major operand (rows = M or N) or an MN-major
// operand (rows = K).
__device__ __forceinline__ uint32_t rs_off(int rows, int row, int col) {
    return (uint32_t)(col >> 6) * (uint32_t)rows * 128u + sw128_offset(row, col & 63);
}

__device__ __forceinline__ uint4 pack8(const float *v) {
    uint4 u;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    return u;
}

__device__ __forceinline__ void unpack8(uint4 u, float *v) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

// 8 consecutive columns (col % 8 == 0) as one 16-byte store.
__device__ __forceinline__ void st_bf16x8(uint8_t *tile, int rows, int row, int col,
                                          const float *v) {
    *reinterpret_cast<uint4 *>(tile + rs_off(rows, row, col)) = pack8(v);
}

// K-major operand descriptor for K-step s (16 elements) of an RS tile,
// starting at row row0.
__device__ __forceinline__ uint64_t kdesc(const uint8_t *tile, int rows, int row0, int s) {
    return smem_desc_sw128(smem_u32(tile) + (uint32_t)(s >> 2) * rows * 128u + row0 * 128u +
                               (uint32_t)(s & 3) * 32u,
                           16, 1024);
}

// MN-major operand descriptor for K-step s (rows row0+16s .. +15) of an RS tile.
__device__ __forceinline__ uint64_t mdesc(const uint8_t *tile, int rows, int row0, int s) {
    return smem_desc_sw128(smem_u32(tile) + (uint32_t)row0 * 128u + (uint32_t)s * 2048u,
                           (uint32_t)rows * 128u, 1024);
}

// Descriptor of the same operand `units` x 16 bytes further on: the start
// address occupies the low 14 bits and never carries out of them here
// (shared-memory addresses are below 256 KB).
__device__ __forceinline__ uint64_t dstep(uint64_t d, uint32_t units) { return d + units; }

// K-steps of a K-major RS operand: +32 bytes inside a 64-column block, then
// the next column block (rows x 128 bytes further on).
__device__ __forceinline__ uint32_t kstep_units(int rows, int s) {
    return (uint32_t)(s >> 2) * (uint32_t)rows * 8u + (uint32_t)(s & 3) * 2u;
}

// Row of a TMEM accumulator held by this thread (lane quarter q = warp % 4),
// or -1.  M = 128: row = lane; M = 64: rows 16q..16q+15 sit in lanes 0..15
// of quarter q.
__device__ __forceinline__ int acc_row(int M, int q, int lane) {
    if (M == 128) return 32 * q + lane;
    return lane < 16 ? 16 * q + lane : -1;
}

// NC (16 or 32) consecutive TMEM columns of this thread's lane, one wait.
template <int NC>
__device__ __forceinline__ void tmem_cols(uint32_t taddr, float (&v)[NC]) {
    if constexpr (NC == 32) tmem_ld32(taddr, v);
    else tmem_ld16(taddr, v);
}

// The backward pass's per-chunk matrices in the workspace -- the state and
// its gradient at every chunk start (fp32 [D][D]), that gradient in bf16
// ([D][D]) and du (bf16 [64][D]) -- are stored by 16-byte units (4 fp32 or
// 8 bf16 of one row), one column of units after another: unit (row r, column
// group g) at index g * rows + r.  A warp whose lanes hold consecutive rows
// (a TMEM lane quarter) then stores one contiguous run of units at a time,
// where row-major storage would have each lane write its own row.
__host__ __device__ __forceinline__ int64_t unit_at(int rows, int r, int g) {
    return (int64_t)g * rows + r;
}

// Per-(chunk, head) record written by the intra-chunk kernel and read by the
// inter-chunk kernel, byte-for-byte the shared-memory image of its operands:
//   WQ    [-W ; Q e^{b}]                 128-row RS tile (W = T (beta K e^{b}));
//                                        A operand of the stacked product
//                                        [-W ; Q e^b] S  (M = 128)
//   UK    [U ; K e^{b_end - b}]          128-row RS tile (U = T (beta V));
//                                        rows 64..127 are the MN-major A
//                                        operand of S += K~^T u
//   AQ    Aq (masked, decayed scores)    64 x 64 RS tile, right after UK so
//                                        that [UK's last 64 rows ; Aq] is a
//                                        128-row operand
//   GEND  e^{b_end} per key channel      fp32 [D]
// Rows past the end of a ragged chunk are zero in every tile.
template <int D>
struct Record {
    static constexpr uint32_t tile64 = C * D * 2;
    static constexpr uint32_t WQ = 0;
    static constexpr uint32_t UK = 2 * tile64;
    static constexpr uint32_t AQ = 4 * tile64;
    static constexpr uint32_t GEND = AQ + 8192;
    static constexpr uint32_t BYTES = (GEND + 4 * D + 1023) & ~1023u;
};

// Workspace of the tensor-core path: the chunk table (written only when the
// backward pass asks for per-chunk states; one {first token,
// length} pair per chunk slot) followed by the records, [slot][head], then
// the flags and counters of the fused launch.
// Sequence n's chunk j occupies slot cu[n]/64 + n + j; slots never collide
// and number at most ntok/64 + N + 1.
struct Workspace {
    static inline int64_t slots(int N, int ntok) { return (int64_t)ntok / C + N + 1; }
    static inline int64_t table_bytes(int N, int ntok) {
        return (slots(N, ntok) * 8 + 1023) & ~int64_t(1023);
    }
    // after the records: one flag per record and two task counters, for the
    // launch that runs the intra-chunk tasks and the recurrence together
    static inline int64_t flag_bytes(int N, int ntok, int H) {
        return ((slots(N, ntok) * H * 4 + 255) & ~int64_t(255)) + 256;
    }
};

}  // namespace tile
}  // namespace la
