// prefill_tc.cu -- chunkwise (gated) delta-rule prefill on tcgen05 tensor
// cores, bf16 I/O, fp32 state and accumulators, dk = dv = D in {64, 128}.
//
// Algorithm ("From GPT-2 to Kimi K3, explained", section DeltaNet
// (Parallelizing Linear Transformers with Delta Rule), eq. 8-10, with the
// cumulative per-key-channel decay of sections Gated DeltaNet and
// KDA / Kimi Linear).  Per chunk of C = 64 tokens, with b = cumulative log
// decay inside the chunk (per key channel):
//   A[r][i]  = beta_r sum_c k_rc k_ic e^{b_rc - b_ic}   (i < r)     UT matrix
//   Aq[r][i] =        sum_c q_rc k_ic e^{b_rc - b_ic}   (i <= r)    scores
//   T  = (I + A)^{-1}                                   blocked forward substitution
//   W  = T (beta K e^{b}),  u = T (beta V) - W S        (eq. 10, then u = U - W S)
//   O  = scale ((Q e^{b}) S + Aq u)                     (eq. 8-9)
//   S <- Diag(e^{b_end}) S + (K e^{b_end - b})^T u
//
// Decay factors.  Only products of alpha are formed, never exponentials of
// cumulative sums: alpha = 1 / (1 + e^g) and 1/alpha = 1 + e^g cost one
// exponential and one reciprocal per element, and every other factor is a
// running product.  Aq and A need e^{b_r - b_i} for i <= r, which does not
// factor into a row term times a column term over a whole chunk without
// overflow.  The chunk is cut into four 16-token blocks; for rows r of block
// R the reference point is the token just before R:
//   row factor  P_r = prod_{t=start(R)}^{r} alpha_t               (<= 1)
//   col factor  prod_{t=i+1}^{start(R)-1} alpha_t   for i < start(R)   (<= 1)
//               1 / prod_{t=start(R)}^{i} alpha_t   for i in R         (>= 1)
// so one tensor-core product per block R (the columns of K scaled for R)
// gives the rows of A and Aq that belong to R.  The reciprocal column factor
// spans at most 16 tokens; it is exact while that 16-token decay of a
// channel stays above ~1e-30 (mean alpha above ~0.013), and is clamped
// (never inf/NaN) beyond.
//
// Mapping: one CTA of 256 threads per (sequence, head) scans the chunks in
// order.  The state S lives in tensor memory (fp32) for the whole sequence;
// a bf16 copy in shared memory feeds the products W S and (Q e^{b}) S.
// Products on tcgen05 (bf16 x bf16 -> fp32 in TMEM), operands staged in
// 128-byte-swizzled shared memory: [Q;K]-hat x K_R^T (4 per chunk), T W-
// and U-products, W S, (Q e^b) S, Aq u, K~^T u.  Raw q, k, v and gate tiles
// arrive by TMA; the next chunk's tiles are in flight while the current
// chunk computes.  The triangular solve runs in fp32 on CUDA cores: the
// four diagonal 16x16 blocks by warp-shuffle forward substitution, the
// off-diagonal blocks by three levels of small block products.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace la {

__device__ unsigned g_tc_error;  // first error code raised by a bounded wait

namespace {

using namespace tc;

constexpr int C = 64;     // tokens per chunk
constexpr int NT = 512;   // threads per CTA (16 warps)
constexpr int TMEM_COLS = 512;
constexpr int LDT = 68;   // fp32 row stride of the A and T scratch (16-byte rows)

// ------------------------------------------------------------- smem layout
// Every operand tile is a "row-swizzled" (RS) tile: `rows` rows of D bf16,
// stored as D/64 column blocks of rows x 128 bytes, 128-byte swizzled with
// 1024-byte atoms.  The same bytes serve as a K-major operand (rows = M or
// N) or an MN-major operand (rows = K).
template <int D, bool GATED>
struct Layout {
    static constexpr uint32_t tile64 = C * D * 2;               // [64][D]
    static constexpr uint32_t RAW_Q = 0;
    static constexpr uint32_t RAW_K = RAW_Q + tile64;
    static constexpr uint32_t RAW_V = RAW_K + tile64;
    static constexpr uint32_t RAW_G = RAW_V + tile64;
    static constexpr uint32_t X = RAW_G + (GATED ? tile64 : 0);
    // X, prologue (gated): fp32 prefix products P and 1/P ([64][D] each),
    // then the block-product operands [Q^; K^] (128 rows) and packed K_R (160)
    static constexpr uint32_t PP = X;
    static constexpr uint32_t PPI = X + 64 * D * 4;
    static constexpr uint32_t QKH = X;
    static constexpr uint32_t KR = X + 128 * D * 2;
    // X during and after the solve
    static constexpr uint32_t T16 = X;                  // T, bf16 [64][64]
    static constexpr uint32_t AQK = X + 8192;           // Aq, bf16 [64][64]
    static constexpr uint32_t SA = X + 16384;           // A, fp32 [64][LDT]
    static constexpr uint32_t ST = SA + 64 * LDT * 4;   // T, fp32 [64][LDT]
    static constexpr uint32_t SX = ST + 64 * LDT * 4;   // merge temps, fp32 (8 KB)
    static constexpr uint32_t SB = (SX + 8192 + 1023) & ~1023u;  // S, bf16 [D][D]
    static constexpr uint32_t X_END_A = GATED ? KR + 160 * D * 2 : X;
    static constexpr uint32_t X_END_P = GATED ? PPI + 64 * D * 4 : X;
    static constexpr uint32_t X_END_C = SB + D * D * 2;
    static constexpr uint32_t X_END0 = X_END_A > X_END_P ? X_END_A : X_END_P;
    static constexpr uint32_t X_END1 = X_END0 > X_END_C ? X_END0 : X_END_C;
    // [Q e^b ; K e^{b_end - b}] (gated) or [q^ ; k^] (ungated), 128 rows
    static constexpr uint32_t PAIR = (X_END1 + 1023) & ~1023u;
    static constexpr uint32_t BKG = PAIR + 2 * tile64;         // beta K e^b, later W
    static constexpr uint32_t BV = BKG + tile64;               // beta V, later u
    static constexpr uint32_t SMALL = BV + tile64;
    static constexpr uint32_t BETA = SMALL;                    // fp32 [64]
    static constexpr uint32_t KN = BETA + 256;                 // fp32 [64]
    static constexpr uint32_t QN = KN + 256;                   // fp32 [64]
    static constexpr uint32_t EB = QN + 256;                   // fp32 [4][D] block decay
    static constexpr uint32_t GEND = EB + 16 * D;              // fp32 [D] chunk decay
    // fp32 [5][4][D] block constants: live only between the decay scan and
    // the operand stage, when the raw gate tile has been consumed
    static constexpr uint32_t KC = RAW_G;
    static_assert(80 * D <= tile64, "block constants fit in the gate tile");
    static constexpr uint32_t BARS = GEND + 4 * D;             // 2 mbarriers + tmem slot
    static constexpr uint32_t TOTAL = BARS + 64;
    static_assert(TOTAL + 1024 <= 227 * 1024, "shared memory budget");
};

// TMEM column map.  S: fp32 state (rows = key channels).  W and U adjacent
// (one N = 2D product writes both), O after them.  A: the block products
// (phase B and C1 only, up to 160 columns), reusing W/U/O's columns.
template <int D>
struct Cols {
    static constexpr uint32_t S = 0, W = D, U = 2 * D, O = 3 * D, A = D;
    static constexpr int MS = D;  // M of the state accumulator
};

__device__ __forceinline__ uint32_t rs_off(int rows, int row, int col) {
    return (uint32_t)(col >> 6) * (uint32_t)rows * 128u + sw128_offset(row, col & 63);
}

// 8 consecutive columns (col % 8 == 0) as one 16-byte store.
__device__ __forceinline__ void st_bf16x8(uint8_t *tile, int rows, int row, int col,
                                          const float *v) {
    uint4 u;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint4 *>(tile + rs_off(rows, row, col)) = u;
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

__device__ __forceinline__ uint4 pack8(const float *v) {
    uint4 u;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    return u;
}

__device__ __forceinline__ float bf(const uint8_t *p) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(p));
}

__device__ __forceinline__ void stbf(uint8_t *p, float v) {
    *reinterpret_cast<__nv_bfloat16 *>(p) = __float2bfloat16_rn(v);
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

struct TcParams {
    const __nv_bfloat16 *beta_logits;
    __nv_bfloat16 *o;
    const int32_t *cu_seqlens;
    const float *init_S;
    float *final_S;
    int H, ntok;
    float scale;
    unsigned flags;
};

__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

// ---- warp-level TF32 products for the small blocks of the triangular solve
// (m16n8k8: A 16x8 row-major, B 8x8 as [k][n], C 16x8; fp32 accumulate).
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const float *A, int lda, const float *B,
                                         int ldb, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const uint32_t a0 = to_tf32(A[g * lda + t]), a1 = to_tf32(A[(g + 8) * lda + t]);
    const uint32_t a2 = to_tf32(A[g * lda + t + 4]), a3 = to_tf32(A[(g + 8) * lda + t + 4]);
    const uint32_t b0 = to_tf32(B[t * ldb + g]), b1 = to_tf32(B[(t + 4) * ldb + g]);
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// C (16x8 tile at Cp, row stride ldc) = sign * d
__device__ __forceinline__ void store_c(float *Cp, int ldc, const float (&d)[4], float sign,
                                        int lane) {
    const int g = lane >> 2, t = lane & 3;
    Cp[g * ldc + 2 * t] = sign * d[0];
    Cp[g * ldc + 2 * t + 1] = sign * d[1];
    Cp[(g + 8) * ldc + 2 * t] = sign * d[2];
    Cp[(g + 8) * ldc + 2 * t + 1] = sign * d[3];
}

template <int D, bool GATED>
__global__ void __launch_bounds__(NT, 1)
    delta_chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_g, TcParams p) {
    using L = Layout<D, GATED>;
    using TC = Cols<D>;
    constexpr int DQ = D / 4;  // TMEM columns per warp in the readbacks
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *rawq = sm + L::RAW_Q, *rawk = sm + L::RAW_K, *rawv = sm + L::RAW_V,
            *rawg = sm + L::RAW_G;
    uint8_t *qkh = sm + L::QKH, *kr = sm + L::KR, *t16 = sm + L::T16, *aqk = sm + L::AQK;
    float *sP = reinterpret_cast<float *>(sm + L::PP);
    float *sPi = reinterpret_cast<float *>(sm + L::PPI);
    float *sA = reinterpret_cast<float *>(sm + L::SA);
    float *sT = reinterpret_cast<float *>(sm + L::ST);
    float *sX = reinterpret_cast<float *>(sm + L::SX);
    uint8_t *sb = sm + L::SB, *pair = sm + L::PAIR, *bkg = sm + L::BKG, *bv = sm + L::BV;
    uint8_t *wt = bkg, *ut = bv;  // W and u tiles reuse beta K e^b and beta V
    float *sbeta = reinterpret_cast<float *>(sm + L::BETA);
    float *skn = reinterpret_cast<float *>(sm + L::KN);
    float *sqn = reinterpret_cast<float *>(sm + L::QN);
    float *sE = reinterpret_cast<float *>(sm + L::EB);
    float *sgend = reinterpret_cast<float *>(sm + L::GEND);
    float *sKC = reinterpret_cast<float *>(sm + L::KC);
    uint64_t *bar_tma = reinterpret_cast<uint64_t *>(sm + L::BARS);
    uint64_t *bar_mma = bar_tma + 1;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar_tma + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qd = warp & 3, cp = warp >> 2;  // TMEM lane quarter, column part
    const int h = blockIdx.x, n = blockIdx.y, H = p.H;
    int t_begin = p.cu_seqlens[n], t_end = p.cu_seqlens[n + 1];
    if (t_begin < 0 || t_end < t_begin || t_end > p.ntok) {
        if (tid == 0) atomicCAS(&g_tc_error, 0u, 100u);
        t_begin = t_end = 0;
    }
    const bool silu = (p.flags & kSiluQK) != 0;
    const bool l2k = (p.flags & kL2NormK) != 0, l2q = (p.flags & kL2NormQ) != 0;
    constexpr uint32_t tx_bytes = (GATED ? 4u : 3u) * L::tile64;

    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        if (GATED) tma_prefetch_desc(&tm_g);
    }
    if (warp == 0) {
        tmem_alloc(tslot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tq = tmem + ((uint32_t)(32 * qd) << 16);  // this warp's lane quarter

    auto issue_tma = [&](int t0) {
        fence_proxy_async();
        mbar_arrive_expect_tx(bar_tma, tx_bytes);
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb) {
            tma_load_3d(rawq + cb * 8192, &tm_q, bar_tma, cb * 64, h, t0);
            tma_load_3d(rawk + cb * 8192, &tm_k, bar_tma, cb * 64, h, t0);
            tma_load_3d(rawv + cb * 8192, &tm_v, bar_tma, cb * 64, h, t0);
            if (GATED) tma_load_3d(rawg + cb * 8192, &tm_g, bar_tma, cb * 64, h, t0);
        }
    };

    // ---- initial state into TMEM (fp32), zero if none
    const int64_t sbase = ((int64_t)n * H + h) * D * D;
    {
        const int row = acc_row(TC::MS, qd, lane);
#pragma unroll
        for (int cb = 0; cb < DQ; cb += 16) {
            const int col = cp * DQ + cb;
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                v[i] = (row >= 0 && p.init_S) ? p.init_S[sbase + (int64_t)row * D + col + i] : 0.0f;
            tmem_st16(tq + TC::S + col, v);
        }
    }
    bool tma_pending = false;
    if (tid == 0 && t_begin < t_end) issue_tma(t_begin);
    tma_pending = t_begin < t_end;
    uint32_t tma_par = 0, mma_par = 0;
    bool failed = false;
    // beta logits of the next chunk, loaded one chunk ahead (threads 0..63)
    float beta_next = 0.0f;
    if (tid < C && t_begin + tid < t_end)
        beta_next = __bfloat162float(p.beta_logits[(int64_t)(t_begin + tid) * H + h]);

    // One thread waits on an mbarrier; the CTA barrier that follows every
    // wait (a __syncthreads_or carrying the outcome) releases the others,
    // who then order their tensor-memory accesses after it.
    auto mma_wait = [&]() -> bool {
        bool ok = true;
        if (tid == 0) ok = mbar_wait(bar_mma, mma_par, &g_tc_error, 2);
        mma_par ^= 1;
        return ok;
    };
    auto phase_sync = [&]() {
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };

    for (int cs = t_begin; cs < t_end; cs += C) {
        const int len = min(C, t_end - cs);
        // ---------------------------------------------- raw tiles of this chunk
        {
            const bool ok = tid == 0 ? mbar_wait(bar_tma, tma_par, &g_tc_error, 1) : true;
            tma_par ^= 1;
            tma_pending = false;
            tc_fence_before();
            if (__syncthreads_or(!ok)) { failed = true; break; }
            tc_fence_after();
        }
        // ---------------------------------------------- A0: beta, row norms
        if (tid < C) {
            sbeta[tid] = tid < len ? __fdividef(1.0f, 1.0f + __expf(-beta_next)) : 0.0f;
            const int tn = cs + C + tid;
            beta_next = tn < t_end ? __bfloat162float(p.beta_logits[(int64_t)tn * H + h]) : 0.0f;
        }
        {
            // 8 threads per row, D/8 channels each, 16-byte loads
            const int r = tid >> 3, part = tid & 7;
            float ssk = 0.0f, ssq = 0.0f;
#pragma unroll
            for (int c = part * (D / 8); c < (part + 1) * (D / 8); c += 8) {
                float kv[8], qv[8];
                unpack8(*reinterpret_cast<const uint4 *>(rawk + rs_off(C, r, c)), kv);
                unpack8(*reinterpret_cast<const uint4 *>(rawq + rs_off(C, r, c)), qv);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (silu) { kv[i] = silu_fast(kv[i]); qv[i] = silu_fast(qv[i]); }
                    ssk += kv[i] * kv[i];
                    ssq += qv[i] * qv[i];
                }
            }
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                ssk += __shfl_xor_sync(0xffffffffu, ssk, o);
                ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
            }
            if (part == 0) {
                const bool valid = r < len;
                skn[r] = valid ? (l2k ? rsqrtf(fmaxf(ssk, 1e-24f)) : 1.0f) : 0.0f;
                sqn[r] = valid ? (l2q ? rsqrtf(fmaxf(ssq, 1e-24f)) : 1.0f) : 0.0f;
            }
        }
        __syncthreads();
        // ---------------------------------------------- A1: operand tiles
        if (!GATED) {
            // [q^; k^] into PAIR, beta k^ into BKG, beta v into BV: 16-byte units
            for (int u = tid; u < C * D / 8; u += NT) {
                const uint32_t off = (uint32_t)u * 16u;                 // offset in a [64][D] tile
                const uint32_t cb = off >> 13, in = off & 8191u;         // column block, offset in it
                const int r = (int)(in >> 7);
                const uint32_t po = cb * (128u * 128u) + in;            // same row in PAIR
                float kv[8], qv[8], vv[8];
                unpack8(*reinterpret_cast<const uint4 *>(rawk + off), kv);
                unpack8(*reinterpret_cast<const uint4 *>(rawq + off), qv);
                unpack8(*reinterpret_cast<const uint4 *>(rawv + off), vv);
                const float kn = skn[r], qn = sqn[r], be = sbeta[r];
                float bk[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (silu) { kv[i] = silu_fast(kv[i]); qv[i] = silu_fast(qv[i]); }
                    kv[i] *= kn;
                    qv[i] *= qn;
                    bk[i] = be * kv[i];
                    vv[i] *= be;
                }
                *reinterpret_cast<uint4 *>(pair + po) = pack8(qv);
                *reinterpret_cast<uint4 *>(pair + po + 64u * 128u) = pack8(kv);
                *reinterpret_cast<uint4 *>(bkg + off) = pack8(bk);
                *reinterpret_cast<uint4 *>(bv + off) = pack8(vv);
            }
            if (tid < D) sgend[tid] = 1.0f;
        } else {
            // One thread per (2 key channels, 8 rows of a 16-token block R); the
            // two 8-row halves of a block sit in lanes l and l^16 of one warp.
            // alpha = 1/(1+e^g), 1/alpha = 1+e^g; P = prefix product of alpha
            // inside the block, Pi = 1/P.  Every operand is (q or k) x (P or Pi)
            // x a per-(block, channel) constant; the within-block suffix is
            // prod_{t>r} alpha_t = E_R / P_r with E_R the block total.
            const bool act = warp < D / 8;
            const int R = (warp * 32 / D) & 3, grp = warp % (D / 32);
            const int hf2 = lane >> 4, c0 = 32 * grp + 2 * (lane & 15);
            const int r0 = 16 * R + 8 * hf2;
            // Rows r0 and r0 + 8 share a swizzle phase, so at step rho the
            // second-half lanes work on row r0 + (rho ^ 4): the two halves of
            // the warp then hit disjoint banks.
            const int pr = 4 * hf2;
            // Addressing: the channel pair is fixed per thread and r0 is a
            // multiple of 8, so row r0 + rho has swizzle phase rho.
            const uint32_t cb = (uint32_t)c0 >> 6, ch = ((uint32_t)c0 >> 3) & 7u;
            const uint32_t cboff64 = cb * 64u * 128u, cboff128 = cb * 128u * 128u,
                           cboff160 = cb * 160u * 128u;
            uint32_t swz[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) swz[j] = ((ch ^ (uint32_t)j) << 4) + ((uint32_t)c0 & 7u) * 2u;
            float P[8][2], Pi[8][2];
#pragma unroll
            for (int rho = 0; rho < 8; ++rho) { P[rho][0] = P[rho][1] = 1.0f; Pi[rho][0] = Pi[rho][1] = 1.0f; }
            if (act) {
                float p0 = 1.0f, p1 = 1.0f, q0 = 1.0f, q1 = 1.0f;
#pragma unroll
                for (int rho = 0; rho < 8; ++rho) {
                    // the scan runs in natural row order (a prefix product);
                    // only the store pass below uses the permuted order
                    const int r = r0 + rho;
                    const __nv_bfloat162 g2 = *reinterpret_cast<const __nv_bfloat162 *>(rawg + cboff64 + r * 128 + swz[rho]);
                    const float2 g = __bfloat1622float2(g2);
                    const float e0 = __expf(fminf(g.x, 80.0f)), e1 = __expf(fminf(g.y, 80.0f));
                    if (r < len) {
                        p0 *= __fdividef(1.0f, 1.0f + e0);
                        p1 *= __fdividef(1.0f, 1.0f + e1);
                        q0 = fminf(q0 * (1.0f + e0), 1e30f);
                        q1 = fminf(q1 * (1.0f + e1), 1e30f);
                    }
                    P[rho][0] = p0; P[rho][1] = p1; Pi[rho][0] = q0; Pi[rho][1] = q1;
                }
            }
            // carry the first half's totals into the second half
            {
                const float t0 = __shfl_sync(0xffffffffu, P[7][0], lane ^ 16);
                const float t1 = __shfl_sync(0xffffffffu, P[7][1], lane ^ 16);
                const float u0 = __shfl_sync(0xffffffffu, Pi[7][0], lane ^ 16);
                const float u1 = __shfl_sync(0xffffffffu, Pi[7][1], lane ^ 16);
                if (hf2) {
#pragma unroll
                    for (int rho = 0; rho < 8; ++rho) {
                        P[rho][0] *= t0; P[rho][1] *= t1;
                        Pi[rho][0] = fminf(Pi[rho][0] * u0, 1e30f);
                        Pi[rho][1] = fminf(Pi[rho][1] * u1, 1e30f);
                    }
                }
            }
            if (act && hf2) {
                sE[R * D + c0] = P[7][0];
                sE[R * D + c0 + 1] = P[7][1];
            }
            __syncthreads();
            if (act) {
                float Gb[2], EaK[2], mt[3][2];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int c = c0 + j;
                    const float E0 = sE[c], E1 = sE[D + c], E2 = sE[2 * D + c], E3 = sE[3 * D + c];
                    Gb[j] = R == 0 ? 1.0f : R == 1 ? E0 : R == 2 ? E0 * E1 : E0 * E1 * E2;
                    EaK[j] = R == 0 ? E0 * E1 * E2 * E3 : R == 1 ? E1 * E2 * E3 : R == 2 ? E2 * E3 : E3;
                    float m = 1.0f;
#pragma unroll
                    for (int t = 0; t < 3; ++t) {
                        const int Rt = R + t;
                        m *= Rt == 0 ? E0 : Rt == 1 ? E1 : Rt == 2 ? E2 : E3;
                        mt[t][j] = m;
                    }
                    if (R == 0 && hf2 == 0) sgend[c] = E0 * E1 * E2 * E3;
                }
                auto st2 = [](uint8_t *p, float a, float b) {
                    *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(a, b);
                };
                uint8_t *const pq_raw = rawq + cboff64, *const pk_raw = rawk + cboff64;
                uint8_t *const p_qh = qkh + cboff128, *const p_kh = qkh + cboff128 + 64 * 128;
                uint8_t *const p_qg = pair + cboff128, *const p_kt = pair + cboff128 + 64 * 128;
                uint8_t *const p_bk = bkg + cboff64, *const p_kr = kr + cboff160;
                // second-half lanes: swap register rows rho <-> rho ^ 4 so the
                // store pass can index P[rho] with a compile-time rho
                if (pr) {
#pragma unroll
                    for (int rho = 0; rho < 4; ++rho) {
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            float t = P[rho][j]; P[rho][j] = P[rho + 4][j]; P[rho + 4][j] = t;
                            t = Pi[rho][j]; Pi[rho][j] = Pi[rho + 4][j]; Pi[rho + 4][j] = t;
                        }
                    }
                }
#pragma unroll
                for (int rho = 0; rho < 8; ++rho) {
                    const int r = r0 + (rho ^ pr);
                    const uint32_t o = (uint32_t)r * 128u + (((ch ^ (uint32_t)(rho ^ pr)) << 4) + ((uint32_t)c0 & 7u) * 2u);
                    float2 qv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(pq_raw + o));
                    float2 kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(pk_raw + o));
                    if (silu) {
                        qv.x = silu_fast(qv.x); qv.y = silu_fast(qv.y);
                        kv.x = silu_fast(kv.x); kv.y = silu_fast(kv.y);
                    }
                    const float qn = sqn[r], kn = skn[r], be = sbeta[r];
                    qv.x *= qn; qv.y *= qn; kv.x *= kn; kv.y *= kn;
                    const float a0 = qv.x * P[rho][0], a1 = qv.y * P[rho][1];     // Q^
                    const float b0 = kv.x * P[rho][0], b1 = kv.y * P[rho][1];     // K^
                    const float k0 = kv.x * Pi[rho][0], k1 = kv.y * Pi[rho][1];   // K_R own block
                    st2(p_qh + o, a0, a1);
                    st2(p_kh + o, b0, b1);
                    st2(p_qg + o, a0 * Gb[0], a1 * Gb[1]);                  // Q e^b
                    st2(p_kt + o, k0 * EaK[0], k1 * EaK[1]);                // K e^{b_end-b}
                    st2(p_bk + o, be * b0 * Gb[0], be * b1 * Gb[1]);        // beta K e^b
                    st2(p_kr + (uint32_t)(8 * R * (R + 1)) * 128u + o, k0, k1);
#pragma unroll
                    for (int t = 0; t < 3; ++t) {
                        const int R2 = R + 1 + t;
                        if (R2 < 4)
                            st2(p_kr + (uint32_t)(8 * R2 * (R2 + 1)) * 128u + o, k0 * mt[t][0], k1 * mt[t][1]);
                    }
                }
            }
            // beta V
            for (int u = tid; u < C * D / 8; u += NT) {
                const uint32_t off = (uint32_t)u * 16u;
                const int r = (int)((off & 8191u) >> 7);
                float vv[8];
                unpack8(*reinterpret_cast<const uint4 *>(rawv + off), vv);
                const float be = sbeta[r];
#pragma unroll
                for (int i = 0; i < 8; ++i) vv[i] *= be;
                *reinterpret_cast<uint4 *>(bv + off) = pack8(vv);
            }
        }
        phase_sync();
        // raw tiles consumed: fetch the next chunk while this one computes
        if (cs + C < t_end) {
            if (tid == 0) issue_tma(cs + C);
            tma_pending = true;
        }
        // ---------------------------------------------- B: block products
        // Issue loops are kept rolled and short: this code runs on one thread,
        // so every instruction of it is fetched without help from other warps.
        if (tid == 0) {
            // gated: the packed K_R tile is one 160-row operand, so all four block
            // products form one N = 160 product (block R at column 8R(R+1));
            // ungated: one product [q^; k^] x k^T (N = 64)
            const uint32_t id = GATED ? idesc_bf16(128, 160, false, false) : idesc_bf16(128, 64, false, false);
            const uint32_t bRows = GATED ? 160u : 128u;
            const uint64_t a0 = GATED ? kdesc(qkh, 128, 0, 0) : kdesc(pair, 128, 0, 0);
            const uint64_t b0 = GATED ? kdesc(kr, 160, 0, 0) : kdesc(pair, 128, 64, 0);
#pragma unroll 1
            for (int kb = 0; kb < D / 64; ++kb) {
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4)
                    mma_bf16(tmem + TC::A, dstep(a0, kb * 128 * 8 + s4 * 2),
                             dstep(b0, kb * bRows * 8 + s4 * 2), id, (kb | s4) != 0);
            }
            mma_commit(bar_mma);
        }
        if (__syncthreads_or(!mma_wait())) { failed = true; break; }
        tc_fence_after();
        // ---------------------------------------------- C1: Aq tile, A rows, T_RR, S to bf16
        // TMEM lanes 0..63 hold rows of Aq, lanes 64..127 rows of A (before
        // beta).  Gated: block R's product sits at column 8R(R+1).  A warp
        // spans two blocks, so it reads both (TMEM addresses stay
        // warp-uniform) and each lane keeps its own.
        //  - every warp: 16 columns (part cp) of its quarter -> Aq tile / A rows
        //  - warps 2, 3 then invert the diagonal 16x16 blocks, read straight
        //    from TMEM: T_RR = (I + A_RR)^{-1}, lane rho of each 16-lane group
        //    owning row rho (forward substitution with shuffles)
        //  - warps 8..15 then copy S to its bf16 operand tile and apply this
        //    chunk's decay e^{b_end} to S in place
        {
            const bool is_q = qd < 2;
            const int rb0 = 32 * (is_q ? qd : qd - 2);
            const int r = rb0 + lane, R = r >> 4, rho = r & 15;
            const int Rw = rb0 >> 4;
            auto colof = [](int Rb) { return GATED ? 8 * Rb * (Rb + 1) : 0; };
            {
                const int col = 16 * cp;
                float v[16];
                if (GATED) {
                    float w0[16], w1[16];
                    // parts beyond a block's product are masked below (col + i > r)
                    tmem_ld16(tq + TC::A + colof(Rw) + col, w0);
                    tmem_ld16(tq + TC::A + colof(Rw + 1) + col, w1);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = (R == Rw) ? w0[i] : w1[i];
                } else {
                    tmem_ld16(tq + TC::A + col, v);
                }
                if (is_q) {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (col + i > r) v[i] = 0.0f;
                    st_bf16x8(aqk, 64, r, col, v);
                    st_bf16x8(aqk, 64, r, col + 8, v + 8);
                } else {
                    const float be = sbeta[r];
                    float4 *dst = reinterpret_cast<float4 *>(sA + r * LDT + col);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float4 f;
                        f.x = (col + 4 * i + 0 < r) ? be * v[4 * i + 0] : 0.0f;
                        f.y = (col + 4 * i + 1 < r) ? be * v[4 * i + 1] : 0.0f;
                        f.z = (col + 4 * i + 2 < r) ? be * v[4 * i + 2] : 0.0f;
                        f.w = (col + 4 * i + 3 < r) ? be * v[4 * i + 3] : 0.0f;
                        dst[i] = f;
                    }
                }
            }
            if (warp == 2 || warp == 3) {
                // diagonal block values, beta-scaled and strict, staged per lane
                // in shared memory so the substitution loop can stay rolled
                float *dgs = sX + (warp - 2) * 32 * 17 + lane * 17;
                {
                    float w0[16], w1[16];
                    tmem_ld16(tq + TC::A + colof(Rw) + 16 * Rw, w0);
                    tmem_ld16(tq + TC::A + colof(Rw + 1) + 16 * (Rw + 1), w1);
                    const float be = sbeta[r];
#pragma unroll
                    for (int m = 0; m < 16; ++m) dgs[m] = (m < rho) ? be * ((R == Rw) ? w0[m] : w1[m]) : 0.0f;
                }
                float t[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) t[j] = (j == rho) ? 1.0f : 0.0f;
                const int gbase = lane & 16;
#pragma unroll 1
                for (int m = 0; m < 15; ++m) {
                    const float a = dgs[m];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float tm = __shfl_sync(0xffffffffu, t[j], gbase + m);
                        if (j <= m) t[j] -= a * tm;
                    }
                }
                float4 *dst = reinterpret_cast<float4 *>(sT + r * LDT);
#pragma unroll
                for (int j = 0; j < 16; ++j) dst[j] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int j = 0; j < 16; j += 4) dst[(16 * R + j) >> 2] = make_float4(t[j], t[j + 1], t[j + 2], t[j + 3]);
            } else if (warp >= 8) {
                const int c = acc_row(TC::MS, qd, lane);
                const float gd = c >= 0 ? sgend[c] : 1.0f;
                const int half = (warp >> 2) & 1;
#pragma unroll
                for (int cb = 0; cb < D / 2; cb += 32) {
                    const int col = half * (D / 2) + cb;
                    float v[32];
                    tmem_ld32(tq + TC::S + col, v);
                    if (c >= 0) {
#pragma unroll
                        for (int i = 0; i < 32; i += 8) st_bf16x8(sb, D, c, col + i, v + i);
                    }
                    if (GATED) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] *= gd;
                        tmem_st16(tq + TC::S + col, *reinterpret_cast<float(*)[16]>(v));
                        tmem_st16(tq + TC::S + col + 16, *reinterpret_cast<float(*)[16]>(v + 16));
                    }
                }
            }
        }
        __syncthreads();
        // ---------------------------------------------- C2: off-diagonal blocks of T
        // Two merges, as warp-level TF32 products (the blocks are 16 and 32
        // wide; T is rounded to bf16 afterwards, coarser than TF32).
        // (1) T_10 = -T_11 (A_10 T_00), T_32 = -T_33 (A_32 T_22)   (warps 0, 1)
        // (2) with T_TT = T[0:32,0:32], T_BB = T[32:64,32:64]:
        //     T[32:64, 0:32] = -T_BB (A[32:64, 0:32] T_TT)           (warps 0..7)
        {
            constexpr int LX = 24, LY = 40;
            float *sX1 = sX;                 // [2][16][LX]
            float *sY = sX + 2 * 16 * LX;    // [32][LY]
            if (warp < 2) {
                const int b = warp, R = 1 + 2 * b, J = 2 * b;
                float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const float *Ab = sA + (16 * R) * LDT + 16 * J + 8 * ks;
                    const float *Bb = sT + (16 * J + 8 * ks) * LDT + 16 * J;
                    mma_tf32(d0, Ab, LDT, Bb, LDT, lane);
                    mma_tf32(d1, Ab, LDT, Bb + 8, LDT, lane);
                }
                store_c(sX1 + b * 16 * LX, LX, d0, 1.0f, lane);
                store_c(sX1 + b * 16 * LX + 8, LX, d1, 1.0f, lane);
                __syncwarp();
                float e0[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const float *Ab = sT + (16 * R) * LDT + 16 * R + 8 * ks;
                    const float *Bb = sX1 + b * 16 * LX + (8 * ks) * LX;
                    mma_tf32(e0, Ab, LDT, Bb, LX, lane);
                    mma_tf32(e1, Ab, LDT, Bb + 8, LX, lane);
                }
                store_c(sT + (16 * R) * LDT + 16 * J, LDT, e0, -1.0f, lane);
                store_c(sT + (16 * R) * LDT + 16 * J + 8, LDT, e1, -1.0f, lane);
            }
            __syncthreads();
            const int mt = (warp >> 2) & 1, nt = warp & 3;
            if (warp < 8) {
                float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_tf32(d, sA + (32 + 16 * mt) * LDT + 8 * ks, LDT,
                             sT + (8 * ks) * LDT + 8 * nt, LDT, lane);
                store_c(sY + (16 * mt) * LY + 8 * nt, LY, d, 1.0f, lane);
            }
            __syncthreads();
            if (warp < 8) {
                float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_tf32(d, sT + (32 + 16 * mt) * LDT + 32 + 8 * ks, LDT,
                             sY + (8 * ks) * LY + 8 * nt, LY, lane);
                store_c(sT + (32 + 16 * mt) * LDT + 8 * nt, LDT, d, -1.0f, lane);
            }
            __syncthreads();
        }
        // ---------------------------------------------- C3: T to bf16 operand
        {
            const int r = tid >> 3, c = (tid & 7) * 8;
            st_bf16x8(t16, 64, r, c, sT + r * LDT + c);
        }
        phase_sync();
        // ---------------------------------------------- D: W = T (beta K e^b), u = T (beta V)
        if (tid == 0) {
            // beta K e^b and beta V are adjacent column blocks: one N = 2D
            // product writes W (columns W) and U (columns U = W + D)
            constexpr uint32_t id = idesc_bf16(64, 2 * D, false, true);
            const uint64_t a0 = kdesc(t16, 64, 0, 0), b0 = mdesc(bkg, C, 0, 0);
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4)
                mma_bf16(tmem + TC::W, dstep(a0, s4 * 2), dstep(b0, s4 * 128), id, s4 > 0);
            mma_commit(bar_mma);
        }
        if (__syncthreads_or(!mma_wait())) { failed = true; break; }
        tc_fence_after();
        // ---------------------------------------------- E: W tile
        {
            const int r = acc_row(64, qd, lane);
            constexpr int NC = DQ >= 32 ? 32 : 16;
#pragma unroll
            for (int cb = 0; cb < DQ; cb += NC) {
                const int col = cp * DQ + cb;
                float v[NC];
                tmem_cols<NC>(tq + TC::W + col, v);
                if (r >= 0) {
#pragma unroll
                    for (int i = 0; i < NC; i += 8) st_bf16x8(wt, C, r, col + i, v + i);
                }
            }
        }
        phase_sync();
        // ---------------------------------------------- F: u -= W S, O = (Q e^b) S
        if (tid == 0) {
            constexpr uint32_t idw = idesc_bf16(64, D, false, true, true);
            constexpr uint32_t ido = idesc_bf16(64, D, false, true);
            const uint64_t bS = mdesc(sb, D, 0, 0), aW = kdesc(wt, C, 0, 0), aQ = kdesc(pair, 128, 0, 0);
#pragma unroll 1
            for (int kb = 0; kb < D / 64; ++kb) {
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4) {
                    const uint64_t b = dstep(bS, (kb * 4 + s4) * 128);
                    mma_bf16(tmem + TC::U, dstep(aW, kb * 64 * 8 + s4 * 2), b, idw, 1);
                    mma_bf16(tmem + TC::O, dstep(aQ, kb * 128 * 8 + s4 * 2), b, ido, (kb | s4) != 0);
                }
            }
            mma_commit(bar_mma);
        }
        if (__syncthreads_or(!mma_wait())) { failed = true; break; }
        tc_fence_after();
        // ---------------------------------------------- G: u tile
        {
            const int r = acc_row(64, qd, lane);
            constexpr int NC = DQ >= 32 ? 32 : 16;
#pragma unroll
            for (int cb = 0; cb < DQ; cb += NC) {
                const int col = cp * DQ + cb;
                float v[NC];
                tmem_cols<NC>(tq + TC::U + col, v);
                if (r >= 0) {
#pragma unroll
                    for (int i = 0; i < NC; i += 8) st_bf16x8(ut, C, r, col + i, v + i);
                }
            }
        }
        phase_sync();
        // ---------------------------------------------- H: O += Aq u, S += K~^T u
        if (tid == 0) {
            constexpr uint32_t ido = idesc_bf16(64, D, false, true);
            constexpr uint32_t ids = idesc_bf16(D, D, true, true);
            const uint64_t bU = mdesc(ut, C, 0, 0), aA = kdesc(aqk, 64, 0, 0), aK = mdesc(pair, 128, 64, 0);
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
                const uint64_t b = dstep(bU, s4 * 128);
                mma_bf16(tmem + TC::O, dstep(aA, s4 * 2), b, ido, 1);
                mma_bf16(tmem + TC::S, dstep(aK, s4 * 128), b, ids, 1);
            }
            mma_commit(bar_mma);
        }
        if (__syncthreads_or(!mma_wait())) { failed = true; break; }
        tc_fence_after();
        // ---------------------------------------------- I: O -> global
        {
            const int r = acc_row(64, qd, lane);
            const bool valid = r >= 0 && r < len;
            __nv_bfloat16 *orow = p.o + ((int64_t)(cs + (r < 0 ? 0 : r)) * H + h) * D;
            constexpr int NC = DQ >= 32 ? 32 : 16;
#pragma unroll
            for (int cb = 0; cb < DQ; cb += NC) {
                const int col = cp * DQ + cb;
                float v[NC];
                tmem_cols<NC>(tq + TC::O + col, v);
                if (valid) {
#pragma unroll
                    for (int i = 0; i < NC; ++i) v[i] *= p.scale;
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + col);
#pragma unroll
                    for (int i = 0; i < NC / 8; ++i) dst[i] = pack8(v + 8 * i);
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }

    if (failed && tma_pending && tid == 0) mbar_wait(bar_tma, tma_par, &g_tc_error, 3);
    // ---- final state
    if (p.final_S && !failed) {
        const int row = acc_row(TC::MS, qd, lane);
#pragma unroll
        for (int cb = 0; cb < DQ; cb += 16) {
            const int col = cp * DQ + cb;
            float v[16];
            tmem_ld16(tq + TC::S + col, v);
            if (row >= 0) {
                float4 *dst = reinterpret_cast<float4 *>(p.final_S + sbase + (int64_t)row * D + col);
#pragma unroll
                for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

// ------------------------------------------------------------------- host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// 3-D map over a packed [ntok][H][D] bf16 tensor; box = 64 tokens x 1 head x 64 channels.
bool make_map(CUtensorMap *m, const void *ptr, int D, int H, int ntok) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)(ntok > 0 ? ntok : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool GATED>
cudaError_t launch_t(const PrefillArgs &a, cudaStream_t s) {
    CUtensorMap mq, mk, mv, mg;
    if (!make_map(&mq, a.q, D, a.H, a.ntok) || !make_map(&mk, a.k, D, a.H, a.ntok) ||
        !make_map(&mv, a.v, D, a.H, a.ntok))
        return cudaErrorInvalidValue;
    if (GATED) {
        if (!make_map(&mg, a.gate_logits, D, a.H, a.ntok)) return cudaErrorInvalidValue;
    } else {
        mg = mq;
    }
    TcParams p{static_cast<const __nv_bfloat16 *>(a.beta_logits), static_cast<__nv_bfloat16 *>(a.o),
               a.cu_seqlens, a.init_S, a.final_S, a.H, a.ntok, a.scale, a.flags};
    // At least 120 KB so that one CTA (and its 512 TMEM columns) owns an SM.
    constexpr size_t need = Layout<D, GATED>::TOTAL + 1024;
    const size_t smem = need > 120 * 1024 ? need : 120 * 1024;
    auto kern = delta_chunk_tc_kernel<D, GATED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.H, a.N);
    kern<<<grid, NT, smem, s>>>(mq, mk, mv, mg, p);
    return cudaGetLastError();
}

}  // namespace

bool delta_tc_supported(const PrefillArgs &a) {
    auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    return a.bf16 && a.dk == a.dv && (a.dk == 64 || a.dk == 128) && al16(a.q) && al16(a.k) &&
           al16(a.v) && al16(a.o) && (!a.gate_logits || al16(a.gate_logits)) &&
           (!a.init_S || al16(a.init_S)) && (!a.final_S || al16(a.final_S)) && encode_fn() != nullptr;
}

cudaError_t launch_delta_tc(const PrefillArgs &a, cudaStream_t s) {
    const bool g = a.gate_logits != nullptr;
    if (a.dk == 128) return g ? launch_t<128, true>(a, s) : launch_t<128, false>(a, s);
    return g ? launch_t<64, true>(a, s) : launch_t<64, false>(a, s);
}

unsigned *device_error_word() {
    static unsigned *ptr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (!ptr[dev]) {
        void *a = nullptr;
        if (cudaGetSymbolAddress(&a, g_tc_error) != cudaSuccess) return nullptr;
        ptr[dev] = static_cast<unsigned *>(a);
    }
    return ptr[dev];
}

cudaError_t tc_take_error(cudaStream_t s, unsigned *code) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(code, g_tc_error, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && *code != 0)
        e = cudaMemcpyToSymbolAsync(g_tc_error, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return e;
}

}  // namespace la
