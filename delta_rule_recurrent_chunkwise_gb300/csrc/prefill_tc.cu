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
constexpr int NT = 256;   // threads per CTA
constexpr int TMEM_COLS = 512;

// ------------------------------------------------------------- smem layout
// Every operand tile is a "row-swizzled" (RS) tile: `rows` rows of D bf16,
// stored as D/64 column blocks of rows x 128 bytes, 128-byte swizzled with
// 1024-byte atoms.  The same bytes serve as a K-major operand (rows = M or
// N) or an MN-major operand (rows = K).
template <int D>
struct Layout {
    static constexpr uint32_t tile64 = C * D * 2;               // [64][D]
    static constexpr uint32_t RAW_Q = 0;
    static constexpr uint32_t RAW_K = RAW_Q + tile64;
    static constexpr uint32_t RAW_V = RAW_K + tile64;
    static constexpr uint32_t RAW_G = RAW_V + tile64;
    static constexpr uint32_t X = RAW_G + tile64;
    // X during the block products: [Q^; K^] (128 rows) and packed K_R (160)
    static constexpr uint32_t QKH = X;
    static constexpr uint32_t KR = X + 128 * D * 2;
    // X during and after the solve
    static constexpr uint32_t T16 = X;                 // T, bf16 [64][64]
    static constexpr uint32_t AQK = X + 8192;          // Aq, bf16 [64][64]
    static constexpr uint32_t SA = X + 16384;          // A, fp32 [64][65]
    static constexpr uint32_t ST = SA + 64 * 65 * 4;   // T, fp32 [64][65]
    static constexpr uint32_t SX = ST + 64 * 65 * 4;   // block temp, fp32 [3][16][17]
    static constexpr uint32_t SB = X + 16384;          // S, bf16 [D][D] (after the solve)
    static constexpr uint32_t X_END_A = KR + 160 * D * 2;
    static constexpr uint32_t X_END_B = SX + 3 * 16 * 17 * 4;
    static constexpr uint32_t X_END_C = SB + D * D * 2;
    static constexpr uint32_t X_END0 = X_END_A > X_END_B ? X_END_A : X_END_B;
    static constexpr uint32_t X_END1 = X_END0 > X_END_C ? X_END0 : X_END_C;
    static constexpr uint32_t QG = (X_END1 + 1023) & ~1023u;   // Q e^{b}       [64][D]
    static constexpr uint32_t KT = QG + tile64;                // K e^{b_end-b} [64][D]
    static constexpr uint32_t BKG = KT + tile64;               // beta K e^{b}, later W
    static constexpr uint32_t BV = BKG + tile64;               // beta V, later u
    static constexpr uint32_t SMALL = BV + tile64;
    static constexpr uint32_t BETA = SMALL;                    // fp32 [64]
    static constexpr uint32_t KN = BETA + 256;                 // fp32 [64]
    static constexpr uint32_t QN = KN + 256;                   // fp32 [64]
    static constexpr uint32_t EB = QN + 256;                   // fp32 [4][D] block decay
    static constexpr uint32_t GEND = EB + 16 * D;              // fp32 [D] chunk decay
    static constexpr uint32_t BARS = GEND + 4 * D;             // 2 mbarriers + tmem slot
    static constexpr uint32_t TOTAL = BARS + 64;
    static_assert(TOTAL + 1024 <= 227 * 1024, "shared memory budget");
};

// TMEM column map.  S: fp32 state (rows = key channels).  U: the delta u.
// A: four 64-column block products (phase B only), later O and W.
template <int D>
struct Cols {
    static constexpr uint32_t S = 0, U = D, A = 2 * D, O = 2 * D, W = 3 * D;
    static constexpr int MS = D;  // M of the state accumulator
};

__device__ __forceinline__ uint32_t rs_off(int rows, int row, int col) {
    return (uint32_t)(col >> 6) * (uint32_t)rows * 128u + sw128_offset(row, col & 63);
}

__device__ __forceinline__ void st_bf16(uint8_t *tile, int rows, int row, int col, float v) {
    *reinterpret_cast<__nv_bfloat16 *>(tile + rs_off(rows, row, col)) = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float ld_bf16(const uint8_t *tile, int rows, int row, int col) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(tile + rs_off(rows, row, col)));
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

__device__ __forceinline__ void ld_bf16x8(const uint8_t *tile, int rows, int row, int col,
                                          float *v) {
    uint4 u = *reinterpret_cast<const uint4 *>(tile + rs_off(rows, row, col));
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

// K-major operand descriptor for K-step s (16 elements) of an RS tile.
__device__ __forceinline__ uint64_t kdesc(const uint8_t *tile, int rows, int row0, int s) {
    return smem_desc_sw128(smem_u32(tile) + (uint32_t)(s >> 2) * rows * 128u + row0 * 128u +
                               (uint32_t)(s & 3) * 32u,
                           16, 1024);
}

// MN-major operand descriptor for K-step s (rows 16s..16s+15) of an RS tile.
__device__ __forceinline__ uint64_t mdesc(const uint8_t *tile, int rows, int s) {
    return smem_desc_sw128(smem_u32(tile) + (uint32_t)s * 2048u, (uint32_t)rows * 128u, 1024);
}

// Row of a TMEM accumulator held by this thread (lane quarter q = warp % 4),
// or -1.  M = 128: row = lane; M = 64: rows 16q..16q+15 sit in lanes 0..15
// of quarter q.
__device__ __forceinline__ int acc_row(int M, int q, int lane) {
    if (M == 128) return 32 * q + lane;
    return lane < 16 ? 16 * q + lane : -1;
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

template <int D, bool GATED>
__global__ void __launch_bounds__(NT, 1)
    delta_chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_g, TcParams p) {
    using L = Layout<D>;
    using TC = Cols<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *rawq = sm + L::RAW_Q, *rawk = sm + L::RAW_K, *rawv = sm + L::RAW_V,
            *rawg = sm + L::RAW_G;
    uint8_t *qkh = sm + L::QKH, *kr = sm + L::KR, *t16 = sm + L::T16, *aqk = sm + L::AQK;
    float *sA = reinterpret_cast<float *>(sm + L::SA);
    float *sT = reinterpret_cast<float *>(sm + L::ST);
    float *sX = reinterpret_cast<float *>(sm + L::SX);
    uint8_t *sb = sm + L::SB, *qg = sm + L::QG, *kt = sm + L::KT, *bkg = sm + L::BKG,
            *bv = sm + L::BV;
    uint8_t *wt = bkg, *ut = bv;  // W and u tiles reuse beta K e^b and beta V
    float *sbeta = reinterpret_cast<float *>(sm + L::BETA);
    float *skn = reinterpret_cast<float *>(sm + L::KN);
    float *sqn = reinterpret_cast<float *>(sm + L::QN);
    float *sE = reinterpret_cast<float *>(sm + L::EB);
    float *sgend = reinterpret_cast<float *>(sm + L::GEND);
    uint64_t *bar_tma = reinterpret_cast<uint64_t *>(sm + L::BARS);
    uint64_t *bar_mma = bar_tma + 1;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar_tma + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qd = warp & 3, hf = warp >> 2;
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
        for (int cb = 0; cb < D / 2; cb += 16) {
            const int col = hf * (D / 2) + cb;
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

    auto mma_wait = [&]() -> bool {
        const bool ok = mbar_wait(bar_mma, mma_par, &g_tc_error, 2);
        mma_par ^= 1;
        tc_fence_after();
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
            const bool ok = mbar_wait(bar_tma, tma_par, &g_tc_error, 1);
            tma_par ^= 1;
            tma_pending = false;
            tc_fence_before();
            if (__syncthreads_or(!ok)) { failed = true; break; }
            tc_fence_after();
        }
        // ---------------------------------------------- A0: beta, row norms
        if (tid < C)
            sbeta[tid] = tid < len ? sigmoid_f(__bfloat162float(p.beta_logits[(int64_t)(cs + tid) * H + h]))
                                   : 0.0f;
        {
            const int r = tid >> 2, part = tid & 3;
            float ssk = 0.0f, ssq = 0.0f;
#pragma unroll
            for (int c = part * (D / 4); c < (part + 1) * (D / 4); c += 8) {
                float kv[8], qv[8];
                ld_bf16x8(rawk, C, r, c, kv);
                ld_bf16x8(rawq, C, r, c, qv);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (silu) { kv[i] = silu_fast(kv[i]); qv[i] = silu_fast(qv[i]); }
                    ssk += kv[i] * kv[i];
                    ssq += qv[i] * qv[i];
                }
            }
            ssk += __shfl_xor_sync(0xffffffffu, ssk, 1);
            ssk += __shfl_xor_sync(0xffffffffu, ssk, 2);
            ssq += __shfl_xor_sync(0xffffffffu, ssq, 1);
            ssq += __shfl_xor_sync(0xffffffffu, ssq, 2);
            if (part == 0) {
                const bool valid = r < len;
                skn[r] = valid ? (l2k ? 1.0f / fmaxf(sqrtf(ssk), 1e-12f) : 1.0f) : 0.0f;
                sqn[r] = valid ? (l2q ? 1.0f / fmaxf(sqrtf(ssq), 1e-12f) : 1.0f) : 0.0f;
            }
        }
        __syncthreads();
        // ---------------------------------------------- A1: decay factors, operands
        {
            constexpr int CPT = D / 64;  // channels per thread
            const int cg = tid & 63, R = tid >> 6, c0 = cg * CPT;
            const int rb = 16 * R;
            float al[16][CPT], ai[16][CPT];
            if (GATED) {
                float E[CPT];
#pragma unroll
                for (int j = 0; j < CPT; ++j) E[j] = 1.0f;
#pragma unroll
                for (int rho = 0; rho < 16; ++rho) {
                    const int r = rb + rho;
#pragma unroll
                    for (int j = 0; j < CPT; ++j) {
                        const float g = fminf(ld_bf16(rawg, C, r, c0 + j), 80.0f);
                        const float e = __expf(g);
                        const bool valid = r < len;
                        al[rho][j] = valid ? __fdividef(1.0f, 1.0f + e) : 1.0f;
                        ai[rho][j] = valid ? 1.0f + e : 1.0f;
                        E[j] *= al[rho][j];
                    }
                }
#pragma unroll
                for (int j = 0; j < CPT; ++j) sE[R * D + c0 + j] = E[j];
                __syncthreads();
            }
            float Gb[CPT], Ea[CPT];
#pragma unroll
            for (int j = 0; j < CPT; ++j) {
                Gb[j] = 1.0f;
                Ea[j] = 1.0f;
                if (GATED) {
                    for (int R2 = 0; R2 < 4; ++R2) {
                        const float e = sE[R2 * D + c0 + j];
                        if (R2 < R) Gb[j] *= e;
                        if (R2 > R) Ea[j] *= e;
                    }
                    if (R == 0) sgend[c0 + j] = Gb[j] * sE[c0 + j] * Ea[j];
                } else if (R == 0) {
                    sgend[c0 + j] = 1.0f;
                }
            }
            // forward over the block: prefix products
            float P[CPT], Pi[CPT];
#pragma unroll
            for (int j = 0; j < CPT; ++j) { P[j] = 1.0f; Pi[j] = 1.0f; }
#pragma unroll
            for (int rho = 0; rho < 16; ++rho) {
                const int r = rb + rho;
                const float kn = skn[r], qn = sqn[r], be = sbeta[r];
#pragma unroll
                for (int j = 0; j < CPT; ++j) {
                    const int c = c0 + j;
                    float kv = ld_bf16(rawk, C, r, c), qv = ld_bf16(rawq, C, r, c);
                    if (silu) { kv = silu_fast(kv); qv = silu_fast(qv); }
                    kv *= kn;
                    qv *= qn;
                    if (GATED) {
                        P[j] *= al[rho][j];
                        Pi[j] = fminf(Pi[j] * ai[rho][j], 1e30f);
                    }
                    st_bf16(qkh, 128, r, c, qv * P[j]);
                    st_bf16(qkh, 128, 64 + r, c, kv * P[j]);
                    st_bf16(qg, C, r, c, qv * Gb[j] * P[j]);
                    st_bf16(bkg, C, r, c, be * kv * Gb[j] * P[j]);
                    st_bf16(kr, 160, 8 * R * (R + 1) + r, c, kv * Pi[j]);
                }
            }
            // backward over the block: suffix products
            float Sb[CPT];
#pragma unroll
            for (int j = 0; j < CPT; ++j) Sb[j] = 1.0f;
#pragma unroll
            for (int rho = 15; rho >= 0; --rho) {
                const int r = rb + rho;
                const float kn = skn[r];
#pragma unroll
                for (int j = 0; j < CPT; ++j) {
                    const int c = c0 + j;
                    float kv = ld_bf16(rawk, C, r, c);
                    if (silu) kv = silu_fast(kv);
                    kv *= kn;
                    st_bf16(kt, C, r, c, kv * Sb[j] * Ea[j]);
                    float f = Sb[j];
                    for (int R2 = R + 1; R2 < 4; ++R2) {
                        st_bf16(kr, 160, 8 * R2 * (R2 + 1) + r, c, kv * f);
                        if (GATED) f *= sE[R2 * D + c];
                    }
                    if (GATED) Sb[j] *= al[rho][j];
                }
            }
        }
        // ---------------------------------------------- A2: beta V
        for (int e = tid; e < C * D / 8; e += NT) {
            const uint32_t off = (uint32_t)e * 16u;
            const int row = (int)((off % (uint32_t)(C * 128)) >> 7);
            uint4 u = *reinterpret_cast<const uint4 *>(rawv + off);
            __nv_bfloat162 *hv = reinterpret_cast<__nv_bfloat162 *>(&u);
            const float be = sbeta[row];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float2 f = __bfloat1622float2(hv[i]);
                hv[i] = __floats2bfloat162_rn(f.x * be, f.y * be);
            }
            *reinterpret_cast<uint4 *>(bv + off) = u;
        }
        phase_sync();
        // raw tiles consumed: fetch the next chunk while this one computes
        if (cs + C < t_end) {
            if (tid == 0) issue_tma(cs + C);
            tma_pending = true;
        }
        // ---------------------------------------------- B: block products
        if (tid == 0) {
            constexpr uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
            for (int R = 0; R < 4; ++R)
#pragma unroll
                for (int s = 0; s < D / 16; ++s)
                    mma_bf16(tmem + TC::A + 64 * R, kdesc(qkh, 128, 0, s),
                             kdesc(kr, 160, 8 * R * (R + 1), s), id, s > 0);
            mma_commit(bar_mma);
        }
        if (__syncthreads_or(!mma_wait())) { failed = true; break; }
        // ---------------------------------------------- C1: Aq tile, A rows, diagonal inverses
        // TMEM lanes 0..63 hold rows of Aq, lanes 64..127 rows of A (before
        // beta); row r belongs to block R = r / 16, whose product sits in
        // columns [64 R, 64 R + 64).  A warp covers two blocks, so it reads
        // both (addresses stay warp-uniform) and each lane keeps its own.
        if (hf == 0) {
            const bool is_q = qd < 2;
            const int rb0 = 32 * (is_q ? qd : qd - 2);
            const int r = rb0 + lane, R = r >> 4, rho = r & 15;
            float row[64];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int Rw = (rb0 >> 4) + half;
#pragma unroll
                for (int cb = 0; cb < 64; cb += 16) {
                    float v[16];
                    tmem_ld16(tq + TC::A + 64 * Rw + cb, v);
                    if (R == Rw) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) row[cb + i] = v[i];
                    }
                }
            }
            if (is_q) {
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if (i > r) row[i] = 0.0f;
#pragma unroll
                for (int cb = 0; cb < 64; cb += 8) st_bf16x8(aqk, 64, r, cb, row + cb);
            } else {
                const float be = sbeta[r];
#pragma unroll
                for (int i = 0; i < 64; ++i) sA[r * 65 + i] = (i < r) ? be * row[i] : 0.0f;
                float dg[16];
#pragma unroll
                for (int m = 0; m < 16; ++m) dg[m] = sA[r * 65 + 16 * R + m];
                // T_RR = (I + A_RR)^{-1}: lane rho of each 16-lane group owns row rho
                float t[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) t[j] = (j == rho) ? 1.0f : 0.0f;
                const int gbase = lane & 16;
#pragma unroll
                for (int m = 0; m < 15; ++m) {
#pragma unroll
                    for (int j = 0; j <= m; ++j) {
                        const float tm = __shfl_sync(0xffffffffu, t[j], gbase + m);
                        if (rho > m) t[j] -= dg[m] * tm;
                    }
                }
#pragma unroll
                for (int j = 0; j < 64; ++j) sT[r * 65 + j] = 0.0f;
#pragma unroll
                for (int j = 0; j < 16; ++j) sT[r * 65 + 16 * R + j] = t[j];
            }
        }
        __syncthreads();
        // ---------------------------------------------- C2: off-diagonal blocks of T
        // T_RJ = -T_RR sum_{M=J}^{R-1} A_RM T_MJ, by levels L = R - J.
#pragma unroll 1
        for (int Lv = 1; Lv < 4; ++Lv) {
            const int nb = 4 - Lv;
            for (int e = tid; e < nb * 256; e += NT) {
                const int b = e >> 8, i = (e >> 4) & 15, j = e & 15;
                const int R = Lv + b, J = b;
                float acc = 0.0f;
                for (int m = 16 * J; m < 16 * R; ++m) acc += sA[(16 * R + i) * 65 + m] * sT[m * 65 + 16 * J + j];
                sX[(b * 16 + i) * 17 + j] = acc;
            }
            __syncthreads();
            for (int e = tid; e < nb * 256; e += NT) {
                const int b = e >> 8, i = (e >> 4) & 15, j = e & 15;
                const int R = Lv + b, J = b;
                float acc = 0.0f;
#pragma unroll
                for (int m = 0; m < 16; ++m) acc += sT[(16 * R + i) * 65 + 16 * R + m] * sX[(b * 16 + m) * 17 + j];
                sT[(16 * R + i) * 65 + 16 * J + j] = -acc;
            }
            __syncthreads();
        }
        // ---------------------------------------------- C3: T to bf16 operand
        {
            const int r = tid >> 2, c = (tid & 3) * 16;
            st_bf16x8(t16, 64, r, c, sT + r * 65 + c);
            st_bf16x8(t16, 64, r, c + 8, sT + r * 65 + c + 8);
        }
        phase_sync();
        // ---------------------------------------------- D: W = T (beta K e^b), u = T (beta V)
        if (tid == 0) {
            constexpr uint32_t id = idesc_bf16(64, D, false, true);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t a = kdesc(t16, 64, 0, s);
                mma_bf16(tmem + TC::W, a, mdesc(bkg, C, s), id, s > 0);
                mma_bf16(tmem + TC::U, a, mdesc(bv, C, s), id, s > 0);
            }
            mma_commit(bar_mma);
        }
        if (__syncthreads_or(!mma_wait())) { failed = true; break; }
        // ---------------------------------------------- E: W tile; S -> bf16, decay S
        {
            const int r = acc_row(64, qd, lane);
#pragma unroll
            for (int cb = 0; cb < D / 2; cb += 16) {
                const int col = hf * (D / 2) + cb;
                float v[16];
                tmem_ld16(tq + TC::W + col, v);
                if (r >= 0) {
                    st_bf16x8(wt, C, r, col, v);
                    st_bf16x8(wt, C, r, col + 8, v + 8);
                }
            }
            const int c = acc_row(TC::MS, qd, lane);
            const float gd = c >= 0 ? sgend[c] : 1.0f;
#pragma unroll
            for (int cb = 0; cb < D / 2; cb += 16) {
                const int col = hf * (D / 2) + cb;
                float v[16];
                tmem_ld16(tq + TC::S + col, v);
                if (c >= 0) {
                    st_bf16x8(sb, D, c, col, v);
                    st_bf16x8(sb, D, c, col + 8, v + 8);
                }
                if (GATED) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] *= gd;
                    tmem_st16(tq + TC::S + col, v);
                }
            }
        }
        phase_sync();
        // ---------------------------------------------- F: u -= W S, O = (Q e^b) S
        if (tid == 0) {
            constexpr uint32_t idw = idesc_bf16(64, D, false, true, true);
            constexpr uint32_t ido = idesc_bf16(64, D, false, true);
#pragma unroll
            for (int s = 0; s < D / 16; ++s) {
                const uint64_t bS = mdesc(sb, D, s);
                mma_bf16(tmem + TC::U, kdesc(wt, C, 0, s), bS, idw, 1);
                mma_bf16(tmem + TC::O, kdesc(qg, C, 0, s), bS, ido, s > 0);
            }
            mma_commit(bar_mma);
        }
        if (__syncthreads_or(!mma_wait())) { failed = true; break; }
        // ---------------------------------------------- G: u tile
        {
            const int r = acc_row(64, qd, lane);
#pragma unroll
            for (int cb = 0; cb < D / 2; cb += 16) {
                const int col = hf * (D / 2) + cb;
                float v[16];
                tmem_ld16(tq + TC::U + col, v);
                if (r >= 0) {
                    st_bf16x8(ut, C, r, col, v);
                    st_bf16x8(ut, C, r, col + 8, v + 8);
                }
            }
        }
        phase_sync();
        // ---------------------------------------------- H: O += Aq u, S += K~^T u
        if (tid == 0) {
            constexpr uint32_t ido = idesc_bf16(64, D, false, true);
            constexpr uint32_t ids = idesc_bf16(D, D, true, true);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t bU = mdesc(ut, C, s);
                mma_bf16(tmem + TC::O, kdesc(aqk, 64, 0, s), bU, ido, 1);
                mma_bf16(tmem + TC::S, mdesc(kt, C, s), bU, ids, 1);
            }
            mma_commit(bar_mma);
        }
        if (__syncthreads_or(!mma_wait())) { failed = true; break; }
        // ---------------------------------------------- I: O -> global
        {
            const int r = acc_row(64, qd, lane);
            const bool valid = r >= 0 && r < len;
            __nv_bfloat16 *orow = p.o + ((int64_t)(cs + (r < 0 ? 0 : r)) * H + h) * D;
#pragma unroll
            for (int cb = 0; cb < D / 2; cb += 16) {
                const int col = hf * (D / 2) + cb;
                float v[16];
                tmem_ld16(tq + TC::O + col, v);
                if (valid) {
                    uint4 u[2];
                    __nv_bfloat162 *hv = reinterpret_cast<__nv_bfloat162 *>(u);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        hv[i] = __floats2bfloat162_rn(v[2 * i] * p.scale, v[2 * i + 1] * p.scale);
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + col);
                    dst[0] = u[0];
                    dst[1] = u[1];
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }

    if (failed && tma_pending) mbar_wait(bar_tma, tma_par, &g_tc_error, 3);
    // ---- final state
    if (p.final_S && !failed) {
        const int row = acc_row(TC::MS, qd, lane);
#pragma unroll
        for (int cb = 0; cb < D / 2; cb += 16) {
            const int col = hf * (D / 2) + cb;
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
    const size_t smem = Layout<D>::TOTAL + 1024 > 120 * 1024 ? Layout<D>::TOTAL + 1024 : 120 * 1024;
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
