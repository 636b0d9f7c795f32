// delta_bwd_channel.cu -- per-chunk gradients of the chunkwise delta rule,
// d = dk = dv in {64, 128}, bf16 I/O, with a decay per key channel (the KDA
// form of "From GPT-2 to Kimi K3, explained", section KDA / Kimi Linear), one
// per token, or none.
//
// Forward of one chunk (section DeltaNet (Parallelizing Linear Transformers
// with Delta Rule), eq. 8-10, with the decay folded in), b_r in R^dk the
// inclusive cumulative log decay inside the chunk, b_L its value at the end:
//   (X * Y)_ri = sum_c x_rc y_ic e^{b_rc - b_ic}   (i <= r)   "decayed scores"
//   A = strict_tril(diag(beta) (K * K)),  T = (I + A)^{-1}
//   Bk = diag(beta) (K o e^b),  Bv = diag(beta) V,  u~ = Bv - Bk S,  u = T u~
//   O = scale ((Q o e^b) S + (Q * K) u),  S' = Diag(e^{b_L}) S + (K o e^{b_L-b})^T u
// Given dO' = scale dO, dS' (the next chunk state's gradient) and du =
// (Q * K)^T dO' + (K o e^{b_L - b}) dS' (both from the reverse chain), and T
// from the forward pass:
//   du_T = T^T du,  dV = diag(beta) du_T,  dBk = -du_T S^T,  d(Q o e^b) = dO' S^T
//   dA = -T^T dT T^T with dT = du u~^T, i.e. dA = -strict_tril(du_T u^T)
//   dP = tril(dO' u^T),  d(K o e^{b_L - b}) = u dS'^T,  d e^{b_L} = rowsum(dS' o S)
//   dbeta_r = du_T,r . v_r + dBk_r . (K e^b)_r + sum_i dA_ri (K * K)_ri, whose
//   last term is -(1/beta_r) du_T,r . (A u)_r with A u = u~ - u
//   (since (I + A) u = u~): K * K itself is never formed.
// Through the decayed scores, with G the gradient of X * Y:
//   dX_rc += sum_{i<=r} G_ri y_ic e^{b_rc - b_ic},   db_rc += x_rc dX_rc
//   dY_ic += sum_{r>=i} G_ri x_rc e^{b_rc - b_ic},   db_ic -= y_ic dY_ic
// (G = dP for Q * K; G = diag(beta) dA for K * K).  Every term that moves
// b adds x o dx with the sign of its exponent, so with dK+ the key-gradient
// terms whose factor grows with b and dK- the others:
//   db = q o dQ + k o (dK+ - dK-),   dK = dK+ + dK-
// plus d b_L at the chunk's last row; d log alpha_t = sum_{r>=t} db_r.
//
// Decayed products without overflow.  e^{b_rc - b_ic} (i <= r, exponent <= 0)
// does not split into a row factor and a column factor over a whole chunk.
// The chunk is cut into four 16-token blocks.  For rows r of block R and
// columns i of an earlier block I:
//   e^{b_r - b_i} = e^{b_r - b_s(R)} e^{b_s(R) - b_e(I)} e^{b_e(I) - b_i}
// with s(R) = 16R - 1 (the token before R) and e(I) = 16I + 15 (the end of
// I): three factors <= 1, the middle one per (R, I) and channel.  So each
// (R, I) block of a decayed product is one 16-deep tensor-core step on
// operands scaled once per row, then scaled per output column.  The 16 x 16
// diagonal blocks (i, r in the same block) take e^{b_r - b_i} directly on
// the CUDA cores (exponent <= 0 again), whatever the decay's strength.
//
// Mapping: a persistent grid over (chunk, head) tasks, 16 warps per CTA.
// Products are warp-level bf16 mma.sync (m16n8k16, warp_mma.cuh) on bf16 shared-memory
// operands with fp32 accumulation; the three gradient accumulators dQ, dK+
// and dK- stay in registers from the first product that feeds them to the
// end of the task (warp w owns rows 16 (w / 4) .. +15 and a quarter of the
// columns).  The quantities that cancel in the beta gradient (du_T . u~ and
// du_T . u) are summed in fp32 from fp32 accumulators.

#include "common.cuh"
#include "delta_tc.h"
#include "launch.h"
#include "tc_tile.cuh"
#include "warp_mma.cuh"

namespace la {
namespace {

using tile::C;
using bf16 = __nv_bfloat16;
// Threads per CTA and CTAs per SM: at d = 128 one CTA of 16 warps per SM;
// at d = 64 two CTAs of 8 warps, so that one task's barrier waits overlap
// the other's work (114.7 KB of shared memory and 256 x 128 registers each).
// The warps tile a 64 x D output as 4 row blocks x CG column groups.
template <int D>
struct Cfg {
    static constexpr int NTH = D == 64 ? 256 : 512, CTAS = D == 64 ? 2 : 1;
    static constexpr int NW = NTH / 32, CG = NW / 4;
    static constexpr int NT = D / (8 * CG);   // n8 tiles of a warp's 16 x D/CG block
    static constexpr int RPW = 64 / NW;       // rows per warp in row-wise passes
};
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------ warp products

using wmma16::ld2;
using wmma16::PadView;
using wmma16::st2;
using wmma16::zero;

// Products on padded row-major tiles (warp_mma.cuh): one 16-deep step of a
// 16 x 16 output block, and NT n8 tiles over a k range.
template <bool TA, bool TB>
__device__ __forceinline__ void mma_step(float (&d)[2][4], const bf16 *A, int lda, const bf16 *B,
                                         int ldb, int m0, int n0, int k) {
    wmma16::mma_step<TA, TB>(d, PadView{A, lda}, PadView{B, ldb}, m0, n0, k);
}

template <int NT, bool TA, bool TB>
__device__ __forceinline__ void mma_rows(float (&d)[NT][4], const bf16 *A, int lda, const bf16 *B,
                                         int ldb, int m0, int n0, int k0, int k1) {
    wmma16::mma_rows<NT, TA, TB>(d, PadView{A, lda}, PadView{B, ldb}, m0, n0, k0, k1);
}

// 2^x for x <= 0 (every decay factor here): the hardware approximation,
// relative error ~2^-22, flushing results below the fp32 normal range to 0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 16 bytes global -> shared without a register round trip (zeros when
// !valid; src must still be a mapped address), and the wait for all of this
// thread's outstanding copies.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(wmma16::saddr(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(valid ? 16 : 0)
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)) : "memory");
}

// ------------------------------------------------------------ layout

// Shared memory (bytes).  Persistent through a task: q^, k^ (bf16), b in
// log2 units (fp32), T (bf16, the forward pass's swizzled tile), row and
// channel vectors.  One union region holds each phase's working tiles.
template <int D>
struct Lay {
    static constexpr int XS = D + 8;            // bf16 stride of a 64 x D tile
    static constexpr int XB = 64 * XS * 2;
    static constexpr int SB = D * XS * 2;       // D x D bf16 (S or dS')
    static constexpr int LS = 72;               // bf16 stride of a 64 x 64 tile
    static constexpr int LB = 64 * LS * 2;
    // fp32 stride of the decay table b and of the 64 x D gradients: D + 8
    // words puts the rows of a quad's float2 accesses on distinct banks
    static constexpr int FS = D + 8;
    static constexpr int TR = 0, Q = TR + 8192, K = Q + XB, B = K + XB;
    static constexpr int BETA = B + 64 * FS * 4;         // fp32 [64]
    static constexpr int DBETA = BETA + 256;             // fp32 [64]
    static constexpr int DBL = DBETA + 256;              // fp32 [D]: d b_L
    static constexpr int DGL = DBL + 4 * D;              // fp32 [D]: d e^{b_L}
    static constexpr int MF = DGL + 4 * D;               // fp32 [6][D]: middle factors
    static constexpr int SEG = MF + 24 * D;              // fp32 [threads / D][D]: scan totals
    static constexpr int ROW = SEG + 4 * Cfg<D>::NTH;    // fp32 [2][64]: du_T . u~, du_T . u
    static constexpr int U = ROW + 512;
    // union region, phases 2-3 (the largest)
    static constexpr int O_DO = 0, O_DU = XB, O_DUT = 2 * XB, O_UT = 3 * XB, O_BK = 4 * XB;
    // phase 5: the alpha table (fp32 [64][FS]) in the S / dS' slot
    static constexpr int O_S = 5 * XB, U_BYTES = 5 * XB + (SB > 64 * FS * 4 ? SB : 64 * FS * 4);
    static constexpr int BYTES = U + U_BYTES;
    // phase 6 (dQ, dK and db in fp32) fits inside the union region
    static_assert(3 * 64 * FS * 4 <= U_BYTES, "phase 6");
    static_assert(LB <= XB, "dP and G_A fit in a 64 x D slot");
};
static_assert(Lay<128>::BYTES <= 232448, "shared memory at d = 128");
static_assert(2 * (Lay<64>::BYTES + 1024) <= 233472, "two CTAs per SM at d = 64");

struct Params {
    const bf16 *q, *k, *v, *beta_logits, *gate_logits, *d_o;
    const int2 *table;        // [slots] {first token, length}
    const float *states;      // [slots][H][D][D] S at each chunk start
    const float *dstates;     // [slots][H][D][D] dS' of each chunk (fp32; with decay only)
    const bf16 *dstates16;    // [slots][H][D][D] dS' of each chunk (bf16)
    const bf16 *du;           // [slots][H][64][D] du of each chunk (bf16)
    const uint8_t *tiles;     // [slots][H] T of each chunk (8 KB bf16 swizzled tiles)
    float *dq, *dk, *dv, *d_beta_logits, *d_gate_logits;
    int64_t n_tasks;
    int H;
    float scale;
    unsigned flags;
};

// Inclusive prefix sums down the 64 rows of each of the D columns of
// x (fp32 [64][LDX]), in place; reverse = suffix sums.  All threads of the CTA.
template <int D, int LDX, int NTH>
__device__ __forceinline__ void column_scan(float *x, float *seg, bool reverse) {
    constexpr int NS = NTH / D, RS = 64 / NS;   // segments per column, rows per segment
    const int c = threadIdx.x % D, s = threadIdx.x / D;
    float run = 0.0f;
#pragma unroll
    for (int i = 0; i < RS; ++i) {
        const int r = reverse ? 63 - (s * RS + i) : s * RS + i;
        run += x[r * LDX + c];
        x[r * LDX + c] = run;
    }
    seg[s * D + c] = run;
    __syncthreads();
    float off = 0.0f;
    for (int t = 0; t < s; ++t) off += seg[t * D + c];
#pragma unroll
    for (int i = 0; i < RS; ++i) {
        const int r = reverse ? 63 - (s * RS + i) : s * RS + i;
        x[r * LDX + c] += off;
    }
    __syncthreads();
}

// DECAY = false (no gate): every decay factor is 1, the decayed scores are
// plain products (diagonal blocks included, on the tensor cores) and there
// is no decay gradient.
template <int D, bool DECAY>
__global__ void __launch_bounds__(Cfg<D>::NTH, Cfg<D>::CTAS) delta_bwd_channel_kernel(Params p) {
    using L = Lay<D>;
    constexpr int kNT = Cfg<D>::NTH, NW = Cfg<D>::NW, CG = Cfg<D>::CG, RPW = Cfg<D>::RPW;
    static_assert(kNT % D == 0, "a thread's 16-byte units of S and dS' lie in one row");
    constexpr int XS = L::XS, LS = L::LS, FS = L::FS;
    constexpr int CPL = D / 32;          // channels per lane in row-wise passes
    constexpr int P2 = D / 64;           // ... as pairs 2 lane + 64 m
    constexpr int NT = Cfg<D>::NT;       // n8 tiles of a warp's 16 x D/CG output block
    extern __shared__ __align__(1024) uint8_t smem[];
    bf16 *sQ = reinterpret_cast<bf16 *>(smem + L::Q), *sK = reinterpret_cast<bf16 *>(smem + L::K);
    float *sB = reinterpret_cast<float *>(smem + L::B);
    float *sBeta = reinterpret_cast<float *>(smem + L::BETA);
    float *sDBeta = reinterpret_cast<float *>(smem + L::DBETA);
    float *sDBL = reinterpret_cast<float *>(smem + L::DBL), *sDGL = reinterpret_cast<float *>(smem + L::DGL);
    float *sMF = reinterpret_cast<float *>(smem + L::MF), *sSeg = reinterpret_cast<float *>(smem + L::SEG);
    float *sRow = reinterpret_cast<float *>(smem + L::ROW);
    uint8_t *U = smem + L::U;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int H = p.H;
    const bool scalar_gate = (p.flags & kGateScalar) != 0;
    const bool silu = (p.flags & kSiluQK) != 0;
    // the additive rule: u = v (beta = 1, no delta term: W = 0, A = 0, T = I),
    // so K enters only through the scores and the state update, and there
    // is no beta gradient; wd (0 or 1) weighs every term of the delta part
    const bool additive = (p.flags & kAdditive) != 0;
    const float wd = additive ? 0.0f : 1.0f;
    // this warp's output block of a 64 x D product: rows 16R .. 16R + 15,
    // columns n0 .. n0 + D/CG - 1; of a 64 x 64 product: columns 64/CG cq ..
    const int R = w / CG, cq = w % CG, n0 = cq * (D / CG);
    const int r0 = 16 * R + g, r1 = r0 + 8;   // this lane's two output rows

    // inputs of task nt into L2 (one 128-byte line per request): the token
    // rows of q, k, v, dO and per-channel gate logits, then S, dS', du and T
    auto prefetch_task = [&](int64_t nt) {
        if (nt >= p.n_tasks) return;
        const int64_t ns = nt / H;
        const int nh = (int)(nt % H);
        const int2 e = p.table[ns];
        if (e.y <= 0 || e.y > 64) return;
        constexpr int LPR = D * 2 / 128;   // lines per bf16 row
        const bool pg = p.gate_logits && !scalar_gate;
        for (int u = tid; u < 64 * LPR * 5; u += kNT) {
            const int which = u / (64 * LPR), r = (u / LPR) % 64, l = u % LPR;
            if (r >= e.y || (which == 4 && !pg)) continue;
            const bf16 *base = which == 0 ? p.q : which == 1 ? p.k : which == 2 ? p.v
                             : which == 3 ? p.d_o : p.gate_logits;
            prefetch_l2(base + ((int64_t)(e.x + r) * H + nh) * D + l * 64);
        }
        const int64_t so = (ns * H + nh) * (int64_t)(D * D), uo = (ns * H + nh) * (int64_t)(64 * D);
        constexpr int LSS = D * D / 32, LU = 64 * D / 64, LT = 8192 / 128;   // lines
        for (int u = tid; u < 2 * LSS + LU + LT; u += kNT) {
            const void *q = u < LSS ? (const void *)(p.states + so + u * 32)
                          : u < 2 * LSS ? (const void *)(p.dstates + so + (u - LSS) * 32)
                          : u < 2 * LSS + LU ? (const void *)(p.du + uo + (u - 2 * LSS) * 64)
                                             : (const void *)(p.tiles + (ns * H + nh) * (int64_t)8192 +
                                                              (u - 2 * LSS - LU) * 128);
            prefetch_l2(q);
        }
    };
    prefetch_task(blockIdx.x);

    for (int64_t task = blockIdx.x; task < p.n_tasks; task += gridDim.x) {
        const int64_t slot = task / H;
        const int h = (int)(task % H);
        const int2 te = p.table[slot];
        const int t0 = te.x, len = te.y;
        if (len <= 0) continue;
        auto tok = [&](int r) { return ((int64_t)(t0 + r) * H + h); };
        bf16 *sDO = reinterpret_cast<bf16 *>(U + L::O_DO), *sDU = reinterpret_cast<bf16 *>(U + L::O_DU);
        bf16 *sV = reinterpret_cast<bf16 *>(U + L::O_UT);   // V, until u~ replaces it in place

        // The benchmark's bf16 operands go straight to shared memory by async
        // copies, in flight through phase 0: T (8 KB, one 16-byte unit per
        // thread), dO and V (rows past the end zero) and du, 64 x D each.
#pragma unroll
        for (int k = 0; k < 512 / kNT; ++k) {
            const int u = tid + k * kNT;
            cp_async16(smem + L::TR + u * 16, p.tiles + (slot * H + h) * (int64_t)8192 + u * 16, true);
        }
        {
            // (du by 16-byte units, unit e = row e % 64 of column group e / 64)
            const bf16 *gdu = p.du + (slot * H + h) * (int64_t)(64 * D);
#pragma unroll
            for (int k = 0; k < 64 * D / 8 / kNT; ++k) {
                const int e = tid + k * kNT, r = e / (D / 8), c = 8 * (e % (D / 8));
                cp_async16(sDO + r * XS + c, p.d_o + tok(r < len ? r : 0) * D + c, r < len);
                cp_async16(sV + r * XS + c, p.v + tok(r < len ? r : 0) * D + c, r < len);
                cp_async16(sDU + (e % 64) * XS + 8 * (e / 64), gdu + 8 * e, true);
            }
        }

        // ---- 0. q^, k^ (silu, L2 norm), beta, log2 alpha; b = prefix sums.
        // Lanes take channel pairs 2 lane + 64 m; the warp's four rows are
        // loaded first (bf16 pairs kept packed).
        __nv_bfloat162 rq[RPW][P2], rk[RPW][P2], rg[RPW][P2];
        float rgs[RPW], rbl[RPW];
        const __nv_bfloat162 z2 = __floats2bfloat162_rn(0.0f, 0.0f);
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
            const int r = w + NW * rr;
            const bool ok = r < len;
            const int64_t o = tok(ok ? r : 0) * D;
            using bfp = const __nv_bfloat162 *;
#pragma unroll
            for (int m = 0; m < P2; ++m) {
                const int c = 2 * lane + 64 * m;
                rq[rr][m] = ok ? *reinterpret_cast<bfp>(p.q + o + c) : z2;
                rk[rr][m] = ok ? *reinterpret_cast<bfp>(p.k + o + c) : z2;
                rg[rr][m] = (DECAY && ok && !scalar_gate) ? *reinterpret_cast<bfp>(p.gate_logits + o + c) : z2;
            }
            rgs[rr] = (DECAY && ok && scalar_gate) ? __bfloat162float(p.gate_logits[tok(r)]) : 0.0f;
            rbl[rr] = (ok && !additive) ? __bfloat162float(p.beta_logits[tok(r)]) : 0.0f;
        }
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
            const int r = w + NW * rr;
            const bool ok = r < len;
            float xq[CPL], xk[CPL], lg[CPL];
            const float gs = (DECAY && ok && scalar_gate) ? log_decay_f(rgs[rr]) : 0.0f;
#pragma unroll
            for (int m = 0; m < P2; ++m) {
                const float2 a = __bfloat1622float2(rq[rr][m]), b = __bfloat1622float2(rk[rr][m]);
                xq[2 * m] = a.x; xq[2 * m + 1] = a.y;
                xk[2 * m] = b.x; xk[2 * m + 1] = b.y;
                float2 gl = make_float2(gs, gs);
                if (DECAY && ok && !scalar_gate) {
                    const float2 gg = __bfloat1622float2(rg[rr][m]);
                    gl = make_float2(log_decay_f(gg.x), log_decay_f(gg.y));
                }
                lg[2 * m] = gl.x * kLog2e;
                lg[2 * m + 1] = gl.y * kLog2e;
            }
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                float *x = which ? xk : xq;
                float ss = 0.0f;
#pragma unroll
                for (int m = 0; m < CPL; ++m) {
                    if (silu) x[m] = silu_f(x[m]);
                    ss += x[m] * x[m];
                }
                const bool norm = (p.flags & (which ? kL2NormK : kL2NormQ)) != 0;
                const float inv = norm ? 1.0f / fmaxf(sqrtf(warp_sum(ss)), 1e-12f) : 1.0f;
                bf16 *dst = (which ? sK : sQ) + r * XS;
#pragma unroll
                for (int m = 0; m < P2; ++m)
                    st2(dst + 2 * lane + 64 * m, x[2 * m] * inv, x[2 * m + 1] * inv);
            }
#pragma unroll
            for (int m = 0; m < P2; ++m)
                *reinterpret_cast<float2 *>(sB + r * FS + 2 * lane + 64 * m) = make_float2(lg[2 * m], lg[2 * m + 1]);
            if (lane == 0) sBeta[r] = ok ? (additive ? 1.0f : sigmoid_f(rbl[rr])) : 0.0f;
        }
        if (tid < 64) sDBeta[tid] = 0.0f;
        if (tid < D) sDBL[tid] = sDGL[tid] = 0.0f;
        __syncthreads();
        if constexpr (DECAY) column_scan<D, FS, kNT>(sB, sSeg, false);
        prefetch_task(task + gridDim.x);
        // sB[r][c] = b_rc / ln 2 from here on; b at the token before block R
        auto bs = [&](int Rb, int c) { return Rb == 0 ? 0.0f : sB[(16 * Rb - 1) * FS + c]; };
        auto b2at = [&](int r, int c) { return *reinterpret_cast<const float2 *>(sB + r * FS + c); };
        // 2^x of a decay exponent; exactly 1 without decay (its loads then go unused)
        auto ex2d = [&](float x) { if constexpr (DECAY) return ex2(x); else return 1.0f; };

        // ---- 1. T = (I + A)^{-1} from the forward pass (bf16, one 64-row
        // swizzled tile, already on its way)
        const wmma16::RsView tv{smem + L::TR, 64, 0};

        // ---- 2. S and Bk in (dO, du by the async copies); du_T = T^T du;
        // u~, d(Q e^b), dBk
        bf16 *sDUT = reinterpret_cast<bf16 *>(U + L::O_DUT), *sUT = reinterpret_cast<bf16 *>(U + L::O_UT);
        bf16 *sBK = reinterpret_cast<bf16 *>(U + L::O_BK), *sS = reinterpret_cast<bf16 *>(U + L::O_S);
        const float *gS = p.states + (slot * H + h) * (int64_t)(D * D);
        const float *gDS = p.dstates + (slot * H + h) * (int64_t)(D * D);
        {
            // S: every load of this thread first, then the bf16 stores (S by
            // 16-byte units: unit e is row e % D of column group e / D)
            constexpr int NS = D * D / 4 / kNT;
            float4 sv[NS];
#pragma unroll
            for (int k = 0; k < NS; ++k) sv[k] = reinterpret_cast<const float4 *>(gS)[tid + k * kNT];
            for (int e = tid; e < 64 * D / 4; e += kNT) {
                const int r = e / (D / 4), c = 4 * (e % (D / 4));
                const float be = wd * sBeta[r];   // Bk = 0 for the additive rule
                const float2 k0 = ld2(sK + r * XS + c), k1 = ld2(sK + r * XS + c + 2);
                const float4 b = *reinterpret_cast<const float4 *>(sB + r * FS + c);
                st2(sBK + r * XS + c, be * k0.x * ex2d(b.x), be * k0.y * ex2d(b.y));
                st2(sBK + r * XS + c + 2, be * k1.x * ex2d(b.z), be * k1.y * ex2d(b.w));
            }
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                const int e = tid + k * kNT, r = e % D, c = 4 * (e / D);
                st2(sS + r * XS + c, sv[k].x, sv[k].y);
                st2(sS + r * XS + c + 2, sv[k].z, sv[k].w);
            }
        }
        cp_async_wait_all();   // T, dO, du in (made visible to all by the barrier below)
        if (tid < 64) sRow[tid] = sRow[64 + tid] = 0.0f;
        __syncthreads();
        float aQ[NT][4], aKp[NT][4], aKm[NT][4];   // dQ, dK+, dK- (see the file header)
        zero(aQ);
        zero(aKp);
        zero(aKm);
        // per-row partial sums of this lane's two rows, reduced over the quad and
        // the four column warps of the row block into v[r]
        auto add_rows = [&](float *v, float s0, float s1) {
            s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
            s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
            s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
            s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
            if (t == 0) {
                atomicAdd(&v[r0], s0);
                atomicAdd(&v[r1], s1);
            }
        };
        // du_T = T^T du, kept in fp32 until u is known (T lower: rows r >= 16R
        // of T reach rows of block R)
        float dut[NT][4];
        zero(dut);
        wmma16::mma_rows<NT, true, false>(dut, tv, PadView{sDU, XS}, 16 * R, n0, 16 * R, 64);
        {
            float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int c = n0 + 8 * j + 2 * t;
                st2(sDUT + r0 * XS + c, dut[j][0], dut[j][1]);
                st2(sDUT + r1 * XS + c, dut[j][2], dut[j][3]);
                // dV = beta du_T; dbeta += du_T . v
                if (r0 < len) {
                    const float2 v = ld2(sV + r0 * XS + c);
                    s0 += dut[j][0] * v.x + dut[j][1] * v.y;
                    *reinterpret_cast<float2 *>(p.dv + tok(r0) * D + c) =
                        make_float2(sBeta[r0] * dut[j][0], sBeta[r0] * dut[j][1]);
                }
                if (r1 < len) {
                    const float2 v = ld2(sV + r1 * XS + c);
                    s1 += dut[j][2] * v.x + dut[j][3] * v.y;
                    *reinterpret_cast<float2 *>(p.dv + tok(r1) * D + c) =
                        make_float2(sBeta[r1] * dut[j][2], sBeta[r1] * dut[j][3]);
                }
            }
            add_rows(sDBeta, s0, s1);
        }
        __syncthreads();
        {
            // u~ = beta V - Bk S; sRow[r] = sum_j du_T u~ (fp32)
            float d[NT][4];
            zero(d);
            mma_rows<NT, false, false>(d, sBK, XS, sS, XS, 16 * R, n0, 0, D);
            float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int c = n0 + 8 * j + 2 * t;
                const float2 v0 = ld2(sV + r0 * XS + c), v1 = ld2(sV + r1 * XS + c);   // (zero past the end)
                const float u00 = sBeta[r0] * v0.x - d[j][0], u01 = sBeta[r0] * v0.y - d[j][1];
                const float u10 = sBeta[r1] * v1.x - d[j][2], u11 = sBeta[r1] * v1.y - d[j][3];
                st2(sUT + r0 * XS + c, u00, u01);
                st2(sUT + r1 * XS + c, u10, u11);
                s0 += dut[j][0] * u00 + dut[j][1] * u01;
                s1 += dut[j][2] * u10 + dut[j][3] * u11;
            }
            add_rows(sRow, s0, s1);
            // d(Q e^b) = scale dO S^T: dQ gets e^b times it
            zero(d);
            mma_rows<NT, false, true>(d, sDO, XS, sS, XS, 16 * R, n0, 0, D);
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const float2 b = b2at(r0 + 8 * hr, n0 + 8 * j + 2 * t);
                    aQ[j][2 * hr] = p.scale * ex2d(b.x) * d[j][2 * hr];
                    aQ[j][2 * hr + 1] = p.scale * ex2d(b.y) * d[j][2 * hr + 1];
                }
            // dBk = -du_T S^T: dK+ gets beta e^b dBk; dbeta += dBk . (K e^b)
            zero(d);
            mma_rows<NT, false, true>(d, sDUT, XS, sS, XS, 16 * R, n0, 0, D);
            s0 = s1 = 0.0f;
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int r = r0 + 8 * hr, c = n0 + 8 * j + 2 * t;
                    const float2 b = b2at(r, c), kv = ld2(sK + r * XS + c);
                    const float e0 = ex2d(b.x), e1 = ex2d(b.y);
                    const float dbk0 = -d[j][2 * hr], dbk1 = -d[j][2 * hr + 1];
                    aKp[j][2 * hr] = wd * sBeta[r] * e0 * dbk0;
                    aKp[j][2 * hr + 1] = wd * sBeta[r] * e1 * dbk1;
                    const float sum = dbk0 * kv.x * e0 + dbk1 * kv.y * e1;
                    if (hr) s1 += sum;
                    else s0 += sum;
                }
            add_rows(sDBeta, s0, s1);
        }
        __syncthreads();

        // ---- 3. u = T u~; the A part of dbeta; dA = -strict_tril(du_T u^T)
        // (so G_A = diag(beta) dA) and dP = scale tril(dO u^T); dS' in:
        // d(K e^{b_L - b}) = u dS'^T, d e^{b_L} = rowsum(dS' o S)
        bf16 *sU = sBK;                                             // 64 x D
        bf16 *sGP = sDU;                                            // 64 x 64
        bf16 *sGA = sUT;                                            // 64 x 64, after u
        if constexpr (!DECAY) {
            // dS' (bf16, from the chain) into the S slot, in flight through 3a
            // and 3b (with decay it is staged from fp32 in 3b, beside S)
            const bf16 *gds16 = p.dstates16 + (slot * H + h) * (int64_t)(D * D);
#pragma unroll
            for (int k = 0; k < D * D / 8 / kNT; ++k) {
                const int e = tid + k * kNT;   // row e % D of column group e / D
                cp_async16(sS + (e % D) * XS + 8 * (e / D), gds16 + 8 * e, true);
            }
        }
        {
            float d[NT][4];
            zero(d);
            wmma16::mma_rows<NT, false, false>(d, tv, PadView{sUT, XS}, 16 * R, n0, 0, 16 * R + 16);
            float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int c = n0 + 8 * j + 2 * t;
                st2(sU + r0 * XS + c, d[j][0], d[j][1]);
                st2(sU + r1 * XS + c, d[j][2], d[j][3]);
                s0 += dut[j][0] * d[j][0] + dut[j][1] * d[j][1];
                s1 += dut[j][2] * d[j][2] + dut[j][3] * d[j][3];
            }
            add_rows(sRow + 64, s0, s1);
        }
        __syncthreads();
        // dbeta_r += sum_i dA_ri (K * K)_ri = -(1/beta_r) sum_j du_T_rj (A u)_rj,
        // and A u = u~ - u because (I + A) u = u~
        // (a beta that underflowed to 0 leaves the row's beta-logit gradient 0 anyway)
        if (tid < len && sBeta[tid] > 0.0f && !additive)
            sDBeta[tid] -= (sRow[tid] - sRow[64 + tid]) / sBeta[tid];
        {
            // 64 x 64 products: this warp's columns in 16-wide steps
#pragma unroll
            for (int jp = 0; jp < 64 / (16 * CG); ++jp) {
                const int c0 = (64 / CG) * cq + 16 * jp;
                float e2[2][4] = {}, f2[2][4] = {};
                if (c0 <= 16 * R)   // blocks right of the diagonal block are zero
                    for (int k = 0; k < D; k += 16) {
                        mma_step<false, true>(e2, sDO, XS, sU, XS, 16 * R, c0, k);
                        mma_step<false, true>(f2, sDUT, XS, sU, XS, 16 * R, c0, k);
                    }
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int i = c0 + 8 * j + 2 * t;
                    const float s = p.scale, b0 = -wd * sBeta[r0], b1 = -wd * sBeta[r1];
                    st2(sGP + r0 * LS + i, i <= r0 ? s * e2[j][0] : 0.0f, i + 1 <= r0 ? s * e2[j][1] : 0.0f);
                    st2(sGP + r1 * LS + i, i <= r1 ? s * e2[j][2] : 0.0f, i + 1 <= r1 ? s * e2[j][3] : 0.0f);
                    st2(sGA + r0 * LS + i, i < r0 ? b0 * f2[j][0] : 0.0f, i + 1 < r0 ? b0 * f2[j][1] : 0.0f);
                    st2(sGA + r1 * LS + i, i < r1 ? b1 * f2[j][2] : 0.0f, i + 1 < r1 ? b1 * f2[j][3] : 0.0f);
                }
            }
            if constexpr (DECAY) {
                // dS' in, and d e^{b_L}_c = sum_j dS'_cj S_cj.  Both come by
                // 16-byte units (unit u: row u % D, columns 4 (u / D) ..): the
                // thread's units all lie in row tid % D (the thread count is a
                // multiple of D), whose kNT / D threads add their sums
                float acc = 0.0f;
                for (int u = tid; u < D * D / 4; u += kNT) {
                    const int c = u % D, j = 4 * (u / D);
                    const float4 ds = reinterpret_cast<const float4 *>(gDS)[u];
                    const float4 sv = reinterpret_cast<const float4 *>(gS)[u];
                    acc += ds.x * sv.x + ds.y * sv.y + ds.z * sv.z + ds.w * sv.w;
                    st2(sS + c * XS + j, ds.x, ds.y);
                    st2(sS + c * XS + j + 2, ds.z, ds.w);
                }
                atomicAdd(&sDGL[tid % D], acc);
            }
        }
        cp_async_wait_all();   // dS' in (made visible to all by the barrier below)
        __syncthreads();
        {
            // K~ = K e^{b_L - b}: dK- gets e^{b_L - b} u dS'^T; d b_L += sum_i k~ (u dS'^T)
            float d[NT][4];
            zero(d);
            mma_rows<NT, false, true>(d, sU, XS, sS, XS, 16 * R, n0, 0, D);
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int c = n0 + 8 * j + 2 * t;
                const float2 bl = b2at(63, c), b0 = b2at(r0, c), b1 = b2at(r1, c);
                const float2 k0 = ld2(sK + r0 * XS + c), k1 = ld2(sK + r1 * XS + c);
                aKm[j][0] = ex2d(bl.x - b0.x) * d[j][0];
                aKm[j][1] = ex2d(bl.y - b0.y) * d[j][1];
                aKm[j][2] = ex2d(bl.x - b1.x) * d[j][2];
                aKm[j][3] = ex2d(bl.y - b1.y) * d[j][3];
                if constexpr (!DECAY) continue;   // no d b_L without a gate
                float sx = k0.x * aKm[j][0] + k1.x * aKm[j][2];
                float sy = k0.y * aKm[j][1] + k1.y * aKm[j][3];
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    sx += __shfl_xor_sync(0xffffffffu, sx, o);
                    sy += __shfl_xor_sync(0xffffffffu, sy, o);
                }
                if (g == 0) {
                    atomicAdd(&sDBL[c], sx);
                    atomicAdd(&sDBL[c + 1], sy);
                }
            }
        }
        __syncthreads();

        // ---- 5. through the decayed scores Q * K (gradient dP) and K * K
        // (gradient G_A).  Operands scaled once per row: K_e = k e^{b_e(I) - b}
        // (to the end of the row's block), Q_s, K_s = (q, k) e^{b - b_s(R)} (from
        // the start of the row's block); middle factors m(R, I) = e^{b_s(R) - b_e(I)}.
        // (without decay they are K and Q themselves, and every factor is 1)
        bf16 *sKe = DECAY ? reinterpret_cast<bf16 *>(U + L::O_DUT) : sK;
        bf16 *sQs = DECAY ? reinterpret_cast<bf16 *>(U + L::O_DO) : sQ;
        bf16 *sKs2 = DECAY ? reinterpret_cast<bf16 *>(U + L::O_BK) : sK;
        float *sAl = reinterpret_cast<float *>(U + L::O_S);   // alpha_t = e^{b_t - b_(t-1)}, fp32 [64][FS]
        for (int e = tid; e < (DECAY ? 64 * D / 2 : 0); e += kNT) {
            const int r = e / (D / 2), c = 2 * (e % (D / 2)), Rb = r >> 4;
            const float2 kv = ld2(sK + r * XS + c), qv = ld2(sQ + r * XS + c);
            const float2 b = b2at(r, c), be = b2at(16 * Rb + 15, c);
            const float f0 = ex2(b.x - bs(Rb, c)), f1 = ex2(b.y - bs(Rb, c + 1));
            st2(sKe + r * XS + c, kv.x * ex2(be.x - b.x), kv.y * ex2(be.y - b.y));
            st2(sQs + r * XS + c, qv.x * f0, qv.y * f1);
            st2(sKs2 + r * XS + c, kv.x * f0, kv.y * f1);
            const float2 bp = r > 0 ? b2at(r - 1, c) : make_float2(0.0f, 0.0f);
            *reinterpret_cast<float2 *>(sAl + r * FS + c) = make_float2(ex2(b.x - bp.x), ex2(b.y - bp.y));
        }
        for (int e = tid; e < (DECAY ? 6 * D : 0); e += kNT) {
            const int pi = e / D, c = e % D;
            const int Rb = pi < 1 ? 1 : pi < 3 ? 2 : 3, Ib = pi - Rb * (Rb - 1) / 2;
            sMF[pi * D + c] = ex2(bs(Rb, c) - sB[(16 * Ib + 15) * FS + c]);
        }
        __syncthreads();
        auto mf = [&](int Rb, int Ib, int c) { return sMF[(Rb * (Rb - 1) / 2 + Ib) * D + c]; };
        {
            // off-diagonal blocks (without decay also the diagonal ones, as
            // plain products), two n8 tiles at a time.  Rows of block R:
            //   dQ  += e^{b_r - b_s(R)} sum_{I<R} m(R,I) (dP[R,I] K_e[I])
            //   dK+ += e^{b_r - b_s(R)} sum_{I<R} m(R,I) (G_A[R,I] K_e[I])
            // rows of block I = R of this warp:
            //   dK- += e^{b_e(I) - b_i} sum_{R'>I} m(R',I) (dP[R',I]^T Q_s[R'] + G_A[R',I]^T K_s[R'])
#pragma unroll
            for (int j = 0; j < NT; j += 2) {
                const int nb = n0 + 8 * j;
                float sq[2][4] = {}, sa[2][4] = {}, sm2[2][4] = {};
                for (int Ib = 0; Ib < R + (DECAY ? 0 : 1); ++Ib) {
                    if constexpr (DECAY) {
                        float tq[2][4] = {}, ta[2][4] = {};
                        mma_step<false, false>(tq, sGP, LS, sKe, XS, 16 * R, nb, 16 * Ib);
                        mma_step<false, false>(ta, sGA, LS, sKe, XS, 16 * R, nb, 16 * Ib);
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj)
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float m = mf(R, Ib, nb + 8 * jj + 2 * t + (e & 1));
                                sq[jj][e] = fmaf(m, tq[jj][e], sq[jj][e]);
                                sa[jj][e] = fmaf(m, ta[jj][e], sa[jj][e]);
                            }
                    } else {
                        mma_step<false, false>(sq, sGP, LS, sKe, XS, 16 * R, nb, 16 * Ib);
                        mma_step<false, false>(sa, sGA, LS, sKe, XS, 16 * R, nb, 16 * Ib);
                    }
                }
                for (int Rb = R + (DECAY ? 1 : 0); Rb < 4; ++Rb) {
                    if constexpr (DECAY) {
                        float tb[2][4] = {};
                        mma_step<true, false>(tb, sGP, LS, sQs, XS, 16 * R, nb, 16 * Rb);
                        mma_step<true, false>(tb, sGA, LS, sKs2, XS, 16 * R, nb, 16 * Rb);
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj)
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float m = mf(Rb, R, nb + 8 * jj + 2 * t + (e & 1));
                                sm2[jj][e] = fmaf(m, tb[jj][e], sm2[jj][e]);
                            }
                    } else {
                        mma_step<true, false>(sm2, sGP, LS, sQs, XS, 16 * R, nb, 16 * Rb);
                        mma_step<true, false>(sm2, sGA, LS, sKs2, XS, 16 * R, nb, 16 * Rb);
                    }
                }
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int c = nb + 8 * jj + 2 * t;
                    const float2 bsr = R == 0 ? make_float2(0.0f, 0.0f) : b2at(16 * R - 1, c);
                    const float2 ber = b2at(16 * R + 15, c);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 b = b2at(r0 + 8 * (e >> 1), c);
                        const float bb = (e & 1) ? b.y : b.x;
                        const float fr = ex2d(bb - ((e & 1) ? bsr.y : bsr.x));
                        const float fc = ex2d(((e & 1) ? ber.y : ber.x) - bb);
                        aQ[j + jj][e] = fmaf(fr, sq[jj][e], aQ[j + jj][e]);
                        aKp[j + jj][e] = fmaf(fr, sa[jj][e], aKp[j + jj][e]);
                        aKm[j + jj][e] = fmaf(fc, sm2[jj][e], aKm[j + jj][e]);
                    }
                }
            }
        }
        if constexpr (DECAY) {
            // diagonal blocks exactly, e^{b_r - b_i} as a running product of the
            // per-token decays alpha_t = e^{b_t - b_(t-1)} (all <= 1):
            //   dQ_rc  += sum_{16R <= i <= r} dP_ri k_ic e^{b_rc - b_ic}
            //   dK+_rc += sum_{16R <= i <  r} G_A,ri k_ic e^{b_rc - b_ic}
            //   dK-_ic += sum_{i <= r < 16R+16} (dP_ri q_rc + G_A,ri k_rc) e^{b_rc - b_ic}
            // (per lane 34 (row, partner) steps whatever g)
            auto al2 = [&](int r, int c) { return *reinterpret_cast<const float2 *>(sAl + r * FS + c); };
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int r = r0 + 8 * hr;
                float f[2 * NT];   // e^{b_r - b_i} at the current partner i, i from r down
#pragma unroll
                for (int j = 0; j < 2 * NT; ++j) f[j] = 1.0f;
                for (int i = r; i >= 16 * R; --i) {
                    const float gp = __bfloat162float(sGP[r * LS + i]);
                    const float ga = __bfloat162float(sGA[r * LS + i]);
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        const int c = n0 + 8 * j + 2 * t;
                        const float2 kv = ld2(sK + i * XS + c), al = al2(i, c);
                        const float w0 = kv.x * f[2 * j], w1 = kv.y * f[2 * j + 1];
                        aQ[j][2 * hr] = fmaf(gp, w0, aQ[j][2 * hr]);
                        aQ[j][2 * hr + 1] = fmaf(gp, w1, aQ[j][2 * hr + 1]);
                        aKp[j][2 * hr] = fmaf(ga, w0, aKp[j][2 * hr]);
                        aKp[j][2 * hr + 1] = fmaf(ga, w1, aKp[j][2 * hr + 1]);
                        f[2 * j] *= al.x;   // e^{b_r - b_(i-1)}
                        f[2 * j + 1] *= al.y;
                    }
                }
#pragma unroll
                for (int j = 0; j < 2 * NT; ++j) f[j] = 1.0f;   // e^{b_rr - b_r}, rr from r up
                for (int rr = r; rr < 16 * R + 16; ++rr) {
                    const float gp = __bfloat162float(sGP[rr * LS + r]);
                    const float ga = __bfloat162float(sGA[rr * LS + r]);
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        const int c = n0 + 8 * j + 2 * t;
                        const float2 qv = ld2(sQ + rr * XS + c), kv = ld2(sK + rr * XS + c);
                        if (rr > r) {
                            const float2 al = al2(rr, c);
                            f[2 * j] *= al.x;
                            f[2 * j + 1] *= al.y;
                        }
                        aKm[j][2 * hr] = fmaf(fmaf(gp, qv.x, ga * kv.x), f[2 * j], aKm[j][2 * hr]);
                        aKm[j][2 * hr + 1] = fmaf(fmaf(gp, qv.y, ga * kv.y), f[2 * j + 1], aKm[j][2 * hr + 1]);
                    }
                }
            }
        }
        __syncthreads();

        // ---- 6. dQ, dK = dK+ + dK- and db = q dQ + k (dK+ - dK-) to shared
        // memory; outputs through the prologue; d log alpha by suffix sums
        float *sFQ = reinterpret_cast<float *>(U), *sFK = sFQ + 64 * FS, *sDB = sFK + 64 * FS;
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int r = r0 + 8 * hr, c = n0 + 8 * j + 2 * t;
                const float2 qv = ld2(sQ + r * XS + c), kv = ld2(sK + r * XS + c);
                const float dq0 = aQ[j][2 * hr], dq1 = aQ[j][2 * hr + 1];
                const float p0 = aKp[j][2 * hr], p1 = aKp[j][2 * hr + 1];
                const float m0 = aKm[j][2 * hr], m1 = aKm[j][2 * hr + 1];
                *reinterpret_cast<float2 *>(sFQ + r * FS + c) = make_float2(dq0, dq1);
                *reinterpret_cast<float2 *>(sFK + r * FS + c) = make_float2(p0 + m0, p1 + m1);
                if constexpr (DECAY)
                    *reinterpret_cast<float2 *>(sDB + r * FS + c) =
                        make_float2(qv.x * dq0 + kv.x * (p0 - m0), qv.y * dq1 + kv.y * (p1 - m1));
            }
        __syncthreads();
        if (DECAY && tid < D)
            sDB[63 * FS + tid] += sDBL[tid] + ex2(sB[63 * FS + tid]) * sDGL[tid];
        __nv_bfloat162 xr[RPW][2][P2];   // raw q, k of the warp's rows, loaded first
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
            const int r = w + NW * rr;
#pragma unroll
            for (int which = 0; which < 2; ++which)
#pragma unroll
                for (int m = 0; m < P2; ++m)
                    xr[rr][which][m] = r < len ? *reinterpret_cast<const __nv_bfloat162 *>(
                                                     (which ? p.k : p.q) + tok(r) * D + 2 * lane + 64 * m)
                                               : __floats2bfloat162_rn(0.0f, 0.0f);
        }
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
            const int r = w + NW * rr;
            if (r >= len) continue;
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const float *src = (which ? sFK : sFQ) + r * FS;
                float x[CPL], d[CPL];
#pragma unroll
                for (int m = 0; m < P2; ++m) {
                    const int c = 2 * lane + 64 * m;
                    const float2 xv = __bfloat1622float2(xr[rr][which][m]);
                    const float2 dv = *reinterpret_cast<const float2 *>(src + c);
                    x[2 * m] = xv.x; x[2 * m + 1] = xv.y;
                    d[2 * m] = dv.x; d[2 * m + 1] = dv.y;
                }
                prep_backward<CPL>(x, d, silu, (p.flags & (which ? kL2NormK : kL2NormQ)) != 0);
                float *out = (which ? p.dk : p.dq) + tok(r) * D;
#pragma unroll
                for (int m = 0; m < P2; ++m)
                    *reinterpret_cast<float2 *>(out + 2 * lane + 64 * m) = make_float2(d[2 * m], d[2 * m + 1]);
            }
        }
        if (tid < len) {
            const float be = sBeta[tid];
            p.d_beta_logits[tok(tid)] = additive ? 0.0f : sDBeta[tid] * be * (1.0f - be);
        }
        if constexpr (DECAY) {
            __syncthreads();
            column_scan<D, FS, kNT>(sDB, sSeg, true);   // d log alpha_t = sum_{r >= t} db_r
            // log alpha = -softplus(x): dx = -d(log alpha) sigmoid(x)
            if (!scalar_gate) {
                constexpr int NG = 64 * D / 2 / kNT;   // bf16 pairs per thread, loaded first
                __nv_bfloat162 gg[NG];
#pragma unroll
                for (int k = 0; k < NG; ++k) {
                    const int e = tid + k * kNT, r = e / (D / 2), c = 2 * (e % (D / 2));
                    gg[k] = r < len ? *reinterpret_cast<const __nv_bfloat162 *>(p.gate_logits + tok(r) * D + c)
                                    : __floats2bfloat162_rn(0.0f, 0.0f);
                }
#pragma unroll
                for (int k = 0; k < NG; ++k) {
                    const int e = tid + k * kNT, r = e / (D / 2), c = 2 * (e % (D / 2));
                    if (r >= len) continue;
                    const float2 gv = __bfloat1622float2(gg[k]);
                    const float2 dl = *reinterpret_cast<const float2 *>(sDB + r * FS + c);
                    *reinterpret_cast<float2 *>(p.d_gate_logits + tok(r) * D + c) =
                        make_float2(-dl.x * sigmoid_f(gv.x), -dl.y * sigmoid_f(gv.y));
                }
            } else {
                for (int r = w; r < len; r += NW) {
                    float s = 0.0f;
#pragma unroll
                    for (int m = 0; m < P2; ++m) {
                        const float2 dl = *reinterpret_cast<const float2 *>(sDB + r * FS + 2 * lane + 64 * m);
                        s += dl.x + dl.y;
                    }
                    s = warp_sum(s);
                    if (lane == 0)
                        p.d_gate_logits[tok(r)] = -s * sigmoid_f(__bfloat162float(p.gate_logits[tok(r)]));
                }
            }
        }
        __syncthreads();
    }
}

template <int D, bool DECAY>
cudaError_t launch_d(const Params &p, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    constexpr int bytes = Lay<D>::BYTES;
    if ((e = cudaFuncSetAttribute(delta_bwd_channel_kernel<D, DECAY>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess)
        return e;
    const int64_t slots = (int64_t)sms * Cfg<D>::CTAS;
    const int64_t grid = p.n_tasks < slots ? p.n_tasks : slots;
    if (grid > 0) {
        delta_bwd_channel_kernel<D, DECAY><<<(unsigned)grid, Cfg<D>::NTH, bytes, s>>>(p);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace

cudaError_t launch_delta_bwd_channel(const BwdChannelArgs &a, cudaStream_t s) {
    Params p{static_cast<const bf16 *>(a.q), static_cast<const bf16 *>(a.k),
             static_cast<const bf16 *>(a.v), static_cast<const bf16 *>(a.beta_logits),
             static_cast<const bf16 *>(a.gate_logits), static_cast<const bf16 *>(a.d_o),
             a.table, a.states, a.dstates, a.dstates16, a.du, a.tiles, a.dq, a.dk, a.dv, a.d_beta_logits,
             a.d_gate_logits, a.n_tasks, a.H, a.scale, a.flags};
    const bool decay = a.gate_logits != nullptr;
    if (a.D == 64) return decay ? launch_d<64, true>(p, s) : launch_d<64, false>(p, s);
    if (a.D == 128) return decay ? launch_d<128, true>(p, s) : launch_d<128, false>(p, s);
    return cudaErrorInvalidValue;
}

}  // namespace la
