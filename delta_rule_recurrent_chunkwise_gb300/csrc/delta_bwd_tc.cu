// delta_bwd_tc.cu -- chunkwise backward pass of the delta rule (bf16 I/O,
// dk = dv in {64, 128}, any gate): the forward pass with records, the
// reverse chain over chunks, and the per-chunk gradients for d = 64 without
// a per-channel decay (the other per-chunk kernel, delta_bwd_channel.cu,
// takes d = 128 and the per-channel decay).
//
// The page ("From GPT-2 to Kimi K3, explained", section DeltaNet
// (Parallelizing Linear Transformers with Delta Rule), eq. 8-10) gives the
// chunkwise forward pass; this is its derivative, chunk by chunk.  Per chunk
// of C = 64 tokens, with b_r the cumulative log decay inside the chunk
// (b = 0 without gate), G[r][i] = e^{b_r - b_i} for i <= r, the forward is
//   A = strict_tril(diag(beta) (K K^T o G)),  T = (I + A)^{-1}
//   W = T diag(beta e^b) K,  U = T diag(beta) V,  u = U - W S
//   P = tril(Q K^T o G),  O = scale (diag(e^b) Q S + P u)
//   S' = e^{b_L} S + K^T diag(e^{b_L - b}) u
// and, with dO' = scale dO and dS' the gradient of the next chunk's state:
//   du  = P^T dO' + diag(e^{b_L - b}) K dS'
//   dS  = e^{b_L} dS' + Q^T diag(e^b) dO' - W^T du          (the only chain)
//   dQ  = diag(e^b) dO' S^T + (tril(dO' u^T) o G) K
//   dK  = (tril(dO' u^T) o G)^T Q + diag(e^{b_L - b}) u dS'^T + ...
//   dT  = dW Bk^T + du Bv^T (dW = -du S^T, Bk = diag(beta e^b) K, Bv = diag(beta) V)
//   dA  = strict_tril(-T^T dT T^T), and so on through A, Bk, Bv and the
//         decay factors to dbeta and d log alpha.
// Two launches after the tensor-core forward pass (run with its per-chunk
// records kept and the state at every chunk start written out):
//   delta_bwd_chain_kernel   per (head, sequence, 32 or 64 value columns):
//                            dS from the last chunk to the first, reading
//                            the forward's records (-W, Q e^b, K e^{b_L-b},
//                            P, e^{b_L}); stores dS' (and, for the other
//                            per-chunk kernel, du) of every chunk.
//   delta_bwd_chunk_kernel   every (chunk, head) in parallel: recomputes the
//                            chunk in fp32 from q, k, v and the stored state,
//                            then all gradients above (warp-level TF32
//                            tensor-core products on fp32 shared memory) and
//                            through the prologue (silu, L2 norm, sigmoid,
//                            softplus), written straight to the outputs.

#include "common.cuh"
#include "delta_tc.h"
#include "launch.h"
#include "tc_tile.cuh"
#include "warp_mma.cuh"

namespace la {
namespace {

using tile::C;
constexpr int LDM = 68;                 // fp32 row stride of a 64-wide shared matrix
constexpr int MAT = 64 * LDM;           // floats per 64 x 64 matrix

// One m16n8k8 TF32 product accumulated into d from fragments already in
// registers (fp32 bit patterns: the tensor core reads their top 19 bits).
__device__ __forceinline__ void mma8(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                     uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t bits(float x) { return __float_as_uint(x); }

// Four 8 x 4 fp32 blocks of shared memory in one instruction: ldmatrix moves
// 8 x 8 blocks of 16-bit pairs, i.e. 8 rows x 16 bytes, and gives lane
// (g, t) = (lane / 4, lane % 4) the 32-bit word in row g, column t of each
// block -- the TF32 fragment layout.  p: this lane's row address (16-byte
// aligned); lanes 8j .. 8j + 7 address the rows of block j.
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const float *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
}

// Zero structure a product can skip: op(A) lower (entries k > m are zero) or
// upper (k < m), op(B) upper (k > n), and outputs wanted only on or below the
// diagonal (blocks above it are left unwritten).
enum : int { kFull = 0, kALower = 1, kAUpper = 2, kBUpper = 4, kOutLower = 8 };

// Cm (M x N, row stride LDC) = or += alpha * op(A) op(B), K-deep, over the
// CTA's NWARP warps.  op(A) is A (row stride LDA) or, with TA, its
// transpose; likewise op(B).  Each warp takes 16 x 16 blocks (two 16 x 8
// tiles sharing the A fragment).  With rowscale, the existing C is first
// multiplied by rowscale[row].  Nothing is synchronised.
template <int M, int N, int K, bool TA, bool TB, int LDA, int LDB, int LDC, int NWARP,
          int SHAPE = kFull>
__device__ __forceinline__ void mm(float *Cm, const float *A, const float *B, float alpha,
                                   bool accumulate, const float *rowscale = nullptr) {
    constexpr int AM = TA ? 1 : LDA, AK = TA ? LDA : 1;
    constexpr int BK = TB ? 1 : LDB, BN = TB ? LDB : 1;
    constexpr int NB = (M / 16) * (N / 16);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    for (int blk = w; blk < NB; blk += NWARP) {
        const int m0 = (blk / (N / 16)) * 16, n0 = (blk % (N / 16)) * 16;
        if ((SHAPE & kOutLower) && n0 > m0) continue;
        // k range that can be nonzero for this block
        int klo = 0, khi = K;
        if (SHAPE & kALower) khi = m0 + 16;
        if (SHAPE & kAUpper) klo = m0;
        if ((SHAPE & kBUpper) && n0 + 16 < khi) khi = n0 + 16;
        const float *Ap = A + (m0 + g) * AM + t * AK;
        const float *Bp = B + t * BK + (n0 + g) * BN;
        // ldmatrix row addresses: A row-major (k contiguous), B stored as B^T
        const float *Al = A + (m0 + (lane & 15)) * LDA + (lane >> 4) * 4;
        const float *Bl = B + (n0 + (lane & 7) + ((lane >> 4) << 3)) * LDB + ((lane >> 3) & 1) * 4;
        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k0 = 0; k0 < K; k0 += 8) {
            if (k0 < klo || k0 >= khi) continue;
            uint32_t a[4], b[4];
            if constexpr (!TA) {
                ldsm_x4(a, Al + k0);
            } else {
                a[0] = bits(Ap[k0 * AK]); a[1] = bits(Ap[8 * AM + k0 * AK]);
                a[2] = bits(Ap[(k0 + 4) * AK]); a[3] = bits(Ap[8 * AM + (k0 + 4) * AK]);
            }
            if constexpr (TB) {
                ldsm_x4(b, Bl + k0);
            } else {
                b[0] = bits(Bp[k0 * BK]); b[1] = bits(Bp[(k0 + 4) * BK]);
                b[2] = bits(Bp[k0 * BK + 8 * BN]); b[3] = bits(Bp[(k0 + 4) * BK + 8 * BN]);
            }
            mma8(d0, a, b[0], b[1]);
            mma8(d1, a, b[2], b[3]);
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const float(&d)[4] = half ? d1 : d0;
            float *c0 = Cm + (m0 + g) * LDC + n0 + 8 * half + 2 * t, *c1 = c0 + 8 * LDC;
            if (accumulate) {
                const float s0 = rowscale ? rowscale[m0 + g] : 1.0f;
                const float s1 = rowscale ? rowscale[m0 + g + 8] : 1.0f;
                c0[0] = fmaf(s0, c0[0], alpha * d[0]); c0[1] = fmaf(s0, c0[1], alpha * d[1]);
                c1[0] = fmaf(s1, c1[0], alpha * d[2]); c1[1] = fmaf(s1, c1[1], alpha * d[3]);
            } else {
                c0[0] = alpha * d[0]; c0[1] = alpha * d[1];
                c1[0] = alpha * d[2]; c1[1] = alpha * d[3];
            }
        }
    }
}

struct ChainParams {
    const uint8_t *records;   // [slots][H] forward records
    const __nv_bfloat16 *d_o;
    const int32_t *cu;
    const float *d_final_S;
    float *dstates;           // [slots][H][D][D]: dS' of every chunk
    float *du;                // null, or [slots][H][64][D]: du of every chunk
    float *d_init_S;
    unsigned *err;
    int H, ntok;
    float scale;
    bool gend;                // records carry e^{b_L} (gated); else it is 1
};

// One CTA of 16 warps per (head, sequence).  Shared memory (bytes): two
// record buffers (the operands of one chunk copied from its record: [-W ;
// Q e^b] as a 128-row swizzled tile, K e^{b_L - b} as a 64-row one, Aq, and
// e^{b_L}), two buffers of scale dO, the bf16 copy of dS' and du, barriers.
template <int D> struct ChainCfg {
    static constexpr int NT = 512;
    static constexpr int XS = D + 8;                      // bf16 stride of dO, du, dS'
    static constexpr int WQB = 128 * D * 2, KB = 64 * D * 2, AQB = 64 * 64 * 2, GB = 4 * D;
    static constexpr int TX = WQB + KB + AQB + GB;        // bytes a record copy delivers
    static constexpr int BUF = (TX + 1023) & ~1023;
    static constexpr int DO = 2 * BUF, DOB = 64 * XS * 2;
    static constexpr int DS = DO + 2 * DOB, DU = DS + D * XS * 2, BARS = DU + 64 * XS * 2;
    static constexpr int BYTES = BARS + 64;
    // warp tiles: du (64 x D) in 4 row blocks x 4 column groups; dS (D x D)
    // in D/16 row blocks x 16/(D/16) column groups
    static constexpr int NT_DU = D / 32;
    static constexpr int CG = 16 / (D / 16), NT_DS = D / CG / 8;
    static constexpr int DO_UNITS = 64 * D / 8 / NT;     // 16-byte units of dO per thread
};

// Reverse pass over the chunks of one (head, sequence).  dS (fp32) stays in
// registers for the whole sequence; per chunk c, last to first:
//   store dS' (= dS) of chunk c;  du = Aq^T dO' + K~ dS';
//   dS = Diag(e^{b_L}) dS' + (Q e^b)^T dO' + (-W)^T du
// with bf16 operands (dS' and du rounded for the products only) read by
// ldmatrix straight from the record tiles.  Chunk c - 1's record arrives by
// bulk copy into the other buffer while chunk c computes.
template <int D>
__global__ void __launch_bounds__(ChainCfg<D>::NT, 1) delta_bwd_chain_kernel(ChainParams p) {
    using namespace tc;
    using L = ChainCfg<D>;
    using Rec = tile::Record<D>;
    using wmma16::PadView;
    using wmma16::RsView;
    using bf16 = __nv_bfloat16;
    constexpr int XS = L::XS, NT_DU = L::NT_DU, NT_DS = L::NT_DS;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BARS);
    bf16 *sDS = reinterpret_cast<bf16 *>(smem + L::DS), *sDU = reinterpret_cast<bf16 *>(smem + L::DU);
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int h = blockIdx.x, n = blockIdx.y, H = p.H;
    int t_begin = p.cu[n], t_end = p.cu[n + 1];
    if (t_begin < 0 || t_end < t_begin || t_end > p.ntok) {
        if (tid == 0) atomicCAS(p.err, 0u, 100u);
        t_begin = t_end = 0;
    }
    const int nc = (t_end - t_begin + C - 1) / C;
    const int64_t slot0 = (int64_t)(t_begin / C) + n;
    const int64_t sbase = ((int64_t)n * H + h) * D * D;
    // this warp's blocks: du rows 16 Ru, columns nu ..; dS rows 16 Rs, columns ns ..
    const int Ru = w >> 2, nu = (w & 3) * (D / 4);
    const int Rs = w / L::CG, ns = (w % L::CG) * (D / L::CG);

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int c) {   // thread 0: chunk c's record into buffer c & 1
        uint8_t *buf = smem + (c & 1) * L::BUF;
        const uint8_t *rec = p.records + ((slot0 + c) * H + h) * (int64_t)Rec::BYTES;
        fence_proxy_async();
        mbar_arrive_expect_tx(&bars[c & 1], L::TX);
        bulk_load(buf, rec + Rec::WQ, L::WQB, &bars[c & 1]);
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb)   // rows 64..127 of each 64-column block of [U ; K~]
            bulk_load(buf + L::WQB + cb * 8192, rec + Rec::UK + cb * 16384 + 8192, 8192, &bars[c & 1]);
        bulk_load(buf + L::WQB + L::KB, rec + Rec::AQ, L::AQB, &bars[c & 1]);
        bulk_load(buf + L::WQB + L::KB + L::AQB, rec + Rec::GEND, L::GB, &bars[c & 1]);
    };
    // this thread's 16-byte units of scale * dO (rows past the end are zero)
    uint4 rdo[L::DO_UNITS];
    auto load_do = [&](int c) {
        const int tok0 = t_begin + c * C, len = min(C, t_end - tok0);
#pragma unroll
        for (int k = 0; k < L::DO_UNITS; ++k) {
            const int u = tid + L::NT * k, r = u / (D / 8), c8 = (u % (D / 8)) * 8;
            rdo[k] = r < len ? *reinterpret_cast<const uint4 *>(p.d_o + ((int64_t)(tok0 + r) * H + h) * D + c8)
                             : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    auto store_do = [&](int c) {
        bf16 *dst = reinterpret_cast<bf16 *>(smem + L::DO + (c & 1) * L::DOB);
#pragma unroll
        for (int k = 0; k < L::DO_UNITS; ++k) {
            const int u = tid + L::NT * k, r = u / (D / 8), c8 = (u % (D / 8)) * 8;
            float v[8];
            tile::unpack8(rdo[k], v);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] *= p.scale;
            *reinterpret_cast<uint4 *>(dst + r * XS + c8) = tile::pack8(v);
        }
    };

    // dS' of the last chunk: the final state's gradient
    float ds[NT_DS][4];
#pragma unroll
    for (int j = 0; j < NT_DS; ++j)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int r = 16 * Rs + g + 8 * hr, col = ns + 8 * j + 2 * t;
            const float2 v = p.d_final_S ? *reinterpret_cast<const float2 *>(p.d_final_S + sbase + r * D + col)
                                         : make_float2(0.0f, 0.0f);
            ds[j][2 * hr] = v.x;
            ds[j][2 * hr + 1] = v.y;
        }
    if (nc > 0) {
        if (tid == 0) issue(nc - 1);
        load_do(nc - 1);
    }
    // chunk c is use (nc - 1 - c) / 2 of buffer c & 1: its phase parity
    auto parity = [&](int c) { return (uint32_t)(((nc - 1 - c) >> 1) & 1); };
    int pending = nc > 0 ? nc - 1 : -1;   // a record copy issued and not yet waited for
    for (int c = nc - 1; c >= 0; --c) {
        const int b = c & 1;
        const uint8_t *buf = smem + b * L::BUF;
        const RsView wq{buf, 128, 0}, qe{buf, 128, 64}, kt{buf + L::WQB, 64, 0};
        const RsView aq{buf + L::WQB + L::KB, 64, 0};
        const float *gend = reinterpret_cast<const float *>(buf + L::WQB + L::KB + L::AQB);
        const PadView dO{reinterpret_cast<const bf16 *>(smem + L::DO + b * L::DOB), XS};
        const PadView dSp{sDS, XS}, dU{sDU, XS};
        // 1. dS' of chunk c out (fp32) and in (bf16 operand); this chunk's dO in
        float *dst = p.dstates + ((slot0 + c) * H + h) * (int64_t)(D * D);
#pragma unroll
        for (int j = 0; j < NT_DS; ++j)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int r = 16 * Rs + g + 8 * hr, col = ns + 8 * j + 2 * t;
                *reinterpret_cast<float2 *>(dst + r * D + col) = make_float2(ds[j][2 * hr], ds[j][2 * hr + 1]);
                wmma16::st2(sDS + r * XS + col, ds[j][2 * hr], ds[j][2 * hr + 1]);
            }
        store_do(c);
        const bool ok = mbar_wait(&bars[b], parity(c), p.err, 15u);
        if (__syncthreads_or(!ok)) break;
        pending = -1;
        if (c > 0) {
            if (tid == 0) issue(c - 1);
            pending = c - 1;
            load_do(c - 1);
        }
        // 2. du = Aq^T dO' + K~ dS' (Aq lower: rows r >= i of Aq reach column i)
        {
            float du[NT_DU][4];
            wmma16::zero(du);
            wmma16::mma_rows<NT_DU, true, false>(du, aq, dO, 16 * Ru, nu, 16 * Ru, 64);
            wmma16::mma_rows_c<0, D, NT_DU, false, false>(du, kt, dSp, 16 * Ru, nu);
            float *gdu = p.du ? p.du + ((slot0 + c) * H + h) * (int64_t)(64 * D) : nullptr;
#pragma unroll
            for (int j = 0; j < NT_DU; ++j)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int r = 16 * Ru + g + 8 * hr, col = nu + 8 * j + 2 * t;
                    wmma16::st2(sDU + r * XS + col, du[j][2 * hr], du[j][2 * hr + 1]);
                    if (gdu)
                        *reinterpret_cast<float2 *>(gdu + r * D + col) = make_float2(du[j][2 * hr], du[j][2 * hr + 1]);
                }
        }
        __syncthreads();
        // 3. dS = Diag(e^{b_L}) dS' + (Q e^b)^T dO' + (-W)^T du
        {
            const float g0 = p.gend ? gend[16 * Rs + g] : 1.0f;
            const float g1 = p.gend ? gend[16 * Rs + g + 8] : 1.0f;
#pragma unroll
            for (int j = 0; j < NT_DS; ++j) {
                ds[j][0] *= g0; ds[j][1] *= g0;
                ds[j][2] *= g1; ds[j][3] *= g1;
            }
            wmma16::mma_rows_c<0, 64, NT_DS, true, false>(ds, qe, dO, 16 * Rs, ns);
            wmma16::mma_rows_c<0, 64, NT_DS, true, false>(ds, wq, dU, 16 * Rs, ns);
        }
    }
    // a copy still in flight (only after a failed wait): let it land first
    if (pending >= 0) mbar_wait(&bars[pending & 1], parity(pending), nullptr, 0u);
    if (p.d_init_S) {
#pragma unroll
        for (int j = 0; j < NT_DS; ++j)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int r = 16 * Rs + g + 8 * hr, col = ns + 8 * j + 2 * t;
                *reinterpret_cast<float2 *>(p.d_init_S + sbase + r * D + col) =
                    make_float2(ds[j][2 * hr], ds[j][2 * hr + 1]);
            }
    }
}

struct ChunkParams {
    const __nv_bfloat16 *__restrict__ q, *__restrict__ k, *__restrict__ v;
    const __nv_bfloat16 *__restrict__ beta_logits;
    const __nv_bfloat16 *__restrict__ gate_scalar;   // [ntok][H] or null
    const __nv_bfloat16 *__restrict__ d_o;
    const int2 *table;        // [slots] {first token, length}
    const float *states;      // [slots][H][64][64] S at each chunk start
    const float *dstates;     // [slots][H][64][64] dS' of each chunk
    float *dq, *dk, *dv;      // [ntok][H][64] gradients of the raw inputs
    float *d_beta_logits;     // [ntok][H]
    float *d_gate_logits;     // [ntok][H] (scalar gate) or null
    int64_t n_tasks;
    int H;
    float scale;
    unsigned flags;
};

constexpr int kGradNT = 512;  // 16 warps

struct GradLayout {
    static constexpr int Q = 0, K = Q + MAT, V = K + MAT, DO = V + MAT, S = DO + MAT;
    static constexpr int DS = S + MAT, T = DS + MAT, P = T + MAT, U = P + MAT, W = U + MAT;
    static constexpr int DK = W + MAT;
    static constexpr int BETA = DK + MAT, B = BETA + 64, EB = B + 64, EBL = EB + 64;
    static constexpr int DEB = EBL + 64, DEBL = DEB + 64, DB = DEBL + 64, DBETA = DB + 64;
    static constexpr int DEBLS = DBETA + 64, FLOATS = DEBLS + 4;
};

// Every (chunk, head): the gradients of the chunk's inputs given its starting
// state S and the gradient dS' of the next chunk's state (the formulas at the
// top of this file).
__global__ void __launch_bounds__(kGradNT, 1) delta_bwd_chunk_kernel(ChunkParams p) {
    using L = GradLayout;
    extern __shared__ __align__(16) float sm[];
    float *sQ = sm + L::Q, *sK = sm + L::K, *sV = sm + L::V, *sDO = sm + L::DO, *sS = sm + L::S;
    float *sDS = sm + L::DS, *sT = sm + L::T, *sP = sm + L::P, *sU = sm + L::U, *sW = sm + L::W;
    float *sDK = sm + L::DK;
    float *sBeta = sm + L::BETA, *sB = sm + L::B, *sEB = sm + L::EB, *sEBL = sm + L::EBL;
    float *sDEB = sm + L::DEB, *sDEBL = sm + L::DEBL, *sDB = sm + L::DB, *sDBeta = sm + L::DBETA;
    float *sDEBLs = sm + L::DEBLS;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int H = p.H;
    const bool gated = p.gate_scalar != nullptr;
    const bool silu = (p.flags & kSiluQK) != 0;
    constexpr int NW = kGradNT / 32;
    // rows r = w + 16 rr of a 64-row matrix belong to warp w (columns lane, lane + 32)
    auto row_of = [&](int rr) { return w + NW * rr; };
    int t0 = 0, len = 0;
    int h = 0;
    // rows r < len of a gradient with respect to the prepared q or k (sG),
    // taken through silu / L2 norm of the raw row and written to out
    auto write_prep_grad = [&](const float *sGr, const __nv_bfloat16 *__restrict__ raw,
                               float *out, bool norm) {
        float x[4][2], d[4][2];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            const int r = row_of(rr);
            const int64_t o = (((int64_t)(t0 + (r < len ? r : 0))) * H + h) * 64 + lane;
            x[rr][0] = __bfloat162float(raw[o]);
            x[rr][1] = __bfloat162float(raw[o + 32]);
            d[rr][0] = sGr[r * LDM + lane];
            d[rr][1] = sGr[r * LDM + lane + 32];
        }
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            const int r = row_of(rr);
            if (r >= len) continue;
            prep_backward<2>(x[rr], d[rr], silu, norm);
            float *dst = out + (((int64_t)(t0 + r)) * H + h) * 64 + lane;
            dst[0] = d[rr][0];
            dst[32] = d[rr][1];
        }
    };

    // The next task's inputs (q, k, v, dO rows and the two 16 KB states) are
    // prefetched into L2 while this task computes, one 128-byte line per
    // thread, so its staging phase reads L2 rather than DRAM.
    auto prefetch_task = [&](int64_t nt) {
        if (nt >= p.n_tasks) return;
        const int64_t ns = nt / H;
        const int nh = (int)(nt % H);
        const int2 e = p.table[ns];
        if (e.y <= 0 || e.y > 64) return;
        if (tid < 256) {
            const int r = tid & 63, which = tid >> 6;
            if (r < e.y) {
                const __nv_bfloat16 *base = which == 0 ? p.q : which == 1 ? p.k : which == 2 ? p.v : p.d_o;
                prefetch_l2(base + ((int64_t)(e.x + r) * H + nh) * 64);
            }
        } else {
            const int v = tid - 256;  // 128 lines of each state
            prefetch_l2((v < 128 ? p.states : p.dstates) + (ns * H + nh) * 4096 + (v & 127) * 32);
        }
    };
    static_assert(kGradNT == 512, "one prefetched line per thread");

    for (int64_t task = blockIdx.x; task < p.n_tasks; task += gridDim.x) {
        const int64_t slot = task / H;
        h = (int)(task % H);
        const int2 te = p.table[slot];
        t0 = te.x;
        len = te.y;
        if (len <= 0) continue;

        // ---- 0. stage the chunk (fp32), beta and the log decays: every load
        // of the warp's four rows first, then the feature maps and stores
        float xq[4][2], xk[4][2], xv[4][2], xo[4][2], xb[4], xg[4];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            const int r = row_of(rr);
            const bool ok = r < len;
            const int64_t th = ((int64_t)(t0 + (ok ? r : 0))) * H + h;
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                const int64_t o = th * 64 + lane + 32 * c2;
                xq[rr][c2] = ok ? __bfloat162float(p.q[o]) : 0.0f;
                xk[rr][c2] = ok ? __bfloat162float(p.k[o]) : 0.0f;
                xv[rr][c2] = ok ? __bfloat162float(p.v[o]) : 0.0f;
                xo[rr][c2] = ok ? __bfloat162float(p.d_o[o]) : 0.0f;
            }
            xb[rr] = ok ? __bfloat162float(p.beta_logits[th]) : 0.0f;
            xg[rr] = (ok && gated) ? __bfloat162float(p.gate_scalar[th]) : 0.0f;
        }
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            const int r = row_of(rr);
            const bool ok = r < len;
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                float x0 = which ? xk[rr][0] : xq[rr][0], x1 = which ? xk[rr][1] : xq[rr][1];
                if (silu) { x0 = silu_f(x0); x1 = silu_f(x1); }
                const bool norm = (p.flags & (which ? kL2NormK : kL2NormQ)) != 0;
                const float inv = norm ? 1.0f / fmaxf(sqrtf(warp_sum(x0 * x0 + x1 * x1)), 1e-12f) : 1.0f;
                float *dst = (which ? sK : sQ) + r * LDM;
                dst[lane] = x0 * inv;
                dst[lane + 32] = x1 * inv;
            }
            sV[r * LDM + lane] = xv[rr][0];
            sV[r * LDM + lane + 32] = xv[rr][1];
            sDO[r * LDM + lane] = p.scale * xo[rr][0];
            sDO[r * LDM + lane + 32] = p.scale * xo[rr][1];
            if (lane == 0) {
                sBeta[r] = ok ? sigmoid_f(xb[rr]) : 0.0f;
                sB[r] = (ok && gated) ? log_decay_f(xg[rr]) : 0.0f;
            }
        }
        {
            const float4 *s4 = reinterpret_cast<const float4 *>(p.states + (slot * H + h) * 4096);
            const float4 *d4 = reinterpret_cast<const float4 *>(p.dstates + (slot * H + h) * 4096);
            for (int u = tid; u < 1024; u += kGradNT) {
                const int r = u >> 4, c = (u & 15) * 4;
                *reinterpret_cast<float4 *>(sS + r * LDM + c) = s4[u];
                *reinterpret_cast<float4 *>(sDS + r * LDM + c) = d4[u];
            }
        }
        if (tid < 64) sDEB[tid] = sDEBL[tid] = sDB[tid] = sDBeta[tid] = 0.0f;
        if (tid == 0) sDEBLs[0] = 0.0f;
        __syncthreads();
        prefetch_task(task + gridDim.x);
        if (w == 0) {
            // b = inclusive cumulative log decay; e^b and e^{b_L - b} (exponents <= 0)
            float v0 = sB[lane], v1 = sB[lane + 32];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float a0 = __shfl_up_sync(0xffffffffu, v0, o);
                const float a1 = __shfl_up_sync(0xffffffffu, v1, o);
                if (lane >= o) { v0 += a0; v1 += a1; }
            }
            v1 += __shfl_sync(0xffffffffu, v0, 31);
            const float bL = __shfl_sync(0xffffffffu, v1, 31);
            sB[lane] = v0;
            sB[lane + 32] = v1;
            sEB[lane] = expf(v0);
            sEB[lane + 32] = expf(v1);
            sEBL[lane] = expf(bL - v0);
            sEBL[lane + 32] = expf(bL - v1);
        }
        // ---- 1. K K^T and Q K^T
        mm<64, 64, 64, false, true, LDM, LDM, LDM, NW, kOutLower>(sT, sK, sK, 1.0f, false);
        mm<64, 64, 64, false, true, LDM, LDM, LDM, NW, kOutLower>(sP, sQ, sK, 1.0f, false);
        __syncthreads();
        // A = strict_tril(beta_r K K^T o G), P = tril(Q K^T o G)
        for (int e = tid; e < 4096; e += kGradNT) {
            const int r = e >> 6, i = e & 63;
            const float G = i <= r ? (gated ? expf(sB[r] - sB[i]) : 1.0f) : 0.0f;
            sP[r * LDM + i] = i <= r ? sP[r * LDM + i] * G : 0.0f;
            sT[r * LDM + i] = i < r ? sBeta[r] * sT[r * LDM + i] * G : 0.0f;
        }
        __syncthreads();
        // ---- 2. T = (I + A)^{-1} in place: the four 16 x 16 diagonal blocks
        // by column-wise forward substitution, then block rows 1..3:
        // T_ij = -T_ii sum_{j <= l < i} A_il T_lj (A_il read before it is replaced)
        {
            float t[16];
            const int R = tid >> 4, j = tid & 15;
            if (tid < 64) {
                const float *Ab = sT + (16 * R) * LDM + 16 * R;
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    float a = (r == j) ? 1.0f : 0.0f;
#pragma unroll
                    for (int k = 0; k < r; ++k) a = fmaf(-Ab[r * LDM + k], t[k], a);
                    t[r] = a;
                }
            }
            __syncthreads();
            if (tid < 64) {
#pragma unroll
                for (int r = 0; r < 16; ++r) sT[(16 * R + r) * LDM + 16 * R + j] = t[r];
            }
            __syncthreads();
        }
#pragma unroll 1
        for (int bi = 1; bi < 4; ++bi) {
            float *X = sU;  // [bi][16][16] scratch
            for (int e = tid; e < bi * 256; e += kGradNT) {
                const int bj = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
                float acc = 0.0f;
                for (int l = bj; l < bi; ++l)
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        acc = fmaf(sT[(16 * bi + rr) * LDM + 16 * l + k], sT[(16 * l + k) * LDM + 16 * bj + cc], acc);
                X[e] = acc;
            }
            __syncthreads();
            for (int e = tid; e < bi * 256; e += kGradNT) {
                const int bj = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
                float acc = 0.0f;
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    acc = fmaf(sT[(16 * bi + rr) * LDM + 16 * bi + k], X[(bj << 8) + k * 16 + cc], acc);
                sT[(16 * bi + rr) * LDM + 16 * bj + cc] = -acc;
            }
            __syncthreads();
        }
        // ---- 3. W = T Bk, U = T Bv, u = U - W S
        for (int e = tid; e < 4096; e += kGradNT) {
            const int r = e >> 6, c = e & 63;
            sW[r * LDM + c] = sBeta[r] * sEB[r] * sK[r * LDM + c];
        }
        __syncthreads();
        mm<64, 64, 64, false, false, LDM, LDM, LDM, NW, kALower>(sDK, sT, sW, 1.0f, false);   // W
        __syncthreads();
        for (int e = tid; e < 4096; e += kGradNT) {
            const int r = e >> 6, c = e & 63;
            sW[r * LDM + c] = sBeta[r] * sV[r * LDM + c];
        }
        __syncthreads();
        mm<64, 64, 64, false, false, LDM, LDM, LDM, NW, kALower>(sU, sT, sW, 1.0f, false);    // U
        mm<64, 64, 64, false, false, LDM, LDM, LDM, NW>(sU, sDK, sS, -1.0f, true);   // u
        __syncthreads();
        // ---- 4. K dS', u dS'^T, then du = P^T dO' + diag(e^{b_L - b}) K dS'
        mm<64, 64, 64, false, false, LDM, LDM, LDM, NW>(sW, sK, sDS, 1.0f, false);
        mm<64, 64, 64, false, true, LDM, LDM, LDM, NW>(sDK, sU, sDS, 1.0f, false);
        __syncthreads();
#pragma unroll 1
        for (int rr = 0; rr < 4; ++rr) {
            const int r = row_of(rr);
            const float el = sEBL[r];
            float a = 0.0f, s = 0.0f;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int c = lane + 32 * h2;
                a = fmaf(sW[r * LDM + c], sU[r * LDM + c], a);
                s = fmaf(sDS[r * LDM + c], sS[r * LDM + c], s);
                sW[r * LDM + c] *= el;
                sDK[r * LDM + c] *= el;
            }
            a = warp_sum(a);
            s = warp_sum(s);
            if (lane == 0) {
                sDEBL[r] = a;
                atomicAdd(sDEBLs, s);
            }
        }
        __syncthreads();
        mm<64, 64, 64, true, false, LDM, LDM, LDM, NW, kAUpper>(sW, sP, sDO, 1.0f, true);     // du
        mm<64, 64, 64, false, true, LDM, LDM, LDM, NW, kOutLower>(sDS, sDO, sU, 1.0f, false);   // dO' u^T
        __syncthreads();
        // ---- 5. dP = tril(dO' u^T); decay terms; P <- dP o G
#pragma unroll 1
        for (int rr = 0; rr < 4; ++rr) {
            const int r = row_of(rr);
            float rs = 0.0f;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int i = lane + 32 * h2;
                const float dpr = i <= r ? sDS[r * LDM + i] : 0.0f;
                const float pv = dpr * sP[r * LDM + i];
                if (gated) {
                    rs += pv;
                    if (pv != 0.0f) atomicAdd(&sDB[i], -pv);
                }
                const float G = i <= r ? (gated ? expf(sB[r] - sB[i]) : 1.0f) : 0.0f;
                sP[r * LDM + i] = dpr * G;
            }
            rs = warp_sum(rs);
            if (gated && lane == 0) atomicAdd(&sDB[r], rs);
        }
        __syncthreads();
        mm<64, 64, 64, false, true, LDM, LDM, LDM, NW>(sDS, sDO, sS, 1.0f, false);   // X = dO' S^T
        __syncthreads();
#pragma unroll 1
        for (int rr = 0; rr < 4; ++rr) {
            const int r = row_of(rr);
            const float eb = sEB[r];
            float a = 0.0f;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int c = lane + 32 * h2;
                a = fmaf(sQ[r * LDM + c], sDS[r * LDM + c], a);
                sDS[r * LDM + c] *= eb;
            }
            a = warp_sum(a);
            if (lane == 0) sDEB[r] += a;
        }
        __syncthreads();
        mm<64, 64, 64, false, false, LDM, LDM, LDM, NW, kALower>(sDS, sP, sK, 1.0f, true);    // dQ
        mm<64, 64, 64, true, false, LDM, LDM, LDM, NW, kAUpper>(sDK, sP, sQ, 1.0f, true);     // dK += dP^T Q
        __syncthreads();
        // dq out (through silu / L2 norm); dW = -du S^T
        write_prep_grad(sDS, p.q, p.dq, (p.flags & kL2NormQ) != 0);
        mm<64, 64, 64, false, true, LDM, LDM, LDM, NW>(sQ, sW, sS, -1.0f, false);    // dW
        __syncthreads();
        // ---- 7. dT = dW Bk^T + du Bv^T, dBk = T^T dW, dBv = T^T du
        for (int e = tid; e < 4096; e += kGradNT) {
            const int r = e >> 6, c = e & 63;
            sDS[r * LDM + c] = sBeta[r] * sEB[r] * sK[r * LDM + c];   // Bk
            sP[r * LDM + c] = sBeta[r] * sV[r * LDM + c];             // Bv
        }
        __syncthreads();
        mm<64, 64, 64, false, true, LDM, LDM, LDM, NW>(sS, sQ, sDS, 1.0f, false);    // dT
        mm<64, 64, 64, false, true, LDM, LDM, LDM, NW>(sS, sW, sP, 1.0f, true);
        __syncthreads();
        mm<64, 64, 64, true, false, LDM, LDM, LDM, NW, kAUpper>(sDS, sT, sQ, 1.0f, false);    // dBk
        mm<64, 64, 64, true, false, LDM, LDM, LDM, NW, kAUpper>(sP, sT, sW, 1.0f, false);     // dBv
        __syncthreads();
#pragma unroll 1
        for (int rr = 0; rr < 4; ++rr) {
            const int r = row_of(rr);
            const float be = sBeta[r], eb = sEB[r];
            float bv = 0.0f, bk = 0.0f;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int c = lane + 32 * h2;
                const float dbv = sP[r * LDM + c], dbk = sDS[r * LDM + c];
                bv = fmaf(dbv, sV[r * LDM + c], bv);
                bk = fmaf(dbk, sK[r * LDM + c], bk);
                sDK[r * LDM + c] = fmaf(be * eb, dbk, sDK[r * LDM + c]);
                if (r < len) p.dv[(((int64_t)(t0 + r)) * H + h) * 64 + c] = be * dbv;
            }
            bv = warp_sum(bv);
            bk = warp_sum(bk);
            if (lane == 0) {
                sDBeta[r] += bv + eb * bk;
                sDEB[r] += be * bk;
            }
        }
        __syncthreads();
        // ---- 8. dA = strict_tril(-T^T dT T^T); through A = diag(beta)(K K^T o G)
        mm<64, 64, 64, true, false, LDM, LDM, LDM, NW, kAUpper>(sQ, sT, sS, 1.0f, false);     // T^T dT
        mm<64, 64, 64, false, true, LDM, LDM, LDM, NW, kOutLower>(sP, sK, sK, 1.0f, false);     // K K^T
        __syncthreads();
        mm<64, 64, 64, false, true, LDM, LDM, LDM, NW, kOutLower | kBUpper>(sW, sQ, sT, -1.0f, false);  // dA
        __syncthreads();
#pragma unroll 1
        for (int rr = 0; rr < 4; ++rr) {
            const int r = row_of(rr);
            const float be = sBeta[r];
            float rb = 0.0f, rs = 0.0f;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int i = lane + 32 * h2;
                float mg = 0.0f;
                if (i < r) {
                    const float G = gated ? expf(sB[r] - sB[i]) : 1.0f;
                    const float da = sW[r * LDM + i], kkg = sP[r * LDM + i] * G;
                    rb = fmaf(da, kkg, rb);                     // dbeta_r
                    const float val = be * da * kkg;            // dG o G
                    if (gated) {
                        rs += val;
                        atomicAdd(&sDB[i], -val);
                    }
                    mg = be * da * G;
                }
                sW[r * LDM + i] = mg;
            }
            rb = warp_sum(rb);
            rs = warp_sum(rs);
            if (lane == 0) {
                sDBeta[r] += rb;
                if (gated) atomicAdd(&sDB[r], rs);
            }
        }
        __syncthreads();
        mm<64, 64, 64, false, false, LDM, LDM, LDM, NW, kALower>(sDK, sW, sK, 1.0f, true);    // + M K
        mm<64, 64, 64, true, false, LDM, LDM, LDM, NW, kAUpper>(sDK, sW, sK, 1.0f, true);     // + M^T K
        __syncthreads();
        // ---- 9. outputs: dk (through silu / L2 norm), beta logits, gate logits
        write_prep_grad(sDK, p.k, p.dk, (p.flags & kL2NormK) != 0);
        if (tid < len) {
            const float be = sBeta[tid];
            p.d_beta_logits[((int64_t)(t0 + tid)) * H + h] = sDBeta[tid] * be * (1.0f - be);
        }
        if (gated && w == 0) {
            // db_r, then d log alpha_t = sum_{r >= t} db_r (b is a prefix sum)
            const float bL = sB[63];
            float d0 = sDB[lane] + sDEB[lane] * sEB[lane] - sDEBL[lane] * sEBL[lane];
            float d1 = sDB[lane + 32] + sDEB[lane + 32] * sEB[lane + 32] -
                       sDEBL[lane + 32] * sEBL[lane + 32];
            const float dbl = warp_sum(sDEBL[lane] * sEBL[lane] + sDEBL[lane + 32] * sEBL[lane + 32]) +
                              sDEBLs[0] * expf(bL);
            if (lane == 31) d1 += dbl;
            // suffix sums over 64 entries: d1 within the upper half, then d0 plus d1's total
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float a0 = __shfl_down_sync(0xffffffffu, d0, o);
                const float a1 = __shfl_down_sync(0xffffffffu, d1, o);
                if (lane + o < 32) { d0 += a0; d1 += a1; }
            }
            d0 += __shfl_sync(0xffffffffu, d1, 0);
            // log alpha = -softplus(x): dx = -d(log alpha) sigmoid(x)
            if (lane < len) {
                const int64_t th = ((int64_t)(t0 + lane)) * H + h;
                p.d_gate_logits[th] = -d0 * sigmoid_f(__bfloat162float(p.gate_scalar[th]));
            }
            if (lane + 32 < len) {
                const int64_t th = ((int64_t)(t0 + lane + 32)) * H + h;
                p.d_gate_logits[th] = -d1 * sigmoid_f(__bfloat162float(p.gate_scalar[th]));
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------ host

size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

struct ChunkWs {
    size_t fwd, states, dstates, du, total;
};

ChunkWs chunk_ws(int N, int ntok, int H, int D) {
    const size_t slots = (size_t)tile::Workspace::slots(N, ntok);
    ChunkWs w;
    w.fwd = a256(delta_tc_workspace_bytes(N, ntok, H, D, D, 64, true));
    w.states = a256(slots * H * D * D * sizeof(float));
    w.dstates = w.states;
    w.du = a256(slots * H * 64 * D * sizeof(float));
    w.total = w.fwd + w.states + w.dstates + w.du;
    return w;
}

template <int D>
cudaError_t launch_chain(const ChainParams &cp, int N, int H, cudaStream_t s) {
    using L = ChainCfg<D>;
    const size_t smem = (size_t)L::BYTES;
    cudaError_t e = cudaFuncSetAttribute(delta_bwd_chain_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    delta_bwd_chain_kernel<D><<<dim3(H, N), L::NT, smem, s>>>(cp);
    return cudaGetLastError();
}

}  // namespace

bool delta_bwd_chunked_supported(const BwdArgs &a) {
    return a.bf16 && a.dk == a.dv && (a.dk == 64 || a.dk == 128) && !(a.flags & kAdditive);
}

size_t delta_bwd_chunked_workspace_bytes(int N, int ntok, int H, int D) {
    return chunk_ws(N, ntok, H, D).total;
}

cudaError_t launch_delta_backward_chunked(const BwdArgs &a, cudaStream_t s) {
    const int D = a.dk;
    const ChunkWs w = chunk_ws(a.N, a.ntok, a.H, D);
    uint8_t *base = static_cast<uint8_t *>(a.workspace);
    float *states = reinterpret_cast<float *>(base + w.fwd);
    float *dstates = reinterpret_cast<float *>(base + w.fwd + w.states);
    float *du = reinterpret_cast<float *>(base + w.fwd + w.states + w.dstates);
    unsigned *err = device_error_word();
    if (!err) return cudaErrorInvalidValue;
    // d = 64 without a per-channel decay: the fp32 per-chunk kernel of this
    // file; otherwise the bf16 one with per-channel decay (it needs du)
    const bool channel = D != 64 || (a.gate_logits && !(a.flags & kGateScalar));

    // 1. the forward pass, keeping its records and the state at every chunk start
    PrefillArgs pa{a.q, a.k, a.v, a.beta_logits, a.gate_logits, nullptr, a.cu_seqlens, a.N,
                   a.ntok, a.H, D, D, a.scale, a.flags, a.init_S, nullptr, nullptr, nullptr,
                   true, base, w.fwd};
    pa.chunk_states = states;
    if (!delta_tc_supported(pa)) return cudaErrorInvalidValue;
    cudaError_t e = launch_delta_tc(pa, s);
    if (e != cudaSuccess) return e;

    // 2. dS from the last chunk to the first
    const uint8_t *records = base + tile::Workspace::table_bytes(a.N, a.ntok);
    ChainParams cp{records, static_cast<const __nv_bfloat16 *>(a.d_o), a.cu_seqlens, a.d_final_S,
                   dstates, channel ? du : nullptr, a.d_init_S, err, a.H, a.ntok, a.scale,
                   a.gate_logits != nullptr};
    e = D == 64 ? launch_chain<64>(cp, a.N, a.H, s) : launch_chain<128>(cp, a.N, a.H, s);
    if (e != cudaSuccess) return e;

    // 3. every (chunk, head): the gradients, through the prologue
    const int64_t n_tasks = tile::Workspace::slots(a.N, a.ntok) * a.H;
    const int2 *table = reinterpret_cast<const int2 *>(base);
    if (channel) {
        BwdChannelArgs ca{a.q, a.k, a.v, a.beta_logits, a.gate_logits, a.d_o, table, states,
                          dstates, du, a.dq, a.dk_out, a.dv_out, a.d_beta_logits,
                          a.gate_logits ? a.d_gate_logits : nullptr, n_tasks, a.H, D, a.scale,
                          a.flags};
        return launch_delta_bwd_channel(ca, s);
    }
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    ChunkParams gp{static_cast<const __nv_bfloat16 *>(a.q), static_cast<const __nv_bfloat16 *>(a.k),
                   static_cast<const __nv_bfloat16 *>(a.v),
                   static_cast<const __nv_bfloat16 *>(a.beta_logits),
                   a.gate_logits ? static_cast<const __nv_bfloat16 *>(a.gate_logits) : nullptr,
                   static_cast<const __nv_bfloat16 *>(a.d_o), table,
                   states, dstates, a.dq, a.dk_out, a.dv_out, a.d_beta_logits,
                   a.gate_logits ? a.d_gate_logits : nullptr, n_tasks, a.H, a.scale, a.flags};
    const size_t grad_smem = (size_t)GradLayout::FLOATS * sizeof(float);
    if ((e = cudaFuncSetAttribute(delta_bwd_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)grad_smem)) != cudaSuccess)
        return e;
    const int64_t grid = n_tasks < sms ? n_tasks : sms;
    if (grid > 0) {
        delta_bwd_chunk_kernel<<<(unsigned)grid, kGradNT, grad_smem, s>>>(gp);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace la
