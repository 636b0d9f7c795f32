// delta_inter128_tc.cu -- the state recurrence of the tensor-core delta-rule
// prefill stepping over 128-token chunks (chunk = 128, dk = dv = 64), one CTA
// per (head, sequence).
//
// ("From GPT-2 to Kimi K3, explained", section DeltaNet (Parallelizing
// Linear Transformers with Delta Rule), eq. 8-10: the chunk length C is a
// free parameter, usually 64 or 128; with the cumulative decay of sections
// Gated DeltaNet and KDA / Kimi Linear.)
//
// The intra-chunk kernel writes one record per 64-token chunk (-W, Q e^b,
// U, K~ = K e^{b_end - b}, Aq, e^{b_end}).  A 128-token chunk is the pair
// (chunk 1, chunk 2) of 64-token chunks; its UT/WY form is the two-level
// blocked solve whose diagonal blocks are the two records and whose
// off-diagonal coupling this kernel forms before the pair's step.  With
// S0 the state before the pair, D1 = Diag(e^{b_end}) of chunk 1, D2 that of
// chunk 2, and M = W2 K1~^T (64 x 64):
//   u1 = U1 - W1 S0,   S1 = D1 S0 + K1~^T u1,   u2 = U2 - W2 S1
//   => u2 = (U2 - M U1) - (W2 D1 - M W1) S0
//   O2 = (Q2 e^b) D1 S0 + (Q2 e^b K1~^T) u1 + Aq2 u2
//   S2 = D1 D2 S0 + (K1~ D2)^T u1 + K2~^T u2
// so the 128-token chunk has
//   W' = [W1 ; W2 D1 - M W1]      U' = [U1 ; U2 - M U1]
//   Q' = [Q1 e^b ; Q2 e^b D1]     K' = [K1~ D2 ; K2~]
//   Aq' = [[Aq1, 0], [Q2 e^b K1~^T, Aq2]],   e^{b_end}' = D1 D2
// and one step of the plain recurrence on it:
//   u = U' - W' S0,   O = scale (Q' S0 + Aq' u),   S <- D1 D2 S0 + K'^T u.
// Only S -> u -> S is sequential, once per 128 tokens.
//
// Products (tcgen05, bf16 operands in shared memory, fp32 in TMEM):
//   composition of a pair (a second issuing thread, off the state chain)
//     [Q2 e^b ; -W2] K1~^T  -> [Aq21 ; -M]                          "c1"
//     [x ; -M] [-W1 | U1]   on top of [. ; -W2 D1 | . ; U2]
//                            (x: whatever precedes -M in shared memory)
//                            -> [. ; -W2' | . ; U2']                 "c2"
//   the step
//     U' accumulator += (-W') S0;   O = Q' S0                        "u"
//     S += K'^T u                                                    "s"
//     O += [Aq1 ; Aq21] u[0:64];   X = [Aq21 ; Aq2] u[64:128]        "o"
//     (X lands in the dead u accumulator; O rows 64..127 add its
//     lanes 64..127)
// Warp roles, joined by mbarriers only:
//   warps 0..7    state: u (TMEM) -> bf16 operand tile; S -> bf16 operand
//                 tile, then (gated) S *= e^{b_end}' of the next pair in TMEM
//   warps 8..11   composition: c1 -> Aq21 and -M tiles, accumulator
//                 preloads; c2 -> -W2' tile; U1 preload; (gated) the D1 and
//                 D2 column scalings of Q2 e^b and K1~
//   warps 12..15  O -> scale -> bf16 -> global
//   warp 16       one thread issues the step's products
//   warp 17       one thread issues the composition's products
//   warp 18       one thread bulk-loads the pieces of each pair's two records
// A pair whose second chunk does not exist (a sequence's last 1..64 tokens)
// takes zero tiles in its place and skips the composition products.

#include "common.cuh"
#include "delta_tc.h"
#include "tc_tile.cuh"

namespace la {
namespace {

using namespace tc;
using namespace tile;

constexpr int D = 64;
constexpr int NT = 19 * 32;
constexpr int W_STATE_END = 8, W_COMP = 8, W_OUT = 12, W_ISSUE = 16, W_CISSUE = 17, W_LOAD = 18;
using Rec = Record<64>;

// Pieces of a 64-token record (d = 64): 8 KB tiles of 64 rows.
constexpr uint32_t P_NW = 0, P_QE = 8192, P_U = 16384, P_KT = 24576, P_AQ = Rec::AQ,
                   P_GEND = Rec::GEND, PIECE = 8192;

// Shared memory.  Per pair, one of two buffers (1024-byte aligned tiles):
//   WT  [-W1 ; -W2']  128-row tile (A of the u product)
//   U1  U1            (right after WT: [-W1 | U1] is the MN-major B of c2
//                      with a 16 KB stride between its two column groups)
//   QT  [Q1 e^b ; Q2 e^b]  128-row tile (A of O = Q' S)
//   W2  -W2           (right after QT: [Q2 e^b ; -W2] is the A of c1)
//   KT  [K1~ ; K2~]   128-row tile (MN-major A of the S product)
//   AQ  [Aq1 ; Aq21 ; Aq2]  (A of the two "o" products: rows 0..127 and
//                      rows 64..191 of this stack)
//   U2  U2
// then, once: the bf16 S tile, the bf16 u tile and right after it the -M
// tile (the u tile's rows 64..127 and -M together are the A of c2, whose
// first 64 rows only feed dead accumulator lanes), e^{b_end} of both
// chunks per buffer, mbarriers.
struct Layout {
    static constexpr uint32_t WT = 0, U1 = 16384, QT = 24576, W2 = 40960, KT = 49152,
                              AQ = 65536, U2 = 90112, BUF = 98304;
    static constexpr uint32_t BUF0 = 0;
    static constexpr uint32_t SB = 2 * BUF;              // S, bf16 [64][64]
    static constexpr uint32_t UT = SB + PIECE;           // u, bf16 [128][64]
    static constexpr uint32_t MT = UT + 2 * PIECE;       // -M, bf16 [64][64]
    static constexpr uint32_t G = MT + PIECE;            // fp32 [2 buffers][2 chunks][64]
    static constexpr uint32_t BARS = G + 2 * 2 * 64 * 4;
    static constexpr uint32_t TOTAL = BARS + 256;
    static_assert(QT + 16384 == W2 && WT + 16384 == U1 && UT + 16384 == MT, "stacked operands");
    static_assert(TOTAL + 1024 <= 227 * 1024, "shared memory budget");
};

enum : int {
    B_REC0 = 0, B_REC1, B_FREE0, B_FREE1, B_U, B_S, B_O, B_SREADY, B_UREADY, B_PREADY0,
    B_PREADY1, B_C1, B_CREADY, B_C2, B_OFREE0, B_OFREE1, B_COUNT
};
constexpr uint32_t N_STATE = 8, N_COMP = 4, N_OUT = 4;  // arrivals per phase

// TMEM columns: S (M = 64), two O accumulators, and per buffer a 64-column
// scratch block Wp directly before the U' accumulator, so that [Wp | U] is
// the 128-column accumulator of c2.
struct Cols {
    static constexpr uint32_t S = 0, O0 = 64, WP0 = 192, TOTAL = 512;
    static constexpr uint32_t o(int b) { return O0 + 64u * (uint32_t)b; }
    static constexpr uint32_t wp(int b) { return WP0 + 128u * (uint32_t)b; }
    static constexpr uint32_t u(int b) { return wp(b) + 64u; }
};

struct Inter128Params {
    const uint8_t *records;   // [slots][H] 64-token records
    __nv_bfloat16 *o;
    const int32_t *cu_seqlens;
    const float *init_S;
    float *final_S;
    unsigned *err;
    int H, ntok;
    float scale;
};

// One thread per row of a 64-column bf16 tile: columns [0, 64) of TMEM lane
// `row` into tile row `row` (rows of 128 bytes, 128-byte swizzled).
__device__ __forceinline__ void tmem_row_to_tile(uint32_t taddr, uint8_t *tile, int rows, int row) {
#pragma unroll
    for (int cb = 0; cb < D; cb += 32) {
        float v[32];
        tmem_ld32(taddr + cb, v);
#pragma unroll
        for (int i = 0; i < 32; i += 8) st_bf16x8(tile, rows, row, cb + i, v + i);
    }
}

// Tile row `row` (64 bf16), each column c times f[c] (f null: 1), into
// TMEM columns [0, 64) of this thread's lane.
__device__ __forceinline__ void tile_row_to_tmem(const uint8_t *tile, int rows, int row,
                                                 const float *f, uint32_t taddr) {
#pragma unroll
    for (int cb = 0; cb < D; cb += 16) {
        float v[16];
        unpack8(*reinterpret_cast<const uint4 *>(tile + rs_off(rows, row, cb)), v);
        unpack8(*reinterpret_cast<const uint4 *>(tile + rs_off(rows, row, cb + 8)), v + 8);
        if (f) {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] *= f[cb + i];
        }
        tmem_st16(taddr + cb, v);
    }
}

// Tile row `row` times f[c] per column, in place.
__device__ __forceinline__ void scale_tile_row(uint8_t *tile, int rows, int row, const float *f) {
#pragma unroll
    for (int cb = 0; cb < D; cb += 8) {
        uint4 *p = reinterpret_cast<uint4 *>(tile + rs_off(rows, row, cb));
        float v[8];
        unpack8(*p, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] *= f[cb + i];
        *p = pack8(v);
    }
}

template <bool GATED>
__global__ void __launch_bounds__(NT, 1) delta_inter128_kernel(Inter128Params p) {
    using L = Layout;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sb = sm + L::SB, *ut = sm + L::UT, *mt = sm + L::MT;
    float *gend = reinterpret_cast<float *>(sm + L::G);  // [buffer][chunk][64]
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::BARS);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + B_COUNT);
    int *s_loads = reinterpret_cast<int *>(tslot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qd = warp & 3;  // TMEM lane quarter
    const int h = blockIdx.x, n = blockIdx.y, H = p.H;
    int t_begin = p.cu_seqlens[n], t_end = p.cu_seqlens[n + 1];
    if (t_begin < 0 || t_end < t_begin || t_end > p.ntok) {
        if (tid == 0) atomicCAS(p.err, 0u, 100u);
        t_begin = t_end = 0;
    }
    const int np = (t_end - t_begin + 127) / 128;  // 128-token chunks
    // 64-token chunk j of this sequence sits in slot t_begin / 64 + n + j
    const int64_t slot0 = (int64_t)(t_begin / C) + n;
    auto rec = [&](int j) { return p.records + ((slot0 + j) * H + h) * (int64_t)Rec::BYTES; };
    auto has2 = [&](int c) { return t_begin + 128 * c + 64 < t_end; };
    auto buf = [&](int c) { return sm + L::BUF0 + (uint32_t)(c & 1) * L::BUF; };
    auto g_of = [&](int c, int k) { return gend + ((c & 1) * 2 + k) * 64; };
    auto rec_bar = [&](int c) { return &bars[B_REC0 + (c & 1)]; };
    auto rec_par = [](int c) { return (uint32_t)(c >> 1) & 1u; };
    auto free_bar = [&](int c) { return &bars[B_FREE0 + (c & 1)]; };
    auto ofree = [&](int c) { return &bars[B_OFREE0 + (c & 1)]; };
    // one phase per use of a buffer, so that no waiter can fall two phases
    // behind (the next use of a buffer waits for this pair's step)
    auto pready = [&](int c) { return &bars[B_PREADY0 + (c & 1)]; };

    if (tid == 0) {
        mbar_init(&bars[B_REC0], 1);
        mbar_init(&bars[B_REC1], 1);
        mbar_init(&bars[B_FREE0], 1);
        mbar_init(&bars[B_FREE1], 1);
        mbar_init(&bars[B_U], 1);
        mbar_init(&bars[B_S], 1);
        mbar_init(&bars[B_O], 1);
        mbar_init(&bars[B_SREADY], N_STATE);
        mbar_init(&bars[B_UREADY], N_STATE);
        mbar_init(&bars[B_PREADY0], N_COMP);
        mbar_init(&bars[B_PREADY1], N_COMP);
        mbar_init(&bars[B_C1], 1);
        mbar_init(&bars[B_CREADY], N_COMP);
        mbar_init(&bars[B_C2], 1);
        mbar_init(&bars[B_OFREE0], N_OUT);
        mbar_init(&bars[B_OFREE1], N_OUT);
        fence_mbar_init();
        *s_loads = 0;
    }
    if (warp == 0) {
        tmem_alloc(tslot, Cols::TOTAL);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the records come from the intra-chunk kernel (launched just before)
    grid_wait_prerequisites();
    const uint32_t tmem = *tslot;
    const uint32_t tq = tmem + ((uint32_t)(32 * qd) << 16);  // this warp's lane quarter
    const int64_t sbase = ((int64_t)n * H + h) * D * D;
    auto warp_arrive = [&](uint64_t *bar) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar);
    };

    if (warp == W_LOAD) {
        // ================================================= loader
        // Pair c goes into buffer c % 2 once pair c - 2's products have
        // completed ("free" commit).
        if (lane == 0) {
            const uint64_t pol = l2_evict_first();
            for (int c = 0; c < np; ++c) {
                if (c >= 2 && !mbar_wait(free_bar(c), (uint32_t)((c - 2) >> 1) & 1u, p.err, 60)) break;
                const bool two = has2(c);
                uint8_t *bf = buf(c);
                const uint8_t *r0 = rec(2 * c);
                const uint32_t gb = GATED ? 4u * D : 0u;
                const uint32_t bytes = 5u * PIECE + gb + (two ? 5u * PIECE + gb : 0u);
                fence_proxy_async();
                mbar_arrive_expect_tx(rec_bar(c), bytes);
                bulk_load_hint(bf + L::WT, r0 + P_NW, PIECE, rec_bar(c), pol);
                bulk_load_hint(bf + L::QT, r0 + P_QE, PIECE, rec_bar(c), pol);
                bulk_load_hint(bf + L::U1, r0 + P_U, PIECE, rec_bar(c), pol);
                bulk_load_hint(bf + L::KT, r0 + P_KT, PIECE, rec_bar(c), pol);
                bulk_load_hint(bf + L::AQ, r0 + P_AQ, PIECE, rec_bar(c), pol);
                if (GATED) bulk_load_hint(g_of(c, 0), r0 + P_GEND, gb, rec_bar(c), pol);
                if (two) {
                    const uint8_t *r1 = rec(2 * c + 1);
                    bulk_load_hint(bf + L::W2, r1 + P_NW, PIECE, rec_bar(c), pol);
                    bulk_load_hint(bf + L::QT + PIECE, r1 + P_QE, PIECE, rec_bar(c), pol);
                    bulk_load_hint(bf + L::U2, r1 + P_U, PIECE, rec_bar(c), pol);
                    bulk_load_hint(bf + L::KT + PIECE, r1 + P_KT, PIECE, rec_bar(c), pol);
                    bulk_load_hint(bf + L::AQ + 2 * PIECE, r1 + P_AQ, PIECE, rec_bar(c), pol);
                    if (GATED) bulk_load_hint(g_of(c, 1), r1 + P_GEND, gb, rec_bar(c), pol);
                }
                *s_loads = c + 1;
            }
        }
    } else if (warp == W_ISSUE) {
        // ================================================= the step's products
        if (lane == 0 && np > 0) {
            constexpr uint32_t id128 = idesc_bf16(128, D, false, true);   // K-major A, MN-major B
            constexpr uint32_t ids = idesc_bf16(D, D, true, true);        // S += K'^T u
            const uint64_t bS = mdesc(sb, D, 0, 0);
            const uint64_t bU0 = mdesc(ut, 128, 0, 0), bU1 = mdesc(ut, 128, 64, 0);
            for (int c = 0; c < np; ++c) {
                const int b = c & 1;
                uint8_t *bf = buf(c);
                // S tile of the pair's start; pair composed, U' preloaded
                if (!mbar_wait(&bars[B_SREADY], (uint32_t)c & 1u, p.err, 62)) break;
                if (!mbar_wait(pready(c), rec_par(c), p.err, 63)) break;
                tc_fence_after();
                const uint64_t aW = kdesc(bf + L::WT, 128, 0, 0), aQ = kdesc(bf + L::QT, 128, 0, 0);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tmem + Cols::u(b), dstep(aW, kstep_units(128, s)), dstep(bS, s * 128), id128, 1);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tmem + Cols::o(b), dstep(aQ, kstep_units(128, s)), dstep(bS, s * 128), id128,
                             s > 0);
                mma_commit(&bars[B_U]);
                // u tile written (and the u accumulator read)
                if (!mbar_wait(&bars[B_UREADY], (uint32_t)c & 1u, p.err, 64)) break;
                tc_fence_after();
                const uint64_t aK = mdesc(bf + L::KT, 128, 0, 0);
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_bf16(tmem + Cols::S, dstep(aK, s * 128), dstep(bU0, s * 128), ids, 1);
                mma_commit(&bars[B_S]);
                const uint64_t aA0 = kdesc(bf + L::AQ, 128, 0, 0), aA1 = kdesc(bf + L::AQ + PIECE, 128, 0, 0);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tmem + Cols::o(b), dstep(aA0, s * 2), dstep(bU0, s * 128), id128, 1);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tmem + Cols::u(b), dstep(aA1, s * 2), dstep(bU1, s * 128), id128, s > 0);
                mma_commit(free_bar(c));
                // the output warps have taken pair c - 1 (so seen its "o"
                // phase) before this pair's "o" phase can complete
                if (c >= 1 && !mbar_wait(ofree(c - 1), (uint32_t)(((c - 1) >> 1) + 1) & 1u, p.err, 68))
                    break;
                mma_commit(&bars[B_O]);
            }
        }
    } else if (warp == W_CISSUE) {
        // ================================================= the composition's products
        if (lane == 0) {
            constexpr uint32_t idc1 = idesc_bf16(128, 64, false, false);
            constexpr uint32_t idc2 = idesc_bf16(128, 128, false, true);
            uint32_t ncomp = 0;
            for (int c = 0; c < np && has2(c); ++c) {
                const int b = c & 1;
                uint8_t *bf = buf(c);
                // c1 writes only this buffer's scratch columns, free since pair
                // c - 2's composition (its records were loaded after that
                // pair's step); the composition warps have taken the previous
                // c1 (this thread waited for their "ready" before the previous
                // c2), so the c1 barrier cannot run two phases ahead of them
                if (!mbar_wait(rec_bar(c), rec_par(c), p.err, 65)) break;
                tc_fence_after();
                const uint64_t a1 = kdesc(bf + L::QT + PIECE, 128, 0, 0), b1 = kdesc(bf + L::KT, 128, 0, 0);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tmem + Cols::wp(b), dstep(a1, s * 2), dstep(b1, s * 2), idc1, s > 0);
                mma_commit(&bars[B_C1]);
                if (!mbar_wait(&bars[B_CREADY], ncomp & 1u, p.err, 67)) break;
                tc_fence_after();
                const uint64_t a2 = kdesc(ut + PIECE, 128, 0, 0);  // [u rows 64..127 ; -M]
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tmem + Cols::wp(b), dstep(a2, s * 2),
                             smem_desc_sw128(smem_u32(bf + L::WT) + (uint32_t)s * 2048u, 16384u, 1024u),
                             idc2, 1);
                mma_commit(&bars[B_C2]);
                ++ncomp;
            }
        }
    } else if (warp >= W_COMP && warp < W_OUT) {
        // ================================================= composition warps
        // Warp 8 + q reads and writes TMEM lanes 32q .. 32q + 31.
        uint32_t ncomp = 0;
        for (int c = 0; c < np; ++c) {
            const int b = c & 1;
            uint8_t *bf = buf(c);
            // the pair's records; the U' accumulator of pair c - 2 read out
            if (!mbar_wait(rec_bar(c), rec_par(c), p.err, 70)) break;
            if (!mbar_wait(ofree(c), (uint32_t)(c >> 1) & 1u, p.err, 71)) break;
            tc_fence_after();
            const uint32_t twp = tq + Cols::wp(b), tu = tq + Cols::u(b);
            if (!has2(c)) {
                // no second chunk: zero tiles for -W2', Q2 e^b, K2~, Aq21, Aq2;
                // U' = [U1 ; 0]
                const int t = tid - W_COMP * 32;
                auto zbase = [&](int r) -> uint8_t * {
                    return bf + (r == 0 ? L::WT + PIECE
                                        : r == 1 ? L::QT + PIECE
                                                 : r == 2 ? L::KT + PIECE : L::AQ + (uint32_t)(r - 2) * PIECE);
                };
                for (int i = t; i < 5 * (int)(PIECE / 16); i += 4 * 32)
                    *reinterpret_cast<uint4 *>(zbase(i / (PIECE / 16)) + (i % (PIECE / 16)) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                if (qd < 2) {
                    tile_row_to_tmem(bf + L::U1, 64, 32 * qd + lane, nullptr, tu);
                } else {
                    float z[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) z[i] = 0.0f;
#pragma unroll
                    for (int cb = 0; cb < D; cb += 16) tmem_st16(tu + cb, z);
                }
                fence_proxy_async();
                warp_arrive(pready(c));
                continue;
            }
            // c1: Aq21 in lanes 0..63, -M in lanes 64..127
            if (!mbar_wait(&bars[B_C1], ncomp & 1u, p.err, 72)) break;
            tc_fence_after();
            const float *d1 = GATED ? g_of(c, 0) : nullptr;
            const float *d2 = GATED ? g_of(c, 1) : nullptr;
            if (qd < 2) {
                const int r = 32 * qd + lane;
                tmem_row_to_tile(twp, bf + L::AQ + PIECE, 64, r);  // Aq21 row r
                if (GATED) {
                    scale_tile_row(bf + L::QT + PIECE, 64, r, d1);  // Q2 e^b D1
                    scale_tile_row(bf + L::KT, 64, r, d2);          // K1~ D2
                }
            } else {
                const int r = 32 * (qd - 2) + lane;
                tmem_row_to_tile(twp, mt, 64, r);                   // -M row r
                tile_row_to_tmem(bf + L::W2, 64, r, d1, twp);       // c2 adds onto -W2 D1
                tile_row_to_tmem(bf + L::U2, 64, r, nullptr, tu);   // and onto U2
            }
            fence_proxy_async();
            warp_arrive(&bars[B_CREADY]);
            // c2: -W2' in lanes 64..127 of the W part, U2' in those of U'
            if (!mbar_wait(&bars[B_C2], ncomp & 1u, p.err, 73)) break;
            tc_fence_after();
            if (qd < 2) tile_row_to_tmem(bf + L::U1, 64, 32 * qd + lane, nullptr, tu);
            else tmem_row_to_tile(twp, bf + L::WT + PIECE, 64, 32 * (qd - 2) + lane);
            fence_proxy_async();
            warp_arrive(pready(c));
            ++ncomp;
        }
    } else if (warp < W_STATE_END) {
        // ================================================= state (and u) warps
        const int c0 = 32 * (warp >> 2);             // this warp's column half
        const int srow = acc_row(D, qd, lane);       // state row (key channel), or -1
        const int urow = 32 * qd + lane;             // u row (token of the pair)
        // e^{b_end} of pair c for key channel `row`
        auto decay_of = [&](int c, int row) -> float {
            if (!GATED || row < 0) return 1.0f;
            const float d = g_of(c, 0)[row];
            return has2(c) ? d * g_of(c, 1)[row] : d;
        };
        bool ok = true;
        if (GATED && np > 0) ok = mbar_wait(rec_bar(0), 0, p.err, 74);
        if (ok) {
            // initial state: bf16 operand copy; TMEM state decayed by pair 0's e^{b_end}
            const float gd = np > 0 ? decay_of(0, srow) : 1.0f;
#pragma unroll
            for (int cb = 0; cb < 32; cb += 16) {
                const int col = c0 + cb;
                float v[16];
                if (srow >= 0 && p.init_S) {
                    const float4 *src = reinterpret_cast<const float4 *>(p.init_S + sbase + (int64_t)srow * D + col);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float4 f = src[i];
                        v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = 0.0f;
                }
                if (srow >= 0) {
                    st_bf16x8(sb, D, srow, col, v);
                    st_bf16x8(sb, D, srow, col + 8, v + 8);
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] *= gd;
                tmem_st16(tq + Cols::S + col, v);
            }
            fence_proxy_async();
            warp_arrive(&bars[B_SREADY]);
        }
        for (int c = 0; c < np && ok; ++c) {
            const int b = c & 1;
            // ---- u -> bf16 operand tile
            if (!(ok = mbar_wait(&bars[B_U], (uint32_t)c & 1u, p.err, 75))) break;
            tc_fence_after();
            {
                float v[32];
                tmem_ld32(tq + Cols::u(b) + c0, v);
#pragma unroll
                for (int i = 0; i < 32; i += 8) st_bf16x8(ut, 128, urow, c0 + i, v + i);
            }
            fence_proxy_async();
            warp_arrive(&bars[B_UREADY]);
            // ---- S after this pair
            if (!(ok = mbar_wait(&bars[B_S], (uint32_t)c & 1u, p.err, 76))) break;
            tc_fence_after();
            if (c + 1 < np) {
                float v[32];
                tmem_ld32(tq + Cols::S + c0, v);
                if (srow >= 0) {
#pragma unroll
                    for (int i = 0; i < 32; i += 8) st_bf16x8(sb, D, srow, c0 + i, v + i);
                }
                fence_proxy_async();
                warp_arrive(&bars[B_SREADY]);
                if (GATED) {
                    // decay for the next pair (needs its records' e^{b_end})
                    if (!(ok = mbar_wait(rec_bar(c + 1), rec_par(c + 1), p.err, 77))) break;
                    const float gd = decay_of(c + 1, srow);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= gd;
                    tmem_st16(tq + Cols::S + c0, *reinterpret_cast<float(*)[16]>(v));
                    tmem_st16(tq + Cols::S + c0 + 16, *reinterpret_cast<float(*)[16]>(v + 16));
                }
            }
        }
        // ---- final state
        if (ok && p.final_S) {
#pragma unroll
            for (int cb = 0; cb < 32; cb += 16) {
                float v[16];
                tmem_ld16(tq + Cols::S + c0 + cb, v);
                if (srow >= 0) {
                    float4 *dst = reinterpret_cast<float4 *>(p.final_S + sbase + (int64_t)srow * D + c0 + cb);
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                }
            }
        }
    } else if (warp >= W_OUT && warp < W_ISSUE) {
        // ================================================= output warps
        const int r = 32 * qd + lane;  // row of the 128-token chunk
        warp_arrive(ofree(0));
        warp_arrive(ofree(1));
        for (int c = 0; c < np; ++c) {
            const int b = c & 1;
            if (!mbar_wait(&bars[B_O], (uint32_t)c & 1u, p.err, 78)) break;
            tc_fence_after();
            const int tok = t_begin + 128 * c + r;
            const bool valid = tok < t_end;
#pragma unroll
            for (int cb = 0; cb < D; cb += 32) {
                float v[32];
                tmem_ld32(tq + Cols::o(b) + cb, v);
                if (qd >= 2) {
                    // rows 64..127 also hold Aq2 u2 in the dead u accumulator
                    float x[32];
                    tmem_ld32(tq + Cols::u(b) + cb, x);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] += x[i];
                }
                if (valid) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= p.scale;
                    uint4 *dst = reinterpret_cast<uint4 *>(p.o + ((int64_t)tok * H + h) * D + cb);
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[i] = pack8(v + 8 * i);
                }
            }
            warp_arrive(ofree(c));
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        // the last load into each buffer (earlier ones completed before it was issued)
        const int K = *s_loads;
        for (int j = K - 2 > 0 ? K - 2 : 0; j < K; ++j) mbar_wait(rec_bar(j), rec_par(j), p.err, 69);
    }
    if (warp == 0) tmem_dealloc(tmem, Cols::TOTAL);
}

template <bool GATED>
cudaError_t launch_t(const TcLaunch &x, cudaStream_t s) {
    const PrefillArgs &a = *x.a;
    Inter128Params p{x.records, static_cast<__nv_bfloat16 *>(a.o), a.cu_seqlens, a.init_S,
                     a.final_S, x.err, a.H, a.ntok, a.scale};
    constexpr size_t smem = Layout::TOTAL + 1024;
    auto kern = delta_inter128_kernel<GATED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_programmatic(kern, dim3(a.H, a.N), dim3(NT), smem, s, p);
}

}  // namespace

cudaError_t launch_delta_inter128(const TcLaunch &x, cudaStream_t s) {
    return x.a->gate_logits != nullptr ? launch_t<true>(x, s) : launch_t<false>(x, s);
}

}  // namespace la
