// delta_bwd_tc.cu -- chunkwise backward pass of the delta rule (bf16 I/O,
// dk = dv in {64, 128}, any gate, either update rule): the forward pass with its records, the
// reverse chain over the chunks, then the per-chunk gradients
// (delta_bwd_channel.cu).
//
// The page ("From GPT-2 to Kimi K3, explained", section DeltaNet
// (Parallelizing Linear Transformers with Delta Rule), eq. 8-10) gives the
// chunkwise forward pass; this is its derivative, chunk by chunk.  Per chunk
// of C = 64 tokens, with b_r the cumulative log decay inside the chunk,
//   u = U - W S,  O = scale ((Q e^b) S + Aq u),  S' = Diag(e^{b_L}) S + K~^T u
// (K~ = K e^{b_L - b}), so with dO' = scale dO and dS' the gradient of the
// next chunk's state, the only sequential dependence is
//   du = Aq^T dO' + K~ dS',   dS = Diag(e^{b_L}) dS' + (Q e^b)^T dO' - W^T du.
// Launches:
//   the tensor-core forward pass, keeping its records (-W, Q e^b, U, K~, Aq,
//     e^{b_L}), T of every chunk, and the state at every chunk start;
//   delta_bwd_chain_kernel   one CTA per (head, sequence): dS from the last
//                            chunk to the first on tcgen05, dS in TMEM, the
//                            record tiles as the products' operands in place;
//                            stores dS' and du of every chunk;
//   delta_bwd_channel_kernel every (chunk, head) in parallel: the gradients of
//                            the chunk's inputs and the prologue's derivatives.

#include "common.cuh"
#include "delta_tc.h"
#include "launch.h"
#include "tc_tile.cuh"

namespace la {
namespace {

using tile::C;
struct ChainParams {
    const uint8_t *records;   // [slots][H] forward records
    const __nv_bfloat16 *d_o;
    const int32_t *cu;
    const float *d_final_S;
    // per (slot, head), by 16-byte units (tile::unit_at):
    float *dstates;           // [slots][H] D x D: dS' of every chunk (fp32; gated)
    __nv_bfloat16 *dstates16; // [slots][H] D x D: dS' of every chunk (bf16; no gate)
    __nv_bfloat16 *du;        // null, or [slots][H] 64 x D: du of every chunk (bf16)
    float *d_init_S;
    unsigned *err;
    int H, ntok;
    float scale;
};

// One CTA of 11 warps per (head, sequence).  Shared memory (bytes, from a
// 1024-aligned base): NB record buffers (the operands of one chunk copied
// from its record: [-W ; Q e^b] as a 128-row swizzled tile, K e^{b_L - b}
// as a 64-row one, Aq, e^{b_L}), NB bf16 tiles of scale dO, the bf16
// operand tiles of dS' and du, barriers.  TMEM: dS (fp32, M = D rows) in
// columns 0 .. D-1, du (M = 64) in columns D .. 2D-1.
template <int D> struct ChainCfg {
    static constexpr int NB = D == 64 ? 4 : 2;            // record and dO buffers
    static constexpr int NT = 11 * 32;
    static constexpr int W_DO = 8, N_DO = 2, W_ISSUER = 10;   // dO warps 8, 9; issuing warp
    static constexpr uint32_t WQB = 128 * D * 2, KB = 64 * D * 2, AQB = 64 * 64 * 2, GB = 4 * D;
    static constexpr uint32_t TX = WQB + KB + AQB + GB;   // bytes a record copy delivers
    static constexpr uint32_t BUF = (TX + 1023) & ~1023u;
    static constexpr uint32_t DOB = 64 * D * 2;           // scale dO, bf16 [64][D] tile
    static constexpr uint32_t DO = NB * BUF;
    static constexpr uint32_t DS = DO + NB * DOB;         // dS', bf16 [D][D] tile
    static constexpr uint32_t DU = DS + D * D * 2;        // du, bf16 [64][D] tile
    static constexpr uint32_t BARS = DU + 64 * D * 2;
    static constexpr uint32_t BYTES = BARS + 256;
    static constexpr uint32_t TDS = 0, TDU = D, TCOLS = 2 * D;
    static constexpr int DO_UNITS = 64 * D / 8 / (32 * N_DO);   // 16-byte units of dO per staging thread
    static_assert(BYTES + 1024 <= 232448, "shared memory budget");
    static_assert(NB <= 4, "four mbarrier slots per kind of buffer");
};

// mbarrier slots: per step, then per buffer (REC: record copy landed; DO:
// dO tile written; FREE: every product reading the buffer has completed)
enum : int {
    CB_DSREADY = 0, CB_DU, CB_DUREADY, CB_DS, CB_END, CB_REC0,
    CB_DO0 = CB_REC0 + 4, CB_FREE0 = CB_DO0 + 4, CB_COUNT = CB_FREE0 + 4
};

// Reverse pass over the chunks of one (head, sequence) on the tensor cores.
// Step i handles chunk c = nc - 1 - i; dS (fp32) stays in TMEM throughout:
//   readback warps  dS' (TMEM) -> global (fp32 gated, else bf16) and its bf16
//                   operand tile; gated: dS' *= e^{b_L} back into TMEM
//   issuer          du = Aq^T dO' (ahead, as soon as the chunk's record and
//                   dO' are in) + K~ dS'                          commit "du"
//                   dS += (Q e^b)^T dO'
//   readback warps  du (TMEM) -> bf16 operand tile and global
//   issuer          dS += (-W)^T du                               commit "ds"
// with dO' = scale dO rounded to bf16 by two staging warps, up to NB - 1
// chunks ahead.  Only dS' -> du -> dS is sequential: two product round trips
// per chunk.  Every mbarrier phase is chained so that no waiter can fall two
// phases behind: a phase of DSREADY / DUREADY / DU / DS needs the previous
// phase's waiter to have gone on; a buffer's REC / DO / FREE phase for use
// u + 1 needs its use u to have been waited for.  Every wait is bounded.
// (11 warps, not 13 with four staging warps: an SM sub-partition's 16 K
// registers then hold three warps of up to 168 registers, where the gated
// d = 128 readback -- a row's 64 dS' columns and their scaled copies --
// needs more than the 128 that four warps would leave.)
template <int D, bool GATED>
__global__ void __launch_bounds__(ChainCfg<D>::NT, 1) delta_bwd_chain_kernel(ChainParams p) {
    using namespace tc;
    using namespace tile;
    using L = ChainCfg<D>;
    using Rec = Record<D>;
    constexpr int NB = L::NB, HALF = D / 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::BARS);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + CB_COUNT);
    uint8_t *sds = sm + L::DS, *sdu = sm + L::DU;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, qd = warp & 3;
    const int h = blockIdx.x, n = blockIdx.y, H = p.H;
    int t_begin = p.cu[n], t_end = p.cu[n + 1];
    if (t_begin < 0 || t_end < t_begin || t_end > p.ntok) {
        if (tid == 0) atomicCAS(p.err, 0u, 100u);
        t_begin = t_end = 0;
    }
    const int nc = (t_end - t_begin + C - 1) / C;
    const int64_t slot0 = (int64_t)(t_begin / C) + n;
    const int64_t sbase = ((int64_t)n * H + h) * D * D;
    auto rec_buf = [&](int i) { return sm + (uint32_t)(i % NB) * L::BUF; };
    auto do_buf = [&](int i) { return sm + L::DO + (uint32_t)(i % NB) * L::DOB; };
    auto use_par = [](int i) { return (uint32_t)(i / NB) & 1u; };
    auto gend_of = [&](int i) { return reinterpret_cast<const float *>(rec_buf(i) + L::WQB + L::KB + L::AQB); };
    // step i's record (chunk nc - 1 - i) into buffer i % NB: [-W ; Q e^b],
    // rows 64..127 of each 64-column block of [U ; K~], Aq, e^{b_L}
    auto issue_rec = [&](int i) {
        uint8_t *buf = rec_buf(i);
        uint64_t *bar = &bars[CB_REC0 + i % NB];
        const uint8_t *rec = p.records + ((slot0 + (nc - 1 - i)) * H + h) * (int64_t)Rec::BYTES;
        fence_proxy_async();
        mbar_arrive_expect_tx(bar, L::TX);
        bulk_load(buf, rec + Rec::WQ, L::WQB, bar);
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb)
            bulk_load(buf + L::WQB + cb * 8192, rec + Rec::UK + cb * 16384 + 8192, 8192, bar);
        bulk_load(buf + L::WQB + L::KB, rec + Rec::AQ, L::AQB, bar);
        bulk_load(buf + L::WQB + L::KB + L::AQB, rec + Rec::GEND, L::GB, bar);
    };
    // a wait whose outcome is the same in every lane of the warp (the TMEM
    // accesses after it are warp-collective)
    auto wwait = [&](int bar, uint32_t parity, unsigned code) {
        return __all_sync(0xffffffffu, mbar_wait(&bars[bar], parity, p.err, code));
    };
    auto warp_arrive = [&](int bar) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[bar]);
    };

    if (tid == 0) {
        mbar_init(&bars[CB_DSREADY], 8);
        mbar_init(&bars[CB_DU], 1);
        mbar_init(&bars[CB_DUREADY], 8);
        mbar_init(&bars[CB_DS], 1);
        mbar_init(&bars[CB_END], 1);
        for (int b = 0; b < NB; ++b) {
            mbar_init(&bars[CB_REC0 + b], 1);
            mbar_init(&bars[CB_DO0 + b], L::N_DO);
            mbar_init(&bars[CB_FREE0 + b], 1);
        }
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, L::TCOLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tq = tmem + ((uint32_t)(32 * qd) << 16);  // this warp's lane quarter

    if (warp == L::W_ISSUER) {
        // ================================================= issuer
        if (lane == 0 && nc > 0) {
            constexpr uint32_t id_aq = idesc_bf16(64, D, true, true);   // Aq^T dO'
            constexpr uint32_t id_k = idesc_bf16(64, D, false, true);   // K~ dS'
            constexpr uint32_t id_s = idesc_bf16(D, D, true, true);     // (Q e^b)^T dO', (-W)^T du
            const uint64_t bS = mdesc(sds, D, 0, 0), bU = mdesc(sdu, C, 0, 0);
            int issued = 0, waited = 0;
            for (; issued < NB && issued < nc; ++issued) issue_rec(issued);
            for (int i = 0; i < nc; ++i) {
                const int b = i % NB;
                const uint8_t *rb = rec_buf(i);
                if (!mbar_wait(&bars[CB_REC0 + b], use_par(i), p.err, 40)) break;
                waited = i + 1;
                if (!mbar_wait(&bars[CB_DO0 + b], use_par(i), p.err, 41)) break;
                tc_fence_after();
                const uint64_t bO = mdesc(do_buf(i), C, 0, 0);
                const uint64_t aA = mdesc(rb + L::WQB + L::KB, C, 0, 0);
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4)
                    mma_bf16(tmem + L::TDU, dstep(aA, s4 * 128), dstep(bO, s4 * 128), id_aq, s4 > 0 ? 1u : 0u);
                // dS' of this chunk in TMEM (scaled) and as the bf16 tile
                if (!mbar_wait(&bars[CB_DSREADY], (uint32_t)i & 1u, p.err, 42)) break;
                tc_fence_after();
                const uint64_t aK = kdesc(rb + L::WQB, C, 0, 0);
#pragma unroll
                for (int s = 0; s < D / 16; ++s)
                    mma_bf16(tmem + L::TDU, dstep(aK, kstep_units(C, s)), dstep(bS, s * 128), id_k, 1);
                mma_commit(&bars[CB_DU]);
                const uint64_t aQ = mdesc(rb, 128, 64, 0);
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4)
                    mma_bf16(tmem + L::TDS, dstep(aQ, s4 * 128), dstep(bO, s4 * 128), id_s, 1);
                // step i - 1's products have completed (its "ds" phase came before
                // this step's DSREADY): its buffer takes step i + NB - 1
                if (i >= 1 && issued < nc) issue_rec(issued++);
                if (!mbar_wait(&bars[CB_DUREADY], (uint32_t)i & 1u, p.err, 43)) break;
                tc_fence_after();
                const uint64_t aW = mdesc(rb, 128, 0, 0);
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4)
                    mma_bf16(tmem + L::TDS, dstep(aW, s4 * 128), dstep(bU, s4 * 128), id_s, 1);
                mma_commit(&bars[CB_DS]);
                mma_commit(&bars[CB_FREE0 + b]);
            }
            // every product issued has completed before TMEM is released
            mma_commit(&bars[CB_END]);
            mbar_wait(&bars[CB_END], 0, p.err, 44);
            // record copies still in flight (only after a failed wait); at
            // most one per buffer
            for (int j = waited; j < issued; ++j) mbar_wait(&bars[CB_REC0 + j % NB], use_par(j), nullptr, 0u);
        }
    } else if (warp < 8) {
        // ================================================= readback warps
        const int c0 = (warp >> 2) * HALF;              // this warp's column half
        const int srow = tile::acc_row(D, qd, lane);    // dS row (key channel), or -1
        const int urow = tile::acc_row(C, qd, lane);    // du row (token), or -1
        bool ok = true;
        float v[HALF];                                   // row srow of dS', columns c0 ..
        for (int i = 0; i < nc && ok; ++i) {
            const int c = nc - 1 - i;
            if (i == 0) {
                // dS' of the last chunk: the final state's gradient
#pragma unroll
                for (int cb = 0; cb < HALF; cb += 4) {
                    const float4 f = (srow >= 0 && p.d_final_S)
                                         ? *reinterpret_cast<const float4 *>(p.d_final_S + sbase + (int64_t)srow * D + c0 + cb)
                                         : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    v[cb] = f.x; v[cb + 1] = f.y; v[cb + 2] = f.z; v[cb + 3] = f.w;
                }
            } else {
                if (!(ok = wwait(CB_DS, (uint32_t)(i - 1) & 1u, 45))) break;
                tc_fence_after();
#pragma unroll
                for (int cb = 0; cb < HALF; cb += 32)
                    tmem_ld32(tq + L::TDS + c0 + cb, *reinterpret_cast<float(*)[32]>(v + cb));
            }
            if (srow >= 0) {
#pragma unroll
                for (int cb = 0; cb < HALF; cb += 8) tile::st_bf16x8(sds, D, srow, c0 + cb, v + cb);
            }
            if (GATED) {
                // dS' * e^{b_L} back into TMEM, to accumulate the chunk's products on
                if (!(ok = wwait(CB_REC0 + i % NB, use_par(i), 46))) break;
                const float gd = srow >= 0 ? gend_of(i)[srow] : 1.0f;
#pragma unroll
                for (int cb = 0; cb < HALF; cb += 16) {
                    float x[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) x[j] = v[cb + j] * gd;
                    tmem_st16(tq + L::TDS + c0 + cb, x);
                }
            } else if (i == 0) {
#pragma unroll
                for (int cb = 0; cb < HALF; cb += 16)
                    tmem_st16(tq + L::TDS + c0 + cb, *reinterpret_cast<float(*)[16]>(v + cb));
            }
            fence_proxy_async();
            warp_arrive(CB_DSREADY);
            // dS' of chunk c out, for the per-chunk gradients, while du is formed
            // (16-byte units by column group: each store is a contiguous run)
            if (srow >= 0) {
                const int64_t o = ((slot0 + c) * H + h) * (int64_t)(D * D);
                if (GATED) {   // fp32: the per-chunk kernel also forms rowsum(dS' o S)
                    float4 *dst = reinterpret_cast<float4 *>(p.dstates + o);
#pragma unroll
                    for (int cb = 0; cb < HALF; cb += 4)
                        dst[unit_at(D, srow, (c0 + cb) / 4)] = make_float4(v[cb], v[cb + 1], v[cb + 2], v[cb + 3]);
                } else {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.dstates16 + o);
#pragma unroll
                    for (int cb = 0; cb < HALF; cb += 8) dst[unit_at(D, srow, (c0 + cb) / 8)] = pack8(v + cb);
                }
            }
            // du of the chunk -> bf16 operand tile and global
            if (!(ok = wwait(CB_DU, (uint32_t)i & 1u, 47))) break;
            tc_fence_after();
            float u[HALF];
#pragma unroll
            for (int cb = 0; cb < HALF; cb += 32)
                tmem_ld32(tq + L::TDU + c0 + cb, *reinterpret_cast<float(*)[32]>(u + cb));
            if (urow >= 0) {
#pragma unroll
                for (int cb = 0; cb < HALF; cb += 8) tile::st_bf16x8(sdu, C, urow, c0 + cb, u + cb);
            }
            fence_proxy_async();
            warp_arrive(CB_DUREADY);
            if (urow >= 0 && p.du) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.du + ((slot0 + c) * H + h) * (int64_t)(C * D));
#pragma unroll
                for (int cb = 0; cb < HALF; cb += 8) dst[unit_at(C, urow, (c0 + cb) / 8)] = pack8(u + cb);
            }
        }
        // the gradient of the initial state: dS after chunk 0's step
        if (ok && p.d_init_S) {
            if (nc > 0) {
                if (wwait(CB_DS, (uint32_t)(nc - 1) & 1u, 48)) {
                    tc_fence_after();
#pragma unroll
                    for (int cb = 0; cb < HALF; cb += 32)
                        tmem_ld32(tq + L::TDS + c0 + cb, *reinterpret_cast<float(*)[32]>(v + cb));
                } else {
                    ok = false;
                }
            } else {
#pragma unroll
                for (int cb = 0; cb < HALF; cb += 4) {
                    const float4 f = (srow >= 0 && p.d_final_S)
                                         ? *reinterpret_cast<const float4 *>(p.d_final_S + sbase + (int64_t)srow * D + c0 + cb)
                                         : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    v[cb] = f.x; v[cb + 1] = f.y; v[cb + 2] = f.z; v[cb + 3] = f.w;
                }
            }
            if (ok && srow >= 0) {
                float4 *dst = reinterpret_cast<float4 *>(p.d_init_S + sbase + (int64_t)srow * D + c0);
#pragma unroll
                for (int cb = 0; cb < HALF; cb += 4) dst[cb / 4] = make_float4(v[cb], v[cb + 1], v[cb + 2], v[cb + 3]);
            }
        }
    } else {
        // ================================================= dO staging warps (8, 9)
        const int st = tid - 32 * L::W_DO;   // 0 .. 63
        for (int j = 0; j < nc; ++j) {
            const int b = j % NB;
            // the buffer's previous use (step j - NB) has finished
            if (j >= NB && !wwait(CB_FREE0 + b, use_par(j - NB), 49)) break;
            const int tok0 = t_begin + (nc - 1 - j) * C, len = min(C, t_end - tok0);
            uint4 r[L::DO_UNITS];
#pragma unroll
            for (int k = 0; k < L::DO_UNITS; ++k) {
                const int un = st + 32 * L::N_DO * k, row = un / (D / 8), c8 = (un % (D / 8)) * 8;
                r[k] = row < len ? *reinterpret_cast<const uint4 *>(p.d_o + ((int64_t)(tok0 + row) * H + h) * D + c8)
                                 : make_uint4(0u, 0u, 0u, 0u);
            }
            uint8_t *dst = do_buf(j);
#pragma unroll
            for (int k = 0; k < L::DO_UNITS; ++k) {
                const int un = st + 32 * L::N_DO * k, row = un / (D / 8), c8 = (un % (D / 8)) * 8;
                float x[8];
                tile::unpack8(r[k], x);
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] *= p.scale;
                *reinterpret_cast<uint4 *>(dst + tile::rs_off(C, row, c8)) = tile::pack8(x);
            }
            fence_proxy_async();
            warp_arrive(CB_DO0 + b);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, L::TCOLS);
}

// ------------------------------------------------------------------ host

size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

struct ChunkWs {
    size_t fwd, states, dstates, dstates16, du, tiles, total;
};

ChunkWs chunk_ws(int N, int ntok, int H, int D) {
    const size_t slots = (size_t)tile::Workspace::slots(N, ntok);
    ChunkWs w;
    w.fwd = a256(delta_tc_workspace_bytes(N, ntok, H, D, D, 64, true));
    w.states = a256(slots * H * D * D * sizeof(float));
    w.dstates = w.states;
    w.dstates16 = a256(slots * H * D * D * 2);
    w.du = a256(slots * H * 64 * D * 2);   // du of every chunk, bf16
    w.tiles = a256(slots * H * 8192);   // T of every chunk (bf16 64 x 64)
    w.total = w.fwd + w.states + w.dstates + w.dstates16 + w.du + w.tiles;
    return w;
}

template <int D, bool GATED>
cudaError_t launch_chain(const ChainParams &cp, int N, int H, cudaStream_t s) {
    using L = ChainCfg<D>;
    const size_t smem = (size_t)L::BYTES + 1024;   // + alignment of the base
    auto kern = delta_bwd_chain_kernel<D, GATED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(H, N), L::NT, smem, s>>>(cp);
    return cudaGetLastError();
}

}  // namespace

bool delta_bwd_chunked_supported(const BwdArgs &a) {
    // the kernels move rows in 16-byte units (null pointers pass)
    auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const void *ptrs[] = {a.q, a.k, a.v, a.beta_logits, a.gate_logits, a.d_o, a.d_final_S, a.init_S,
                          a.dq, a.dk_out, a.dv_out, a.d_beta_logits, a.d_gate_logits, a.d_init_S};
    for (const void *p : ptrs)
        if (!al16(p)) return false;
    return a.bf16 && a.dk == a.dv && (a.dk == 64 || a.dk == 128);
}

size_t delta_bwd_chunked_workspace_bytes(int N, int ntok, int H, int D) {
    return chunk_ws(N, ntok, H, D).total;
}

namespace {

// The backward workspace's regions after the forward's own workspace.
struct ChunkPtrs {
    uint8_t *base;
    float *states, *dstates;
    __nv_bfloat16 *dstates16, *du;
    uint8_t *tiles;
};

ChunkPtrs chunk_ptrs(void *workspace, const ChunkWs &w) {
    ChunkPtrs c;
    c.base = static_cast<uint8_t *>(workspace);
    c.states = reinterpret_cast<float *>(c.base + w.fwd);
    c.dstates = reinterpret_cast<float *>(c.base + w.fwd + w.states);
    c.dstates16 = reinterpret_cast<__nv_bfloat16 *>(c.base + w.fwd + w.states + w.dstates);
    c.du = reinterpret_cast<__nv_bfloat16 *>(c.base + w.fwd + w.states + w.dstates + w.dstates16);
    c.tiles = c.base + w.fwd + w.states + w.dstates + w.dstates16 + w.du;
    return c;
}

// The forward pass with everything the gradients need kept in the backward
// workspace: its records and chunk table, T of every chunk and the state at
// every chunk start.  f.o and f.final_S are written when given.
PrefillArgs saving_forward_args(const PrefillArgs &f) {
    const ChunkWs w = chunk_ws(f.N, f.ntok, f.H, f.dk);
    const ChunkPtrs c = chunk_ptrs(f.workspace, w);
    PrefillArgs pa = f;
    pa.workspace = c.base;
    pa.workspace_bytes = w.fwd;
    pa.chunk = tile::C;
    pa.chunk_states = c.states;
    pa.t_out = c.tiles;
    return pa;
}

// The reverse chain and the per-chunk gradients from a workspace that holds
// the forward's saved tensors.
cudaError_t launch_gradients(const BwdArgs &a, cudaStream_t s) {
    const int D = a.dk;
    const ChunkWs w = chunk_ws(a.N, a.ntok, a.H, D);
    const ChunkPtrs c = chunk_ptrs(a.workspace, w);
    unsigned *err = device_error_word();
    if (!err) return cudaErrorInvalidValue;

    // dS from the last chunk to the first
    const uint8_t *records = c.base + tile::Workspace::table_bytes(a.N, a.ntok);
    ChainParams cp{records, static_cast<const __nv_bfloat16 *>(a.d_o), a.cu_seqlens, a.d_final_S,
                   c.dstates, c.dstates16, c.du, a.d_init_S, err, a.H, a.ntok, a.scale};
    const bool gated = a.gate_logits != nullptr;   // records carry e^{b_L}; else it is 1
    cudaError_t e;
    if (D == 64) e = gated ? launch_chain<64, true>(cp, a.N, a.H, s) : launch_chain<64, false>(cp, a.N, a.H, s);
    else e = gated ? launch_chain<128, true>(cp, a.N, a.H, s) : launch_chain<128, false>(cp, a.N, a.H, s);
    if (e != cudaSuccess) return e;

    // every (chunk, head): the gradients, through the prologue
    const int64_t n_tasks = tile::Workspace::slots(a.N, a.ntok) * a.H;
    const int2 *table = reinterpret_cast<const int2 *>(c.base);
    BwdChannelArgs ca{a.q, a.k, a.v, a.beta_logits, a.gate_logits, a.d_o, table, c.states,
                      c.dstates, c.dstates16, c.du, c.tiles, a.dq, a.dk_out, a.dv_out,
                      a.d_beta_logits, a.gate_logits ? a.d_gate_logits : nullptr, n_tasks, a.H, D,
                      a.scale, a.flags};
    return launch_delta_bwd_channel(ca, s);
}

}  // namespace

cudaError_t launch_delta_backward_chunked(const BwdArgs &a, cudaStream_t s) {
    // 1. the forward pass, keeping what the gradients need (no output)
    PrefillArgs f{a.q, a.k, a.v, a.beta_logits, a.gate_logits, nullptr, a.cu_seqlens, a.N,
                  a.ntok, a.H, a.dk, a.dk, a.scale, a.flags, a.init_S, nullptr, nullptr, nullptr,
                  true, a.workspace, 0};
    const PrefillArgs pa = saving_forward_args(f);
    if (!delta_tc_supported(pa)) return cudaErrorInvalidValue;
    cudaError_t e = launch_delta_tc(pa, s);
    // 2, 3. the reverse chain, then every (chunk, head) in parallel
    return e != cudaSuccess ? e : launch_gradients(a, s);
}

bool delta_train_supported(const PrefillArgs &a) {
    return a.bf16 && a.dk == a.dv && (a.dk == 64 || a.dk == 128) &&
           delta_tc_supported(saving_forward_args(a));
}

cudaError_t launch_delta_train_forward(const PrefillArgs &a, cudaStream_t s) {
    const PrefillArgs pa = saving_forward_args(a);
    if (!delta_tc_supported(pa)) return cudaErrorInvalidValue;
    return launch_delta_tc(pa, s);
}

cudaError_t launch_delta_backward_saved(const BwdArgs &a, cudaStream_t s) {
    // The chunk table is rebuilt from this call's cu_seqlens, so the per-chunk
    // kernel's token rows stay inside the tensors whatever the workspace held.
    PrefillArgs f{a.q, a.k, a.v, a.beta_logits, a.gate_logits, nullptr, a.cu_seqlens, a.N,
                  a.ntok, a.H, a.dk, a.dk, a.scale, a.flags, a.init_S, nullptr, nullptr, nullptr,
                  true, a.workspace, 0};
    const PrefillArgs pa = saving_forward_args(f);
    TcLaunch x{};
    x.a = &pa;
    x.slots = tile::Workspace::slots(a.N, a.ntok);
    x.table = static_cast<int2 *>(pa.workspace);
    cudaError_t e = launch_chunk_table(x, s);
    return e != cudaSuccess ? e : launch_gradients(a, s);
}

}  // namespace la
