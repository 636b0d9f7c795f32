// delta_inter_tc.cu -- inter-chunk half of the tensor-core (gated) delta-rule
// prefill: the state recurrence across chunks, one CTA per (head, sequence).
//
// ("From GPT-2 to Kimi K3, explained", section DeltaNet (Parallelizing
// Linear Transformers with Delta Rule), eq. 8-10, with the cumulative decay of
// sections Gated DeltaNet and KDA / Kimi Linear.)  Per chunk, reading the
// record the intra-chunk kernel wrote (-W, U, Aq, Q e^b, K~ = K e^{b_end - b},
// e^{b_end}):
//   u = U - W S                     (S = state at the end of the previous chunk)
//   O = scale ((Q e^b) S + Aq u)
//   S <- Diag(e^{b_end}) S + K~^T u
//
// Three tensor-core products per chunk, all M = 128 where the rows allow,
// into one TMEM accumulator per chunk (two, alternating) whose lanes 0..63
// hold u and lanes 64..127 hold O:
//   [-W ; Q e^b] S         on top of [U ; 0]  ->  [u ; (Q e^b) S]   commit "u"
//   S += K~^T u                                                     commit "s"
//   [anything ; Aq] u      ->  lanes 64..127 += Aq u (lanes 0..63, already
//                              read out, take a harmless sum)       commit "o"
// Only S -> u -> S is sequential.  Warp roles, synchronised by mbarriers:
//   warps 0..7     state: S (TMEM fp32) -> bf16 operand tile for the next
//                  chunk, then (gated) S *= e^{b_end} of the next chunk in
//                  TMEM; the four on lanes 0..63 first turn u into its bf16
//                  operand tile
//   warps 8, 9     put U of the chunk into accumulator lanes 0..63
//   warps 10, 11   O (lanes 64..127) -> scale -> bf16 -> global, then zero
//                  those lanes for the chunk after next
//   warp 12        one thread issues the products
// (13 warps: a 16th would cost the register budget of 20.)
// The fp32 state lives in tensor memory for the whole sequence; records
// stream in by bulk copies up to NB - 1 chunks ahead.

#include "common.cuh"
#include "delta_tc.h"
#include "tc_tile.cuh"

namespace la {
namespace {

using namespace tc;
using namespace tile;

constexpr int NT = 13 * 32;
constexpr int W_ISSUER = 12;

template <int D>
struct Layout {
    using Rec = Record<D>;
    // record buffers: loads run up to NB - 1 chunks ahead of the recurrence
    static constexpr int NB = D == 64 ? 4 : 2;
    static constexpr uint32_t REC0 = 0;
    static constexpr uint32_t SB = NB * Rec::BYTES;      // S, bf16 [D][D] RS tile
    static constexpr uint32_t UT = SB + D * D * 2;        // u, bf16 [64][D] RS tile
    static constexpr uint32_t BARS = UT + C * D * 2;      // mbarriers, tmem slot, load counts
    static constexpr uint32_t TOTAL = BARS + 128;
    static_assert(TOTAL + 1024 <= 227 * 1024, "shared memory budget");
};

// mbarrier slots (B_REC0 .. B_REC0 + NB - 1: record buffers)
enum : int {
    B_U = 0, B_S, B_O, B_SREADY, B_UREADY, B_UPRE, B_OFREE0, B_OFREE1, B_REC0,
    B_COUNT = B_REC0 + 4
};
constexpr uint32_t N_STATE = 8, N_UPRE = 2, N_OUT = 2;  // arrivals per phase

// TMEM columns: S (M = D rows = key channels), then two [u ; O] accumulators.
template <int D>
struct Cols {
    static constexpr uint32_t S = 0, ACC = D, TOTAL = D == 64 ? 256 : 512;
};

struct InterParams {
    const uint8_t *records;   // [slots][H] records
    __nv_bfloat16 *o;         // null: outputs not written
    float *states;            // null, or the state at each chunk start [slot][H][D][D]
    const int32_t *cu_seqlens;
    const float *init_S;
    float *final_S;
    unsigned *err;
    int H, ntok;
    float scale;
};

template <int D, bool GATED>
__global__ void __launch_bounds__(NT, 1) delta_inter_kernel(InterParams p) {
    using L = Layout<D>;
    using Rec = Record<D>;
    using TC = Cols<D>;
    constexpr int NB = L::NB;
    constexpr int HALF = D / 2;  // columns per thread in every readback (two column halves)
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sb = sm + L::SB, *ut = sm + L::UT;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::BARS);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + B_COUNT);
    int *s_loads = reinterpret_cast<int *>(tslot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qd = warp & 3;                  // TMEM lane quarter
    const int c0 = ((warp >> 2) & 1) * HALF;  // state warps: this warp's column half
    const int h = blockIdx.x, n = blockIdx.y, H = p.H;
    int t_begin = p.cu_seqlens[n], t_end = p.cu_seqlens[n + 1];
    if (t_begin < 0 || t_end < t_begin || t_end > p.ntok) {
        if (tid == 0) atomicCAS(p.err, 0u, 100u);
        t_begin = t_end = 0;
    }
    const int nc = (t_end - t_begin + C - 1) / C;
    const int64_t slot0 = (int64_t)(t_begin / C) + n;
    auto rec_src = [&](int c) { return p.records + ((slot0 + c) * H + h) * (int64_t)Rec::BYTES; };
    auto buf = [&](int c) { return sm + L::REC0 + (uint32_t)(c % NB) * Rec::BYTES; };
    auto rec_bar = [&](int c) { return &bars[B_REC0 + c % NB]; };
    auto rec_par = [](int c) { return (uint32_t)(c / NB) & 1u; };
    // Record loads (one bulk copy each): the issuer starts records 0 .. NB-1,
    // output warp 10 loads record c + NB into chunk c's buffer once chunk c
    // is finished with it, so the records loaded are always 0 .. K-1; both
    // count theirs (s_loads) for the final wait.
    auto issue_rec = [&](int c) {
        fence_proxy_async();
        mbar_arrive_expect_tx(rec_bar(c), Rec::BYTES);
        bulk_load_hint(buf(c), rec_src(c), Rec::BYTES, rec_bar(c), l2_evict_first());
    };

    if (tid == 0) {
        for (int b = 0; b < NB; ++b) mbar_init(&bars[B_REC0 + b], 1);
        mbar_init(&bars[B_U], 1);
        mbar_init(&bars[B_S], 1);
        mbar_init(&bars[B_O], 1);
        mbar_init(&bars[B_SREADY], N_STATE);
        mbar_init(&bars[B_UREADY], N_STATE);
        mbar_init(&bars[B_UPRE], N_UPRE);
        mbar_init(&bars[B_OFREE0], N_OUT);
        mbar_init(&bars[B_OFREE1], N_OUT);
        fence_mbar_init();
        s_loads[0] = s_loads[1] = 0;
    }
    if (warp == 0) {
        tmem_alloc(tslot, TC::TOTAL);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the records come from the intra-chunk kernel (launched just before)
    grid_wait_prerequisites();
    const uint32_t tmem = *tslot;
    const uint32_t tq = tmem + ((uint32_t)(32 * qd) << 16);  // this warp's lane quarter
    auto acc = [&](int c) { return (uint32_t)(TC::ACC + (c & 1) * D); };
    const int64_t sbase = ((int64_t)n * H + h) * D * D;
    // 16 consecutive fp32 state entries (row srow, columns col..col+15) at the
    // start of chunk c, for the backward pass (16-byte units by column group,
    // so the warp's lanes, on consecutive rows, store contiguous runs)
    auto store_state = [&](int c, int srow, int col, const float *v) {
        float4 *dst = reinterpret_cast<float4 *>(p.states + ((slot0 + c) * H + h) * (int64_t)(D * D));
#pragma unroll
        for (int i = 0; i < 4; ++i)
            dst[unit_at(D, srow, col / 4 + i)] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    };
    // one lane of each warp arrives once the warp's work is ordered before it
    auto warp_arrive = [&](uint64_t *bar) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar);
    };

    if (warp == W_ISSUER) {
        // ================================================= issuer
        if (lane == 0 && nc > 0) {
            constexpr uint32_t id128 = idesc_bf16(128, D, false, true);
            constexpr uint32_t ids = idesc_bf16(D, D, true, true);
            const uint64_t bS = mdesc(sb, D, 0, 0), bU = mdesc(ut, C, 0, 0);
            for (int c = 0; c < NB && c < nc; ++c) issue_rec(c);
            s_loads[0] = NB < nc ? NB : nc;
            for (int c = 0; c < nc; ++c) {
                uint8_t *rb = buf(c);
                const uint32_t ta = tmem + acc(c);
                // the state tile, U in lanes 0..63 (and zeros below it), the record
                if (!mbar_wait(&bars[B_SREADY], (uint32_t)c & 1u, p.err, 5)) break;
                if (!mbar_wait(&bars[B_UPRE], (uint32_t)c & 1u, p.err, 6)) break;
                if (!mbar_wait(rec_bar(c), rec_par(c), p.err, 4)) break;
                tc_fence_after();
                const uint64_t aWQ = kdesc(rb + Rec::WQ, 128, 0, 0);
#pragma unroll 1
                for (int kb = 0; kb < D / 64; ++kb) {
#pragma unroll
                    for (int s4 = 0; s4 < 4; ++s4) {
                        const int s = 4 * kb + s4;
                        mma_bf16(ta, dstep(aWQ, kstep_units(128, s)), dstep(bS, s * 128), id128, 1);
                    }
                }
                mma_commit(&bars[B_U]);
                // u tile ready, state decayed for this chunk
                if (!mbar_wait(&bars[B_UREADY], (uint32_t)c & 1u, p.err, 7)) break;
                tc_fence_after();
                const uint64_t aK = mdesc(rb + Rec::UK, 128, 64, 0);
                const uint64_t aA = kdesc(rb + Rec::AQ - 8192, 128, 0, 0);
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4)
                    mma_bf16(tmem + TC::S, dstep(aK, s4 * 128), dstep(bU, s4 * 128), ids, 1);
                mma_commit(&bars[B_S]);
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4)
                    mma_bf16(ta, dstep(aA, s4 * 2), dstep(bU, s4 * 128), id128, 1);
                // The output warps must have taken chunk c - 1 (so seen its "o"
                // phase) before this chunk's "o" phase can complete.
                if (c >= 1 &&
                    !mbar_wait(&bars[B_OFREE0 + ((c - 1) & 1)], (uint32_t)(((c - 1) >> 1) + 1) & 1u, p.err, 8))
                    break;
                mma_commit(&bars[B_O]);
            }
        }
    } else if (warp < 8) {
        // ================================================= state (and u) warps
        const int srow = acc_row(D, qd, lane);     // state row (key channel), or -1
        const bool u_warp = qd < 2;
        const int urow = 32 * qd + lane;           // u row (token) for u_warp
        bool ok = true;
        // initial state: bf16 operand copy; TMEM state decayed by chunk 0's e^{b_end}
        if (GATED && nc > 0) ok = mbar_wait(rec_bar(0), 0, p.err, 10);
        if (ok) {
            const float gd = (GATED && nc > 0 && srow >= 0)
                                 ? reinterpret_cast<const float *>(buf(0) + Rec::GEND)[srow]
                                 : 1.0f;
#pragma unroll
            for (int cb = 0; cb < HALF; cb += 16) {
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
                    if (p.states) store_state(0, srow, col, v);
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] *= gd;
                tmem_st16(tq + TC::S + col, v);
            }
            fence_proxy_async();
            warp_arrive(&bars[B_SREADY]);
        }
        for (int c = 0; c < nc && ok; ++c) {
            // ---- u -> bf16 operand tile (lanes 0..63 of the accumulator)
            if (u_warp) {
                if (!(ok = mbar_wait(&bars[B_U], (uint32_t)c & 1u, p.err, 11))) break;
                tc_fence_after();
#pragma unroll
                for (int cb = 0; cb < HALF; cb += 32) {
                    float v[32];
                    tmem_ld32(tq + acc(c) + c0 + cb, v);
#pragma unroll
                    for (int i = 0; i < 32; i += 8) st_bf16x8(ut, C, urow, c0 + cb + i, v + i);
                }
                fence_proxy_async();
            }
            warp_arrive(&bars[B_UREADY]);
            // ---- S after this chunk
            if (!(ok = mbar_wait(&bars[B_S], (uint32_t)c & 1u, p.err, 12))) break;
            tc_fence_after();
            if (c + 1 < nc) {
#pragma unroll
                for (int cb = 0; cb < HALF; cb += 32) {
                    float v[32];
                    tmem_ld32(tq + TC::S + c0 + cb, v);
                    if (srow >= 0) {
#pragma unroll
                        for (int i = 0; i < 32; i += 8) st_bf16x8(sb, D, srow, c0 + cb + i, v + i);
                        if (p.states) {
                            store_state(c + 1, srow, c0 + cb, v);
                            store_state(c + 1, srow, c0 + cb + 16, v + 16);
                        }
                    }
                }
                fence_proxy_async();
                warp_arrive(&bars[B_SREADY]);
                if (GATED) {
                    // decay for the next chunk (needs its record's e^{b_end});
                    // the state is read again rather than held in registers
                    if (!(ok = mbar_wait(rec_bar(c + 1), rec_par(c + 1), p.err, 13))) break;
                    const float gd = srow >= 0
                                         ? reinterpret_cast<const float *>(buf(c + 1) + Rec::GEND)[srow]
                                         : 1.0f;
#pragma unroll
                    for (int cb = 0; cb < HALF; cb += 32) {
                        float v[32];
                        tmem_ld32(tq + TC::S + c0 + cb, v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] *= gd;
                        tmem_st16(tq + TC::S + c0 + cb, *reinterpret_cast<float(*)[16]>(v));
                        tmem_st16(tq + TC::S + c0 + cb + 16, *reinterpret_cast<float(*)[16]>(v + 16));
                    }
                }
            }
        }
        // ---- final state
        if (ok && p.final_S) {
#pragma unroll
            for (int cb = 0; cb < HALF; cb += 16) {
                float v[16];
                tmem_ld16(tq + TC::S + c0 + cb, v);
                if (srow >= 0) {
                    float4 *dst = reinterpret_cast<float4 *>(p.final_S + sbase + (int64_t)srow * D + c0 + cb);
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                }
            }
        }
    } else if (qd < 2) {
        // ================================================= U pre-load (warps 8, 9)
        const int urow = 32 * qd + lane;
        for (int c = 0; c < nc; ++c) {
            // the issuer has taken the previous chunk's U (so phases cannot run
            // ahead of it); this accumulator drained and zeroed (chunk c - 2)
            if (c >= 1 && !mbar_wait(&bars[B_U], (uint32_t)(c - 1) & 1u, p.err, 15)) break;
            if (!mbar_wait(&bars[B_OFREE0 + (c & 1)], (uint32_t)(c >> 1) & 1u, p.err, 16)) break;
            if (!mbar_wait(rec_bar(c), rec_par(c), p.err, 17)) break;
            tc_fence_after();
            const uint8_t *uk = buf(c) + Rec::UK;
#pragma unroll
            for (int cb = 0; cb < D; cb += 16) {
                float v[16];
                unpack8(*reinterpret_cast<const uint4 *>(uk + rs_off(128, urow, cb)), v);
                unpack8(*reinterpret_cast<const uint4 *>(uk + rs_off(128, urow, cb + 8)), v + 8);
                tmem_st16(tq + acc(c) + cb, v);
            }
            warp_arrive(&bars[B_UPRE]);
        }
    } else {
        // ================================================= output warps (10, 11)
        const int orow = 32 * (qd - 2) + lane;  // row of O in the chunk
        int refills = 0;
        // both accumulators' O lanes start at zero
        {
            float z[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) z[i] = 0.0f;
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
                for (int cb = 0; cb < D; cb += 16) tmem_st16(tq + acc(b) + cb, z);
            warp_arrive(&bars[B_OFREE0]);
            warp_arrive(&bars[B_OFREE1]);
        }
        for (int c = 0; c < nc; ++c) {
            if (!mbar_wait(&bars[B_O], (uint32_t)c & 1u, p.err, 14)) break;
            tc_fence_after();
            const int tok0 = t_begin + c * C;
            const bool valid = orow < t_end - tok0;
#pragma unroll
            for (int cb = 0; cb < D; cb += 32) {
                float v[32];
                tmem_ld32(tq + acc(c) + cb, v);
                if (valid && p.o) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= p.scale;
                    uint4 *dst = reinterpret_cast<uint4 *>(p.o + ((int64_t)(tok0 + orow) * H + h) * D + cb);
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[i] = pack8(v + 8 * i);
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0.0f;
                tmem_st16(tq + acc(c) + cb, *reinterpret_cast<float(*)[16]>(v));
                tmem_st16(tq + acc(c) + cb + 16, *reinterpret_cast<float(*)[16]>(v + 16));
            }
            warp_arrive(&bars[B_OFREE0 + (c & 1)]);
            // every product that reads record c has completed ("o" is the last
            // commit of chunk c): its buffer takes record c + NB
            if (warp == 10 && lane == 0 && c + NB < nc) {
                issue_rec(c + NB);
                ++refills;
            }
        }
        if (warp == 10 && lane == 0) s_loads[1] = refills;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        // the last load into each buffer (earlier ones completed before it was issued)
        const int K = s_loads[0] + s_loads[1];
        for (int j = K - NB > 0 ? K - NB : 0; j < K; ++j) mbar_wait(rec_bar(j), rec_par(j), p.err, 9);
    }
    if (warp == 0) tmem_dealloc(tmem, TC::TOTAL);
}

template <int D, bool GATED>
cudaError_t launch_t(const TcLaunch &x, cudaStream_t s) {
    const PrefillArgs &a = *x.a;
    InterParams p{x.records, static_cast<__nv_bfloat16 *>(a.o), a.chunk_states, a.cu_seqlens,
                  a.init_S, a.final_S, x.err, a.H, a.ntok, a.scale};
    constexpr size_t smem = Layout<D>::TOTAL + 1024;
    auto kern = delta_inter_kernel<D, GATED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.H, a.N);
    return launch_programmatic(kern, grid, dim3(NT), smem, s, p);
}

}  // namespace

cudaError_t launch_delta_inter(const TcLaunch &x, cudaStream_t s) {
    const bool g = x.a->gate_logits != nullptr;
    if (x.a->dk == 128) return g ? launch_t<128, true>(x, s) : launch_t<128, false>(x, s);
    return g ? launch_t<64, true>(x, s) : launch_t<64, false>(x, s);
}

}  // namespace la
