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
//                            chunk to the first, dS in registers, the record
//                            tiles read in place; stores dS' and du of every
//                            chunk;
//   delta_bwd_channel_kernel every (chunk, head) in parallel: the gradients of
//                            the chunk's inputs and the prologue's derivatives.

#include "common.cuh"
#include "delta_tc.h"
#include "launch.h"
#include "tc_tile.cuh"
#include "warp_mma.cuh"

namespace la {
namespace {

using tile::C;
struct ChainParams {
    const uint8_t *records;   // [slots][H] forward records
    const __nv_bfloat16 *d_o;
    const int32_t *cu;
    const float *d_final_S;
    float *dstates;           // [slots][H][D][D]: dS' of every chunk (fp32; gated)
    __nv_bfloat16 *dstates16; // [slots][H][D][D]: dS' of every chunk (bf16; no gate)
    __nv_bfloat16 *du;        // null, or [slots][H][64][D]: du of every chunk (bf16)
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
        bf16 *dst16 = p.dstates16 + ((slot0 + c) * H + h) * (int64_t)(D * D);
#pragma unroll
        for (int j = 0; j < NT_DS; ++j)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int r = 16 * Rs + g + 8 * hr, col = ns + 8 * j + 2 * t;
                if (p.gend)   // gated: fp32 (the per-chunk kernel also forms rowsum(dS' o S))
                    *reinterpret_cast<float2 *>(dst + r * D + col) = make_float2(ds[j][2 * hr], ds[j][2 * hr + 1]);
                else
                    wmma16::st2(dst16 + r * D + col, ds[j][2 * hr], ds[j][2 * hr + 1]);
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
            bf16 *gdu = p.du ? p.du + ((slot0 + c) * H + h) * (int64_t)(64 * D) : nullptr;
#pragma unroll
            for (int j = 0; j < NT_DU; ++j)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int r = 16 * Ru + g + 8 * hr, col = nu + 8 * j + 2 * t;
                    wmma16::st2(sDU + r * XS + col, du[j][2 * hr], du[j][2 * hr + 1]);
                    if (gdu) wmma16::st2(gdu + r * D + col, du[j][2 * hr], du[j][2 * hr + 1]);
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
    return a.bf16 && a.dk == a.dv && (a.dk == 64 || a.dk == 128);
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
    __nv_bfloat16 *dstates16 = reinterpret_cast<__nv_bfloat16 *>(base + w.fwd + w.states + w.dstates);
    __nv_bfloat16 *du = reinterpret_cast<__nv_bfloat16 *>(base + w.fwd + w.states + w.dstates + w.dstates16);
    uint8_t *tiles = base + w.fwd + w.states + w.dstates + w.dstates16 + w.du;
    unsigned *err = device_error_word();
    if (!err) return cudaErrorInvalidValue;

    // 1. the forward pass, keeping its records and the state at every chunk start
    PrefillArgs pa{a.q, a.k, a.v, a.beta_logits, a.gate_logits, nullptr, a.cu_seqlens, a.N,
                   a.ntok, a.H, D, D, a.scale, a.flags, a.init_S, nullptr, nullptr, nullptr,
                   true, base, w.fwd};
    pa.chunk_states = states;
    pa.t_out = tiles;
    if (!delta_tc_supported(pa)) return cudaErrorInvalidValue;
    cudaError_t e = launch_delta_tc(pa, s);
    if (e != cudaSuccess) return e;

    // 2. dS from the last chunk to the first
    const uint8_t *records = base + tile::Workspace::table_bytes(a.N, a.ntok);
    ChainParams cp{records, static_cast<const __nv_bfloat16 *>(a.d_o), a.cu_seqlens, a.d_final_S,
                   dstates, dstates16, du, a.d_init_S, err, a.H, a.ntok, a.scale,
                   a.gate_logits != nullptr};
    e = D == 64 ? launch_chain<64>(cp, a.N, a.H, s) : launch_chain<128>(cp, a.N, a.H, s);
    if (e != cudaSuccess) return e;

    // 3. every (chunk, head): the gradients, through the prologue
    const int64_t n_tasks = tile::Workspace::slots(a.N, a.ntok) * a.H;
    const int2 *table = reinterpret_cast<const int2 *>(base);
    BwdChannelArgs ca{a.q, a.k, a.v, a.beta_logits, a.gate_logits, a.d_o, table, states, dstates,
                      dstates16, du, tiles, a.dq, a.dk_out, a.dv_out, a.d_beta_logits,
                      a.gate_logits ? a.d_gate_logits : nullptr, n_tasks, a.H, D, a.scale, a.flags};
    return launch_delta_bwd_channel(ca, s);
}

}  // namespace la
