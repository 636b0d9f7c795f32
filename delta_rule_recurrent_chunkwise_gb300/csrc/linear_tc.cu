// linear_tc.cu -- ELU+1 causal linear attention on the tensor cores (bf16
// I/O, dk = dv = 64): one CTA per (head, sequence), chunk after chunk.
//
// ("From GPT-2 to Kimi K3, explained", section Linear attention: feature map
// phi = elu + 1, state S = sum phi(k) v^T, normaliser z = sum phi(k), output
// phi(q)^T S / phi(q)^T z; chunked as in section DeltaNet (Parallelizing
// Linear Transformers with Delta Rule).)  With V' = [V | 1] the normaliser
// is column 64 of the state S' = [S | z] (dk x 72) and the denominator
// column 64 of the output, so one chunk of 64 tokens is four products
// (M = 64, N = 64 or 72, K = 64):
//   P           = tril(phi(Q) phi(K)^T)          (i <= r)
//   [num | den] = phi(Q) S'_c + P V'
//   O           = num / den
//   S'_{c+1}    = S'_c + phi(K)^T V'
// The product P V' of chunk c is issued together with chunk c + 1's other
// products, so a chunk costs one tensor-core round trip, and the CTA turns
// chunk c + 1's raw q, k into phi(q), phi(k) (a second pair of tiles) while
// chunk c's products run.  Raw q, k, v arrive by TMA three chunks ahead
// (four stages).  The state stays fp32 in TMEM; its bf16 copy is the
// operand of the next chunk's phi(Q) S'.

#include "common.cuh"
#include "delta_tc.h"
#include "launch.h"
#include "tc_tile.cuh"

namespace la {
namespace {

using namespace tc;
using namespace tile;

constexpr int D = 64, NT = 512, NSTAGE = 4;
constexpr int NX = 72;                // state / output columns: 64 values, the normaliser, 7 zero
constexpr uint32_t TILE = 8192;       // bf16 [64][64], 128-byte swizzled

struct LinTcLayout {
    static constexpr uint32_t STAGE = 3 * TILE;            // raw q, k, v (TMA)
    static constexpr uint32_t ONES = NSTAGE * STAGE;       // rows [1, 0, .., 0]: V' columns 64..
    static constexpr uint32_t FQ = ONES + TILE;            // phi(q), phi(k) of even chunks,
    static constexpr uint32_t FK = FQ + TILE;              //   then of odd chunks (+ 2 TILE)
    static constexpr uint32_t PT = FK + 3 * TILE;          // P
    static constexpr uint32_t SB = PT + TILE;              // S' in bf16: two 64-column blocks
    static constexpr uint32_t BARS = SB + 2 * TILE;        // 4 TMA barriers, 1 product barrier
    static constexpr uint32_t TOTAL = BARS + 64;
    static_assert(TOTAL + 1024 <= 227 * 1024, "shared memory budget");
};

// TMEM columns (M = 64 accumulators: rows in lanes 0..15 of each quarter)
constexpr uint32_t C_P = 0, C_O0 = 64, C_S = 224, TMEM_COLS = 512;
__device__ __forceinline__ uint32_t c_o(int b) { return C_O0 + 80u * (uint32_t)b; }

struct LinTcParams {
    const int32_t *cu_seqlens;
    __nv_bfloat16 *o;
    const float *init_S, *init_z;
    float *final_S, *final_z;
    unsigned *err;
    int H, ntok;
};

__global__ void __launch_bounds__(NT, 1)
    linear_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, LinTcParams p) {
    using L = LinTcLayout;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *pt = sm + L::PT, *sbf = sm + L::SB, *ones = sm + L::ONES;
    auto fq = [&](int c) { return sm + L::FQ + (uint32_t)(c & 1) * 2 * TILE; };
    auto fk = [&](int c) { return sm + L::FK + (uint32_t)(c & 1) * 2 * TILE; };
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::BARS);  // [0..3] stages, [4] products
    uint64_t *bar_mma = bars + NSTAGE;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + NSTAGE + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qd = warp & 3, c0 = 16 * (warp >> 2);  // lane quarter, 16-column quarter
    const int h = blockIdx.x, n = blockIdx.y, H = p.H;
    int t_begin = p.cu_seqlens[n], t_end = p.cu_seqlens[n + 1];
    if (t_begin < 0 || t_end < t_begin || t_end > p.ntok) {
        if (tid == 0) atomicCAS(p.err, 0u, 100u);
        t_begin = t_end = 0;
    }
    const int nc = (t_end - t_begin + C - 1) / C;
    auto stage = [&](int c) { return sm + (uint32_t)(c % NSTAGE) * L::STAGE; };
    const int64_t sbase = ((int64_t)n * H + h) * D * D, zbase = ((int64_t)n * H + h) * D;
    const int arow = acc_row(64, qd, lane);  // accumulator row of this lane, or -1

    if (tid == 0) {
        for (int s = 0; s < NSTAGE; ++s) mbar_init(&bars[s], 1);
        mbar_init(&bars[NSTAGE], 2);  // products: one commit from each issuing thread
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    if (warp == 0) {
        tmem_alloc(tslot, TMEM_COLS);
        tmem_relinquish();
    }
    // V' columns 64..127: 1 in column 64, zeros after it
    for (int x = tid; x < (int)(TILE / 16); x += NT)
        *reinterpret_cast<uint4 *>(ones + 16 * x) = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    if (tid < C) *reinterpret_cast<__nv_bfloat16 *>(ones + rs_off(64, tid, 0)) = __float2bfloat16_rn(1.0f);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    grid_wait_prerequisites();
    const uint32_t tmem = *tslot;
    const uint32_t tq = tmem + ((uint32_t)(32 * qd) << 16);
    const uint64_t pol = l2_evict_first();

    auto issue_tma = [&](int c) {
        uint8_t *st = stage(c);
        uint64_t *bar = &bars[c % NSTAGE];
        const int t0 = t_begin + c * C;
        fence_proxy_async();  // earlier generic reads of this stage come first
        mbar_arrive_expect_tx(bar, 3 * TILE);
        tma_load_3d_hint(st, &tm_q, bar, 0, h, t0, pol);
        tma_load_3d_hint(st + TILE, &tm_k, bar, 0, h, t0, pol);
        tma_load_3d_hint(st + 2 * TILE, &tm_v, bar, 0, h, t0, pol);
    };
    int issued = 0;  // chunks whose raw tiles have been requested (thread 0)
    if (tid == 0)
        for (; issued < NSTAGE - 1 && issued < nc; ++issued) issue_tma(issued);

    // initial state: fp32 in TMEM (column 64 = z), bf16 operand copy
    {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            v[i] = (arow >= 0 && p.init_S) ? p.init_S[sbase + (int64_t)arow * D + c0 + i] : 0.0f;
        if (arow >= 0)
#pragma unroll
            for (int i = 0; i < 16; i += 8) st_bf16x8(sbf, 64, arow, c0 + i, v + i);
        tmem_st16(tq + C_S + c0, v);
        if (c0 == 0) {
            float z[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) z[i] = 0.0f;
            if (arow >= 0 && p.init_z) z[0] = p.init_z[zbase + arow];
            if (arow >= 0) st_bf16x8(sbf, 64, arow, 64, z);
            tmem_st16(tq + C_S + 64, z);
        }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    constexpr uint32_t idP = idesc_bf16(64, 64, false, false);   // phi(Q) phi(K)^T
    constexpr uint32_t idQS = idesc_bf16(64, NX, false, true);   // phi(Q) S', P V'
    constexpr uint32_t idS = idesc_bf16(64, NX, true, true);     // phi(K)^T V'
    uint32_t mma_par = 0;
    int waited = 0;  // chunks whose raw tiles have been consumed
    bool ok = true;
    // chunk c's raw tiles -> phi(q), phi(k) (rows past the chunk's end zeroed);
    // false if the tiles never arrived
    // (every thread waits for the tiles itself, so that the conversion does
    // not wait for the threads issuing products; a failed wait is carried to
    // the round's next CTA barrier)
    auto make_phi = [&](int c) -> bool {
        if (!mbar_wait(&bars[c % NSTAGE], (uint32_t)(c / NSTAGE) & 1u, p.err, 80)) return false;
        waited = c + 1;
        const int len = min(C, t_end - (t_begin + c * C));
        const uint8_t *st = stage(c);
        uint8_t *dq = fq(c), *dk = fk(c);
        for (int x = tid; x < 2 * (int)(TILE / 16); x += NT) {
            const int which = x / (int)(TILE / 16), xi = x % (int)(TILE / 16), row = xi >> 3;
            float f[8];
            unpack8(*reinterpret_cast<const uint4 *>(st + which * TILE + 16 * xi), f);
            // elu + 1 with the fast exponential: the result is rounded to bf16
#pragma unroll
            for (int i = 0; i < 8; ++i) f[i] = row < len ? (f[i] > 0.0f ? f[i] + 1.0f : __expf(f[i])) : 0.0f;
            *reinterpret_cast<uint4 *>((which ? dk : dq) + 16 * xi) = pack8(f);
        }
        fence_proxy_async();
        return true;
    };
    if (nc > 0) {
        const bool w_ok = make_phi(0);
        tc_fence_before();
        ok = !__syncthreads_or(!w_ok);
        tc_fence_after();
    }
    // Round c: chunk c's products (c < nc) with chunk c - 1's P V'; meanwhile
    // phi of chunk c + 1; then chunk c's scores and state to bf16 and chunk
    // c - 1's outputs.
    for (int c = 0; c <= nc && ok; ++c) {
        const bool cur = c < nc;
        // two threads in different warps issue: thread 0 chunk c - 1's P V'
        // and chunk c's scores, thread 32 chunk c's phi(Q) S' and state update
        if (tid == 0) {
            if (c >= 1) {
                // chunk c - 1: O += P V'
                const uint8_t *vt = stage(c - 1) + 2 * TILE;
                const uint32_t lbo = (uint32_t)(ones - vt);
                const uint64_t aP = kdesc(pt, 64, 0, 0);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tmem + c_o((c - 1) & 1), dstep(aP, s * 2),
                             smem_desc_sw128(smem_u32(vt) + (uint32_t)s * 2048u, lbo, 1024u), idQS, 1);
            }
            if (cur) {
                const uint64_t aQ = kdesc(fq(c), 64, 0, 0), bK = kdesc(fk(c), 64, 0, 0);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tmem + C_P, dstep(aQ, s * 2), dstep(bK, s * 2), idP, s > 0);
            }
            mma_commit(bar_mma);
        } else if (tid == 32) {
            if (cur) {
                const uint64_t aQ = kdesc(fq(c), 64, 0, 0), aK = mdesc(fk(c), 64, 0, 0);
                const uint8_t *vt = stage(c) + 2 * TILE;
                const uint32_t lbo = (uint32_t)(ones - vt);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tmem + c_o(c & 1), dstep(aQ, s * 2),
                             smem_desc_sw128(smem_u32(sbf) + (uint32_t)s * 2048u, TILE, 1024u), idQS, s > 0);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tmem + C_S, dstep(aK, s * 128),
                             smem_desc_sw128(smem_u32(vt) + (uint32_t)s * 2048u, lbo, 1024u), idS, 1);
            }
            mma_commit(bar_mma);
        }
        // the next chunk's phi tiles (the pair last read by round c - 1's products)
        bool r_ok = c + 1 < nc ? make_phi(c + 1) : true;
        if (tid == 0) r_ok = mbar_wait(bar_mma, mma_par, p.err, 81) && r_ok;
        mma_par ^= 1u;
        if (__syncthreads_or(!r_ok)) { ok = false; break; }
        tc_fence_after();
        // chunk c - 1's stage is free (its last products have completed): the
        // raw tiles of chunk c + 3 go into it
        if (tid == 0 && issued < nc && issued <= c + NSTAGE - 1) issue_tma(issued++);
        if (cur) {
            // ---- P (masked i <= r) and S'_{c+1} to their bf16 operand tiles
            float v[16];
            tmem_ld16(tq + C_P + c0, v);
            if (arow >= 0) {
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = (c0 + i <= arow) ? v[i] : 0.0f;
#pragma unroll
                for (int i = 0; i < 16; i += 8) st_bf16x8(pt, 64, arow, c0 + i, v + i);
            }
            tmem_ld16(tq + C_S + c0, v);
            if (arow >= 0)
#pragma unroll
                for (int i = 0; i < 16; i += 8) st_bf16x8(sbf, 64, arow, c0 + i, v + i);
            if (c0 == 0) {
                float z[16];
                tmem_ld16(tq + C_S + 64, z);
#pragma unroll
                for (int i = 1; i < 16; ++i) z[i] = 0.0f;
                if (arow >= 0) st_bf16x8(sbf, 64, arow, 64, z);
            }
        }
        if (c >= 1) {
            // ---- outputs of chunk c - 1: num / den
            const int pc = c - 1, tok0 = t_begin + pc * C;
            float v[16], d[16];
            tmem_ld16(tq + c_o(pc & 1) + c0, v);
            tmem_ld16(tq + c_o(pc & 1) + 64, d);
            if (arow >= 0 && tok0 + arow < t_end) {
                const float inv = 1.0f / d[0];
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] *= inv;
                uint4 *dst = reinterpret_cast<uint4 *>(p.o + ((int64_t)(tok0 + arow) * H + h) * D + c0);
#pragma unroll
                for (int i = 0; i < 2; ++i) dst[i] = pack8(v + 8 * i);
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    // ---- final state
    if (ok && (p.final_S || p.final_z)) {
        float v[16];
        tmem_ld16(tq + C_S + c0, v);
        if (arow >= 0 && p.final_S)
#pragma unroll
            for (int i = 0; i < 16; ++i) p.final_S[sbase + (int64_t)arow * D + c0 + i] = v[i];
        if (c0 == 0) {
            float z[16];
            tmem_ld16(tq + C_S + 64, z);
            if (arow >= 0 && p.final_z) p.final_z[zbase + arow] = z[0];
        }
    }
    // a failed wait may leave raw-tile loads in flight: let them land
    if (tid == 0)
        for (int j = waited; j < issued; ++j)
            mbar_wait(&bars[j % NSTAGE], (uint32_t)(j / NSTAGE) & 1u, p.err, 82);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

bool linear_tc_supported(const PrefillArgs &a) {
    auto al16 = [](const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
    return a.bf16 && a.dk == D && a.dv == D && al16(a.q) && al16(a.k) && al16(a.v) && al16(a.o);
}

cudaError_t launch_linear_tc(const PrefillArgs &a, cudaStream_t s) {
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, a.q, D, a.H, a.ntok) || !make_map(&mk, a.k, D, a.H, a.ntok) ||
        !make_map(&mv, a.v, D, a.H, a.ntok))
        return cudaErrorInvalidValue;
    unsigned *err = device_error_word();
    if (!err) return cudaErrorInvalidValue;
    LinTcParams p{a.cu_seqlens, static_cast<__nv_bfloat16 *>(a.o), a.init_S, a.init_z,
                  a.final_S, a.final_z, err, a.H, a.ntok};
    constexpr size_t smem = LinTcLayout::TOTAL + 1024;
    cudaError_t e = cudaFuncSetAttribute(linear_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    linear_tc_kernel<<<dim3(a.H, a.N), NT, smem, s>>>(mq, mk, mv, p);
    return cudaGetLastError();
}

}  // namespace la
