// delta_bwd.cu -- gradients of the (gated) delta rule with respect to q, k,
// v, the beta and gate logits and the initial state.
//
// The page ("From GPT-2 to Kimi K3, explained", section DeltaNet
// (Parallelizing Linear Transformers with Delta Rule)) gives the forward
// pass only and motivates its chunked form by training.  The backward pass
// is the chain rule through each statement of the token step in reverse:
//   o_t = scale S_t^T q_t        dq_t = scale S_t do_t;   dS += scale q_t do_t^T
//   S_t = S' + k_t u_t^T         dk_t += dS u_t;  du = dS^T k_t
//   u_t = beta (v_t - S'^T k_t)  dbeta = du.(v_t - S'^T k_t);  dv_t = beta du;
//                                dk_t -= beta S' du;  dS' = dS - beta k_t du^T
//   S' = Diag(alpha_t) S_{t-1}   dalpha = rowsum(dS' o S_{t-1});  dS <- Diag(alpha) dS'
// then through the prologue (sigmoid beta, -softplus log-decay, silu and
// L2 normalisation of q and k).  The additive rule (u_t = v_t, section Gated
// DeltaNet) drops the read path: beta = 1 and the terms weighted by beta S'
// and beta k vanish; it has no beta gradient.
//
// Every column j of S evolves on its own: u_t[j], the j-th column of S and of
// dS depend on column j and on the shared per-token q, k, alpha, beta only.
// Only dq, dk, dalpha and dbeta sum over the columns.  So:
//
//  1. delta_bwd_ckpt_kernel: grid (column group, head, sequence), one warp
//     per column (its dk rows spread over the lanes); runs the forward token
//     loop and stores S at the start of every 64-token chunk (fp32,
//     transposed: [slot][head][dv][dk], slot = cu[n]/64 + n + chunk).
//  2. delta_bwd_kernel: same grid, launched as clusters of all the column
//     groups of one (sequence, head).  Chunks in reverse; in each, a forward
//     pass from the checkpoint keeps S every 8 tokens in shared memory, then
//     each 8-token block is recomputed with its states in registers and swept
//     backwards.  The per-token column sums (dq^, dk^, dalpha, dbeta) are
//     added over the CTA's warps in shared memory, then over the cluster's
//     CTAs through distributed shared memory, and written once per token to
//     a fp32 workspace: no global atomics, the same result on every run.
//  3. delta_bwd_prologue_kernel: one warp per (token, head): the prologue's
//     derivatives, written to dq, dk, d_beta_logits, d_gate_logits.
//
// The cost is a token-serial loop per column (as the decode step, but
// backward and with the forward recomputed twice): this is the direct CUDA
// form of the gradient, not the chunkwise tensor-core form.

#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"

namespace cg = cooperative_groups;

namespace la {
namespace {

constexpr int kC = 64;      // tokens per checkpointed chunk
constexpr int kE = 8;       // tokens per register-resident block
constexpr int kNW = 16;     // warps (= columns) per CTA
constexpr int kNT = kNW * 32;

struct BwdParams {
    const void *q, *k, *v, *beta_logits, *gate_logits, *d_o;
    const float *d_final_S, *init_S;
    const int32_t *cu;
    float *dq, *dk, *dv, *d_beta_logits, *d_gate_logits, *d_init_S;
    float *ckpt;     // [slots][H][dv][dk]
    float *sums;     // [ntok][H][3][dk] : dq^, dk^, d log alpha (per key channel)
    float *dbeta;    // [ntok][H]
    unsigned *err;
    int N, H, ntok;
    float scale;
    unsigned flags;
};

__device__ __forceinline__ bool seq_bounds(const BwdParams &p, int n, int64_t &c0, int64_t &L) {
    c0 = p.cu[n];
    const int64_t c1 = p.cu[n + 1];
    if (c0 < 0 || c1 < c0 || c1 > p.ntok) return false;
    L = c1 - c0;
    return true;
}

// Stage one chunk of per-token operands in shared memory: the prepared key
// (and query) rows, alpha per key channel, beta, and this CTA's columns of v
// (and of the output gradient).
template <typename IO, int DK, int DV>
__device__ void stage_chunk(const BwdParams &p, int64_t t0, int Lc, int h, int j0, bool with_q,
                            float *sQ, float *sK, float *sA, float *sB, float *sV, float *sDO) {
    constexpr int R = DK / 32;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const bool silu = (p.flags & kSiluQK) != 0;
    const bool scalar = (p.flags & kGateScalar) != 0;
    for (int s = w; s < Lc; s += kNW) {
        const int64_t th = (t0 + s) * p.H + h;
        for (int which = 0; which < (with_q ? 2 : 1); ++which) {
            const IO *src = static_cast<const IO *>(which ? p.q : p.k) + th * DK;
            const bool norm = (p.flags & (which ? kL2NormQ : kL2NormK)) != 0;
            float x[R], ss = 0.0f;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                x[r] = to_f32(src[lane + 32 * r]);
                if (silu) x[r] = silu_f(x[r]);
                ss += x[r] * x[r];
            }
            const float inv = norm ? 1.0f / fmaxf(sqrtf(warp_sum(ss)), 1e-12f) : 1.0f;
            float *dst = (which ? sQ : sK) + s * DK;
#pragma unroll
            for (int r = 0; r < R; ++r) dst[lane + 32 * r] = x[r] * inv;
        }
        const IO *g = static_cast<const IO *>(p.gate_logits);
#pragma unroll
        for (int r = 0; r < R; ++r)
            sA[s * DK + lane + 32 * r] =
                !g ? 1.0f : decay_f(to_f32(scalar ? g[th] : g[th * DK + lane + 32 * r]));
        if (lane == 0)
            sB[s] = (p.flags & kAdditive)
                        ? 1.0f
                        : sigmoid_f(to_f32(static_cast<const IO *>(p.beta_logits)[th]));
    }
    for (int idx = threadIdx.x; idx < Lc * kNW; idx += kNT) {
        const int s = idx / kNW, c = idx % kNW;
        const int64_t o = ((t0 + s) * p.H + h) * DV + j0 + c;
        sV[idx] = to_f32(static_cast<const IO *>(p.v)[o]);
        if (sDO) sDO[idx] = to_f32(static_cast<const IO *>(p.d_o)[o]);
    }
}

// One forward token step of column j (rows lane + 32 r): S <- Diag(a) S,
// r = S^T k (all lanes), u = beta (v - r) (u = v for the additive rule),
// S += k u.
template <int DK>
__device__ __forceinline__ void fwd_step(float (&S)[DK / 32], const float *a, const float *kk,
                                         float beta, float v, bool additive, float &rr,
                                         float &uu) {
    constexpr int R = DK / 32;
    const int lane = threadIdx.x & 31;
    float acc = 0.0f;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        S[r] *= a[lane + 32 * r];
        acc = fmaf(kk[lane + 32 * r], S[r], acc);
    }
    rr = warp_sum(acc);
    uu = additive ? v : beta * (v - rr);
#pragma unroll
    for (int r = 0; r < R; ++r) S[r] = fmaf(kk[lane + 32 * r], uu, S[r]);
}

// Shared-memory footprint of the staged chunk (fp32): q^, k^, alpha rows,
// beta, and this CTA's columns of v and of the output gradient.
template <int DK>
struct Stage {
    static constexpr int Q = 0, K = Q + kC * DK, A = K + kC * DK, B = A + kC * DK;
    static constexpr int V = B + kC, DO = V + kC * kNW, FLOATS = DO + kC * kNW;
};

template <typename IO, int DK, int DV>
__global__ void __launch_bounds__(kNT, 1) delta_bwd_ckpt_kernel(BwdParams p) {
    constexpr int R = DK / 32;
    using L = Stage<DK>;
    extern __shared__ __align__(16) float smem[];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int h = blockIdx.y, n = blockIdx.z;
    const int j0 = blockIdx.x * kNW, j = j0 + w;
    const bool additive = (p.flags & kAdditive) != 0;
    int64_t c0, len;
    if (!seq_bounds(p, n, c0, len)) {
        if (threadIdx.x == 0 && blockIdx.x == 0) atomicCAS(p.err, 0u, 100u);
        return;
    }
    const int64_t slot0 = c0 / kC + n;
    float S[R];
#pragma unroll
    for (int r = 0; r < R; ++r)
        S[r] = p.init_S ? p.init_S[(((int64_t)n * p.H + h) * DK + lane + 32 * r) * DV + j] : 0.0f;
    const int nc = (int)((len + kC - 1) / kC);
    for (int c = 0; c < nc; ++c) {
        float *ck = p.ckpt + (((slot0 + c) * p.H + h) * DV + j) * DK;
#pragma unroll
        for (int r = 0; r < R; ++r) ck[lane + 32 * r] = S[r];
        const int Lc = (int)(len - (int64_t)c * kC < kC ? len - (int64_t)c * kC : kC);
        __syncthreads();  // the previous chunk's operands are no longer read
        stage_chunk<IO, DK, DV>(p, c0 + (int64_t)c * kC, Lc, h, j0, false, nullptr,
                                smem + L::K, smem + L::A, smem + L::B, smem + L::V, nullptr);
        __syncthreads();
        for (int s = 0; s < Lc; ++s) {
            float rr, uu;
            fwd_step<DK>(S, smem + L::A + s * DK, smem + L::K + s * DK, smem[L::B + s],
                         smem[L::V + s * kNW + w], additive, rr, uu);
        }
    }
}

template <int DK>
struct BwdLayout {
    using L = Stage<DK>;
    static constexpr int SUB = L::FLOATS;                      // [warp][chunk/kE][DK]
    static constexpr int ACC = SUB + kNW * (kC / kE) * DK;     // two accumulator buffers
    static constexpr int ACCB = kE * 3 * DK + kE;              // [kE][3][DK] then dbeta[kE]
    static constexpr int FLOATS = ACC + 2 * ACCB;
};

template <typename IO, int DK, int DV>
__global__ void __launch_bounds__(kNT, 1) delta_bwd_kernel(BwdParams p) {
    constexpr int R = DK / 32, G = DV / kNW, TPC = kE / G;
    static_assert(kE % G == 0, "each CTA of a cluster reduces whole tokens");
    using L = Stage<DK>;
    using B = BwdLayout<DK>;
    extern __shared__ __align__(16) float smem[];
    cg::cluster_group cl = cg::this_cluster();
    const int rank = (int)cl.block_rank();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int h = blockIdx.y, n = blockIdx.z;
    const int j0 = blockIdx.x * kNW, j = j0 + w;
    const bool additive = (p.flags & kAdditive) != 0;
    int64_t c0, len;
    // The same sequence for every CTA of the cluster: all leave here together.
    if (!seq_bounds(p, n, c0, len)) return;

    for (int i = threadIdx.x; i < 2 * B::ACCB; i += kNT) smem[B::ACC + i] = 0.0f;
    cl.sync();

    float dS[R];
#pragma unroll
    for (int r = 0; r < R; ++r)
        dS[r] = p.d_final_S
                    ? p.d_final_S[(((int64_t)n * p.H + h) * DK + lane + 32 * r) * DV + j]
                    : 0.0f;
    const int64_t slot0 = c0 / kC + n;
    const int nc = (int)((len + kC - 1) / kC);
    unsigned m = 0;  // blocks done: selects the accumulator buffer
    for (int c = nc - 1; c >= 0; --c) {
        const int64_t t0 = c0 + (int64_t)c * kC;
        const int Lc = (int)(len - (int64_t)c * kC < kC ? len - (int64_t)c * kC : kC);
        __syncthreads();
        stage_chunk<IO, DK, DV>(p, t0, Lc, h, j0, true, smem + L::Q, smem + L::K, smem + L::A,
                                smem + L::B, smem + L::V, smem + L::DO);
        __syncthreads();
        const float *sQ = smem + L::Q, *sK = smem + L::K, *sA = smem + L::A;
        const float *sB = smem + L::B, *sV = smem + L::V, *sDO = smem + L::DO;

        // Forward from the chunk's checkpoint, keeping S every kE tokens.
        float *sub = smem + B::SUB + w * (kC / kE) * DK;
        float S[R];
        const float *ck = p.ckpt + (((slot0 + c) * p.H + h) * DV + j) * DK;
#pragma unroll
        for (int r = 0; r < R; ++r) S[r] = ck[lane + 32 * r];
        for (int s = 0; s < Lc; ++s) {
            if ((s % kE) == 0) {
#pragma unroll
                for (int r = 0; r < R; ++r) sub[(s / kE) * DK + lane + 32 * r] = S[r];
            }
            float rr, uu;
            fwd_step<DK>(S, sA + s * DK, sK + s * DK, sB[s], sV[s * kNW + w], additive, rr, uu);
        }
        __syncwarp();

        for (int b = (Lc + kE - 1) / kE - 1; b >= 0; --b, ++m) {
            float *acc = smem + B::ACC + (m & 1u) * B::ACCB;
            // Recompute the block with every state in registers.
            float hist[kE][R], rr[kE], uu[kE];
#pragma unroll
            for (int r = 0; r < R; ++r) S[r] = sub[b * DK + lane + 32 * r];
#pragma unroll
            for (int e = 0; e < kE; ++e) {
                const int s = b * kE + e;
                if (s < Lc) {
#pragma unroll
                    for (int r = 0; r < R; ++r) hist[e][r] = S[r];
                    fwd_step<DK>(S, sA + s * DK, sK + s * DK, sB[s], sV[s * kNW + w], additive,
                                 rr[e], uu[e]);
                }
            }
            // Sweep it backwards.
#pragma unroll
            for (int e = kE - 1; e >= 0; --e) {
                const int s = b * kE + e;
                if (s >= Lc) continue;
                const float *a = sA + s * DK, *kk = sK + s * DK, *qq = sQ + s * DK;
                const float beta = sB[s], dov = sDO[s * kNW + w];
                const float bread = additive ? 0.0f : beta;   // weight of the read path
                float *ae = acc + e * 3 * DK;
                float Sd[R], pdu = 0.0f;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int i = lane + 32 * r;
                    Sd[r] = a[i] * hist[e][r];
                    const float St = fmaf(kk[i], uu[e], Sd[r]);   // S_t, after the write
                    atomicAdd(&ae[i], p.scale * St * dov);         // dq^
                    dS[r] = fmaf(p.scale * qq[i], dov, dS[r]);
                    pdu = fmaf(dS[r], kk[i], pdu);
                }
                const float du = warp_sum(pdu);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int i = lane + 32 * r;
                    atomicAdd(&ae[DK + i], fmaf(dS[r], uu[e], -bread * Sd[r] * du)); // dk^
                    const float dSp = fmaf(-bread * kk[i], du, dS[r]);              // dS'
                    atomicAdd(&ae[2 * DK + i], dSp * Sd[r]);     // d log alpha = dalpha alpha
                    dS[r] = a[i] * dSp;
                }
                if (lane == 0) {
                    p.dv[((t0 + s) * p.H + h) * DV + j] = beta * du;
                    atomicAdd(&acc[kE * 3 * DK + e], du * (sV[s * kNW + w] - rr[e]));
                }
            }
            cl.sync();  // every CTA's sums of this block are complete
            // CTA `rank` finishes tokens rank, rank + G, ...: adds the G
            // partial sums in rank order, clears them for the block after next.
            for (int idx = threadIdx.x; idx < TPC * (3 * DK + 1); idx += kNT) {
                const int e = rank + G * (idx / (3 * DK + 1)), f = idx % (3 * DK + 1);
                const int s = b * kE + e;
                if (s >= Lc) continue;
                float *mine = acc + (f < 3 * DK ? e * 3 * DK + f : kE * 3 * DK + e);
                float sum = 0.0f;
                for (int c2 = 0; c2 < G; ++c2) {
                    float *rem = cl.map_shared_rank(mine, c2);
                    sum += *rem;
                    *rem = 0.0f;
                }
                const int64_t th = (t0 + s) * p.H + h;
                if (f < 3 * DK) p.sums[th * 3 * DK + f] = sum;
                else p.dbeta[th] = sum;
            }
        }
    }
    if (p.d_init_S) {
#pragma unroll
        for (int r = 0; r < R; ++r)
            p.d_init_S[(((int64_t)n * p.H + h) * DK + lane + 32 * r) * DV + j] = dS[r];
    }
    cl.sync();  // no CTA leaves while another may still read its shared memory
}

// One warp per (token, head): the column sums through the prologue.  Tokens
// outside every sequence are skipped (their rows stay as the caller left them).
template <typename IO, int DK>
__global__ void __launch_bounds__(256) delta_bwd_prologue_kernel(BwdParams p) {
    constexpr int R = DK / 32;
    const int lane = threadIdx.x & 31;
    const int64_t th = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (th >= (int64_t)p.ntok * p.H) return;
    const int64_t t = th / p.H;
    // the sequence holding token t: last n with cu[n] <= t
    int lo = 0, hi = p.N;
    while (hi - lo > 1) {
        const int mid = (lo + hi) / 2;
        if (p.cu[mid] <= t) lo = mid; else hi = mid;
    }
    if (!(p.cu[lo] <= t && t < p.cu[lo + 1])) return;

    const float *sum = p.sums + th * 3 * DK;
    if (lane == 0) {
        if (p.flags & kAdditive) {
            p.d_beta_logits[th] = 0.0f;   // the additive rule has no beta
        } else {
            const float beta = sigmoid_f(to_f32(static_cast<const IO *>(p.beta_logits)[th]));
            p.d_beta_logits[th] = p.dbeta[th] * beta * (1.0f - beta);
        }
    }
    const IO *g = static_cast<const IO *>(p.gate_logits);
    if (g) {
        if (p.flags & kGateScalar) {
            float da = 0.0f;
#pragma unroll
            for (int r = 0; r < R; ++r) da += sum[2 * DK + lane + 32 * r];
            da = warp_sum(da);
            if (lane == 0) p.d_gate_logits[th] = -da * sigmoid_f(to_f32(g[th]));
        } else {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int i = lane + 32 * r;
                // log alpha = -softplus(x): d x = -d(log alpha) sigmoid(x)
                p.d_gate_logits[th * DK + i] = -sum[2 * DK + i] * sigmoid_f(to_f32(g[th * DK + i]));
            }
        }
    }
    const bool silu = (p.flags & kSiluQK) != 0;
    for (int which = 0; which < 2; ++which) {
        const IO *src = static_cast<const IO *>(which ? p.k : p.q) + th * DK;
        float x[R], d[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            x[r] = to_f32(src[lane + 32 * r]);
            d[r] = sum[(which ? DK : 0) + lane + 32 * r];
        }
        prep_backward<R>(x, d, silu, (p.flags & (which ? kL2NormK : kL2NormQ)) != 0);
        float *dst = (which ? p.dk : p.dq) + th * DK;
#pragma unroll
        for (int r = 0; r < R; ++r) dst[lane + 32 * r] = d[r];
    }
}

// ------------------------------------------------------------------ host

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsParts {
    size_t ckpt, sums, dbeta, total;
};

WsParts ws_parts(int N, int ntok, int H, int dk, int dv) {
    const size_t slots = (size_t)ntok / kC + (size_t)N + 1;
    WsParts w;
    w.ckpt = align256(slots * H * dk * dv * sizeof(float));
    w.sums = align256((size_t)ntok * H * 3 * dk * sizeof(float));
    w.dbeta = align256((size_t)ntok * H * sizeof(float));
    w.total = w.ckpt + w.sums + w.dbeta;
    return w;
}

template <typename IO, int DK, int DV>
cudaError_t launch_t(const BwdArgs &a, BwdParams p, cudaStream_t s) {
    constexpr int G = DV / kNW;
    const size_t ck_smem = (size_t)Stage<DK>::FLOATS * sizeof(float);
    const size_t bw_smem = (size_t)BwdLayout<DK>::FLOATS * sizeof(float);
    auto ck = delta_bwd_ckpt_kernel<IO, DK, DV>;
    auto bw = delta_bwd_kernel<IO, DK, DV>;
    cudaError_t e = cudaFuncSetAttribute(ck, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ck_smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bw, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bw_smem);
    if (e != cudaSuccess) return e;
    const dim3 grid(G, a.H, a.N);
    ck<<<grid, kNT, ck_smem, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kNT);
    cfg.dynamicSmemBytes = bw_smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if ((e = cudaOccupancyMaxActiveClusters(&clusters, bw, &cfg)) != cudaSuccess) return e;
    if (clusters < 1) return cudaErrorInvalidConfiguration;
    if ((e = cudaLaunchKernelEx(&cfg, bw, p)) != cudaSuccess) return e;

    const int64_t rows = (int64_t)a.ntok * a.H;
    if (rows > 0) {
        delta_bwd_prologue_kernel<IO, DK><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(p);
        e = cudaGetLastError();
    }
    return e;
}

template <typename IO>
cudaError_t dispatch(const BwdArgs &a, BwdParams p, cudaStream_t s) {
    if (a.dk == 128 && a.dv == 128) return launch_t<IO, 128, 128>(a, p, s);
    if (a.dk == 128 && a.dv == 64) return launch_t<IO, 128, 64>(a, p, s);
    if (a.dk == 64 && a.dv == 128) return launch_t<IO, 64, 128>(a, p, s);
    return launch_t<IO, 64, 64>(a, p, s);
}

}  // namespace

size_t delta_bwd_workspace_bytes(int N, int ntok, int H, int dk, int dv) {
    // enough for either form (the chunkwise one exists for dk = dv)
    const size_t serial = ws_parts(N, ntok, H, dk, dv).total;
    const size_t chunked = dk == dv ? delta_bwd_chunked_workspace_bytes(N, ntok, H, dk) : 0;
    return serial > chunked ? serial : chunked;
}

cudaError_t launch_delta_backward(const BwdArgs &a, cudaStream_t s) {
    if (delta_bwd_chunked_supported(a)) return launch_delta_backward_chunked(a, s);
    const WsParts w = ws_parts(a.N, a.ntok, a.H, a.dk, a.dv);
    uint8_t *base = static_cast<uint8_t *>(a.workspace);
    BwdParams p{a.q, a.k, a.v, a.beta_logits, a.gate_logits, a.d_o, a.d_final_S, a.init_S,
                a.cu_seqlens, a.dq, a.dk_out, a.dv_out, a.d_beta_logits, a.d_gate_logits,
                a.d_init_S, reinterpret_cast<float *>(base),
                reinterpret_cast<float *>(base + w.ckpt),
                reinterpret_cast<float *>(base + w.ckpt + w.sums), device_error_word(), a.N, a.H,
                a.ntok, a.scale, a.flags};
    if (!p.err) return cudaErrorInvalidValue;
    return a.bf16 ? dispatch<__nv_bfloat16>(a, p, s) : dispatch<float>(a, p, s);
}

}  // namespace la
