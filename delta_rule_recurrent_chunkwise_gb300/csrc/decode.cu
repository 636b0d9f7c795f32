// decode.cu -- one recurrent decode step of the (gated) delta rule.
//
// Operation ("From GPT-2 to Kimi K3, explained", sections DeltaNet (Fast
// Weight Programmers) and Gated DeltaNet, with the per-key-channel decay of
// section KDA / Kimi Linear), per (sequence, head), state S in R^{dk x dv}:
//   S' = Diag(alpha) S
//   u  = beta (v - S'^T k)
//   S  <- S' + k u^T                      (in place)
//   o  = scale S^T q = scale (S'^T q + (q.k) u)
// (the additive rule of section Gated DeltaNet takes u = v instead)
// The last identity lets one pass over S produce both reductions S'^T k and
// S'^T q, so the state is read once and written once: the step streams
// 8 * dk * dv bytes of fp32 state per head and is bound by HBM bandwidth.
//
// Layout: the dv columns of S are independent, so each (sequence, head) is
// split into SPLIT column slices, one CTA of 256 threads each.  A thread
// owns a float4 column group of `RPT` rows of its slice and keeps them in
// registers between the read and the write; all loads are issued before the
// prologue runs so that each thread's whole share is in flight at once.
// With 32 KB per CTA and ~60 registers per thread, four CTAs share an SM,
// so one CTA's write phase overlaps the others' reads.
//
// Slot map (optional): with `slots` set, sequence n's state is entry
// slots[n] of a pool of n_slots states [n_slots][H][dk][dv]; a negative
// entry marks a padding sequence (no state or output is touched), an entry
// >= n_slots records code 100 in the error word and touches nothing.

#include "common.cuh"
#include "launch.h"

namespace la {
namespace {

struct DecodeParams {
    const void *q, *k, *v, *beta_logits, *gate_logits;
    void *o;
    float *state;
    const int32_t *slots;  // nullable: state of sequence n is slot n
    int64_t n_slots;
    unsigned *err;
    int H;
    float scale;
    unsigned flags;
};

constexpr int kSplit = 2;  // column slices per (sequence, head)

template <typename IO, int DK, int DV>
__global__ void __launch_bounds__(256, 4) decode_step_kernel(DecodeParams p) {
    constexpr int NT = 256;
    constexpr int DVS = DV / kSplit;    // columns of this CTA's slice
    constexpr int C4 = DVS / 4;         // float4 column groups per slice row
    constexpr int RPP = NT / C4;        // rows covered by one pass of the block
    constexpr int RPT = DK / RPP;       // rows held by each thread
    constexpr int C4F = DV / 4;         // float4 groups per full state row
    static_assert(DK % RPP == 0, "shape");

    __shared__ float sk[DK], sq[DK], sa[DK], sv[DVS], su[DVS];
    __shared__ __align__(16) float red_k[RPP][DVS];
    __shared__ __align__(16) float red_q[RPP][DVS];
    __shared__ float s_beta, s_qk;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t nh = blockIdx.x / kSplit;
    const int j0 = (blockIdx.x % kSplit) * DVS;   // first column of the slice
    const int col4 = tid % C4, row0 = tid / C4;
    int64_t sh = nh;                               // (state slot, head) of this CTA
    if (p.slots) {
        const int64_t n = nh / p.H, slot = p.slots[n];
        if (slot < 0) return;                      // padding sequence
        if (slot >= p.n_slots) {
            if (tid == 0) atomicCAS(p.err, 0u, 100u);
            return;
        }
        sh = slot * p.H + (nh - n * p.H);
    }
    float4 *S4 = reinterpret_cast<float4 *>(p.state + sh * (int64_t)(DK * DV) + j0);

    // 1. put this thread's share of the state in flight (streaming loads).
    float4 s[RPT];
#pragma unroll
    for (int m = 0; m < RPT; ++m) s[m] = __ldcs(S4 + (row0 + m * RPP) * C4F + col4);

    // 2. prologue: feature map / L2 norm of q and k, beta, per-channel decay.
    const IO *q = static_cast<const IO *>(p.q) + nh * DK;
    const IO *k = static_cast<const IO *>(p.k) + nh * DK;
    const IO *v = static_cast<const IO *>(p.v) + nh * DV;
    const bool silu = (p.flags & kSiluQK) != 0;
    if (tid < DK) {
        float kv = to_f32(k[tid]), qv = to_f32(q[tid]);
        if (silu) { kv = silu_f(kv); qv = silu_f(qv); }
        sk[tid] = kv;
        sq[tid] = qv;
        const int64_t gi = (p.flags & kGateScalar) ? nh : nh * DK + tid;  // scalar: one per head
        sa[tid] = p.gate_logits ? decay_f(to_f32(static_cast<const IO *>(p.gate_logits)[gi])) : 1.0f;
    }
    if (tid < DVS) sv[tid] = to_f32(v[j0 + tid]);
    __syncthreads();
    if (warp < 2) {
        float *x = warp == 0 ? sk : sq;
        const bool norm = (p.flags & (warp == 0 ? kL2NormK : kL2NormQ)) != 0;
        float ss = 0.0f;
        for (int i = lane; i < DK; i += 32) ss += x[i] * x[i];
        ss = warp_sum(ss);
        const float inv = norm ? 1.0f / fmaxf(sqrtf(ss), 1e-12f) : 1.0f;
        for (int i = lane; i < DK; i += 32) x[i] *= inv;
    } else if (warp == 2 && lane == 0) {
        s_beta = (p.flags & kAdditive) ? 1.0f
                                       : sigmoid_f(to_f32(static_cast<const IO *>(p.beta_logits)[nh]));
    }
    __syncthreads();
    if (warp == 0) {
        float d = 0.0f;
        for (int i = lane; i < DK; i += 32) d += sq[i] * sk[i];
        d = warp_sum(d);
        if (lane == 0) s_qk = d;
    }

    // 3. decay the rows, partial reductions S'^T k and S'^T q over own rows.
    float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
        const int r = row0 + m * RPP;
        const float a = sa[r], kr = sk[r], qr = sq[r];
        s[m].x *= a; s[m].y *= a; s[m].z *= a; s[m].w *= a;
        pk.x += kr * s[m].x; pk.y += kr * s[m].y; pk.z += kr * s[m].z; pk.w += kr * s[m].w;
        pq.x += qr * s[m].x; pq.y += qr * s[m].y; pq.z += qr * s[m].z; pq.w += qr * s[m].w;
    }
    reinterpret_cast<float4 *>(&red_k[row0][0])[col4] = pk;
    reinterpret_cast<float4 *>(&red_q[row0][0])[col4] = pq;
    __syncthreads();

    // 4. column totals, the delta u and the output.
    if (tid < DVS) {
        float rk = 0.0f, rq = 0.0f;
#pragma unroll
        for (int i = 0; i < RPP; ++i) { rk += red_k[i][tid]; rq += red_q[i][tid]; }
        const float u = s_beta * (sv[tid] - ((p.flags & kAdditive) ? 0.0f : rk));
        su[tid] = u;
        static_cast<IO *>(p.o)[nh * DV + j0 + tid] = from_f32<IO>(p.scale * (rq + s_qk * u));
    }
    __syncthreads();

    // 5. write S' + k u^T back in place.
    const float4 u4 = reinterpret_cast<const float4 *>(su)[col4];
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
        const int r = row0 + m * RPP;
        const float kr = sk[r];
        float4 w = s[m];
        w.x += kr * u4.x; w.y += kr * u4.y; w.z += kr * u4.z; w.w += kr * u4.w;
        __stcs(S4 + r * C4F + col4, w);
    }
}

template <typename IO, int DK, int DV>
cudaError_t launch_t(const DecodeArgs &a, cudaStream_t s) {
    DecodeParams p{a.q, a.k, a.v, a.beta_logits, a.gate_logits, a.o, a.state,
                   a.slots, a.n_slots, a.err, a.H, a.scale, a.flags};
    const unsigned grid = (unsigned)((int64_t)a.N * a.H * kSplit);
    decode_step_kernel<IO, DK, DV><<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

template <typename IO>
cudaError_t dispatch(const DecodeArgs &a, cudaStream_t s) {
    if (a.dk == 128 && a.dv == 128) return launch_t<IO, 128, 128>(a, s);
    if (a.dk == 128 && a.dv == 64) return launch_t<IO, 128, 64>(a, s);
    if (a.dk == 64 && a.dv == 128) return launch_t<IO, 64, 128>(a, s);
    return launch_t<IO, 64, 64>(a, s);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s) {
    return a.bf16 ? dispatch<__nv_bfloat16>(a, s) : dispatch<float>(a, s);
}

}  // namespace la
