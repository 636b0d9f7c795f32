// prefill_simt.cu -- fp32 CUDA-core chunkwise prefill kernels.
//
// These kernels compute every product in fp32 FMA (no tensor cores), which
// is what fp32 I/O at a 1e-4 relative tolerance needs.  One CTA of 256
// threads scans one (sequence, head, 32-wide dv slice) chunk by chunk; the
// dv columns of the state are independent, so slicing dv multiplies the
// number of concurrent scans without any exchange.
//
// Chunked forms ("From GPT-2 to Kimi K3, explained", section DeltaNet
// (Parallelizing Linear Transformers with Delta Rule)): inside a chunk the
// masked q k^T scores act on the chunk's own values, across chunks
// everything is folded into the state and read back with one product.
//
// Delta rule (eq. 8-10 of that section, extended with the cumulative
// per-key-channel decay of sections Gated DeltaNet and KDA / Kimi Linear):
// with b = inclusive cumulative sum of log alpha inside the chunk,
//   A[r][i]  = beta_r sum_c k_rc k_ic e^{b_rc - b_ic}      (i < r)
//   Aq[r][i] =        sum_c q_rc k_ic e^{b_rc - b_ic}      (i <= r)
//   T        = (I + A)^{-1}                               (forward substitution)
//   u        = T (beta (V - (K e^{b}) S))                 (= U - W S of eq. 8-10)
//   (additive rule: A = 0, beta = 1 and no read, so u = V)
//   O        = scale ((Q e^{b}) S + Aq u)
//   S       <- Diag(e^{b_end}) S + (K e^{b_end - b})^T u
// Every exponent used is a difference b_r - b_i with i <= r, so it is <= 0:
// nothing overflows however strong the decay.  The tail chunk of a sequence
// is padded with k = q = v = 0, beta = 0, log alpha = 0, which leaves the
// state and the valid rows unchanged.

#include "common.cuh"
#include "launch.h"

namespace la {
namespace {

constexpr int kC = 64;    // tokens per chunk
constexpr int kDVS = 32;  // dv columns per CTA
constexpr int kNT = 256;  // threads per CTA

struct SimtParams {
    const void *q, *k, *v, *beta_logits, *gate_logits;
    void *o;
    const int32_t *cu_seqlens;
    unsigned *err;
    int H, dv, ntok;
    float scale;
    unsigned flags;
    const float *init_S, *init_z;
    float *final_S, *final_z;
};

template <int DK>
constexpr size_t delta_smem_floats() {
    return 3 * (size_t)kC * (DK + 1) + 2 * (size_t)kC * (kDVS + 1) + 2 * (size_t)kC * (kC + 1) +
           (size_t)DK * (kDVS + 1) + kC + DK;
}

template <typename IO, int DK>
__global__ void __launch_bounds__(kNT) delta_chunk_simt_kernel(SimtParams p) {
    constexpr int C = kC, DVS = kDVS, NT = kNT;
    constexpr int LDK = DK + 1, LDV = DVS + 1, LDC = C + 1;
    extern __shared__ float smem[];
    float *sK = smem;              // [C][LDK]  k (prepared) -> K e^{b_end - b}
    float *sQ = sK + C * LDK;      // [C][LDK]  q (prepared) -> Q e^{b}
    float *sB = sQ + C * LDK;      // [C][LDK]  b = cumsum log alpha -> K e^{b}
    float *sV = sB + C * LDK;      // [C][LDV]  v -> beta (v - K e^{b} S)
    float *sU = sV + C * LDV;      // [C][LDV]  u
    float *sA = sU + C * LDV;      // [C][LDC]  A -> T
    float *sAq = sA + C * LDC;     // [C][LDC]  Aq
    float *sS = sAq + C * LDC;     // [DK][LDV] state slice
    float *sBeta = sS + DK * LDV;  // [C]
    float *sGend = sBeta + C;      // [DK]      b_end, then e^{b_end}

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = blockIdx.z, h = blockIdx.y, j0 = blockIdx.x * DVS;
    const int H = p.H, dv = p.dv;
    const bool gated = p.gate_logits != nullptr;
    const bool gate_scalar = (p.flags & kGateScalar) != 0;  // gate [ntok][H]
    const bool silu = (p.flags & kSiluQK) != 0;
    const bool additive = (p.flags & kAdditive) != 0;  // u = v: no delta term, no beta
    const IO *Q = static_cast<const IO *>(p.q), *K = static_cast<const IO *>(p.k);
    const IO *V = static_cast<const IO *>(p.v);
    const IO *BL = static_cast<const IO *>(p.beta_logits);
    const IO *GL = static_cast<const IO *>(p.gate_logits);
    IO *O = static_cast<IO *>(p.o);
    int t_begin = p.cu_seqlens[n], t_end = p.cu_seqlens[n + 1];
    if (t_begin < 0 || t_end < t_begin || t_end > p.ntok) {
        if (tid == 0 && p.err) atomicCAS(p.err, 0u, 100u);
        t_begin = t_end = 0;
    }
    const int64_t sbase = ((int64_t)n * H + h) * DK * dv + j0;

    for (int e = tid; e < DK * DVS; e += NT) {
        const int c = e / DVS, j = e % DVS;
        sS[c * LDV + j] = p.init_S ? p.init_S[sbase + (int64_t)c * dv + j] : 0.0f;
    }

    for (int cs = t_begin; cs < t_end; cs += C) {
        const int len = min(C, t_end - cs);
        __syncthreads();
        // ---- load the chunk (padded rows are zero; log alpha = 0 there)
        for (int e = tid; e < C * DK; e += NT) {
            const int r = e / DK, c = e % DK;
            const bool ok = r < len;
            const int64_t g = ((int64_t)(cs + r) * H + h) * DK + c;
            sK[r * LDK + c] = ok ? to_f32(K[g]) : 0.0f;
            sQ[r * LDK + c] = ok ? to_f32(Q[g]) : 0.0f;
            if (gated)
                sB[r * LDK + c] = ok ? log_decay_f(to_f32(GL[gate_scalar ? (int64_t)(cs + r) * H + h : g]))
                                     : 0.0f;
        }
        for (int e = tid; e < C * DVS; e += NT) {
            const int r = e / DVS, j = e % DVS;
            sV[r * LDV + j] = r < len ? to_f32(V[((int64_t)(cs + r) * H + h) * dv + j0 + j]) : 0.0f;
        }
        if (tid < C)
            sBeta[tid] = tid >= len ? 0.0f
                         : additive ? 1.0f
                                    : sigmoid_f(to_f32(BL[(int64_t)(cs + tid) * H + h]));
        __syncthreads();
        // ---- prologue: silu, L2 norms (one warp per row), decay cumsum
        for (int r = warp; r < C; r += NT / 32) {
            float sk = 0.0f, sq = 0.0f;
            for (int c = lane; c < DK; c += 32) {
                float kv = sK[r * LDK + c], qv = sQ[r * LDK + c];
                if (silu) { kv = silu_f(kv); qv = silu_f(qv); sK[r * LDK + c] = kv; sQ[r * LDK + c] = qv; }
                sk += kv * kv;
                sq += qv * qv;
            }
            sk = warp_sum(sk);
            sq = warp_sum(sq);
            const float ik = (p.flags & kL2NormK) ? 1.0f / fmaxf(sqrtf(sk), 1e-12f) : 1.0f;
            const float iq = (p.flags & kL2NormQ) ? 1.0f / fmaxf(sqrtf(sq), 1e-12f) : 1.0f;
            for (int c = lane; c < DK; c += 32) { sK[r * LDK + c] *= ik; sQ[r * LDK + c] *= iq; }
        }
        if (gated) {
            for (int c = tid; c < DK; c += NT) {
                float acc = 0.0f;
                for (int r = 0; r < C; ++r) { acc += sB[r * LDK + c]; sB[r * LDK + c] = acc; }
                sGend[c] = acc;
            }
        }
        __syncthreads();
        // ---- A (strict, beta-scaled rows) and Aq (inclusive)
        for (int e = tid; e < C * C; e += NT) {
            const int r = e / C, i = e % C;
            float akk = 0.0f, aqk = 0.0f;
            if (i <= r) {
                const float *kr = sK + r * LDK, *ki = sK + i * LDK, *qr = sQ + r * LDK;
                if (gated) {
                    const float *br = sB + r * LDK, *bi = sB + i * LDK;
                    for (int c = 0; c < DK; ++c) {
                        const float f = ki[c] * expf(br[c] - bi[c]);
                        akk += kr[c] * f;
                        aqk += qr[c] * f;
                    }
                } else {
                    for (int c = 0; c < DK; ++c) { akk += kr[c] * ki[c]; aqk += qr[c] * ki[c]; }
                }
            }
            sA[r * LDC + i] = (i < r && !additive) ? sBeta[r] * akk : 0.0f;
            sAq[r * LDC + i] = aqk;
        }
        __syncthreads();
        // ---- T = (I + A)^{-1}: T[i][j] = -(A[i][j] + sum_{j<m<i} A[i][m] T[m][j])
        for (int i = 1; i < C; ++i) {
            float tv = 0.0f;
            if (tid < i) {
                float acc = sA[i * LDC + tid];
                for (int m = tid + 1; m < i; ++m) acc += sA[i * LDC + m] * sA[m * LDC + tid];
                tv = -acc;
            }
            __syncthreads();
            if (tid < i) sA[i * LDC + tid] = tv;
            __syncthreads();
        }
        if (tid < C) sA[tid * LDC + tid] = 1.0f;
        // ---- decay factors: Q e^{b}, K e^{b} (into sB), K e^{b_end - b}
        if (gated) {
            for (int e = tid; e < C * DK; e += NT) {
                const int r = e / DK, c = e % DK;
                const float b = sB[r * LDK + c], kk = sK[r * LDK + c];
                sQ[r * LDK + c] *= expf(b);
                sB[r * LDK + c] = kk * expf(b);
                sK[r * LDK + c] = kk * expf(sGend[c] - b);
            }
        }
        __syncthreads();
        if (gated && tid < DK) sGend[tid] = expf(sGend[tid]);
        const float *sKg = gated ? sB : sK;
        // ---- R = beta (V - (K e^{b}) S)
        for (int e = tid; e < C * DVS; e += NT) {
            const int r = e / DVS, j = e % DVS;
            float acc = 0.0f;
            for (int c = 0; c < DK; ++c) acc += sKg[r * LDK + c] * sS[c * LDV + j];
            sV[r * LDV + j] = sBeta[r] * (sV[r * LDV + j] - (additive ? 0.0f : acc));
        }
        __syncthreads();
        // ---- u = T R
        for (int e = tid; e < C * DVS; e += NT) {
            const int r = e / DVS, j = e % DVS;
            float acc = 0.0f;
            for (int i = 0; i <= r; ++i) acc += sA[r * LDC + i] * sV[i * LDV + j];
            sU[r * LDV + j] = acc;
        }
        __syncthreads();
        // ---- O = scale ((Q e^{b}) S + Aq u)
        for (int e = tid; e < C * DVS; e += NT) {
            const int r = e / DVS, j = e % DVS;
            if (r < len) {
                float acc = 0.0f;
                for (int c = 0; c < DK; ++c) acc += sQ[r * LDK + c] * sS[c * LDV + j];
                for (int i = 0; i <= r; ++i) acc += sAq[r * LDC + i] * sU[i * LDV + j];
                O[((int64_t)(cs + r) * H + h) * dv + j0 + j] = from_f32<IO>(p.scale * acc);
            }
        }
        __syncthreads();
        // ---- S <- Diag(e^{b_end}) S + (K e^{b_end - b})^T u
        for (int e = tid; e < DK * DVS; e += NT) {
            const int c = e / DVS, j = e % DVS;
            float acc = 0.0f;
            for (int i = 0; i < C; ++i) acc += sK[i * LDK + c] * sU[i * LDV + j];
            const float g = gated ? sGend[c] : 1.0f;
            sS[c * LDV + j] = g * sS[c * LDV + j] + acc;
        }
    }
    __syncthreads();
    if (p.final_S) {
        for (int e = tid; e < DK * DVS; e += NT) {
            const int c = e / DVS, j = e % DVS;
            p.final_S[sbase + (int64_t)c * dv + j] = sS[c * LDV + j];
        }
    }
}

// ELU+1 linear attention ("From GPT-2 to Kimi K3, explained", section Linear
// attention, chunked as in the next section):
//   A = tril(phi(Q) phi(K)^T)                           (inclusive)
//   O = (phi(Q) S + A V) / (phi(Q) z + A 1)
//   S <- S + phi(K)^T V,   z <- z + sum_i phi(k_i)
// One CTA of 256 threads per (sequence, head, 16 value columns), chunk after
// chunk.  Narrow value slices give more CTAs to short batches; each CTA
// forms the chunk's score matrix itself (4 x 4 register tiles of the lower
// triangle, float4 operands), then every thread owns 4 output columns of one
// row, and the denominator is summed over the row's 4 threads.
constexpr int kLJ = 16;  // value columns per CTA

template <int DK>
struct LinLayout {
    static constexpr int LDQ = DK + 4;   // phi(q), phi(k) rows: 16-byte aligned, float4 columns conflict-free
    static constexpr int LDP = kC + 4;
    static constexpr int Q = 0, K = Q + kC * LDQ, P = K + kC * LDQ, V = P + kC * LDP;
    static constexpr int HS = V + kC * kLJ, Z = HS + DK * kLJ, FLOATS = Z + DK;
};

__device__ __forceinline__ float dot4(const float4 a, const float4 b) {
    return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

__device__ __forceinline__ void axpy4(float4 &acc, float s, const float4 v) {
    acc.x = fmaf(s, v.x, acc.x);
    acc.y = fmaf(s, v.y, acc.y);
    acc.z = fmaf(s, v.z, acc.z);
    acc.w = fmaf(s, v.w, acc.w);
}

template <typename IO, int DK>
__global__ void __launch_bounds__(kNT) linear_chunk_simt_kernel(SimtParams p) {
    using L = LinLayout<DK>;
    constexpr int C = kC, NT = kNT, LDQ = L::LDQ, LDP = L::LDP, LJ = kLJ;
    extern __shared__ __align__(16) float smem[];
    float *sQ = smem + L::Q, *sK = smem + L::K, *sP = smem + L::P, *sV = smem + L::V;
    float *sH = smem + L::HS, *sZ = smem + L::Z;

    const int tid = threadIdx.x;
    const int n = blockIdx.z, h = blockIdx.y, j0 = blockIdx.x * LJ;
    const int H = p.H, dv = p.dv;
    const IO *Q = static_cast<const IO *>(p.q), *K = static_cast<const IO *>(p.k);
    const IO *V = static_cast<const IO *>(p.v);
    IO *O = static_cast<IO *>(p.o);
    int t_begin = p.cu_seqlens[n], t_end = p.cu_seqlens[n + 1];
    if (t_begin < 0 || t_end < t_begin || t_end > p.ntok) {
        if (tid == 0 && p.err) atomicCAS(p.err, 0u, 100u);
        t_begin = t_end = 0;
    }
    const int64_t sbase = ((int64_t)n * H + h) * DK * dv + j0;
    const int64_t zbase = ((int64_t)n * H + h) * DK;

    for (int e = tid; e < DK * LJ; e += NT) {
        const int c = e / LJ, j = e % LJ;
        sH[e] = p.init_S ? p.init_S[sbase + (int64_t)c * dv + j] : 0.0f;
    }
    for (int c = tid; c < DK; c += NT) sZ[c] = p.init_z ? p.init_z[zbase + c] : 0.0f;

    // The raw q, k and value-slice elements of a chunk, held in registers:
    // the next chunk's are loaded (all at once) while this one computes.
    constexpr int QU = C * DK / 4 / NT;   // 4-element units of q (and k) per thread
    static_assert(QU * NT * 4 == C * DK && C * LJ / 4 == NT, "load mapping");
    float rq[QU][4], rk[QU][4], rv[4];
    auto load_raw = [&](int cs) {
        const int len = min(C, t_end - cs);
#pragma unroll
        for (int u = 0; u < QU; ++u) {
            const int e = tid + u * NT, r = e / (DK / 4), c = (e % (DK / 4)) * 4;
            const int64_t g = ((int64_t)(cs + (r < len ? r : 0)) * H + h) * DK + c;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                rq[u][i] = r < len ? to_f32(Q[g + i]) : 0.0f;
                rk[u][i] = r < len ? to_f32(K[g + i]) : 0.0f;
            }
        }
        const int r = tid / (LJ / 4), j = (tid % (LJ / 4)) * 4;
        const int64_t g = ((int64_t)(cs + (r < len ? r : 0)) * H + h) * dv + j0 + j;
#pragma unroll
        for (int i = 0; i < 4; ++i) rv[i] = r < len ? to_f32(V[g + i]) : 0.0f;
    };
    if (t_begin < t_end) load_raw(t_begin);

    for (int cs = t_begin; cs < t_end; cs += C) {
        const int len = min(C, t_end - cs);
        __syncthreads();
        // phi(q), phi(k) (zero rows past the chunk's end) and the value slice
#pragma unroll
        for (int u = 0; u < QU; ++u) {
            const int e = tid + u * NT, r = e / (DK / 4), c = (e % (DK / 4)) * 4;
            const bool ok = r < len;
            const float4 fq = make_float4(ok ? elu1_f(rq[u][0]) : 0.f, ok ? elu1_f(rq[u][1]) : 0.f,
                                          ok ? elu1_f(rq[u][2]) : 0.f, ok ? elu1_f(rq[u][3]) : 0.f);
            const float4 fk = make_float4(ok ? elu1_f(rk[u][0]) : 0.f, ok ? elu1_f(rk[u][1]) : 0.f,
                                          ok ? elu1_f(rk[u][2]) : 0.f, ok ? elu1_f(rk[u][3]) : 0.f);
            *reinterpret_cast<float4 *>(sQ + r * LDQ + c) = fq;
            *reinterpret_cast<float4 *>(sK + r * LDQ + c) = fk;
        }
        *reinterpret_cast<float4 *>(sV + (tid / (LJ / 4)) * LJ + (tid % (LJ / 4)) * 4) =
            make_float4(rv[0], rv[1], rv[2], rv[3]);
        __syncthreads();
        if (cs + C < t_end) load_raw(cs + C);   // in flight during this chunk's products
        // scores A[r][i] = phi(q_r) . phi(k_i), i <= r: thread (tr, tc) takes
        // rows 4 tr .. 4 tr + 3 and columns 4 tc .. 4 tc + 3 (tiles above the
        // diagonal are never read)
        {
            const int tr = tid >> 4, tc = tid & 15;
            if (tc <= tr) {
                float acc[4][4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
#pragma unroll 4
                for (int c = 0; c < DK; c += 4) {
                    float4 a[4], b[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        a[i] = *reinterpret_cast<const float4 *>(sQ + (4 * tr + i) * LDQ + c);
                        b[i] = *reinterpret_cast<const float4 *>(sK + (4 * tc + i) * LDQ + c);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[i][j] += dot4(a[i], b[j]);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = 4 * tr + i;
                    float4 o4;
                    o4.x = (4 * tc + 0 <= r) ? acc[i][0] : 0.0f;
                    o4.y = (4 * tc + 1 <= r) ? acc[i][1] : 0.0f;
                    o4.z = (4 * tc + 2 <= r) ? acc[i][2] : 0.0f;
                    o4.w = (4 * tc + 3 <= r) ? acc[i][3] : 0.0f;
                    *reinterpret_cast<float4 *>(sP + r * LDP + 4 * tc) = o4;
                }
            }
        }
        __syncthreads();
        // outputs: thread (r, jq) owns columns jq .. jq + 3 of row r; the
        // row's four threads split the denominator's sums and add them up
        {
            const int r = tid >> 2, part = tid & 3, jq = part * 4;
            float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
            float den = 0.0f;
            const float *qr = sQ + r * LDQ, *pr = sP + r * LDP;
#pragma unroll 8
            for (int c = 0; c < DK; ++c) axpy4(num, qr[c], *reinterpret_cast<const float4 *>(sH + c * LJ + jq));
            for (int c = part; c < DK; c += 4) den = fmaf(qr[c], sZ[c], den);
            for (int i = 0; i <= r; ++i) axpy4(num, pr[i], *reinterpret_cast<const float4 *>(sV + i * LJ + jq));
            for (int i = part; i <= r; i += 4) den += pr[i];
            den += __shfl_xor_sync(0xffffffffu, den, 1);
            den += __shfl_xor_sync(0xffffffffu, den, 2);
            if (r < len) {
                const float inv = 1.0f / den;
                IO *dst = O + ((int64_t)(cs + r) * H + h) * dv + j0 + jq;
                dst[0] = from_f32<IO>(num.x * inv);
                dst[1] = from_f32<IO>(num.y * inv);
                dst[2] = from_f32<IO>(num.z * inv);
                dst[3] = from_f32<IO>(num.w * inv);
            }
        }
        __syncthreads();
        // state slice and normaliser: S += phi(K)^T V, z += sum of phi(k)
        for (int e = tid; e < DK * (LJ / 4); e += NT) {
            const int c = e / (LJ / 4), jq = (e % (LJ / 4)) * 4;
            float4 acc = *reinterpret_cast<const float4 *>(sH + c * LJ + jq);
#pragma unroll 8
            for (int i = 0; i < C; ++i) axpy4(acc, sK[i * LDQ + c], *reinterpret_cast<const float4 *>(sV + i * LJ + jq));
            *reinterpret_cast<float4 *>(sH + c * LJ + jq) = acc;
        }
        for (int c = tid; c < DK; c += NT) {
            float acc = sZ[c];
            for (int i = 0; i < C; ++i) acc += sK[i * LDQ + c];
            sZ[c] = acc;
        }
    }
    __syncthreads();
    if (p.final_S)
        for (int e = tid; e < DK * LJ; e += NT) {
            const int c = e / LJ, j = e % LJ;
            p.final_S[sbase + (int64_t)c * dv + j] = sH[e];
        }
    if (p.final_z && blockIdx.x == 0)
        for (int c = tid; c < DK; c += NT) p.final_z[zbase + c] = sZ[c];
}

// Short sequences (at most kPMax chunks each): one 512-thread CTA per
// (sequence, head, chunk, 16 value columns), all chunks of a sequence side by
// side.  A chunk's starting state is the initial state plus the earlier
// chunks' phi(K)^T V (at most kPMax - 1 of them, recomputed by the CTA), so
// no chunk waits for another; the CTA of a sequence's last chunk also writes
// the final state.  Narrow value slices keep each CTA's serial work short
// (the recomputed sums and the outputs scale with the slice; only the
// chunk's 64 x 64 scores are repeated per slice).  fp32 throughout.
constexpr int kPMax = 8;    // chunks per sequence for the chunk-parallel form
constexpr int kPJ = 16;     // value columns per CTA
constexpr int kPNT = 512;   // threads per CTA

template <int DK>
struct PLayout {
    static constexpr int LDK = DK + 4, LDV = kPJ + 4, LDP = kC + 4;
    static constexpr int K = 0, V = K + kC * LDK, Q = V + kC * LDV, P = Q + kC * LDK,
                         S = P + kC * LDP, Z = S + DK * LDV, FLOATS = Z + DK;
};

template <typename IO, int DK>
__global__ void __launch_bounds__(kPNT) linear_prefix_simt_kernel(SimtParams p, int cmax) {
    using L = PLayout<DK>;
    constexpr int C = kC, NT = kPNT, LDK = L::LDK, LDV = L::LDV, LDP = L::LDP, J = kPJ;
    constexpr int CPT = J * DK / NT;     // state columns per thread (one state row each)
    constexpr int UK = C * DK / NT;      // phi(k) (and phi(q)) elements per thread per chunk
    constexpr int UV = C * J / NT;       // value elements per thread per chunk
    static_assert(CPT == 2 || CPT == 4, "state mapping");
    extern __shared__ __align__(16) float smem[];
    float *sK = smem + L::K, *sV = smem + L::V, *sQ = smem + L::Q, *sP = smem + L::P;
    float *sS = smem + L::S, *sZ = smem + L::Z;

    const int tid = threadIdx.x;
    const int c = blockIdx.x % cmax, j0 = (blockIdx.x / cmax) * J;
    const int h = blockIdx.y, n = blockIdx.z, H = p.H, dv = p.dv;
    const IO *Q = static_cast<const IO *>(p.q), *K = static_cast<const IO *>(p.k);
    const IO *V = static_cast<const IO *>(p.v);
    IO *O = static_cast<IO *>(p.o);
    int t_begin = p.cu_seqlens[n], t_end = p.cu_seqlens[n + 1];
    if (t_begin < 0 || t_end < t_begin || t_end > p.ntok || t_end - t_begin > kPMax * C) {
        if (tid == 0 && p.err) atomicCAS(p.err, 0u, 100u);
        t_begin = t_end = 0;
    }
    const int nc = (t_end - t_begin + C - 1) / C;
    // chunk 0 of an empty sequence still writes the final state (= initial)
    if (c >= (nc > 0 ? nc : 1)) return;
    const int64_t sbase = ((int64_t)n * H + h) * DK * dv + j0;
    const int64_t zbase = ((int64_t)n * H + h) * DK;

    // raw chunk elements in registers, loaded one chunk ahead
    float rk[UK], rv[UV], rq[UK];
    auto load_kv = [&](int j) {
        const int cs = t_begin + j * C, len = min(C, t_end - cs);
#pragma unroll
        for (int u = 0; u < UK; ++u) {
            const int e = tid + u * NT, r = e / DK, col = e % DK;
            rk[u] = r < len ? to_f32(K[((int64_t)(cs + r) * H + h) * DK + col]) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < UV; ++u) {
            const int e = tid + u * NT, r = e / J, col = e % J;
            rv[u] = r < len ? to_f32(V[((int64_t)(cs + r) * H + h) * dv + j0 + col]) : 0.0f;
        }
    };
    // phi(k) (0 past the chunk's end) and the value slice into shared memory
    auto stage_kv = [&](int j) {
        const int len = min(C, t_end - (t_begin + j * C));
#pragma unroll
        for (int u = 0; u < UK; ++u) {
            const int e = tid + u * NT, r = e / DK, col = e % DK;
            sK[r * LDK + col] = r < len ? elu1_f(rk[u]) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < UV; ++u) {
            const int e = tid + u * NT, r = e / J, col = e % J;
            sV[r * LDV + col] = rv[u];
        }
    };
    // state row srow, columns scol .. scol + CPT - 1 of the slice, in registers
    const int srow = tid / (J / CPT), scol = (tid % (J / CPT)) * CPT;
    float acc[CPT];
    float zacc = 0.0f;  // thread tid < DK: z[tid]
#pragma unroll
    for (int i = 0; i < CPT; ++i)
        acc[i] = p.init_S ? p.init_S[sbase + (int64_t)srow * dv + scol + i] : 0.0f;
    if (tid < DK) zacc = p.init_z ? p.init_z[zbase + tid] : 0.0f;
    // S += phi(K)^T V, z += column sums of phi(K), from the staged chunk
    auto accumulate = [&]() {
#pragma unroll 8
        for (int i = 0; i < C; ++i) {
            const float kk = sK[i * LDK + srow];
            if constexpr (CPT == 4) {
                const float4 v4 = *reinterpret_cast<const float4 *>(sV + i * LDV + scol);
                acc[0] = fmaf(kk, v4.x, acc[0]);
                acc[1] = fmaf(kk, v4.y, acc[1]);
                acc[2] = fmaf(kk, v4.z, acc[2]);
                acc[3] = fmaf(kk, v4.w, acc[3]);
            } else {
                const float2 v2 = *reinterpret_cast<const float2 *>(sV + i * LDV + scol);
                acc[0] = fmaf(kk, v2.x, acc[0]);
                acc[1] = fmaf(kk, v2.y, acc[1]);
            }
        }
        if (tid < DK)
            for (int i = 0; i < C; ++i) zacc += sK[i * LDK + tid];
    };

    // ---- the state at this chunk's start
    if (nc > 0) load_kv(0);
    for (int j = 0; j < c; ++j) {
        __syncthreads();
        stage_kv(j);
        __syncthreads();
        load_kv(j + 1);  // the next chunk (this CTA's own at j + 1 == c) in flight
        accumulate();
    }
    if (nc == 0) {
        // empty sequence: the final state is the initial one
        if (p.final_S)
#pragma unroll
            for (int i = 0; i < CPT; ++i) p.final_S[sbase + (int64_t)srow * dv + scol + i] = acc[i];
        if (p.final_z && j0 == 0 && tid < DK) p.final_z[zbase + tid] = zacc;
        return;
    }
    // ---- this chunk: phi(q), phi(k), v, and the state into shared memory
    const int cs = t_begin + c * C, len = min(C, t_end - cs);
#pragma unroll
    for (int u = 0; u < UK; ++u) {
        const int e = tid + u * NT, r = e / DK, col = e % DK;
        rq[u] = r < len ? to_f32(Q[((int64_t)(cs + r) * H + h) * DK + col]) : 0.0f;
    }
    __syncthreads();
    stage_kv(c);
#pragma unroll
    for (int u = 0; u < UK; ++u) {
        const int e = tid + u * NT, r = e / DK, col = e % DK;
        sQ[r * LDK + col] = r < len ? elu1_f(rq[u]) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < CPT; ++i) sS[srow * LDV + scol + i] = acc[i];
    if (tid < DK) sZ[tid] = zacc;
    __syncthreads();
    // scores P[r][i] = phi(q_r) . phi(k_i), i <= r (else 0): thread (tr, tc)
    // takes rows 2 tr, 2 tr + 1 and columns tc, tc + 16, tc + 32, tc + 48;
    // tiles wholly above the diagonal only write zeros
    {
        const int tr = tid >> 4, tc = tid & 15;
        float pa[2][4];
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) pa[a][b] = 0.0f;
        const int nb = min(4, (2 * tr + 1 - tc) / 16 + 1);  // column groups reaching the diagonal
        if (tc <= 2 * tr + 1) {
#pragma unroll 2
            for (int k0 = 0; k0 < DK; k0 += 4) {
                const float4 q0 = *reinterpret_cast<const float4 *>(sQ + (2 * tr) * LDK + k0);
                const float4 q1 = *reinterpret_cast<const float4 *>(sQ + (2 * tr + 1) * LDK + k0);
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    if (b < nb) {
                        const float4 kb = *reinterpret_cast<const float4 *>(sK + (tc + 16 * b) * LDK + k0);
                        pa[0][b] += dot4(q0, kb);
                        pa[1][b] += dot4(q1, kb);
                    }
                }
            }
        }
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int r = 2 * tr + a, i = tc + 16 * b;
                sP[r * LDP + i] = i <= r ? pa[a][b] : 0.0f;
            }
    }
    __syncthreads();
    // outputs: thread (r, part) owns columns 2 part, 2 part + 1 of row r; the
    // row's eight threads (consecutive lanes) split the denominator's sums
    {
        const int r = tid >> 3, part = tid & 7, jq = 2 * part;
        float n0 = 0.0f, n1 = 0.0f, den = 0.0f;
        const float *qr = sQ + r * LDK, *pr = sP + r * LDP;
#pragma unroll 8
        for (int k0 = 0; k0 < DK; ++k0) {
            const float a = qr[k0];
            const float2 s2 = *reinterpret_cast<const float2 *>(sS + k0 * LDV + jq);
            n0 = fmaf(a, s2.x, n0);
            n1 = fmaf(a, s2.y, n1);
        }
        for (int k0 = part; k0 < DK; k0 += 8) den = fmaf(qr[k0], sZ[k0], den);
        for (int i = 0; i <= r; ++i) {
            const float a = pr[i];
            const float2 v2 = *reinterpret_cast<const float2 *>(sV + i * LDV + jq);
            n0 = fmaf(a, v2.x, n0);
            n1 = fmaf(a, v2.y, n1);
        }
        for (int i = part; i <= r; i += 8) den += pr[i];
        den += __shfl_xor_sync(0xffffffffu, den, 1);
        den += __shfl_xor_sync(0xffffffffu, den, 2);
        den += __shfl_xor_sync(0xffffffffu, den, 4);
        if (r < len) {
            const float inv = 1.0f / den;
            IO *dst = O + ((int64_t)(cs + r) * H + h) * dv + j0 + jq;
            dst[0] = from_f32<IO>(n0 * inv);
            dst[1] = from_f32<IO>(n1 * inv);
        }
    }
    // ---- the last chunk's CTA: the final state
    if (c == nc - 1 && (p.final_S || p.final_z)) {
        accumulate();  // reads the staged phi(k), v of this chunk (unchanged since)
        if (p.final_S)
#pragma unroll
            for (int i = 0; i < CPT; ++i) p.final_S[sbase + (int64_t)srow * dv + scol + i] = acc[i];
        if (p.final_z && j0 == 0 && tid < DK) p.final_z[zbase + tid] = zacc;
    }
}

SimtParams to_params(const PrefillArgs &a) {
    return SimtParams{a.q, a.k, a.v, a.beta_logits, a.gate_logits, a.o, a.cu_seqlens,
                      device_error_word(), a.H, a.dv, a.ntok, a.scale, a.flags, a.init_S,
                      a.init_z, a.final_S, a.final_z};
}

template <typename Kern>
cudaError_t launch_kernel(Kern kern, size_t smem, const PrefillArgs &a, cudaStream_t s,
                          int dvs = kDVS) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.dv / dvs, a.H, a.N);
    kern<<<grid, kNT, smem, s>>>(to_params(a));
    return cudaGetLastError();
}

template <typename IO>
cudaError_t delta_dispatch(const PrefillArgs &a, cudaStream_t s) {
    if (a.dk == 128)
        return launch_kernel(delta_chunk_simt_kernel<IO, 128>, delta_smem_floats<128>() * 4, a, s);
    return launch_kernel(delta_chunk_simt_kernel<IO, 64>, delta_smem_floats<64>() * 4, a, s);
}

template <typename IO, int DK>
cudaError_t launch_prefix(const PrefillArgs &a, cudaStream_t s) {
    auto kern = linear_prefix_simt_kernel<IO, DK>;
    constexpr size_t smem = PLayout<DK>::FLOATS * 4;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int cmax = a.max_chunks > 0 ? a.max_chunks : 1;
    dim3 grid((a.dv / kPJ) * cmax, a.H, a.N);
    kern<<<grid, kPNT, smem, s>>>(to_params(a), cmax);
    return cudaGetLastError();
}

template <typename IO>
cudaError_t linear_dispatch(const PrefillArgs &a, cudaStream_t s) {
    // every sequence known to span at most kPMax chunks: the chunk-parallel form
    static_assert(kPMax == kLinearParallelMaxChunks, "one limit for the dispatch");
    if (a.max_chunks >= 0 && a.max_chunks <= kPMax)
        return a.dk == 128 ? launch_prefix<IO, 128>(a, s) : launch_prefix<IO, 64>(a, s);
    if (a.dk == 128)
        return launch_kernel(linear_chunk_simt_kernel<IO, 128>, LinLayout<128>::FLOATS * 4, a, s, kLJ);
    return launch_kernel(linear_chunk_simt_kernel<IO, 64>, LinLayout<64>::FLOATS * 4, a, s, kLJ);
}

}  // namespace

cudaError_t launch_delta_simt(const PrefillArgs &a, cudaStream_t s) {
    return a.bf16 ? delta_dispatch<__nv_bfloat16>(a, s) : delta_dispatch<float>(a, s);
}

cudaError_t launch_linear_simt(const PrefillArgs &a, cudaStream_t s) {
    return a.bf16 ? linear_dispatch<__nv_bfloat16>(a, s) : linear_dispatch<float>(a, s);
}

}  // namespace la
