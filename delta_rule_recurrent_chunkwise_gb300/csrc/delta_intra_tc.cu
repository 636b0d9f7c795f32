// delta_intra_tc.cu -- intra-chunk half of the tensor-core (gated) delta-rule
// prefill: everything that depends on one chunk alone, for all chunks of all
// sequences and heads at once.  bf16 I/O, fp32 accumulators, dk = dv = D in
// {64, 128}, chunk C = 64.
//
// Algorithm ("From GPT-2 to Kimi K3, explained", section DeltaNet
// (Parallelizing Linear Transformers with Delta Rule), eq. 8-10, with the
// cumulative per-key-channel decay of sections Gated DeltaNet and
// KDA / Kimi Linear).  Per chunk, with b = cumulative log decay inside the
// chunk (per key channel):
//   A[r][i]  = beta_r sum_c k_rc k_ic e^{b_rc - b_ic}   (i < r)     UT matrix
//   Aq[r][i] =        sum_c q_rc k_ic e^{b_rc - b_ic}   (i <= r)    scores
//   T  = (I + A)^{-1}                                   blocked forward substitution
//   W  = T (beta K e^{b}),  U = T (beta V)              (eq. 10)
// plus the operands the state recurrence needs: Q e^{b}, K e^{b_end - b} and
// e^{b_end}.  None of it depends on the state, so every (chunk, head) is an
// independent task; the inter-chunk kernel then carries the state through
// the chunks with u = U - W S, O = (Q e^b) S + Aq u, S <- e^{b_end} S + K~^T u.
// The additive rule (section Gated DeltaNet: the decayed state plus k v^T at
// full strength, no delta) is the same pipeline with A = 0 (so T = I),
// beta = 1 and W = 0: then U = V and u = V.
//
// Decay factors.  Only products of alpha are formed, never exponentials of
// cumulative sums: alpha = 1 / (1 + e^g) and 1/alpha = 1 + e^g cost one
// exponential and one reciprocal per element, and every other factor is a
// running product.  Aq and A need e^{b_r - b_i} for i <= r, which does not
// factor into a row term times a column term over a whole chunk without
// overflow.  The chunk is cut into four 16-token blocks; for rows r of block
// R the reference point is the token just before R:
//   row factor  P_r = prod_{t=start(R)}^{r} alpha_t               (<= 1)
//   col factor  prod_{t=i+1}^{start(R)-1} alpha_t   for i < start(R)   (<= 1)
//               1 / prod_{t=start(R)}^{i} alpha_t   for i in R         (>= 1)
// so one tensor-core product per block R (the columns of K scaled for R)
// gives the rows of A and Aq that belong to R.  Keys of earlier blocks are
// decayed to the end of their block by suffix products (<= 1), so only a
// key's own block uses the reciprocal 1/P; that stays exact while the
// channel's 16-token decay stays above 1e-36.  Channels below it ("strong",
// fast forgetting) contribute zero to the tensor-core product and get their
// own-block scores from an exact CUDA-core pass (running products of alpha,
// taken only for tasks that have such a channel).
//
// Mapping: a persistent grid walks the (chunk slot, head) tasks; the next
// task's raw q, k, v, gate tiles arrive by TMA while the current one
// computes.  Every phase is short and bound by latency and by its CTA
// barriers (several phases keep only a few warps busy), so where shared
// memory and tensor memory allow (d = 64 without gate) the CTA is 256
// threads and two of them share an SM, each filling the other's idle
// phases; otherwise one CTA of 512 threads per SM.  Products on tcgen05 (bf16 x bf16
// -> fp32 in TMEM): [Q;K]-hat x K_R^T (one N = 160 product when gated) and
// T x [beta K e^b | beta V] (one N = 2D product).  The triangular solve runs
// in fp32 on CUDA cores: the four diagonal 16x16 blocks by column-wise
// forward substitution, the off-diagonal blocks by warp-level TF32 products.
// The finished operands leave as one record per task by bulk copies.

#include <cuda.h>

#include "common.cuh"
#include "delta_tc.h"
#include "tc_tile.cuh"

namespace la {
namespace {

using namespace tc;
using namespace tile;

constexpr int LDT = 68;          // fp32 row stride of the A and T scratch (16-byte rows)
constexpr uint32_t TC_A = 0, TC_W = 0;  // TMEM columns; U follows W

// ------------------------------------------------------------- smem layout
template <int D, bool GATED>
struct Layout {
    static constexpr uint32_t tile64 = C * D * 2;               // [64][D]
    // Raw q and k, interleaved per 64-column block so that [q; k] is one
    // 128-row RS tile: column block cb holds q rows 0..63, then k rows
    // 0..63 (rows 64..127), 16 KB per block.  That tile is the A operand and
    // its k half the B operand of the first product when it runs on the raw
    // inputs.
    static constexpr uint32_t RAW_QK = 0;
    static constexpr uint32_t RAW_V = RAW_QK + 2 * tile64;
    static constexpr uint32_t RAW_G = RAW_V + tile64;
    static constexpr uint32_t X = RAW_G + (GATED ? tile64 : 0);
    // X, prologue: the block-product operand [Q^; K^] (128 rows; gated or
    // silu only) and, gated, the packed K_R tile (160 rows)
    static constexpr uint32_t QKH = X;
    static constexpr uint32_t KR = X + 128 * D * 2;
    // X during and after the solve
    static constexpr uint32_t SA = X;                   // A, fp32 [64][LDT]
    static constexpr uint32_t T16 = X;                  // [T; T], bf16 [128][64] (A dead by then)
    static constexpr uint32_t ST = SA + 64 * LDT * 4;   // T, fp32 [64][LDT]
    static constexpr uint32_t AQK = ST + 64 * LDT * 4;  // Aq, bf16 [64][64]
    static constexpr uint32_t SX = AQK + 8192;          // solve temps, fp32 (7 KB)
    static constexpr uint32_t SX_BYTES = 7 * 1024;
    static_assert(128 * 128 <= 64 * LDT * 4, "[T; T] fits in the dead A scratch");
    static constexpr uint32_t X_END_A = GATED ? KR + 160 * D * 2 : KR;
    static constexpr uint32_t X_END_C = SX + SX_BYTES;
    static constexpr uint32_t X_END = X_END_A > X_END_C ? X_END_A : X_END_C;
    // The record's first four tiles, contiguous as in the record:
    //   WQ = [beta K e^b, later -W (rows 0..63) ; Q e^b (rows 64..127)]
    //   UK = [beta V, later U      (rows 0..63) ; K e^{b_end - b} (rows 64..127)]
    // (ungated: e^b = 1).  Rows 0..63 of WQ and UK, 16 KB apart per
    // 64-column block, are also the B operand [beta K e^b | beta V].
    static constexpr uint32_t WQ = (X_END + 1023) & ~1023u;
    static constexpr uint32_t UK = WQ + 2 * tile64;
    static constexpr uint32_t SMALL = UK + 2 * tile64;
    static constexpr uint32_t BETA = SMALL;                    // fp32 [64]
    static constexpr uint32_t KN = BETA + 256;                 // fp32 [64]
    static constexpr uint32_t QN = KN + 256;                   // fp32 [64]
    static constexpr uint32_t EB = QN + 256;                   // fp32 [4][D] block decay (gated)
    static constexpr uint32_t GEND = EB + (GATED ? 16 * D : 0);  // fp32 [D] chunk decay
    // scalar gate (one decay per token): log alpha, then cumulative b, and
    // the row factors e^b, e^{b_end - b}
    static constexpr uint32_t SLB = GEND + 4 * D;              // fp32 [64]
    static constexpr uint32_t SEB = SLB + 256;                 // fp32 [64]
    static constexpr uint32_t SEK = SEB + 256;                 // fp32 [64]
    // gated: exact own-block scores of fast-decaying channels (Aq part, then
    // K K^T part, [4][16][16] each) and the flag that some channel needs them
    static constexpr uint32_t DIAG = SEK + 256;
    static constexpr uint32_t SFLAG = DIAG + (GATED ? 2u * 4u * 256u * 4u : 0u);
    // cu_seqlens copied once per CTA (batches of up to CU_MAX - 1 sequences),
    // so that the binary search naming a slot's sequence reads shared memory
    static constexpr int CU_MAX = 256;
    static constexpr uint32_t CU = SFLAG + 16;                 // int32 [CU_MAX]
    static constexpr uint32_t INFO = CU + 4 * CU_MAX;          // int4: next task
    static constexpr uint32_t NIDX = INFO + 16;                // int64: its index
    static constexpr uint32_t FST = NIDX + 16;                 // int64 [4]: the fetcher's task state
    static constexpr uint32_t BAR_TMA = FST + 32;              // mbarrier: raw tiles
    static constexpr uint32_t BAR_MMA = BAR_TMA + 8;           // mbarrier: tensor-core products
    static constexpr uint32_t TASK_BYTES = (BAR_MMA + 8 + 1023) & ~1023u;
    static_assert(UK - WQ == Record<D>::UK, "record image");
    // threads per CTA, CTAs per SM, TMEM columns (block products, then W | U)
    static constexpr bool SMALL_CTA = D == 64 && !GATED;
    static constexpr int NT = SMALL_CTA ? 256 : 512;
    static constexpr int CTAS_PER_SM = SMALL_CTA ? 2 : 1;
    static constexpr uint32_t TMEM_COLS = SMALL_CTA ? 128 : 256;
    // tasks side by side in one CTA (lockstep) and threads / warps per task
    static constexpr int P = 1;
    static constexpr int NTC = NT / P, NW = NTC / 32;
    static constexpr uint32_t TCOLS = TMEM_COLS / P;
    static constexpr uint32_t COMMON = P * TASK_BYTES;         // TMEM address slot
    static constexpr uint32_t TOTAL = COMMON + 64;
    static_assert(TOTAL + 1024 <= 227 * 1024, "shared memory budget");
    static_assert(CTAS_PER_SM * (TOTAL + 2048) <= 228 * 1024, "CTAs per SM");
    static_assert(TCOLS >= (GATED ? 160u : 64u) && TCOLS >= 2u * D, "TMEM columns per task");
};

// Offsets of raw q and k elements inside the interleaved RAW_QK tile.
__device__ __forceinline__ uint32_t qoff(int r, int c) { return rs_off(128, r, c); }
__device__ __forceinline__ uint32_t koff(int r, int c) { return rs_off(128, r + 64, c); }

__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

// ---- warp-level TF32 products for the small blocks of the triangular solve
// (m16n8k8: A 16x8 row-major, B 8x8 as [k][n], C 16x8; fp32 accumulate).
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const float *A, int lda, const float *B,
                                         int ldb, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const uint32_t a0 = to_tf32(A[g * lda + t]), a1 = to_tf32(A[(g + 8) * lda + t]);
    const uint32_t a2 = to_tf32(A[g * lda + t + 4]), a3 = to_tf32(A[(g + 8) * lda + t + 4]);
    const uint32_t b0 = to_tf32(B[t * ldb + g]), b1 = to_tf32(B[(t + 4) * ldb + g]);
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// C (16x8 tile at Cp, row stride ldc) = sign * d
__device__ __forceinline__ void store_c(float *Cp, int ldc, const float (&d)[4], float sign,
                                        int lane) {
    const int g = lane >> 2, t = lane & 3;
    Cp[g * ldc + 2 * t] = sign * d[0];
    Cp[g * ldc + 2 * t + 1] = sign * d[1];
    Cp[(g + 8) * ldc + 2 * t] = sign * d[2];
    Cp[(g + 8) * ldc + 2 * t + 1] = sign * d[3];
}

// Exact own-block scores for the fast-decaying ("strong") channels of a
// gated chunk: warp w takes block R = w / (D/32) and channels
// 32 (w % (D/32)) + lane; for i <= r in the block it adds
//   sum_c q^_rc k^_ic prod_{t=i+1}^{r} alpha_tc   (Aq part, sDiag[0..1023])
//   sum_c k^_rc k^_ic prod_{t=i+1}^{r} alpha_tc   (A part,  sDiag[1024..])
// over the warp's strong channels, the decay as a running product down each
// column (factors <= 1).  Out of line: it runs only for chunks that have such
// a channel and must not raise the register count of the common path.
template <int D>
__device__ __noinline__ void exact_own_block(const uint8_t *rawqk, const uint8_t *rawg,
                                             const float *sqn,
                                             const float *skn, const float *sE, float *sDiag,
                                             int lw, int lane, int len, bool silu) {
    constexpr int CG = D / 32;
    const int R = lw / CG, c = 32 * (lw % CG) + lane;
    const bool st = sE[R * D + c] < 1e-36f;
    if (!__any_sync(0xffffffffu, st)) return;
    float al[16], kh[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const int row = 16 * R + r;
        const uint32_t o = tile::rs_off(tile::C, row, c);
        const float g = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(rawg + o));
        float kv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(rawqk + koff(row, c)));
        if (silu) kv = kv / (1.0f + expf(-kv));
        al[r] = row < len ? decay_f(g) : 1.0f;
        kh[r] = kv * skn[row];
    }
    float *dq = sDiag + R * 256, *dk = sDiag + 1024 + R * 256;
#pragma unroll 1
    for (int i = 0; i < 16; ++i) {
        float pr = st ? kh[i] : 0.0f;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            if (r < i) continue;
            if (r > i) pr *= al[r];
            const int row = 16 * R + r;
            float qv = __bfloat162float(
                *reinterpret_cast<const __nv_bfloat16 *>(rawqk + qoff(row, c)));
            if (silu) qv = qv / (1.0f + expf(-qv));
            const float sq = warp_sum(qv * sqn[row] * pr);
            const float sk = warp_sum(kh[r] * pr);
            if (lane == 0) {
                atomicAdd(&dq[r * 16 + i], sq);
                atomicAdd(&dk[r * 16 + i], sk);
            }
        }
    }
}

struct IntraParams {
    const __nv_bfloat16 *beta_logits;
    const __nv_bfloat16 *gate_scalar;  // [ntok][H] with a scalar gate (ungated kernel), else null
    const int32_t *cu_seqlens;         // [N + 1]
    uint8_t *records;       // [slots][H] records
    uint8_t *t_out;         // null, or [slots][H] T tiles (8 KB) for the backward pass
    unsigned *err;
    int64_t n_tasks;        // slots * H
    int N, H, ntok;
    unsigned flags;
};


// Barriers of the threads that run one task loop: the whole CTA, or one of
// the CTA's 256-thread halves (named barrier 1 + half), when a CTA runs two
// independent task loops.  Every barrier of a loop is reached by all of its
// threads the same number of times.
struct CtaBarrier {
    __device__ __forceinline__ int thread() const { return threadIdx.x; }
    __device__ __forceinline__ void sync() const { __syncthreads(); }
    __device__ __forceinline__ bool sync_or(bool pred) const { return __syncthreads_or(pred) != 0; }
};

struct HalfBarrier {
    int id;  // 1 or 2
    __device__ __forceinline__ int thread() const { return threadIdx.x & 255; }
    __device__ __forceinline__ void sync() const {
        asm volatile("bar.sync %0, 256;" ::"r"(id) : "memory");
    }
    __device__ __forceinline__ bool sync_or(bool pred) const {
        uint32_t r;
        asm volatile(
            "{\n\t.reg .pred ip, op;\n\t"
            "setp.ne.u32 ip, %1, 0;\n\t"
            "bar.red.or.pred op, %2, 256, ip;\n\t"
            "selp.u32 %0, 1, 0, op;\n\t}"
            : "=r"(r)
            : "r"((uint32_t)pred), "r"(id)
            : "memory");
        return r != 0;
    }
};

// Task source of the fused launch (intra-chunk work and the recurrence in
// one grid): tasks are taken from two global counters in chunk-major order,
// [0, cutoff) by every CTA and [cutoff, n_tasks) by the CTAs that do not
// turn to the recurrence afterwards, and every finished record is published
// through a flag.
struct FusedSched {
    unsigned *flags = nullptr;     // [slots * H]: record written and visible
    unsigned *counters = nullptr;  // [2] task counters (zeroed before the launch)
    int share_1024 = 0;            // cutoff = n_tasks * share_1024 / 1024
    int n_chain_ctas = 0;          // CTAs 0 .. n_chain_ctas - 1 run the recurrence afterwards
};

// Every (chunk slot, head) task this task loop is given.  FUSED selects the
// task source of the fused launch (chain_slot: this loop turns to the
// recurrence after the shared range); otherwise the CTA walks its fixed
// stride of the task list.  SCALAR: one decay per token and head (ungated
// layout plus per-row factors).  The loop owns the shared-memory region
// sbase (Layout::TOTAL bytes, 1024-byte aligned), the TMEM columns from
// tmem on and the barriers of `bar`; it returns after its last barrier, with
// every load and store it issued complete.
template <int D, bool GATED, bool SCALAR, bool FUSED, class Bar>
__device__ __forceinline__ void intra_run(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                                          const CUtensorMap &tm_v, const CUtensorMap &tm_g,
                                          const IntraParams &p, const FusedSched &fs,
                                          uint8_t *const sbase, const uint32_t tmem,
                                          const Bar bar, const bool chain_slot) {
    using L = Layout<D, GATED>;
    using Rec = Record<D>;
    constexpr int P = L::P, NTC = L::NTC, NW = L::NW;
    static_assert(!FUSED || P == 1, "the fused task source hands out one task at a time");
    const int tid = bar.thread(), warp = tid >> 5, lane = tid & 31;
    // this thread's task slot in the CTA, its warp and thread index within it
    const int kslot = warp / NW, lw = warp % NW, ltid = tid % NTC;
    const bool leader = ltid == 0;
    // issues the next task's raw-tile loads in the middle of a task (thread 0
    // issues the first tensor-core product right then; the loads' proxy fence
    // would hold it up)
    const bool fetcher = ltid == 32;
    uint8_t *sm = sbase + kslot * L::TASK_BYTES;
    uint8_t *rawqk = sm + L::RAW_QK, *rawv = sm + L::RAW_V, *rawg = sm + L::RAW_G;
    uint8_t *qkh = sm + L::QKH, *kr = sm + L::KR, *t16 = sm + L::T16, *aqk = sm + L::AQK;
    float *sA = reinterpret_cast<float *>(sm + L::SA);
    float *sT = reinterpret_cast<float *>(sm + L::ST);
    float *sX = reinterpret_cast<float *>(sm + L::SX);
    uint8_t *wq = sm + L::WQ, *uk = sm + L::UK;
    float *sbeta = reinterpret_cast<float *>(sm + L::BETA);
    float *skn = reinterpret_cast<float *>(sm + L::KN);
    float *sqn = reinterpret_cast<float *>(sm + L::QN);
    float *sE = reinterpret_cast<float *>(sm + L::EB);
    float *sgend = reinterpret_cast<float *>(sm + L::GEND);
    int4 *sinfo = reinterpret_cast<int4 *>(sm + L::INFO);
    float *sLb = reinterpret_cast<float *>(sm + L::SLB);
    float *sEb = reinterpret_cast<float *>(sm + L::SEB);
    float *sEk = reinterpret_cast<float *>(sm + L::SEK);
    float *sDiag = reinterpret_cast<float *>(sm + L::DIAG);
    int *sflag = reinterpret_cast<int *>(sm + L::SFLAG);
    static_assert(!(GATED && SCALAR), "a scalar gate uses the ungated layout");
    constexpr bool scalar = SCALAR;
    uint64_t *bar_tma = reinterpret_cast<uint64_t *>(sm + L::BAR_TMA);
    uint64_t *bar_mma = reinterpret_cast<uint64_t *>(sbase + L::BAR_MMA);

    const int qd = lw & 3, cp = lw >> 2;  // TMEM lane quarter, column part
    const int H = p.H;
    const bool silu = (p.flags & kSiluQK) != 0;
    // The first product [q; k] k^T runs on the raw tiles as soon as they land
    // (the norms, beta and scalar decays are applied as it is read out of
    // TMEM) unless silu or a per-channel gate changes the operands themselves.
    const bool raw_p1 = !GATED && !silu;
    const bool additive = (p.flags & kAdditive) != 0;  // A = 0, W = 0, beta = 1: u = V
    const bool l2k = (p.flags & kL2NormK) != 0, l2q = (p.flags & kL2NormQ) != 0;
    constexpr uint32_t tx_bytes = (GATED ? 4u : 3u) * L::tile64;

    if (leader) mbar_init(bar_tma, 1);
    if (tid == 0) {
        mbar_init(bar_mma, 1);
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        if (GATED) tma_prefetch_desc(&tm_g);
    }
    if (leader) fence_mbar_init();
    tc_fence_before();
    bar.sync();
    tc_fence_after();
    // this task's TMEM columns, and this warp's lane quarter of them
    const uint32_t tq = tmem + kslot * L::TCOLS + ((uint32_t)(32 * qd) << 16);
    // shared-memory region and TMEM columns of task slot kk (for the issuing thread)
    auto task_sm = [&](int kk) { return sbase + kk * L::TASK_BYTES; };
    auto task_tmem = [&](int kk) { return tmem + kk * L::TCOLS; };

    // Task -> {first token, length, head, slot}; length 0 marks a task with
    // no chunk (or an entry out of range).  Sequence n's chunk j has slot
    // f(n) + j, f(n) = cu[n] / 64 + n (f grows by at least nc(n) from one
    // sequence to the next, so slots never collide).
    // Order: with cu_seqlens in shared memory (up to CU_MAX - 1 sequences)
    // the tasks run chunk-major, t = j' N H + n H + h with j' = j in the
    // fused launch (its recurrence needs chunk 0 first) and j' = J - 1 - j
    // otherwise (the first chunks' records, which the recurrence kernel reads
    // first, are then the last written), J = the longest sequence's chunk
    // count.  Otherwise
    // t = slot * H + head, and a slot's sequence is the last n with
    // f(n) <= slot, found by binary search over cu_seqlens.
    const int *scu = reinterpret_cast<const int *>(sbase + L::CU);
    const bool cu_in_smem = p.N < L::CU_MAX - 1;  // entry CU_MAX - 1 holds J
    auto cu_at = [&](int n) { return cu_in_smem ? scu[n] : p.cu_seqlens[n]; };
    int J = 0;  // chunks of the longest sequence (chunk-major order)
    auto task_at = [&](int64_t t, int64_t n_tasks) -> int4 {
        const int4 none = make_int4(0, 0, 0, 0);
        if (t < 0 || t >= n_tasks || p.N < 1) return none;
        int n, h, j;
        if (cu_in_smem) {
            const int64_t NH = (int64_t)p.N * H;
            // fused: forward, the recurrence running alongside needs chunk 0 first
            j = FUSED ? (int)(t / NH) : J - 1 - (int)(t / NH);
            const int rem = (int)(t % NH);
            n = rem / H;
            h = rem - n * H;
        } else {
            const int64_t slot = t / H;
            h = (int)(t - slot * H);
            auto f = [&](int m) { return (int64_t)(cu_at(m) / C) + m; };
            if (f(0) > slot) return none;
            int lo = 0, hi = p.N - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (f(mid) <= slot) lo = mid;
                else hi = mid - 1;
            }
            n = lo;
            j = (int)(slot - f(lo));
        }
        const int a = cu_at(n), e = cu_at(n + 1);
        if (a < 0 || e < a || e > p.ntok) return none;  // reported by the inter-chunk kernel
        if (j < 0 || j >= (e - a + C - 1) / C) return none;  // past the sequence's chunks
        const int x = a + j * C;
        const int len = e - x < C ? e - x : C;
        const int64_t slot = (int64_t)(a / C) + n + j;
        if (slot >= p.n_tasks / H) return none;
        return make_int4(x, len, h, (int)slot);
    };
    const uint64_t pol = l2_evict_first();  // inputs and records pass through L2 once
    auto issue_tma = [&](int t0, int hh) {
        fence_proxy_async();
        mbar_arrive_expect_tx(bar_tma, tx_bytes);
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb) {
            tma_load_3d_hint(rawqk + cb * 16384, &tm_q, bar_tma, cb * 64, hh, t0, pol);
            tma_load_3d_hint(rawqk + cb * 16384 + 8192, &tm_k, bar_tma, cb * 64, hh, t0, pol);
            tma_load_3d_hint(rawv + cb * 8192, &tm_v, bar_tma, cb * 64, hh, t0, pol);
            if (GATED) tma_load_3d_hint(rawg + cb * 8192, &tm_g, bar_tma, cb * 64, hh, t0, pol);
        }
    };
    auto load_beta = [&](const int4 &ti) -> float {
        return (!additive && ltid < C && ltid < ti.y)
                   ? __bfloat162float(p.beta_logits[(int64_t)(ti.x + ltid) * H + ti.z])
                   : 0.0f;
    };
    auto load_gate = [&](const int4 &ti) -> float {  // scalar gate logit of row ltid
        return (scalar && ltid < C && ltid < ti.y)
                   ? __bfloat162float(p.gate_scalar[(int64_t)(ti.x + ltid) * H + ti.z])
                   : 0.0f;
    };

    // Each task's leader thread waits for its raw tiles and issues its
    // products; the fetcher issues the next task's raw-tile loads, stores the
    // record and hands out the task indices: the current one (g) and, held
    // in its own shared-memory slots, the next two (the next one's tiles are
    // loaded during the current task).  Without FUSED the
    // CTA takes task groups g = blockIdx.x, + gridDim.x, ...; task slot kslot
    // of group g is task g * P + kslot.
    // cu_seqlens and the inputs may come from the previous launch; the
    // inter-chunk kernel may be scheduled as SMs free up (it waits for this
    // grid to finish)
    grid_wait_prerequisites();
    grid_launch_dependents();
    int64_t n_tasks = p.n_tasks;
    if (cu_in_smem) {
        int *cu_w = reinterpret_cast<int *>(sbase + L::CU);
        for (int n = tid; n <= p.N; n += L::NT) cu_w[n] = p.cu_seqlens[n];
        if (tid == 0) cu_w[L::CU_MAX - 1] = 0;
        bar.sync();
        int jmax = 0;
        for (int n = tid; n < p.N; n += L::NT) {
            const int a = cu_w[n], e = cu_w[n + 1];
            if (a >= 0 && e >= a) jmax = max(jmax, (e - a + C - 1) / C);
        }
        jmax = __reduce_max_sync(0xffffffffu, jmax);
        if (lane == 0 && jmax > 0) atomicMax(cu_w + L::CU_MAX - 1, jmax);
        bar.sync();
        J = cu_w[L::CU_MAX - 1];
        n_tasks = (int64_t)J * p.N * H;
    }
    const int64_t n_groups = (n_tasks + P - 1) / P;
    const bool chain_cta = FUSED && chain_slot;
    const int64_t cutoff = FUSED ? n_tasks * fs.share_1024 / 1024 : 0;
    // The fetcher's own state, kept in shared memory rather than in
    // registers every thread would carry: the next two task indices, the
    // next group of the static order (or, fused, -1 once the shared range is
    // used up) and the record waiting to be published.
    int64_t *fst = reinterpret_cast<int64_t *>(sm + L::FST);
    enum { F_NXT = 0, F_AFT = 1, F_STATIC = 2, F_PUB = 3 };
    auto next_group = [&]() -> int64_t {
        if constexpr (FUSED) {
            if (fst[F_STATIC] >= 0) {
                const int64_t t = atomicAdd(fs.counters, 1u);
                if (t < cutoff) return t;
                fst[F_STATIC] = -1;
            }
            if (chain_cta) return -1;
            const int64_t t = cutoff + atomicAdd(fs.counters + 1, 1u);
            return t < n_tasks ? t : -1;
        } else {
            const int64_t gg = fst[F_STATIC];
            fst[F_STATIC] = gg + gridDim.x;
            return gg < n_groups ? gg : -1;
        }
    };
    int64_t *snidx = reinterpret_cast<int64_t *>(sm + L::NIDX);
    if (fetcher) {
        fst[F_STATIC] = FUSED ? 0 : (int64_t)blockIdx.x;
        fst[F_PUB] = -1;
        const int64_t g0 = next_group();
        fst[F_NXT] = g0 >= 0 ? next_group() : -1;
        fst[F_AFT] = fst[F_NXT] >= 0 ? next_group() : -1;
        *snidx = g0;
    }
    bar.sync();
    int64_t g = *snidx;                        // -1: no task left
    int4 cur = task_at(g * P + kslot, n_tasks);
    // fetcher: the next task becomes the one whose tiles load now (its info
    // and index to shared memory)
    auto advance = [&]() -> int4 {
        const int64_t ni = fst[F_NXT];
        const int4 nxt = task_at(ni * P + kslot, n_tasks);
        *sinfo = nxt;
        *snidx = ni;
        const int64_t ai = fst[F_AFT];
        fst[F_NXT] = ai;
        fst[F_AFT] = ai >= 0 ? next_group() : -1;
        return nxt;
    };
    // fetcher (fused): the record stored last is complete; publish it
    auto publish = [&]() {
        const int64_t pub = fst[F_PUB];
        if (pub >= 0) {
            fence_proxy_async_global();
            st_release_gpu(fs.flags + pub, 1u);
            fst[F_PUB] = -1;
        }
    };
    bool tma_pending = false;  // meaningful in the leader, who waits for the loads
    if (leader && cur.y > 0) {
        issue_tma(cur.x, cur.z);
        tma_pending = true;
    }
    float beta_cur = load_beta(cur);  // threads 0..63 of the task
    float gate_cur = load_gate(cur);
    uint32_t tma_par = 0, mma_par = 0;
    bool failed = false;

    // One thread waits on an mbarrier; the CTA barrier that follows every
    // wait (a __syncthreads_or carrying the outcome) releases the others,
    // who then order their tensor-memory accesses after it.
    auto mma_wait = [&]() -> bool {
        bool ok = true;
        if (tid == 0) ok = mbar_wait(bar_mma, mma_par, p.err, 2);
        mma_par ^= 1;
        return ok;
    };
    auto phase_sync = [&]() {
        fence_proxy_async();
        tc_fence_before();
        bar.sync();
        tc_fence_after();
    };
    // B: the block products, one thread.  Gated: the packed K_R tile is one
    // 160-row operand, so all four block products form one N = 160 product
    // (block R at column 8R(R+1)); ungated: one product [q; k] x k^T
    // (N = 64) on the raw tiles, or on [q^; k^] (QKH) with silu.  Issue loops
    // are kept rolled and short: this code runs on one thread, so every
    // instruction of it is fetched without help from other warps.
    auto issue_p1 = [&]() {
        const uint32_t id = GATED ? idesc_bf16(128, 160, false, false) : idesc_bf16(128, 64, false, false);
        const int bRows = GATED ? 160 : 128;
#pragma unroll 1
        for (int kk = 0; kk < P; ++kk) {
            uint8_t *tsm = task_sm(kk);
            const uint8_t *qk = raw_p1 ? tsm + L::RAW_QK : tsm + L::QKH;
            const uint64_t a0 = kdesc(qk, 128, 0, 0);
            const uint64_t b0 = GATED ? kdesc(tsm + L::KR, 160, 0, 0) : kdesc(qk, 128, 64, 0);
#pragma unroll 1
            for (int kb = 0; kb < D / 64; ++kb) {
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4)
                    mma_bf16(task_tmem(kk) + TC_A, dstep(a0, kstep_units(128, 4 * kb + s4)),
                             dstep(b0, kstep_units(bRows, 4 * kb + s4)), id, (kb | s4) != 0);
            }
        }
        mma_commit(bar_mma);
    };

    while (g >= 0) {
        // one task per CTA: cur is the same in every thread
        const bool any_task = P == 1 ? cur.y > 0 : bar.sync_or(cur.y > 0);
        if (!any_task) {
            // empty slots only: nothing to compute, start the next tasks' loads
            if (fetcher) {
                if constexpr (FUSED) {
                    bulk_wait_all();
                    publish();
                }
                advance();
            }
            bar.sync();
            if (leader && sinfo->y > 0) {
                issue_tma(sinfo->x, sinfo->z);
                tma_pending = true;
            }
            cur = *sinfo;
            g = *snidx;
            beta_cur = load_beta(cur);
            gate_cur = load_gate(cur);
            bar.sync();
            continue;
        }
        // A slot with no task (len 0) runs along on whatever its buffers
        // hold; nothing of it is stored.
        const int len = cur.y, h = cur.z;
        // ---------------------------------------------- raw tiles of this chunk
        {
            bool ok = true;
            if (leader && len > 0) {
                ok = mbar_wait(bar_tma, tma_par, p.err, 1);
                tma_par ^= 1;
                tma_pending = false;
                // the first product needs nothing but the raw tiles: it runs
                // while the CUDA cores work through the prologue below
                if (ok && raw_p1) issue_p1();
            }
            tc_fence_before();
            if (bar.sync_or(!ok)) { failed = true; break; }
            tc_fence_after();
        }
        // ---------------------------------------------- A0: beta, row norms
        if (GATED && ltid == 0) *sflag = 0;
        if (ltid < C)
            sbeta[ltid] = ltid >= len ? 0.0f : additive ? 1.0f : __fdividef(1.0f, 1.0f + __expf(-beta_cur));
        if (scalar && ltid < C) sLb[ltid] = ltid < len ? log_decay_f(gate_cur) : 0.0f;  // log alpha
        {
            // TPR threads per row, D/TPR channels each, 16-byte loads
            constexpr int TPR = NTC / C;
            const int r = ltid / TPR, part = ltid % TPR;
            float ssk = 0.0f, ssq = 0.0f;
#pragma unroll
            for (int c = part * (D / TPR); c < (part + 1) * (D / TPR); c += 8) {
                float kv[8], qv[8];
                unpack8(*reinterpret_cast<const uint4 *>(rawqk + koff(r, c)), kv);
                unpack8(*reinterpret_cast<const uint4 *>(rawqk + qoff(r, c)), qv);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (silu) { kv[i] = silu_fast(kv[i]); qv[i] = silu_fast(qv[i]); }
                    ssk += kv[i] * kv[i];
                    ssq += qv[i] * qv[i];
                }
            }
#pragma unroll
            for (int o = 1; o < TPR; o <<= 1) {
                ssk += __shfl_xor_sync(0xffffffffu, ssk, o);
                ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
            }
            if (part == 0) {
                const bool valid = r < len;
                skn[r] = valid ? (l2k ? rsqrtf(fmaxf(ssk, 1e-24f)) : 1.0f) : 0.0f;
                sqn[r] = valid ? (l2q ? rsqrtf(fmaxf(ssq, 1e-24f)) : 1.0f) : 0.0f;
            }
        }
        if (fetcher) bulk_wait_read();  // previous record's sources are rewritten below
        bar.sync();
        // ---------------------------------------------- A1: operand tiles
        if (!GATED) {
            if (scalar) {
                // b_r = sum_{t<=r} log alpha_t inside the chunk (warp 0, two rows
                // per lane); row factors e^{b_r} and e^{b_end - b_r} (both <= 1)
                if (warp == 0) {
                    const float l0 = sLb[2 * lane], l1 = sLb[2 * lane + 1];
                    float x = l0 + l1;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float y = __shfl_up_sync(0xffffffffu, x, o);
                        if (lane >= o) x += y;
                    }
                    const float b1 = x, b0 = x - l1;
                    const float bend = __shfl_sync(0xffffffffu, x, 31);  // b of row 63 = b_end
                    sLb[2 * lane] = b0;
                    sLb[2 * lane + 1] = b1;
                    sEb[2 * lane] = __expf(b0);
                    sEb[2 * lane + 1] = __expf(b1);
                    sEk[2 * lane] = __expf(bend - b0);
                    sEk[2 * lane + 1] = __expf(bend - b1);
                }
                bar.sync();
                if (ltid < D) sgend[ltid] = sEb[63];  // e^{b_end}, the same for every channel
            }
            // beta k^, q^ into WQ; beta v, k^ into UK; with silu also [q^; k^]
            // into QKH (the first product's operand; without silu that
            // product runs on the raw tiles): 16-byte units
            for (int u = ltid; u < C * D / 8; u += NTC) {
                const uint32_t off = (uint32_t)u * 16u;                 // offset in a [64][D] tile
                const uint32_t cb = off >> 13, in = off & 8191u;         // column block, offset in it
                const int r = (int)(in >> 7);
                const uint32_t po = cb * (128u * 128u) + in;            // same row, 128-row tile
                float kv[8], qv[8], vv[8];
                unpack8(*reinterpret_cast<const uint4 *>(rawqk + po + 64u * 128u), kv);
                unpack8(*reinterpret_cast<const uint4 *>(rawqk + po), qv);
                unpack8(*reinterpret_cast<const uint4 *>(rawv + off), vv);
                const float kn = skn[r], qn = sqn[r], be = sbeta[r];
                float bk[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (silu) { kv[i] = silu_fast(kv[i]); qv[i] = silu_fast(qv[i]); }
                    kv[i] *= kn;
                    qv[i] *= qn;
                    bk[i] = be * kv[i];
                    vv[i] *= be;
                }
                const uint4 qh = pack8(qv), kh = pack8(kv);
                if (!raw_p1) {
                    *reinterpret_cast<uint4 *>(qkh + po) = qh;
                    *reinterpret_cast<uint4 *>(qkh + po + 64u * 128u) = kh;
                }
                *reinterpret_cast<uint4 *>(uk + po) = pack8(vv);
                if (scalar) {
                    // Q e^b, beta K e^b, K e^{b_end - b}: one factor per row
                    const float eb = sEb[r], ek = sEk[r];
#pragma unroll
                    for (int i = 0; i < 8; ++i) { bk[i] *= eb; qv[i] *= eb; kv[i] *= ek; }
                    *reinterpret_cast<uint4 *>(wq + po) = pack8(bk);
                    *reinterpret_cast<uint4 *>(wq + po + 64u * 128u) = pack8(qv);
                    *reinterpret_cast<uint4 *>(uk + po + 64u * 128u) = pack8(kv);
                } else {
                    *reinterpret_cast<uint4 *>(wq + po) = pack8(bk);
                    *reinterpret_cast<uint4 *>(wq + po + 64u * 128u) = qh;
                    *reinterpret_cast<uint4 *>(uk + po + 64u * 128u) = kh;
                }
            }
            if (!scalar && ltid < D) sgend[ltid] = 1.0f;
        } else {
            // One thread per (2 key channels, 8 rows of a 16-token block R); the
            // two 8-row halves of a block sit in lanes l and l^16 of one warp.
            // alpha = 1/(1+e^g); P = prefix product of alpha inside the block,
            // Sf = suffix product prod_{t>r} alpha_t inside the block.  Every
            // operand is (q or k) x (P, Sf or, for a key's own block, 1/P) x a
            // per-(block, channel) product of block totals.
            static_assert(NW * 8 >= D, "one thread per (channel pair, 8 rows)");
            const bool act = lw < D / 8;
            const int R = (lw * 32 / D) & 3, grp = lw % (D / 32);
            const int hf2 = lane >> 4, c0 = 32 * grp + 2 * (lane & 15);
            const int r0 = 16 * R + 8 * hf2;
            // Rows r0 and r0 + 8 share a swizzle phase, so at step rho the
            // second-half lanes work on row r0 + (rho ^ 4): the two halves of
            // the warp then hit disjoint banks.
            const int pr = 4 * hf2;
            // Addressing: the channel pair is fixed per thread and r0 is a
            // multiple of 8, so row r0 + rho has swizzle phase rho.
            const uint32_t cb = (uint32_t)c0 >> 6, ch = ((uint32_t)c0 >> 3) & 7u;
            const uint32_t cboff64 = cb * 64u * 128u, cboff128 = cb * 128u * 128u,
                           cboff160 = cb * 160u * 128u;
            // byte offset of the channel pair in row phase j (the 16-byte chunk
            // index is XOR-ed with the row's swizzle phase)
            auto swz = [&](int j) { return ((ch ^ (uint32_t)j) << 4) + ((uint32_t)c0 & 7u) * 2u; };
            float P[8][2], Sf[8][2];
#pragma unroll
            for (int rho = 0; rho < 8; ++rho) {
                P[rho][0] = P[rho][1] = 1.0f;
                Sf[rho][0] = Sf[rho][1] = 1.0f;
            }
            if (act) {
                float p0 = 1.0f, p1 = 1.0f, a[8][2];
#pragma unroll
                for (int rho = 0; rho < 8; ++rho) {
                    // the scan runs in natural row order (a prefix product);
                    // only the store pass below uses the permuted order
                    const int r = r0 + rho;
                    const __nv_bfloat162 g2 = *reinterpret_cast<const __nv_bfloat162 *>(rawg + cboff64 + r * 128 + swz(rho));
                    const float2 g = __bfloat1622float2(g2);
                    const float e0 = __expf(fminf(g.x, 80.0f)), e1 = __expf(fminf(g.y, 80.0f));
                    a[rho][0] = a[rho][1] = 1.0f;
                    if (r < len) {
                        a[rho][0] = __fdividef(1.0f, 1.0f + e0);
                        a[rho][1] = __fdividef(1.0f, 1.0f + e1);
                        p0 *= a[rho][0];
                        p1 *= a[rho][1];
                    }
                    P[rho][0] = p0; P[rho][1] = p1;
                }
                // within-half suffix products prod_{t > r} alpha_t (<= 1)
#pragma unroll
                for (int rho = 6; rho >= 0; --rho) {
                    Sf[rho][0] = Sf[rho + 1][0] * a[rho + 1][0];
                    Sf[rho][1] = Sf[rho + 1][1] * a[rho + 1][1];
                }
            }
            // carry the first half's totals into the second half
            {
                const float t0 = __shfl_sync(0xffffffffu, P[7][0], lane ^ 16);
                const float t1 = __shfl_sync(0xffffffffu, P[7][1], lane ^ 16);
                if (hf2) {
#pragma unroll
                    for (int rho = 0; rho < 8; ++rho) { P[rho][0] *= t0; P[rho][1] *= t1; }
                } else {
                    // first half: the suffix runs on through the second half
#pragma unroll
                    for (int rho = 0; rho < 8; ++rho) { Sf[rho][0] *= t0; Sf[rho][1] *= t1; }
                }
            }
            if (act && hf2) {
                sE[R * D + c0] = P[7][0];
                sE[R * D + c0 + 1] = P[7][1];
            }
            bar.sync();
            if (act) {
                // Gb: decay of the blocks before R; Ea: of the blocks after R;
                // mt[t]: of blocks R+1 .. R+t (keys of R used by block R+1+t).
                // A channel whose block total falls below 1e-36 ("strong")
                // gets its own-block scores from the exact path instead.
                float Gb[2], Ea[2], mt[3][2], invE[2];
                bool strong[2];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int c = c0 + j;
                    const float E0 = sE[c], E1 = sE[D + c], E2 = sE[2 * D + c], E3 = sE[3 * D + c];
                    Gb[j] = R == 0 ? 1.0f : R == 1 ? E0 : R == 2 ? E0 * E1 : E0 * E1 * E2;
                    Ea[j] = R == 0 ? E1 * E2 * E3 : R == 1 ? E2 * E3 : R == 2 ? E3 : 1.0f;
                    float m = 1.0f;
#pragma unroll
                    for (int t = 0; t < 3; ++t) {
                        mt[t][j] = m;
                        const int Rt = R + 1 + t;
                        m *= Rt == 1 ? E1 : Rt == 2 ? E2 : Rt == 3 ? E3 : 1.0f;
                    }
                    const float ER = sE[R * D + c];
                    strong[j] = ER < 1e-36f;
                    // 1/P_r = Sf_r / E_R: one reciprocal per channel
                    invE[j] = strong[j] ? 0.0f : __fdividef(1.0f, ER);
                    if (R == 0 && hf2 == 0) sgend[c] = E0 * E1 * E2 * E3;
                }
                if (strong[0] || strong[1]) atomicOr(sflag, 1);
                // 32-bit shared-memory addresses keep the six destinations in
                // six registers (generic pointers would take twelve)
                auto st2 = [](uint32_t a, float x, float y) {
                    const __nv_bfloat162 v = __floats2bfloat162_rn(x, y);
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(a), "r"(*reinterpret_cast<const uint32_t *>(&v))
                                 : "memory");
                };
                uint8_t *const pq_raw = rawqk + cboff128, *const pk_raw = rawqk + cboff128 + 64 * 128;
                const uint32_t p_qh = smem_u32(qkh) + cboff128, p_kh = smem_u32(qkh) + cboff128 + 64 * 128;
                const uint32_t p_qg = smem_u32(wq) + cboff128 + 64 * 128, p_kt = smem_u32(uk) + cboff128 + 64 * 128;
                const uint32_t p_bk = smem_u32(wq) + cboff128, p_kr = smem_u32(kr) + cboff160;
                // second-half lanes: swap register rows rho <-> rho ^ 4 so the
                // store pass can index P[rho] with a compile-time rho
                if (pr) {
#pragma unroll
                    for (int rho = 0; rho < 4; ++rho) {
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            float t = P[rho][j]; P[rho][j] = P[rho + 4][j]; P[rho + 4][j] = t;
                            t = Sf[rho][j]; Sf[rho][j] = Sf[rho + 4][j]; Sf[rho + 4][j] = t;
                        }
                    }
                }
#pragma unroll
                for (int rho = 0; rho < 8; ++rho) {
                    const int r = r0 + (rho ^ pr);
                    const uint32_t o = (uint32_t)r * 128u + (((ch ^ (uint32_t)(rho ^ pr)) << 4) + ((uint32_t)c0 & 7u) * 2u);
                    float2 qv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(pq_raw + o));
                    float2 kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(pk_raw + o));
                    if (silu) {
                        qv.x = silu_fast(qv.x); qv.y = silu_fast(qv.y);
                        kv.x = silu_fast(kv.x); kv.y = silu_fast(kv.y);
                    }
                    const float qn = sqn[r], kn = skn[r], be = sbeta[r];
                    qv.x *= qn; qv.y *= qn; kv.x *= kn; kv.y *= kn;
                    const float a0 = qv.x * P[rho][0], a1 = qv.y * P[rho][1];     // Q^
                    const float b0 = kv.x * P[rho][0], b1 = kv.y * P[rho][1];     // K^
                    // keys decayed to the end of their block (suffix, <= 1)
                    const float s0 = kv.x * Sf[rho][0], s1 = kv.y * Sf[rho][1];
                    // K_R own block: k / P = k Sf / E_R (E_R >= 1e-36 keeps it in
                    // range); zero for strong channels
                    const float k0 = s0 * invE[0], k1 = s1 * invE[1];
                    st2(p_qh + o, a0, a1);
                    st2(p_kh + o, b0, b1);
                    st2(p_qg + o, a0 * Gb[0], a1 * Gb[1]);                  // Q e^b
                    st2(p_kt + o, s0 * Ea[0], s1 * Ea[1]);                  // K e^{b_end-b}
                    st2(p_bk + o, be * b0 * Gb[0], be * b1 * Gb[1]);        // beta K e^b
                    st2(p_kr + (uint32_t)(8 * R * (R + 1)) * 128u + o, k0, k1);
#pragma unroll
                    for (int t = 0; t < 3; ++t) {
                        const int R2 = R + 1 + t;
                        if (R2 < 4)
                            st2(p_kr + (uint32_t)(8 * R2 * (R2 + 1)) * 128u + o, s0 * mt[t][0], s1 * mt[t][1]);
                    }
                }
            }
            // beta V
            for (int u = ltid; u < C * D / 8; u += NTC) {
                const uint32_t off = (uint32_t)u * 16u;
                const int r = (int)((off & 8191u) >> 7);
                float vv[8];
                unpack8(*reinterpret_cast<const uint4 *>(rawv + off), vv);
                const float be = sbeta[r];
#pragma unroll
                for (int i = 0; i < 8; ++i) vv[i] *= be;
                *reinterpret_cast<uint4 *>(uk + (off >> 13) * (128u * 128u) + (off & 8191u)) = pack8(vv);
            }
        }
        phase_sync();
        if constexpr (GATED) {
            // Exact own-block scores of the channels whose 16-token block decay
            // fell below 1e-36 (their 1/P factor would leave the fp32 range):
            // sum_c q^_rc k^_ic prod_{t=i+1}^{r} alpha_tc for i <= r in one
            // block, with the decay as a running product down each column
            // (every factor <= 1).  One warp per (block, 32 channels); the
            // tensor-core product holds zero for these channels.
            if (*sflag) {
                for (int u = ltid; u < 2048; u += NTC) sDiag[u] = 0.0f;
                bar.sync();
                if (lw < 4 * (D / 32))
                    exact_own_block<D>(rawqk, rawg, sqn, skn, sE, sDiag, lw, lane, len, silu);
                bar.sync();
            }
        }
        // Raw tiles consumed by the CUDA cores: fetch the next task's while
        // this one computes -- at once when the first product reads the
        // operand tiles, after it has completed when it reads the raw tiles.
        if (fetcher) {
            const int4 nxt = advance();
            if (!raw_p1 && nxt.y > 0) issue_tma(nxt.x, nxt.z);
        }
        // ---------------------------------------------- B: block products
        if (!raw_p1 && tid == 0) issue_p1();
        {
            const bool mma_failed = bar.sync_or(!mma_wait());
            if (mma_failed) {
                // the leader must wait for loads in flight before leaving
                tma_pending = !raw_p1 && sinfo->y > 0;
                failed = true;
                break;
            }
            if (raw_p1 && fetcher && sinfo->y > 0) issue_tma(sinfo->x, sinfo->z);
            tma_pending = sinfo->y > 0;
            // the previous task's record stores, issued a task phase ago
            if constexpr (FUSED) {
                if (fetcher) {
                    bulk_wait_all();
                    publish();
                }
            }
        }
        tc_fence_after();
        // the next task is known to every thread now: prefetch its beta
        const int4 nx = *sinfo;
        const int64_t nx_g = *snidx;
        const float beta_nx = load_beta(nx);
        const float gate_nx = load_gate(nx);
        // ---------------------------------------------- C1: Aq tile, A rows
        // TMEM lanes 0..63 hold rows of Aq, lanes 64..127 rows of A (before
        // beta).  Gated: block R's product sits at column 8R(R+1).  A warp
        // spans two blocks, so it reads both (TMEM addresses stay
        // warp-uniform) and each lane keeps its own.
        // Every warp: 64 / (NW / 4) columns (part cp) of its quarter -> Aq
        // tile / A rows (beta-scaled, strictly lower, fp32).
        {
            const bool is_q = qd < 2;
            const int rb0 = 32 * (is_q ? qd : qd - 2);
            const int r = rb0 + lane, R = r >> 4;
            const int Rw = rb0 >> 4;
            const bool diag_on = GATED && *sflag != 0;
            auto colof = [](int Rb) { return GATED ? 8 * Rb * (Rb + 1) : 0; };
#pragma unroll
            for (int sub = 0; sub < 16 / NW; ++sub) {
                const int col = 16 * (cp + sub * (NW / 4));
                float v[16];
                if (GATED) {
                    float w0[16], w1[16];
                    // parts beyond a block's product are masked below (col + i > r)
                    tmem_ld16(tq + TC_A + colof(Rw) + col, w0);
                    tmem_ld16(tq + TC_A + colof(Rw + 1) + col, w1);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = (R == Rw) ? w0[i] : w1[i];
                    if (diag_on && (col >> 4) == R) {
                        // own block of row r: add the exact part of strong channels
                        const float *dg = sDiag + (is_q ? 0 : 1024) + R * 256 + (r & 15) * 16;
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] += dg[i];
                    }
                } else {
                    tmem_ld16(tq + TC_A + col, v);
                    if (raw_p1) {
                        // raw operands: the row's and the key's norm factors
                        // (zero for rows past the end of the chunk)
                        const float rf = is_q ? sqn[r] : skn[r];
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] *= rf * skn[col + i];
                    }
                    if (scalar) {
                        // e^{b_r - b_i} for i <= r (exponent <= 0); later columns are masked
                        const float br = sLb[r];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            v[i] *= (col + i <= r) ? __expf(br - sLb[col + i]) : 0.0f;
                    }
                }
                if (is_q) {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (col + i > r) v[i] = 0.0f;
                    st_bf16x8(aqk, 64, r, col, v);
                    st_bf16x8(aqk, 64, r, col + 8, v + 8);
                } else {
                    const float be = additive ? 0.0f : sbeta[r];
                    float4 *dst = reinterpret_cast<float4 *>(sA + r * LDT + col);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float4 f;
                        f.x = (col + 4 * i + 0 < r) ? be * v[4 * i + 0] : 0.0f;
                        f.y = (col + 4 * i + 1 < r) ? be * v[4 * i + 1] : 0.0f;
                        f.z = (col + 4 * i + 2 < r) ? be * v[4 * i + 2] : 0.0f;
                        f.w = (col + 4 * i + 3 < r) ? be * v[4 * i + 3] : 0.0f;
                        dst[i] = f;
                    }
                }
            }
        }
        bar.sync();
        // ---------------------------------------------- C1b: diagonal blocks and T_10, T_32
        // Warp b (0, 1) takes blocks J = 2b and R = 2b + 1.
        // (a) T_JJ, T_RR = (I + A_XX)^{-1} by column-oriented forward
        //     substitution: lane (block, j) owns column j of its block and
        //     needs only its own earlier entries (A broadcast from shared
        //     memory), so there is no cross-lane exchange on the chain:
        //     T[r][j] = [r == j] - sum_{k<r} A[r][k] T[k][j].  The lanes of
        //     block R also zero the block above it (rows of J, columns of R),
        //     which the merges below read.
        // (b) T_RJ = -T_RR (A_RJ T_JJ) in the same warp, as warp-level TF32
        //     products (T is rounded to bf16 afterwards, coarser than TF32).
        // No T entry right of these blocks is ever read; C3 writes zeros there.
        {
            constexpr int LX = 24;
            float *sX1 = sX;                 // [2][16][LX]
            if (lw < 2) {
                const int b = lw;
                {
                    const int Rb = 2 * b + (lane >> 4), j = lane & 15;
                    const float *Ab = sA + (16 * Rb) * LDT + 16 * Rb;
                    float t[16];
#pragma unroll
                    for (int r = 0; r < 16; ++r) {
                        float a0 = (r == j) ? 1.0f : 0.0f, a1 = 0.0f;
#pragma unroll
                        for (int k = 0; k < r; ++k) {
                            if (k & 1) a1 = fmaf(-Ab[r * LDT + k], t[k], a1);
                            else a0 = fmaf(-Ab[r * LDT + k], t[k], a0);
                        }
                        t[r] = a0 + a1;
                    }
                    float *Tb = sT + (16 * Rb) * LDT + 16 * Rb + j;
#pragma unroll
                    for (int r = 0; r < 16; ++r) Tb[r * LDT] = t[r];
                    if (lane >= 16) {
                        float *Tz = sT + (16 * (Rb - 1)) * LDT + 16 * Rb + j;
#pragma unroll
                        for (int r = 0; r < 16; ++r) Tz[r * LDT] = 0.0f;
                    }
                }
                __syncwarp();
                const int R = 1 + 2 * b, J = 2 * b;
                float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const float *Ab = sA + (16 * R) * LDT + 16 * J + 8 * ks;
                    const float *Bb = sT + (16 * J + 8 * ks) * LDT + 16 * J;
                    mma_tf32(d0, Ab, LDT, Bb, LDT, lane);
                    mma_tf32(d1, Ab, LDT, Bb + 8, LDT, lane);
                }
                store_c(sX1 + b * 16 * LX, LX, d0, 1.0f, lane);
                store_c(sX1 + b * 16 * LX + 8, LX, d1, 1.0f, lane);
                __syncwarp();
                float e0[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const float *Ab = sT + (16 * R) * LDT + 16 * R + 8 * ks;
                    const float *Bb = sX1 + b * 16 * LX + (8 * ks) * LX;
                    mma_tf32(e0, Ab, LDT, Bb, LX, lane);
                    mma_tf32(e1, Ab, LDT, Bb + 8, LX, lane);
                }
                store_c(sT + (16 * R) * LDT + 16 * J, LDT, e0, -1.0f, lane);
                store_c(sT + (16 * R) * LDT + 16 * J + 8, LDT, e1, -1.0f, lane);
            }
            bar.sync();
            // ------------------------------------------ C2: lower-left 32 x 32 block of T
            // With T_TT = T[0:32,0:32], T_BB = T[32:64,32:64]:
            //   T[32:64, 0:32] = -T_BB (A[32:64, 0:32] T_TT).
            // Warp nt (0..3) takes the 8 columns 8 nt .. 8 nt + 7: it forms
            // those columns of Y = A[32:64, 0:32] T_TT itself (in its own
            // shared-memory slice, so only the warp synchronises) and then
            // T_BB Y for them.
            constexpr int LYW = 8;
            float *sYw = sX + 2 * 16 * LX + lw * 32 * LYW;  // [32][LYW] per warp
            if (lw < 4) {
                const int nt = lw;
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_tf32(d, sA + (32 + 16 * mt) * LDT + 8 * ks, LDT,
                                 sT + (8 * ks) * LDT + 8 * nt, LDT, lane);
                    store_c(sYw + (16 * mt) * LYW, LYW, d, 1.0f, lane);
                }
                __syncwarp();
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_tf32(d, sT + (32 + 16 * mt) * LDT + 32 + 8 * ks, LDT,
                                 sYw + (8 * ks) * LYW, LYW, lane);
                    store_c(sT + (32 + 16 * mt) * LDT + 8 * nt, LDT, d, -1.0f, lane);
                }
            }
            static_assert((2 * 16 * LX + 4 * 32 * LYW) * 4 <= L::SX_BYTES, "solve temps");
            bar.sync();
        }
        // ---------------------------------------------- C3: [T; T] to the bf16 operand
        // (A is dead: the tile takes its place.)  Blocks right of the
        // diagonal are zero.  T twice makes the W | U product M = 128, so its
        // readback below uses all 128 TMEM lanes.
        for (int u = ltid; u < 64 * 8; u += NTC) {
            const int r = u >> 3, c = (u & 7) * 8;
            uint4 pk = make_uint4(0u, 0u, 0u, 0u);  // bf16 zeros
            if ((c >> 4) <= (r >> 4)) pk = pack8(sT + r * LDT + c);
            *reinterpret_cast<uint4 *>(t16 + rs_off(128, r, c)) = pk;
            *reinterpret_cast<uint4 *>(t16 + rs_off(128, r + 64, c)) = pk;
        }
        phase_sync();
        // ---------------------------------------------- D: W = T (beta K e^b), U = T (beta V)
        if (tid == 0) {
            // beta K e^b and beta V are adjacent column blocks: one N = 2D
            // product with A = [T; T] writes [W | U] into TMEM lanes 0..63
            // and again into lanes 64..127
            constexpr uint32_t id = idesc_bf16(128, 2 * D, false, true);
#pragma unroll 1
            for (int kk = 0; kk < P; ++kk) {
                const uint64_t a0 = kdesc(task_sm(kk) + L::T16, 128, 0, 0);
                // [beta K e^b | beta V]: rows 0..63 of WQ then UK, 16 KB per column block
                const uint64_t b0 = mdesc(task_sm(kk) + L::WQ, 128, 0, 0);
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4)
                    mma_bf16(task_tmem(kk) + TC_W, dstep(a0, s4 * 2), dstep(b0, s4 * 128), id, s4 > 0);
            }
            mma_commit(bar_mma);
        }
        if (bar.sync_or(!mma_wait())) { failed = true; break; }
        tc_fence_after();
        // ---------------------------------------------- E: W and U tiles
        {
            // lanes 0..63 read W (columns 0..D-1), lanes 64..127 U (columns
            // D..2D-1), each in NW / 4 parts of CPP columns; -W into rows
            // 0..63 of WQ, U into rows 0..63 of UK
            constexpr int CPP = D / (NW / 4);
            constexpr int CB = CPP >= 32 ? 32 : 16;
            const bool is_w = qd < 2;
            const int r = 32 * (qd & 1) + lane;
            const int c0 = cp * CPP;
            uint8_t *dst = is_w ? wq : uk;
            const float sgn = is_w ? (additive ? 0.0f : -1.0f) : 1.0f;
            const uint32_t tc0 = TC_W + (is_w ? 0u : (uint32_t)D) + (uint32_t)c0;
#pragma unroll
            for (int cb = 0; cb < CPP; cb += CB) {
                float v[CB];
                tmem_cols<CB>(tq + tc0 + cb, v);
#pragma unroll
                for (int i = 0; i < CB; ++i) v[i] *= sgn;
#pragma unroll
                for (int i = 0; i < CB; i += 8) st_bf16x8(dst, 128, r, c0 + cb + i, v + i);
            }
        }
        phase_sync();
        // ---------------------------------------------- F: record out
        // (by the fetcher, so that the leader goes straight on to the next
        // task's raw tiles)
        if (fetcher && len > 0) {
            uint8_t *rec = p.records + ((int64_t)cur.w * H + h) * Rec::BYTES;
            bulk_store_hint(rec + Rec::WQ, wq, 4 * L::tile64, pol);
            bulk_store_hint(rec + Rec::AQ, aqk, 8192, pol);
            if (GATED || scalar) bulk_store_hint(rec + Rec::GEND, sgend, 4 * D, pol);
            // the backward pass's copy of T: rows 0..63 of [T; T], a 64-row tile
            if (p.t_out) bulk_store_hint(p.t_out + ((int64_t)cur.w * H + h) * 8192, t16, 8192, pol);
            bulk_commit();
            if constexpr (FUSED) fst[F_PUB] = (int64_t)cur.w * H + h;
        }
        cur = nx;
        beta_cur = beta_nx;
        gate_cur = gate_nx;
        g = nx_g;
    }

    if (leader && failed && tma_pending) mbar_wait(bar_tma, tma_par, p.err, 3);
    if (fetcher) {
        bulk_wait_all();
        if constexpr (FUSED) publish();
    }
    tc_fence_before();
    bar.sync();
    tc_fence_after();
}

template <int D, bool GATED, bool SCALAR>
__global__ void __launch_bounds__(Layout<D, GATED>::NT, Layout<D, GATED>::CTAS_PER_SM)
    delta_intra_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_g, IntraParams p) {
    using L = Layout<D, GATED>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *const sbase = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sbase + L::COMMON);
    if ((threadIdx.x >> 5) == 0) {
        tmem_alloc(tslot, L::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    intra_run<D, GATED, SCALAR, false>(tm_q, tm_k, tm_v, tm_g, p, FusedSched{}, sbase, tmem,
                                       CtaBarrier{}, false);
    if ((threadIdx.x >> 5) == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

// ================================================================ fused launch
// The recurrence of one (sequence, head) inside the fused launch, on the 8
// warps of a d = 64 intra-chunk CTA once its share of intra-chunk tasks is
// done.  It computes what delta_inter_kernel computes, with the same three
// products per chunk into the same TMEM accumulators (lanes 0..63 u, lanes
// 64..127 O), and takes each record as soon as the task that wrote it has
// published it:
//   u = U - W S;  O = scale ((Q e^b) S + Aq u);  S <- Diag(e^{b_end}) S + K~^T u
// Roles, joined by mbarriers (every phase chained so that no waiter can
// fall two phases behind, as in the inter-chunk kernel):
//   warps 0..3  state, lane quarter w: S -> bf16 operand tile; with a gate,
//               S *= e^{b_end} of the next chunk in TMEM.  Warps 0, 1 (lanes
//               0..63) also turn u into its bf16 tile and put the next
//               chunk's U into the accumulator.
//   warp 4      one thread issues the products
//   warp 5      one thread loads each record into one of two buffers once
//               its flag is set
//   warps 6, 7  O (lanes 64..127) -> scale -> bf16 -> global, then zero
struct ChainParams {
    const uint8_t *records;   // [slots][H] records
    const unsigned *flags;    // [slots * H] set once a record is complete
    __nv_bfloat16 *o;
    const float *init_S;
    float *final_S;
    unsigned *err;
    int H, ntok;
    float scale;
};

struct ChainLayout {
    using Rec = Record<64>;
    static constexpr int NB = 2;
    static constexpr uint32_t REC0 = 0;
    static constexpr uint32_t SB = NB * Rec::BYTES;      // S, bf16 [64][64] RS tile
    static constexpr uint32_t UT = SB + 64 * 64 * 2;      // u, bf16 [64][64] RS tile
    static constexpr uint32_t BARS = UT + 64 * 64 * 2;    // mbarriers
    static constexpr uint32_t END = BARS + 128;
    // below the intra-chunk role's cu_seqlens copy, which the recurrence reads
    static_assert(END <= Layout<64, false>::CU, "recurrence buffers overlap the cu_seqlens copy");
    static_assert(SB % 1024 == 0 && UT % 1024 == 0, "swizzled tiles on 1024-byte boundaries");
};

enum : int {
    FB_U = 0, FB_S, FB_O, FB_SREADY, FB_UREADY, FB_UPRE, FB_OFREE0, FB_OFREE1, FB_REC0, FB_REC1,
    FB_COUNT
};

template <bool GATED>
__device__ __forceinline__ void chain_run(uint8_t *sm, uint32_t tmem, const ChainParams &p,
                                          const int *cu, int chain, const HalfBarrier bar) {
    using Lc = ChainLayout;
    using Rec = Record<64>;
    constexpr int D = 64;
    constexpr uint32_t S_COL = 0, ACC = 64;
    uint8_t *sb = sm + Lc::SB, *ut = sm + Lc::UT;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + Lc::BARS);
    const int tid = bar.thread(), warp = tid >> 5, lane = tid & 31;
    const int qd = warp & 3;
    const int H = p.H, n = chain / H, h = chain - n * H;
    int t_begin = cu[n], t_end = cu[n + 1];
    if (t_begin < 0 || t_end < t_begin || t_end > p.ntok) {
        if (tid == 0) atomicCAS(p.err, 0u, 100u);
        t_begin = t_end = 0;
    }
    const int nc = (t_end - t_begin + C - 1) / C;
    const int64_t slot0 = (int64_t)(t_begin / C) + n;
    auto rec_src = [&](int c) { return p.records + ((slot0 + c) * H + h) * (int64_t)Rec::BYTES; };
    auto buf = [&](int c) { return sm + Lc::REC0 + (uint32_t)(c & 1) * Rec::BYTES; };
    auto rec_bar = [&](int c) { return &bars[FB_REC0 + (c & 1)]; };
    auto rec_par = [](int c) { return (uint32_t)(c >> 1) & 1u; };
    auto ofree = [&](int c) { return &bars[FB_OFREE0 + (c & 1)]; };
    auto acc = [&](int c) { return ACC + (uint32_t)(c & 1) * D; };
    const uint32_t tq = tmem + ((uint32_t)(32 * qd) << 16);
    const int64_t sbase = ((int64_t)n * H + h) * D * D;

    if (tid == 0) {
        mbar_init(&bars[FB_U], 1);
        mbar_init(&bars[FB_S], 1);
        mbar_init(&bars[FB_O], 1);
        mbar_init(&bars[FB_SREADY], 4);
        mbar_init(&bars[FB_UREADY], 4);
        mbar_init(&bars[FB_UPRE], 2);
        mbar_init(&bars[FB_OFREE0], 2);
        mbar_init(&bars[FB_OFREE1], 2);
        mbar_init(&bars[FB_REC0], 1);
        mbar_init(&bars[FB_REC1], 1);
        fence_mbar_init();
    }
    tc_fence_before();
    bar.sync();
    tc_fence_after();
    auto warp_arrive = [&](uint64_t *bar) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar);
    };
    // U rows of chunk c into accumulator lanes 0..63 (warps 0, 1)
    auto preload_u = [&](int c) {
        const uint8_t *uk = buf(c) + Rec::UK;
        const int urow = 32 * qd + lane;
#pragma unroll
        for (int cb = 0; cb < D; cb += 16) {
            float v[16];
            unpack8(*reinterpret_cast<const uint4 *>(uk + rs_off(128, urow, cb)), v);
            unpack8(*reinterpret_cast<const uint4 *>(uk + rs_off(128, urow, cb + 8)), v + 8);
            tmem_st16(tq + acc(c) + cb, v);
        }
    };

    if (warp == 5) {
        // ====================================================== loader
        if (lane == 0) {
            int issued0 = -1, issued1 = -1;  // last chunk loaded into each buffer
            bool ok = true;
            for (int c = 0; c < nc && ok; ++c) {
                // chunk c - 2 drained: its buffer is free
                if (c >= 2 && !(ok = mbar_wait(ofree(c), (uint32_t)(c >> 1) & 1u, p.err, 40))) break;
                if (!(ok = wait_flag(p.flags + (slot0 + c) * H + h, p.err, 41))) break;
                fence_proxy_async_global();
                fence_proxy_async();
                mbar_arrive_expect_tx(rec_bar(c), Rec::BYTES);
                bulk_load_hint(buf(c), rec_src(c), Rec::BYTES, rec_bar(c), l2_evict_first());
                if (c & 1) issued1 = c;
                else issued0 = c;
            }
            if (!ok) {
                // whatever happened elsewhere, no load may still be writing
                // into shared memory when the CTA leaves
                if (issued0 >= 0) mbar_wait(rec_bar(issued0), rec_par(issued0), p.err, 43);
                if (issued1 >= 0) mbar_wait(rec_bar(issued1), rec_par(issued1), p.err, 43);
            }
        }
    } else if (warp == 4) {
        // ====================================================== issuer
        if (lane == 0 && nc > 0) {
            constexpr uint32_t id128 = idesc_bf16(128, D, false, true);
            constexpr uint32_t ids = idesc_bf16(D, D, true, true);
            const uint64_t bS = mdesc(sb, D, 0, 0), bU = mdesc(ut, C, 0, 0);
            for (int c = 0; c < nc; ++c) {
                uint8_t *rb = buf(c);
                const uint32_t ta = tmem + acc(c);
                if (!mbar_wait(&bars[FB_SREADY], (uint32_t)c & 1u, p.err, 44)) break;
                if (!mbar_wait(&bars[FB_UPRE], (uint32_t)c & 1u, p.err, 45)) break;
                if (!mbar_wait(rec_bar(c), rec_par(c), p.err, 46)) break;
                tc_fence_after();
                const uint64_t aWQ = kdesc(rb + Rec::WQ, 128, 0, 0);
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4)
                    mma_bf16(ta, dstep(aWQ, kstep_units(128, s4)), dstep(bS, s4 * 128), id128, 1);
                mma_commit(&bars[FB_U]);
                if (!mbar_wait(&bars[FB_UREADY], (uint32_t)c & 1u, p.err, 47)) break;
                tc_fence_after();
                const uint64_t aK = mdesc(rb + Rec::UK, 128, 64, 0);
                const uint64_t aA = kdesc(rb + Rec::AQ - 8192, 128, 0, 0);
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4)
                    mma_bf16(tmem + S_COL, dstep(aK, s4 * 128), dstep(bU, s4 * 128), ids, 1);
                mma_commit(&bars[FB_S]);
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4)
                    mma_bf16(ta, dstep(aA, s4 * 2), dstep(bU, s4 * 128), id128, 1);
                // the output warps have taken chunk c - 1 before chunk c's
                // output phase can complete
                if (c >= 1 &&
                    !mbar_wait(ofree(c - 1), (uint32_t)(((c - 1) >> 1) + 1) & 1u, p.err, 48))
                    break;
                mma_commit(&bars[FB_O]);
            }
        }
    } else if (warp < 4) {
        // ====================================================== state (and u)
        const int srow = acc_row(D, qd, lane);   // state row (key channel), or -1
        const bool u_warp = qd < 2;
        const int urow = 32 * qd + lane;
        bool ok = true;
        if (GATED && nc > 0) ok = mbar_wait(rec_bar(0), 0, p.err, 50);
        if (ok) {
            const float gd = (GATED && nc > 0 && srow >= 0)
                                 ? reinterpret_cast<const float *>(buf(0) + Rec::GEND)[srow]
                                 : 1.0f;
#pragma unroll
            for (int cb = 0; cb < D; cb += 16) {
                float v[16];
                if (srow >= 0 && p.init_S) {
                    const float4 *src = reinterpret_cast<const float4 *>(p.init_S + sbase + (int64_t)srow * D + cb);
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
                    st_bf16x8(sb, D, srow, cb, v);
                    st_bf16x8(sb, D, srow, cb + 8, v + 8);
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] *= gd;
                tmem_st16(tq + S_COL + cb, v);
            }
            fence_proxy_async();
            warp_arrive(&bars[FB_SREADY]);
            if (u_warp && nc > 0) {
                ok = mbar_wait(ofree(0), 0, p.err, 51) && mbar_wait(rec_bar(0), 0, p.err, 52);
                if (ok) {
                    tc_fence_after();
                    preload_u(0);
                    warp_arrive(&bars[FB_UPRE]);
                }
            }
        }
        for (int c = 0; c < nc && ok; ++c) {
            if (u_warp) {
                if (!(ok = mbar_wait(&bars[FB_U], (uint32_t)c & 1u, p.err, 53))) break;
                tc_fence_after();
#pragma unroll
                for (int cb = 0; cb < D; cb += 32) {
                    float v[32];
                    tmem_ld32(tq + acc(c) + cb, v);
#pragma unroll
                    for (int i = 0; i < 32; i += 8) st_bf16x8(ut, C, urow, cb + i, v + i);
                }
                fence_proxy_async();
            }
            // every state warp: u tile written, and S decayed for this chunk
            warp_arrive(&bars[FB_UREADY]);
            if (u_warp && c + 1 < nc) {
                if (!(ok = mbar_wait(ofree(c + 1), (uint32_t)((c + 1) >> 1) & 1u, p.err, 54))) break;
                if (!(ok = mbar_wait(rec_bar(c + 1), rec_par(c + 1), p.err, 55))) break;
                tc_fence_after();
                preload_u(c + 1);
                warp_arrive(&bars[FB_UPRE]);
            }
            if (!(ok = mbar_wait(&bars[FB_S], (uint32_t)c & 1u, p.err, 56))) break;
            tc_fence_after();
            if (c + 1 < nc) {
                float v[32];
#pragma unroll
                for (int cb = 0; cb < D; cb += 32) {
                    tmem_ld32(tq + S_COL + cb, v);
                    if (srow >= 0) {
#pragma unroll
                        for (int i = 0; i < 32; i += 8) st_bf16x8(sb, D, srow, cb + i, v + i);
                    }
                }
                fence_proxy_async();
                warp_arrive(&bars[FB_SREADY]);
                if (GATED) {
                    if (!(ok = mbar_wait(rec_bar(c + 1), rec_par(c + 1), p.err, 57))) break;
                    const float gd = srow >= 0
                                         ? reinterpret_cast<const float *>(buf(c + 1) + Rec::GEND)[srow]
                                         : 1.0f;
#pragma unroll
                    for (int cb = 0; cb < D; cb += 32) {
                        tmem_ld32(tq + S_COL + cb, v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] *= gd;
                        tmem_st16(tq + S_COL + cb, *reinterpret_cast<float(*)[16]>(v));
                        tmem_st16(tq + S_COL + cb + 16, *reinterpret_cast<float(*)[16]>(v + 16));
                    }
                }
            }
        }
        if (ok && p.final_S) {
#pragma unroll
            for (int cb = 0; cb < D; cb += 16) {
                float v[16];
                tmem_ld16(tq + S_COL + cb, v);
                if (srow >= 0) {
                    float4 *dst = reinterpret_cast<float4 *>(p.final_S + sbase + (int64_t)srow * D + cb);
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                }
            }
        }
    } else {
        // ====================================================== output (warps 6, 7)
        const int orow = 32 * (qd - 2) + lane;
        {
            float z[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) z[i] = 0.0f;
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
                for (int cb = 0; cb < D; cb += 16) tmem_st16(tq + acc(b) + cb, z);
            warp_arrive(&bars[FB_OFREE0]);
            warp_arrive(&bars[FB_OFREE1]);
        }
        for (int c = 0; c < nc; ++c) {
            if (!mbar_wait(&bars[FB_O], (uint32_t)c & 1u, p.err, 58)) break;
            tc_fence_after();
            const int tok0 = t_begin + c * C;
            const bool valid = orow < t_end - tok0;
#pragma unroll
            for (int cb = 0; cb < D; cb += 32) {
                float v[32];
                tmem_ld32(tq + acc(c) + cb, v);
                if (valid) {
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
            warp_arrive(ofree(c));
        }
    }
}

// Intra-chunk tasks and the recurrence in one cooperative grid (d = 64, no
// gate or a scalar gate), one 512-thread CTA per SM made of two independent
// 256-thread task loops, each with its own shared-memory region, TMEM
// columns and named barrier (the same resources as two CTAs of the
// two-launch path).  Every loop takes intra-chunk tasks in chunk-major order
// from the shared counters; the second loop of CTAs 0 .. n_chain_ctas - 1
// stops after the first share of them and runs the recurrence of one
// (sequence, head), consuming records as the other loops publish them.
// Intra-chunk work never waits for the recurrence and the cooperative launch
// keeps every CTA resident, so every wait ends.
template <bool SCALAR>
__global__ void __launch_bounds__(512, 1)
    delta_fused_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_g, IntraParams p, FusedSched fs,
                       ChainParams cp) {
    using L = Layout<64, false>;
    static_assert(L::NT == 256 && L::TCOLS == 128, "two 256-thread loops of 128 TMEM columns");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *const sbase = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int half = threadIdx.x >> 8;
    uint8_t *const sm = sbase + half * L::TASK_BYTES;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sbase + 2 * L::TASK_BYTES);
    // TMEM: columns 0..127 and 128..255 for the two task loops, 256..511 for
    // the recurrence (S, two [u ; O] accumulators)
    if (threadIdx.x < 32) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const HalfBarrier bar{1 + half};
    const bool chain_slot = half == 1 && (int)blockIdx.x < fs.n_chain_ctas;
    intra_run<64, false, SCALAR, true>(tm_q, tm_k, tm_v, tm_g, p, fs, sm, tmem + 128u * half, bar,
                                       chain_slot);
    if (chain_slot && (int)blockIdx.x < p.N * p.H)
        chain_run<SCALAR>(sm, tmem + 256u, cp, reinterpret_cast<const int *>(sm + L::CU),
                          blockIdx.x, bar);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x < 32) tmem_dealloc(tmem, 512);
}

// The chunk table the backward pass's kernels read (the forward kernels find
// their chunks from cu_seqlens).  One warp per sequence: the table entries
// of its chunk slots, then zeros
// for the (at most two) unused slots before the next sequence's first one.
__global__ void chunk_table_kernel(const int32_t *cu, int N, int ntok, int64_t slots,
                                   int2 *table) {
    grid_launch_dependents();  // the intra-chunk kernel may start its prologue
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= N) return;
    const int n = (int)gw;
    const int a = cu[n], e = cu[n + 1];
    if (n == 0 && a >= 0 && a <= ntok)
        for (int64_t s = lane; s < a / C; s += 32) table[s] = make_int2(0, 0);
    if (a < 0 || e < a || e > ntok) return;  // reported by the inter-chunk kernel
    const int64_t b = (int64_t)(a / C) + n;
    const int nc = (e - a + C - 1) / C;
    for (int j = lane; j < nc; j += 32) table[b + j] = make_int2(a + C * j, min(C, e - a - C * j));
    const int64_t gap_end = n + 1 < N ? (int64_t)(e / C) + n + 1 : slots;
    for (int64_t s = b + nc + lane; s < gap_end; s += 32) table[s] = make_int2(0, 0);
}

template <int D, bool GATED, bool SCALAR>
cudaError_t launch_t(const TcLaunch &x, cudaStream_t s) {
    IntraParams p{static_cast<const __nv_bfloat16 *>(x.a->beta_logits),
                  SCALAR ? static_cast<const __nv_bfloat16 *>(x.a->gate_logits) : nullptr,
                  x.a->cu_seqlens, x.records, x.a->t_out,
                  x.err, x.slots * x.a->H, x.a->N, x.a->H, x.a->ntok, x.a->flags};
    using L = Layout<D, GATED>;
    // Shared memory caps the CTAs per SM at CTAS_PER_SM, which keeps their
    // TMEM allocations within the SM's 512 columns.
    constexpr size_t need = L::TOTAL + 1024;
    constexpr size_t floor_ = L::CTAS_PER_SM == 1 ? 120 * 1024 : 77 * 1024;
    const size_t smem = need > floor_ ? need : floor_;
    auto kern = delta_intra_kernel<D, GATED, SCALAR>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    const int64_t groups = (p.n_tasks + L::P - 1) / L::P;
    const int64_t slots = (int64_t)x.sms * L::CTAS_PER_SM;
    const unsigned grid = (unsigned)(groups < slots ? groups : slots);
    if (grid == 0) return cudaSuccess;
    return launch_programmatic(kern, dim3(grid), dim3(L::NT), smem, s, x.mq, x.mk, x.mv, x.mg, p);
}

// Share of the intra-chunk tasks (in 1/1024) that the recurrence CTAs also
// take before they turn to their chains: about half lets the recurrence
// start when it can keep pace with the remaining tasks.
constexpr int kFusedShare1024 = 512;

// Dynamic shared memory of the fused kernel: two task loops' regions, the
// TMEM address slot and alignment slack.
constexpr size_t fused_smem_bytes() { return 2 * (size_t)Layout<64, false>::TASK_BYTES + 64 + 1024; }
static_assert(fused_smem_bytes() <= 227 * 1024, "two task loops in one CTA");

template <bool SCALAR>
cudaError_t launch_fused_t(const TcLaunch &x, cudaStream_t s, int grid) {
    const PrefillArgs &a = *x.a;
    IntraParams p{static_cast<const __nv_bfloat16 *>(a.beta_logits),
                  SCALAR ? static_cast<const __nv_bfloat16 *>(a.gate_logits) : nullptr,
                  a.cu_seqlens, x.records, a.t_out, x.err, x.slots * a.H, a.N, a.H, a.ntok, a.flags};
    FusedSched fs;
    fs.flags = x.flags;
    fs.counters = x.counters;
    fs.share_1024 = kFusedShare1024;
    fs.n_chain_ctas = a.N * a.H;
    ChainParams cp{x.records, x.flags, static_cast<__nv_bfloat16 *>(a.o), a.init_S, a.final_S,
                   x.err, a.H, a.ntok, a.scale};
    const size_t smem = fused_smem_bytes();
    auto kern = delta_fused_kernel<SCALAR>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(512);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, x.mq, x.mk, x.mv, x.mg, p, fs, cp);
}

// CTAs of the fused kernel (one per SM) when the device can hold them all at
// once, else 0.
template <bool SCALAR>
int fused_resident_ctas(int sms) {
    const size_t smem = fused_smem_bytes();
    auto kern = delta_fused_kernel<SCALAR>;
    // two CTAs per SM need the largest shared-memory carveout
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return 0;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 512, smem) != cudaSuccess)
        return 0;
    return per_sm >= 1 ? sms : 0;
}

}  // namespace

// The one-launch path is not dispatched: one run of it (three back-to-back
// calls of an 8 x 2048-token, 12-head problem) ended in a device fault whose
// cause has not been found, while a rerun with bounds-checked accesses was
// clean.  Until the cause is known every call takes the two launches.
constexpr bool kFusedDispatch = false;

bool delta_fused_eligible(int N, int H, int dk, int dv, bool gate, bool scalar, bool chunk_states,
                          int sms) {
    if (!kFusedDispatch) return false;
    if (dk != 64 || dv != 64 || (gate && !scalar) || chunk_states) return false;
    if (N < 1 || N >= Layout<64, false>::CU_MAX - 1 || sms < 1) return false;
    const int grid = scalar ? fused_resident_ctas<true>(sms) : fused_resident_ctas<false>(sms);
    // one recurrence per CTA (in its second task loop)
    return grid > 0 && (int64_t)N * H <= grid;
}

bool delta_fused_supported(const TcLaunch &x) {
    const PrefillArgs &a = *x.a;
    const bool scalar = a.gate_logits != nullptr && (a.flags & kGateScalar);
    return x.flags && x.counters &&
           delta_fused_eligible(a.N, a.H, a.dk, a.dv, a.gate_logits != nullptr, scalar,
                                a.chunk_states != nullptr, x.sms);
}

cudaError_t launch_delta_fused(const TcLaunch &x, cudaStream_t s) {
    const PrefillArgs &a = *x.a;
    const bool scalar = a.gate_logits != nullptr && (a.flags & kGateScalar);
    const int grid = scalar ? fused_resident_ctas<true>(x.sms) : fused_resident_ctas<false>(x.sms);
    if (grid <= 0) return cudaErrorNotSupported;
    cudaError_t e = cudaMemsetAsync(x.flags, 0, x.flag_bytes, s);
    if (e != cudaSuccess) return e;
    return scalar ? launch_fused_t<true>(x, s, grid) : launch_fused_t<false>(x, s, grid);
}

cudaError_t launch_chunk_table(const TcLaunch &x, cudaStream_t s) {
    const int64_t threads = (int64_t)x.a->N * 32;
    const unsigned blocks = (unsigned)((threads + 255) / 256);
    chunk_table_kernel<<<blocks, 256, 0, s>>>(x.a->cu_seqlens, x.a->N, x.a->ntok, x.slots,
                                              x.table);
    return cudaGetLastError();
}

cudaError_t launch_delta_intra(const TcLaunch &x, cudaStream_t s) {
    // per-channel gate: the gated kernel; scalar gate: the ungated one, which
    // applies the per-row decay itself
    const bool sc = x.a->gate_logits != nullptr && (x.a->flags & kGateScalar);
    const bool g = x.a->gate_logits != nullptr && !sc;
    if (x.a->dk == 128)
        return g ? launch_t<128, true, false>(x, s)
                 : sc ? launch_t<128, false, true>(x, s) : launch_t<128, false, false>(x, s);
    return g ? launch_t<64, true, false>(x, s)
             : sc ? launch_t<64, false, true>(x, s) : launch_t<64, false, false>(x, s);
}

}  // namespace la
