// api.cu -- the C ABI (include/linattn.h): argument validation on the host,
// then launches on the caller's stream.  Nothing here allocates, frees or
// synchronises (la_check_device excepted), and no exception escapes.

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "../../include/linattn.h"
#include "launch.h"
#include "tc.cuh"

namespace {

// Waits on an mbarrier that nothing arrives on: the bounded wait every
// kernel of the library uses runs out, records its code in the device error
// word and returns, and the kernel ends normally.
__global__ void wait_selftest_kernel(unsigned *err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        la::tc::mbar_init(&bar, 1);
        la::tc::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) la::tc::mbar_wait(&bar, 0, err, 99u);
}

bool head_size_ok(int d) { return d == 64 || d == 128; }

bool dtype_ok(la_dtype io) { return io == LA_F32 || io == LA_BF16; }

la_status check_cu_host(const int32_t *cu_host, int N, int ntok) {
    if (!cu_host) return LA_OK;
    if (cu_host[0] < 0 || cu_host[N] > ntok) return LA_ERR_INVALID_ARG;
    for (int n = 0; n < N; ++n)
        if (cu_host[n + 1] < cu_host[n]) return LA_ERR_INVALID_ARG;
    return LA_OK;
}

la_status from_cuda(cudaError_t e) { return e == cudaSuccess ? LA_OK : LA_ERR_CUDA; }

// Host checks shared by the delta-rule prefill entry points (workspace aside).
la_status check_delta_args(const void *q, const void *k, const void *v, const void *beta_logits,
                           const void *gate_logits, const void *o, la_dtype io,
                           const int32_t *cu_seqlens,
                           const int32_t *cu_seqlens_host, int N, int ntok, int H, int dk,
                           int dv, int chunk, float scale, unsigned flags) {
    if (!q || !k || !v || !o || !cu_seqlens || N < 1 || ntok < 0 || H < 1 || !dtype_ok(io))
        return LA_ERR_INVALID_ARG;
    if (!beta_logits && !(flags & LA_ADDITIVE)) return LA_ERR_INVALID_ARG;
    if (dk < 1 || dv < 1 || chunk < 1 || !std::isfinite(scale)) return LA_ERR_INVALID_ARG;
    if (flags & ~(LA_L2NORM_K | LA_L2NORM_Q | LA_SILU_QK | LA_GATE_SCALAR | LA_ADDITIVE))
        return LA_ERR_INVALID_ARG;
    if ((flags & LA_GATE_SCALAR) && !gate_logits) return LA_ERR_INVALID_ARG;
    if (!head_size_ok(dk) || !head_size_ok(dv)) return LA_ERR_UNSUPPORTED;
    // chunk 128: the tensor-core path (bf16 I/O) with dk = dv = 64
    if (chunk != 64 && !(chunk == 128 && io == LA_BF16 && dk == 64 && dv == 64))
        return LA_ERR_UNSUPPORTED;
    if (N > 65535 || H > 65535) return LA_ERR_UNSUPPORTED;
    return check_cu_host(cu_seqlens_host, N, ntok);
}

la_status check_decode_args(const void *q, const void *k, const void *v, const void *beta_logits,
                            const void *gate_logits, const void *o, la_dtype io, int N, int H,
                            int dk, int dv, float scale, unsigned flags, const float *state) {
    if (!q || !k || !v || !o || !state || N < 1 || H < 1 || !dtype_ok(io))
        return LA_ERR_INVALID_ARG;
    if (!beta_logits && !(flags & LA_ADDITIVE)) return LA_ERR_INVALID_ARG;
    if (dk < 1 || dv < 1 || !std::isfinite(scale)) return LA_ERR_INVALID_ARG;
    if (flags & ~(LA_L2NORM_K | LA_L2NORM_Q | LA_SILU_QK | LA_GATE_SCALAR | LA_ADDITIVE))
        return LA_ERR_INVALID_ARG;
    if ((flags & LA_GATE_SCALAR) && !gate_logits) return LA_ERR_INVALID_ARG;
    if (!head_size_ok(dk) || !head_size_ok(dv)) return LA_ERR_UNSUPPORTED;
    if ((int64_t)N * H * 2 > 0x7fffffffLL) return LA_ERR_UNSUPPORTED;
    return LA_OK;
}

}  // namespace

extern "C" {

const char *la_status_string(la_status s) {
    switch (s) {
        case LA_OK: return "LA_OK";
        case LA_ERR_INVALID_ARG: return "LA_ERR_INVALID_ARG: invalid argument";
        case LA_ERR_UNSUPPORTED: return "LA_ERR_UNSUPPORTED: no kernel for this configuration";
        case LA_ERR_CUDA: return "LA_ERR_CUDA: CUDA runtime or launch error";
        case LA_ERR_TIMEOUT: return "LA_ERR_TIMEOUT: a bounded in-kernel wait expired";
        case LA_ERR_TOO_LARGE:
            return "LA_ERR_TOO_LARGE: scratch needed exceeds the library's static buffer";
    }
    return "LA_ERR_UNKNOWN";
}

la_status la_prefill_linear(const void *q, const void *k, const void *v, void *o, la_dtype io,
                            const int32_t *cu_seqlens, const int32_t *cu_seqlens_host, int N,
                            int ntok, int H, int dk, int dv, const float *init_S,
                            const float *init_z, float *final_S, float *final_z, void *stream) {
    if (!q || !k || !v || !o || !cu_seqlens || N < 1 || ntok < 0 || H < 1 || !dtype_ok(io))
        return LA_ERR_INVALID_ARG;
    if (dk < 1 || dv < 1) return LA_ERR_INVALID_ARG;
    if (!head_size_ok(dk) || !head_size_ok(dv) || N > 65535 || H > 65535) return LA_ERR_UNSUPPORTED;
    if (la_status st = check_cu_host(cu_seqlens_host, N, ntok)) return st;
    la::PrefillArgs a{q, k, v, nullptr, nullptr, o, cu_seqlens, N, ntok, H, dk, dv, 1.0f, 0u,
                      init_S, init_z, final_S, final_z, io == LA_BF16};
    // longest sequence in chunks: from the host copy of cu_seqlens, else
    // bounded by the packed total
    if (cu_seqlens_host) {
        int longest = 0;
        for (int n = 0; n < N; ++n)
            longest = std::max(longest, cu_seqlens_host[n + 1] - cu_seqlens_host[n]);
        a.max_chunks = (longest + 63) / 64;
    } else if (ntok <= la::kLinearParallelMaxChunks * 64) {
        a.max_chunks = (ntok + 63) / 64;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // short sequences: the chunk-parallel CUDA-core kernel (fp32 or bf16);
    // longer bf16 ones at d = 64: the tensor cores; else the CUDA-core scan
    const bool short_seqs = a.max_chunks >= 0 && a.max_chunks <= la::kLinearParallelMaxChunks;
    if (!short_seqs && la::linear_tc_supported(a)) return from_cuda(la::launch_linear_tc(a, s));
    return from_cuda(la::launch_linear_simt(a, s));
}

size_t la_prefill_delta_workspace_size(int N, int ntok, int H, int dk, int dv, int chunk,
                                       la_dtype io) {
    if (!dtype_ok(io)) return 0;
    return la::delta_tc_workspace_bytes(N, ntok, H, dk, dv, chunk, io == LA_BF16);
}

la_status la_prefill_delta(const void *q, const void *k, const void *v, const void *beta_logits,
                           const void *gate_logits, void *o, la_dtype io,
                           const int32_t *cu_seqlens, const int32_t *cu_seqlens_host, int N,
                           int ntok, int H, int dk, int dv, int chunk, float scale,
                           unsigned flags, const float *init_S, float *final_S, void *workspace,
                           size_t workspace_bytes, void *stream) {
    if (la_status st = check_delta_args(q, k, v, beta_logits, gate_logits, o, io, cu_seqlens, cu_seqlens_host,
                                        N, ntok, H, dk, dv, chunk, scale, flags))
        return st;
    const size_t ws_need = la_prefill_delta_workspace_size(N, ntok, H, dk, dv, chunk, io);
    if (ws_need > 0 && (!workspace || workspace_bytes < ws_need ||
                        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return LA_ERR_INVALID_ARG;
    la::PrefillArgs a{q, k, v, beta_logits, gate_logits, o, cu_seqlens, N, ntok, H, dk, dv, scale,
                      flags, init_S, nullptr, final_S, nullptr, io == LA_BF16, workspace,
                      workspace_bytes};
    a.chunk = chunk;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (la::delta_tc_supported(a)) return from_cuda(la::launch_delta_tc(a, s));
    // the CUDA-core kernels step over 64-token chunks only
    if (chunk != 64) return LA_ERR_UNSUPPORTED;
    return from_cuda(la::launch_delta_simt(a, s));
}

int la_prefill_delta_launches(int N, int ntok, int H, int dk, int dv, int chunk, la_dtype io,
                              unsigned flags, int has_gate) {
    const void *g = has_gate ? reinterpret_cast<const void *>(16) : nullptr;
    const void *x = reinterpret_cast<const void *>(16);
    if (check_delta_args(x, x, x, x, g, x, io, reinterpret_cast<const int32_t *>(x), nullptr, N,
                         ntok, H, dk, dv, chunk, 1.0f, flags) != LA_OK)
        return 0;
    return la::delta_tc_launches(N, ntok, H, dk, dv, chunk, io == LA_BF16, has_gate != 0,
                                 has_gate && (flags & LA_GATE_SCALAR));
}

la_status la_prefill_delta_static(const void *q, const void *k, const void *v,
                                  const void *beta_logits, const void *gate_logits, void *o,
                                  la_dtype io, const int32_t *cu_seqlens,
                                  const int32_t *cu_seqlens_host, int N, int ntok, int H, int dk,
                                  int dv, int chunk, float scale, unsigned flags,
                                  const float *init_S, float *final_S, void *stream) {
    static_assert(la::kStaticScratchBytes == LA_STATIC_SCRATCH_BYTES, "static scratch size");
    if (la_status st = check_delta_args(q, k, v, beta_logits, gate_logits, o, io, cu_seqlens, cu_seqlens_host,
                                        N, ntok, H, dk, dv, chunk, scale, flags))
        return st;
    const size_t need = la_prefill_delta_workspace_size(N, ntok, H, dk, dv, chunk, io);
    if (need > la::kStaticScratchBytes) return LA_ERR_TOO_LARGE;
    void *ws = nullptr;
    if (need > 0 && !(ws = la::static_scratch())) return LA_ERR_CUDA;
    return la_prefill_delta(q, k, v, beta_logits, gate_logits, o, io, cu_seqlens, cu_seqlens_host,
                            N, ntok, H, dk, dv, chunk, scale, flags, init_S, final_S, ws,
                            ws ? la::kStaticScratchBytes : 0, stream);
}

la_status la_decode_step(const void *q, const void *k, const void *v, const void *beta_logits,
                         const void *gate_logits, void *o, la_dtype io, int N, int H, int dk,
                         int dv, float scale, unsigned flags, float *state, void *stream) {
    if (la_status st = check_decode_args(q, k, v, beta_logits, gate_logits, o, io, N, H, dk, dv,
                                         scale, flags, state))
        return st;
    la::DecodeArgs a{q, k, v, beta_logits, gate_logits, o, N, H, dk, dv, scale, flags, state,
                     io == LA_BF16};
    return from_cuda(la::launch_decode(a, static_cast<cudaStream_t>(stream)));
}

la_status la_decode_step_slots(const void *q, const void *k, const void *v,
                               const void *beta_logits, const void *gate_logits, void *o,
                               la_dtype io, int N, int H, int dk, int dv, float scale,
                               unsigned flags, float *state_pool, int n_slots,
                               const int32_t *state_indices, void *stream) {
    if (la_status st = check_decode_args(q, k, v, beta_logits, gate_logits, o, io, N, H, dk, dv,
                                         scale, flags, state_pool))
        return st;
    if (!state_indices || n_slots < 1) return LA_ERR_INVALID_ARG;
    la::DecodeArgs a{q, k, v, beta_logits, gate_logits, o, N, H, dk, dv, scale, flags,
                     state_pool, io == LA_BF16, state_indices, n_slots, la::device_error_word()};
    if (!a.err) return LA_ERR_CUDA;
    return from_cuda(la::launch_decode(a, static_cast<cudaStream_t>(stream)));
}

size_t la_backward_delta_workspace_size(int N, int ntok, int H, int dk, int dv) {
    if (N < 1 || ntok < 0 || H < 1 || !head_size_ok(dk) || !head_size_ok(dv)) return 0;
    return la::delta_bwd_workspace_bytes(N, ntok, H, dk, dv);
}

la_status la_backward_delta(const void *q, const void *k, const void *v, const void *beta_logits,
                            const void *gate_logits, const void *d_o, const float *d_final_S,
                            la_dtype io, const int32_t *cu_seqlens,
                            const int32_t *cu_seqlens_host, int N, int ntok, int H, int dk,
                            int dv, float scale, unsigned flags, const float *init_S, float *dq,
                            float *dk_out, float *dv_out, float *d_beta_logits,
                            float *d_gate_logits, float *d_init_S, void *workspace,
                            size_t workspace_bytes, void *stream) {
    if (la_status st = check_delta_args(q, k, v, beta_logits, gate_logits, d_o, io, cu_seqlens,
                                        cu_seqlens_host, N, ntok, H, dk, dv, 64, scale, flags))
        return st;
    if (!dq || !dk_out || !dv_out || !d_beta_logits || (gate_logits && !d_gate_logits))
        return LA_ERR_INVALID_ARG;
    const size_t need = la::delta_bwd_workspace_bytes(N, ntok, H, dk, dv);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return LA_ERR_INVALID_ARG;
    la::BwdArgs a{q, k, v, beta_logits, gate_logits, d_o, d_final_S, init_S, cu_seqlens, N, ntok,
                  H, dk, dv, scale, flags, dq, dk_out, dv_out, d_beta_logits, d_gate_logits,
                  d_init_S, workspace, io == LA_BF16};
    return from_cuda(la::launch_delta_backward(a, static_cast<cudaStream_t>(stream)));
}

la_status la_prefill_delta_train(const void *q, const void *k, const void *v,
                                 const void *beta_logits, const void *gate_logits, void *o,
                                 la_dtype io, const int32_t *cu_seqlens,
                                 const int32_t *cu_seqlens_host, int N, int ntok, int H, int dk,
                                 int dv, float scale, unsigned flags, const float *init_S,
                                 float *final_S, void *saved, size_t saved_bytes, void *stream) {
    if (la_status st = check_delta_args(q, k, v, beta_logits, gate_logits, o, io, cu_seqlens,
                                        cu_seqlens_host, N, ntok, H, dk, dv, 64, scale, flags))
        return st;
    if (io != LA_BF16 || dk != dv) return LA_ERR_UNSUPPORTED;
    const size_t need = la::delta_bwd_workspace_bytes(N, ntok, H, dk, dv);
    if (!saved || saved_bytes < need || (reinterpret_cast<uintptr_t>(saved) & 255u))
        return LA_ERR_INVALID_ARG;
    la::PrefillArgs a{q, k, v, beta_logits, gate_logits, o, cu_seqlens, N, ntok, H, dk, dv, scale,
                      flags, init_S, nullptr, final_S, nullptr, true, saved, saved_bytes};
    if (!la::delta_train_supported(a)) return LA_ERR_UNSUPPORTED;
    return from_cuda(la::launch_delta_train_forward(a, static_cast<cudaStream_t>(stream)));
}

la_status la_backward_delta_saved(const void *q, const void *k, const void *v,
                                  const void *beta_logits, const void *gate_logits,
                                  const void *d_o, const float *d_final_S, la_dtype io,
                                  const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                                  int N, int ntok, int H, int dk, int dv, float scale,
                                  unsigned flags, const float *init_S, float *dq, float *dk_out,
                                  float *dv_out, float *d_beta_logits, float *d_gate_logits,
                                  float *d_init_S, void *saved, size_t saved_bytes, void *stream) {
    if (la_status st = check_delta_args(q, k, v, beta_logits, gate_logits, d_o, io, cu_seqlens,
                                        cu_seqlens_host, N, ntok, H, dk, dv, 64, scale, flags))
        return st;
    if (!dq || !dk_out || !dv_out || !d_beta_logits || (gate_logits && !d_gate_logits))
        return LA_ERR_INVALID_ARG;
    if (io != LA_BF16 || dk != dv) return LA_ERR_UNSUPPORTED;   // as la_prefill_delta_train
    const size_t need = la::delta_bwd_workspace_bytes(N, ntok, H, dk, dv);
    if (!saved || saved_bytes < need || (reinterpret_cast<uintptr_t>(saved) & 255u))
        return LA_ERR_INVALID_ARG;
    la::BwdArgs a{q, k, v, beta_logits, gate_logits, d_o, d_final_S, init_S, cu_seqlens, N, ntok,
                  H, dk, dv, scale, flags, dq, dk_out, dv_out, d_beta_logits, d_gate_logits,
                  d_init_S, saved, true};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // unaligned gradient tensors: the token-serial form, recomputing the forward
    if (!la::delta_bwd_chunked_supported(a)) return from_cuda(la::launch_delta_backward(a, s));
    return from_cuda(la::launch_delta_backward_saved(a, s));
}

la_status la_selftest_wait_timeout(void *stream) {
    unsigned *err = la::device_error_word();
    if (!err) return LA_ERR_CUDA;
    wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err);
    return from_cuda(cudaGetLastError());
}

la_status la_check_device(void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return LA_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    unsigned code = 0;
    if (la::tc_take_error(s, &code) != cudaSuccess) return LA_ERR_CUDA;
    if (code == 100u) return LA_ERR_INVALID_ARG;  // cu_seqlens or a state slot out of range
    if (code != 0u) return LA_ERR_TIMEOUT;
    return LA_OK;
}

}  // extern "C"
