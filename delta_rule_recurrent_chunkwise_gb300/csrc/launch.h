// launch.h -- internal launchers behind the C ABI (host side, no validation:
// api.cu checks every argument before calling these).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace la {

struct PrefillArgs {
    const void *q, *k, *v, *beta_logits, *gate_logits;
    void *o;
    const int32_t *cu_seqlens;
    int N, ntok, H, dk, dv;
    float scale;
    unsigned flags;
    const float *init_S, *init_z;
    float *final_S, *final_z;
    bool bf16;
    void *workspace;          // device scratch (tensor-core delta path)
    size_t workspace_bytes;
    // Tensor-core delta path only, for the backward pass: the state at the
    // start of every chunk, fp32 [slot][H][dk][dv] (slot as in the chunk
    // table), or null.  With it, o may be null (no output written).
    float *chunk_states = nullptr;
    // Backward pass only: the UT matrix T = (I + A)^{-1} of every chunk,
    // bf16, one 64 x 64 row-swizzled tile (8 KB) per (slot, head), or null.
    uint8_t *t_out = nullptr;
    // Tokens per chunk of the recurrence: 64, or 128 on the tensor-core path
    // with dk = dv = 64 (the records stay per 64 tokens; the recurrence pairs
    // them).
    int chunk = 64;
    // ELU+1 prefill: the most 64-token chunks any sequence spans, when known
    // on the host (-1: unknown); up to 8 selects the chunk-parallel kernel.
    int max_chunks = -1;
};

struct DecodeArgs {
    const void *q, *k, *v, *beta_logits, *gate_logits;
    void *o;
    int N, H, dk, dv;
    float scale;
    unsigned flags;
    float *state;
    bool bf16;
    const int32_t *slots = nullptr;  // optional slot map into a state pool
    int64_t n_slots = 0;
    unsigned *err = nullptr;         // device error word (slot map only)
};

// Gradients of the delta rule (token-serial, column per warp, clusters).
struct BwdArgs {
    const void *q, *k, *v, *beta_logits, *gate_logits, *d_o;
    const float *d_final_S, *init_S;
    const int32_t *cu_seqlens;
    int N, ntok, H, dk, dv;
    float scale;
    unsigned flags;
    float *dq, *dk_out, *dv_out, *d_beta_logits, *d_gate_logits, *d_init_S;
    void *workspace;
    bool bf16;
};
size_t delta_bwd_workspace_bytes(int N, int ntok, int H, int dk, int dv);
cudaError_t launch_delta_backward(const BwdArgs &a, cudaStream_t s);
// Chunkwise form (bf16, dk = dv in {64, 128}, any gate, either rule, every
// tensor 16-byte aligned): the tensor-core forward with chunk states, a
// reverse dS chain and a parallel per-chunk gradient kernel that also takes
// the prologue's derivatives.
bool delta_bwd_chunked_supported(const BwdArgs &a);
size_t delta_bwd_chunked_workspace_bytes(int N, int ntok, int H, int D);
cudaError_t launch_delta_backward_chunked(const BwdArgs &a, cudaStream_t s);
// The same split for training: the forward pass (a.workspace = a backward
// workspace of delta_bwd_workspace_bytes) writing o and final_S as asked and
// keeping the records, T and the chunk-start states there; then the
// gradients from that workspace, without the forward recomputation.
bool delta_train_supported(const PrefillArgs &a);
cudaError_t launch_delta_train_forward(const PrefillArgs &a, cudaStream_t s);
cudaError_t launch_delta_backward_saved(const BwdArgs &a, cudaStream_t s);

// fp32 SIMT chunk kernels (any I/O dtype).
cudaError_t launch_linear_simt(const PrefillArgs &a, cudaStream_t s);
// ELU+1 prefill on the tensor cores (bf16 I/O, dk = dv = 64, 16-byte aligned
// tensors): one CTA per (head, sequence), used for sequences longer than
// the chunk-parallel CUDA-core kernel takes.
bool linear_tc_supported(const PrefillArgs &a);
cudaError_t launch_linear_tc(const PrefillArgs &a, cudaStream_t s);
constexpr int kLinearParallelMaxChunks = 8;  // the chunk-parallel kernel's limit
cudaError_t launch_delta_simt(const PrefillArgs &a, cudaStream_t s);
// tcgen05 tensor-core chunk kernels (bf16 I/O, dk == dv in {64, 128}): the
// intra-chunk kernel and the inter-chunk kernel, with the per-chunk records
// in the caller's workspace (and a chunk table for the backward pass).
size_t delta_tc_workspace_bytes(int N, int ntok, int H, int dk, int dv, int chunk, bool bf16);
bool delta_tc_supported(const PrefillArgs &a);
// Kernels one la_prefill_delta call launches for these sizes (aligned
// tensors, a workspace of the queried size): 1 or 2 on the tensor-core path,
// 1 on the CUDA-core path.
int delta_tc_launches(int N, int ntok, int H, int dk, int dv, int chunk, bool bf16, bool gate,
                      bool scalar);
cudaError_t launch_delta_tc(const PrefillArgs &a, cudaStream_t s);
// Static device scratch behind la_prefill_delta_static (static_scratch.cu,
// a module of its own; per device, the address is looked up on first use).
constexpr size_t kStaticScratchBytes = size_t(256) << 20;
void *static_scratch();
// Device address of the library's error word on the current device (kernels
// record the first failure there; la_check_device reads and clears it).
unsigned *device_error_word();
// Reads and clears the device error word (synchronises s).
cudaError_t tc_take_error(cudaStream_t s, unsigned *code);
// HBM-streaming decode step.
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s);

}  // namespace la
