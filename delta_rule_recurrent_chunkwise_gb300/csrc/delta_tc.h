// delta_tc.h -- host-side interface between the launches of the
// tensor-core delta-rule prefill: intra-chunk kernel (every (chunk, head)
// task in parallel) and inter-chunk kernel (the state recurrence, one CTA
// per (head, sequence)), plus the chunk table the backward pass reads.
#pragma once

#include <cuda.h>

#include "launch.h"

namespace la {

struct TcLaunch {
    CUtensorMap mq, mk, mv, mg;  // TMA maps over q, k, v, gate (intra-chunk kernel)
    const PrefillArgs *a;
    int2 *table;                 // workspace: [slots] chunk table (backward pass)
    uint8_t *records;            // workspace: [slots][H] per-chunk records
    unsigned *flags;             // workspace: [slots * H] record-published flags (fused launch)
    unsigned *counters;          // workspace: [2] task counters (fused launch), right after flags
    size_t flag_bytes;           // bytes of flags and counters (zeroed before a fused launch)
    int64_t slots;
    unsigned *err;               // device error word
    int sms;                     // multiprocessors of the current device
};

// Launch with the programmatic-stream-serialisation attribute: the kernel
// may start while the previous kernel on the stream finishes, and must wait
// (griddepcontrol.wait) before reading that kernel's output.
template <typename... KArgs, typename... Args>
cudaError_t launch_programmatic(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// TMA map over a packed [ntok][H][D] bf16 tensor (box 64 tokens x 1 head x
// 64 channels, 128-byte swizzle); false if the driver refuses it.
bool make_map(CUtensorMap *m, const void *ptr, int D, int H, int ntok);

cudaError_t launch_chunk_table(const TcLaunch &x, cudaStream_t s);
// One cooperative launch running the intra-chunk tasks and the recurrence
// together (d = 64, no gate or a scalar gate, when the grid holds the chains).
bool delta_fused_supported(const TcLaunch &x);
bool delta_fused_eligible(int N, int H, int dk, int dv, bool gate, bool scalar, bool chunk_states,
                          int sms);
cudaError_t launch_delta_fused(const TcLaunch &x, cudaStream_t s);
cudaError_t launch_delta_intra(const TcLaunch &x, cudaStream_t s);
cudaError_t launch_delta_inter(const TcLaunch &x, cudaStream_t s);
// The recurrence over 128-token chunks (pairs of 64-token records; d = 64).
cudaError_t launch_delta_inter128(const TcLaunch &x, cudaStream_t s);

// Per-chunk gradients of the chunkwise backward pass (bf16, d = dk = dv in
// {64, 128}, a decay per key channel, per token or none): every (chunk,
// head) from its inputs, its starting state, the reverse chain's dS' and du,
// and the forward pass's T.
struct BwdChannelArgs {
    const void *q, *k, *v, *beta_logits, *gate_logits, *d_o;
    const int2 *table;        // [slots] {first token, length}
    const float *states;      // [slots][H][D][D] S at each chunk start
    const float *dstates;     // [slots][H][D][D] dS' of each chunk (fp32; gated only)
    const __nv_bfloat16 *dstates16;  // [slots][H][D][D] dS' of each chunk (bf16)
    const __nv_bfloat16 *du;  // [slots][H][64][D] du of each chunk (bf16)
    const uint8_t *tiles;     // [slots][H] T of each chunk, 8 KB bf16 swizzled tiles
    float *dq, *dk, *dv, *d_beta_logits, *d_gate_logits;
    int64_t n_tasks;
    int H, D;
    float scale;
    unsigned flags;
};
cudaError_t launch_delta_bwd_channel(const BwdChannelArgs &a, cudaStream_t s);

}  // namespace la
