// prefill_tc.cu -- host side of the tensor-core (gated) delta-rule prefill:
// TMA maps, workspace layout and the launches (intra-chunk kernel, then
// inter-chunk kernel; a chunk table first when the backward pass asks for
// per-chunk states), plus the library's device error word.  The kernels live
// in delta_intra_tc.cu and delta_inter_tc.cu; the static scratch buffer of
// la_prefill_delta_static in static_scratch.cu.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "delta_tc.h"
#include "launch.h"
#include "tc_tile.cuh"

namespace la {

__device__ unsigned g_tc_error;  // first error code raised in a kernel

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

}  // namespace

// 3-D map over a packed [ntok][H][D] bf16 tensor; box = 64 tokens x 1 head x 64 channels.
bool make_map(CUtensorMap *m, const void *ptr, int D, int H, int ntok) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)(ntok > 0 ? ntok : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// Per-device values cached on first use.  Host threads racing on a first
// call store the same value; a failed query is retried on the next call.
int sm_count() {
    static std::atomic<int> count[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int c = count[dev].load(std::memory_order_acquire);
    if (!c) {
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        count[dev].store(c, std::memory_order_release);
    }
    return c;
}

size_t record_bytes(int D) {
    return D == 128 ? tile::Record<128>::BYTES : tile::Record<64>::BYTES;
}

}  // namespace

size_t delta_tc_workspace_bytes(int N, int ntok, int H, int dk, int dv, int chunk, bool bf16) {
    // chunk 128 (d = 64 only) keeps the 64-token records: the same workspace
    const bool chunk_ok = chunk == tile::C || (chunk == 2 * tile::C && dk == 64);
    if (!bf16 || dk != dv || (dk != 64 && dk != 128) || !chunk_ok || N < 1 || ntok < 0 || H < 1)
        return 0;
    const int64_t slots = tile::Workspace::slots(N, ntok);
    return (size_t)tile::Workspace::table_bytes(N, ntok) + (size_t)slots * H * record_bytes(dk) +
           (size_t)tile::Workspace::flag_bytes(N, ntok, H);
}

bool delta_tc_supported(const PrefillArgs &a) {
    auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const size_t ws = delta_tc_workspace_bytes(a.N, a.ntok, a.H, a.dk, a.dv, a.chunk, a.bf16);
    // per-chunk states (the backward pass) are kept at 64-token chunks only
    if (a.chunk != tile::C && a.chunk_states) return false;
    return ws > 0 && a.workspace && a.workspace_bytes >= ws &&
           (reinterpret_cast<uintptr_t>(a.workspace) & 255u) == 0 && al16(a.q) && al16(a.k) &&
           al16(a.v) && al16(a.o) && (!a.gate_logits || al16(a.gate_logits)) &&
           (!a.init_S || al16(a.init_S)) && (!a.final_S || al16(a.final_S)) &&
           encode_fn() != nullptr && sm_count() > 0;
}

cudaError_t launch_delta_tc(const PrefillArgs &a, cudaStream_t s) {
    TcLaunch x;
    const int D = a.dk;
    if (!make_map(&x.mq, a.q, D, a.H, a.ntok) || !make_map(&x.mk, a.k, D, a.H, a.ntok) ||
        !make_map(&x.mv, a.v, D, a.H, a.ntok))
        return cudaErrorInvalidValue;
    if (a.gate_logits && !(a.flags & kGateScalar)) {  // a scalar gate is read without TMA
        if (!make_map(&x.mg, a.gate_logits, D, a.H, a.ntok)) return cudaErrorInvalidValue;
    } else {
        x.mg = x.mq;
    }
    x.a = &a;
    x.slots = tile::Workspace::slots(a.N, a.ntok);
    x.table = static_cast<int2 *>(a.workspace);
    x.records = static_cast<uint8_t *>(a.workspace) + tile::Workspace::table_bytes(a.N, a.ntok);
    x.flags = reinterpret_cast<unsigned *>(x.records + x.slots * a.H * (int64_t)record_bytes(D));
    x.counters = x.flags + (((x.slots * a.H * 4 + 255) & ~int64_t(255)) / 4);
    x.flag_bytes = (size_t)tile::Workspace::flag_bytes(a.N, a.ntok, a.H);
    x.err = device_error_word();
    x.sms = sm_count();
    if (!x.err) return cudaErrorInvalidValue;
    // d = 64 without a per-channel gate: both halves in one cooperative
    // launch when the device holds the whole grid (else the two launches)
    if (a.chunk == tile::C && delta_fused_supported(x)) {
        const cudaError_t ef = launch_delta_fused(x, s);
        if (ef == cudaSuccess) return ef;
        cudaGetLastError();  // clear the refused launch; fall back below
    }
    // The chunk table is read only by the backward pass's kernels (which ask
    // for per-chunk states); the intra-chunk kernel finds its chunks from
    // cu_seqlens itself.
    cudaError_t e = a.chunk_states ? launch_chunk_table(x, s) : cudaSuccess;
    if (e == cudaSuccess) e = launch_delta_intra(x, s);
    if (e == cudaSuccess)
        e = a.chunk == 2 * tile::C ? launch_delta_inter128(x, s) : launch_delta_inter(x, s);
    return e;
}

int delta_tc_launches(int N, int ntok, int H, int dk, int dv, int chunk, bool bf16, bool gate,
                      bool scalar) {
    if (delta_tc_workspace_bytes(N, ntok, H, dk, dv, chunk, bf16) == 0) return 1;  // CUDA-core kernel
    if (chunk != tile::C) return 2;
    return delta_fused_eligible(N, H, dk, dv, gate, scalar, false, sm_count()) ? 1 : 2;
}

unsigned *device_error_word() {
    static std::atomic<void *> addr[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    void *p = addr[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_tc_error) != cudaSuccess) return nullptr;
        addr[dev].store(p, std::memory_order_release);
    }
    return static_cast<unsigned *>(p);
}

cudaError_t tc_take_error(cudaStream_t s, unsigned *code) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(code, g_tc_error, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && *code != 0)
        e = cudaMemcpyToSymbolAsync(g_tc_error, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return e;
}

}  // namespace la
