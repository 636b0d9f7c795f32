// delta_tc.h -- host-side interface between the three launches of the
// tensor-core delta-rule prefill: chunk table, intra-chunk kernel (every
// (chunk, head) task in parallel) and inter-chunk kernel (the state
// recurrence, one CTA per (head, sequence)).
#pragma once

#include <cuda.h>

#include "launch.h"

namespace la {

struct TcLaunch {
    CUtensorMap mq, mk, mv, mg;  // TMA maps over q, k, v, gate (intra-chunk kernel)
    const PrefillArgs *a;
    int2 *table;                 // workspace: [slots] chunk table
    uint8_t *records;            // workspace: [slots][H] per-chunk records
    int64_t slots;
    unsigned *err;               // device error word
    int sms;                     // multiprocessors of the current device
};

cudaError_t launch_chunk_table(const TcLaunch &x, cudaStream_t s);
cudaError_t launch_delta_intra(const TcLaunch &x, cudaStream_t s);
cudaError_t launch_delta_inter(const TcLaunch &x, cudaStream_t s);

}  // namespace la
