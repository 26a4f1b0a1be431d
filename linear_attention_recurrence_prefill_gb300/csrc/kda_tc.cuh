// kda_tc.cuh -- entry points of the tcgen05 tensor-core prefill path.
#pragma once

#include "kda_common.cuh"

namespace kda {

// True when the tensor-core path is built for this head size, dtype and chunk
// option (0 = default chunk).
bool tc_prefill_supported(int d, int dtype, int chunk);

// Workspace bytes the tensor-core path needs for these sizes.
size_t tc_workspace_bytes(int T_total, int N, int H, int d, const kda_options* opt);

// Kernels one tensor-core prefill call enqueues (with cu_seqlens; a call of
// equal-length sequences skips the first, the chunk bases), and its chunk length.
int tc_launches(int T_total, int N, int H, int d, const kda_options* opt);
int tc_chunk(const kda_options* opt);

// Enqueue the tensor-core prefill on stream s (arguments already checked).
cudaError_t launch_prefill_tc(const PrefillArgs& a, const kda_options* opt, cudaStream_t s);

}  // namespace kda
