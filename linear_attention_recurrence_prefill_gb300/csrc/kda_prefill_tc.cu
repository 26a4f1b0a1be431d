// kda_prefill_tc.cu -- tcgen05 tensor-core prefill (not built yet: the entry
// points report the path as unavailable so that dispatch uses the SIMT path).
#include "kda_tc.cuh"

namespace kda {

bool tc_prefill_supported(int, int, int) { return false; }

size_t tc_workspace_bytes(int, int, int, int, const kda_options*) { return 0; }

int tc_launches(int, int, int, int, const kda_options*) { return 0; }
int tc_chunk(const kda_options*) { return 64; }

cudaError_t launch_prefill_tc(const PrefillArgs&, const kda_options*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace kda
