// kda_prefill_noalloc.cu -- kda_prefill_noalloc: the tensor-core prefill with
// its scratch memory in a fixed array that lives inside the library, for
// callers that cannot allocate device memory themselves.
//
// The scratch is a file-scope device array of KDA_NOALLOC_SCRATCH_BYTES
// (64 MiB).  Every GPU that loads libkda.so holds it until the process exits.
// In host code the array's name is only a host-side stand-in, never a device
// address, so its device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and handed to the kernels.
#include <string.h>

#include "kda_common.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (set up on the
// first call per device).  Returns nullptr if the runtime refuses.
void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace
}  // namespace kda

extern "C" int kda_prefill_noalloc(const void* q, const void* k, const void* v,
                                   const float* log_alpha, const void* beta, const float* S0,
                                   const int32_t* cu_seqlens, int N, void* o, float* S_T,
                                   int T_total, int H, int d_k, int d_v, int dtype,
                                   const kda_options* opt, kda_stream_t stream) {
  kda_options op;
  if (opt) memcpy(&op, opt, sizeof(op));
  else kda_options_init(&op);
  if (op.impl != KDA_IMPL_AUTO && op.impl != KDA_IMPL_TC) return KDA_ERR_UNSUPPORTED;
  op.impl = KDA_IMPL_TC;
  if (N < 1 || H < 1 || T_total < 0) return KDA_ERR_SHAPE;
  if (dtype != KDA_BF16 || d_k != 128 || d_v != 128) return KDA_ERR_UNSUPPORTED;
  // sizes whose scratch does not fit the built-in array are refused up front
  const size_t need = kda_prefill_workspace_size(T_total, N, H, d_k, d_v, &op);
  if (need == 0 || need > (size_t)KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_WORKSPACE;
  void* scratch = kda::scratch_address();
  if (!scratch) return KDA_ERR_CUDA;
  op.workspace = scratch;
  op.workspace_bytes = (size_t)KDA_NOALLOC_SCRATCH_BYTES;
  // Every byte the kernels read from the scratch is written earlier in the
  // same call (chunk table, then one operand block per chunk and head), so
  // nothing has to be cleared between calls.
  return kda_prefill(q, k, v, log_alpha, beta, S0, cu_seqlens, N, o, S_T, T_total, H, d_k, d_v,
                     dtype, &op, stream);
}
