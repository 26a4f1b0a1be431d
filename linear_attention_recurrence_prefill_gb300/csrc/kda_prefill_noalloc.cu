// kda_prefill_noalloc.cu -- kda_prefill_noalloc: the tensor-core prefill with
// its scratch memory in a fixed array that lives inside the library, for
// callers that cannot allocate device memory themselves.
//
// The scratch is a file-scope device array of KDA_NOALLOC_SCRATCH_BYTES
// (64 MiB).  Every GPU that loads libkda.so holds it until the process exits.
// In host code the array's name is only a host-side stand-in, never a device
// address, so its device address is looked up with cudaGetSymbolAddress, with
// the device current, once per device (and again only if the device's context
// was replaced, e.g. after a device reset), and handed to the kernels.
#include <string.h>

#include <mutex>

#include "kda_common.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};
unsigned long long g_scratch_ctx[kMaxDevices] = {0};

// Device address of the scratch array on the current device (set up on the
// first call per device and context).  Returns nullptr if the runtime refuses.
void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  const unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> g(g_scratch_mutex);
  if (id != 0 && g_scratch_ctx[dev] == id && g_scratch_addr[dev]) return g_scratch_addr[dev];
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
  g_scratch_addr[dev] = p;
  g_scratch_ctx[dev] = current_context_id();
  return p;
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
  // only the tensor-core path (chunk 64) uses scratch; anything else is not
  // offered here
  if (op.impl != KDA_IMPL_AUTO && op.impl != KDA_IMPL_TC) return KDA_ERR_UNSUPPORTED;
  if (op.chunk != 0 && op.chunk != 64) return KDA_ERR_UNSUPPORTED;
  op.impl = KDA_IMPL_TC;
  // the same argument checks as kda_prefill, before anything is sized
  int path = 0;
  int rc = kda::check_prefill(q, k, v, log_alpha, beta, S0, cu_seqlens, N, o, S_T, T_total, H,
                              d_k, d_v, dtype, &op, &path, nullptr);
  if (rc != KDA_OK) return rc;
  if (path != KDA_IMPL_TC) return KDA_ERR_UNSUPPORTED;
  // sizes whose scratch does not fit the built-in array are refused up front
  const size_t need = kda::tc_workspace_bytes(T_total, N, H, d_k, &op);
  if (need == 0) return KDA_ERR_UNSUPPORTED;
  if (need > (size_t)KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_WORKSPACE;
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
