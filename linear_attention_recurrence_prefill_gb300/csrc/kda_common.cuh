// kda_common.cuh -- small device helpers and launch prototypes shared by the
// translation units of libkda.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

// ---------------------------------------------------------------- element I/O
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------- arguments
// Everything a prefill kernel needs, passed by value.  Sizes that can exceed
// 2^31 elements are indexed in 64-bit inside the kernels.
struct PrefillArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* log_alpha;
  const void* beta;
  const float* S0;
  const int32_t* cu_seqlens;
  void* o;
  float* S_T;
  const void* gate;
  const float* norm_weight;
  int* status;
  int N, T_total, H, d;
  int l2norm_qk, beta_is_logit, decay_mode;
  float g_min, q_scale, eps_l2, eps_norm;
  float* snapshots;          // NULL: no state snapshots
  int snapshot_every;        // tokens between snapshots (a multiple of 64)
  int snapshot_slots;        // slots per sequence in `snapshots`
};

// Slot of the snapshot taken after `done` tokens of a sequence, or -1.
__device__ __forceinline__ int snapshot_slot(const PrefillArgs& a, int done) {
  if (!a.snapshots || done <= 0 || done % a.snapshot_every != 0) return -1;
  const int m = done / a.snapshot_every - 1;
  return m < a.snapshot_slots ? m : -1;
}

struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* log_alpha;
  const void* beta;
  float* S;
  void* o;
  const void* gate;
  const float* norm_weight;
  int N, H, d;
  int l2norm_qk, beta_is_logit, decay_mode;
  float g_min, q_scale, eps_l2, eps_norm;
};

// log alpha of token-head row `row` (token * H + head), key channel c, under
// the decay mode (KDA_DECAY_*), before the floor.
// Written without branches so that the load issues with the token's others.
__device__ __forceinline__ float log_alpha_at(const float* la, int mode, size_t row, int d,
                                              int c) {
  const size_t off = mode == KDA_DECAY_CHANNEL ? row * d + c : row;
  return mode == KDA_DECAY_NONE ? 0.f : la[off];
}

// Token range [t0, t1) of sequence n.
__device__ __forceinline__ void seq_range(const int32_t* cu, int N, int T_total, int n,
                                          int& t0, int& t1) {
  if (cu) {
    t0 = cu[n];
    t1 = cu[n + 1];
  } else {
    const int L = T_total / N;
    t0 = n * L;
    t1 = t0 + L;
  }
}

// ---------------------------------------------------------------- launchers
// Each returns a cudaError_t from the launch.
cudaError_t launch_prefill_simt(const PrefillArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_gated_rmsnorm(const void* o, const void* gate, const float* w, void* y,
                                 long long rows_heads, int d, float eps, int dtype,
                                 cudaStream_t s);

// Device address of the library's status word on the current device.
int* status_word();

// Unique id of the calling thread's current CUDA context, 0 if there is none
// (or the driver cannot say).  Device addresses of the library's own device
// variables are cached per (device, context id): a device reset creates a new
// context, in which those variables live at new addresses.
unsigned long long current_context_id();

// Every host-side check of kda_prefill (everything but the workspace): returns
// KDA_OK and the path (KDA_IMPL_SIMT or KDA_IMPL_TC) and the number of
// snapshot slots per sequence, or the status code kda_prefill returns.
int check_prefill(const void* q, const void* k, const void* v, const float* log_alpha,
                  const void* beta, const float* S0, const int32_t* cu_seqlens, int N,
                  const void* o, const float* S_T, int T_total, int H, int d_k, int d_v,
                  int dtype, const kda_options* op, int* path_out, int* snap_slots_out);

}  // namespace kda
