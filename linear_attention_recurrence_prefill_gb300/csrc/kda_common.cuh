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
  int decay_from_logit;      // 1: log_alpha holds decay logits
  const float* decay_scale;  // A [H] or NULL
  const float* decay_bias;   // b [H][d] or NULL
  const float* conv_weight;  // [3][H][d][4] or NULL (no short convolution)
  const void* conv_state;    // [N][3][3][H][d] (dtype) or NULL (zeros)
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
  int decay_from_logit;
  const float* decay_scale;
  const float* decay_bias;
  const float* conv_weight;
  void* conv_state;          // read and advanced by one token
};

// log alpha from the decay logit z of key channel c of head h: the bounded
// sigmoid g_min * sigmoid(A_h (z + b_{h,c})), within [g_min, 0].
__device__ __forceinline__ float log_alpha_from_logit(float z, const float* scale,
                                                      const float* bias, int h, int d, int c,
                                                      float g_min) {
  const float A = scale ? scale[h] : 1.f;
  const float b = bias ? bias[(size_t)h * d + c] : 0.f;
  return g_min / (1.f + __expf(-A * (z + b)));
}

// e^t for t in [-80, 80] from IEEE fp32 operations only, so that any
// implementation of the same steps gets the same bits: Cody and Waite's range
// reduction t = n ln2 + r (n = rint(t log2 e); ln2 split into a 14-bit head,
// exact in n * head, and a tail), the Taylor polynomial of e^r to degree 6
// (|r| <= 0.35) by Horner's rule, then the exact scaling by 2^n.
__device__ __forceinline__ float exp_ieee(float t) {
  const float n = rintf(t * 0x1.715476p+0f);
  float r = fmaf(-n, 0x1.62e4p-1f, t);
  r = fmaf(-n, 0x1.7f7d1cp-20f, r);
  float p = 0x1.6c16c2p-10f;      // 1/720
  p = fmaf(p, r, 0x1.111112p-7f);  // 1/120
  p = fmaf(p, r, 0x1.555556p-5f);  // 1/24
  p = fmaf(p, r, 0x1.555556p-3f);  // 1/6
  p = fmaf(p, r, 0.5f);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  return p * __int_as_float(((int)n + 127) << 23);
}

// The short convolution of one channel (taps w.x .. w.w weigh the rows oldest
// first: x0 three tokens back, x3 the token's own row) followed by Swish,
// y sigmoid(y) with sigmoid(y) = 1 / (1 + e^-y), the exponent clamped to
// [-80, 80].  Every path computes it in this one fixed fp32 order (IEEE
// multiply, fused multiply-add and division), so the value each path stores in
// the data type is the same to the bit.
__device__ __forceinline__ float conv4_swish(float4 w, float x0, float x1, float x2, float x3) {
  float y = w.w * x3;
  y = fmaf(w.z, x2, y);
  y = fmaf(w.y, x1, y);
  y = fmaf(w.x, x0, y);
  const float t = fminf(fmaxf(-y, -80.f), 80.f);
  return y * __fdiv_rn(1.0f, 1.0f + exp_ieee(t));
}

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
