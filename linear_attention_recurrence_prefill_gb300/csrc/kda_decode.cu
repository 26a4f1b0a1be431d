// kda_decode.cu -- one recurrent KDA token for N sequences (state in place),
// and the standalone per-head RMSNorm x sigmoid-gate epilogue.
//
// Decode is bound by HBM: each head's d x d fp32 state is read once and
// written once.  One CTA per (sequence, head); the state sits in registers as
// float4 rows between the read pass and the write pass, loaded and stored as
// coalesced 16-byte accesses (a warp covers whole 512-byte rows for d = 128).
//
// With S' = Diag(a) S (fade), u = S'^T k and r = S'^T q are both reductions over
// the key channels, taken in the same pass.  Then
//   S_new = S' + beta k (v - u)^T     and     o = S_new^T q = r + (k.q) beta (v - u)
// so q reads the updated state without a second pass over it ("Kimi K3,
// explained", section "Kimi Delta Attention: making the radical option work":
// k and v update S(t-1), q reads the updated S(t)).
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kDecThreads = 256;

// kConv: the short convolution runs on the token's q, k, v first (a separate
// instantiation, so that the default one carries none of its registers).
template <int D, typename T, bool kConv>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(DecodeArgs a) {
  constexpr int C4 = D / 4;               // float4 per state row
  constexpr int RPP = kDecThreads / C4;   // rows per pass
  constexpr int PASSES = D / RPP;         // passes over the rows
  static_assert(RPP * C4 == kDecThreads && PASSES * RPP == D, "decode tiling");

  __shared__ float sq[D], sk[D], sa[D], sv[D], so[D];
  __shared__ __align__(16) float sw[D];  // read as float4
  __shared__ __align__(16) float red_u[RPP][D];
  __shared__ __align__(16) float red_r[RPP][D];
  __shared__ float misc[8];

  const int tid = threadIdx.x;
  const int unit = blockIdx.x;  // n * H + h
  const int c4 = tid % C4, r0 = tid / C4;

  float4* Sp = reinterpret_cast<float4*>(a.S) + (size_t)unit * (size_t)(D * C4);
  float4 s[PASSES];
#pragma unroll
  for (int p = 0; p < PASSES; ++p) s[p] = Sp[(size_t)(r0 + p * RPP) * C4 + c4];

  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  const size_t base = (size_t)unit * D;
  // every global load of the token (and beta) is issued before the first barrier
  float qv = 0.f, kv = 0.f, vv = 0.f, lav = 0.f, bv = 0.f;
  float win[3][3];  // short convolution: raw rows of the 3 previous tokens
  float4 cw[3];     // and this channel's taps
  T* cs = static_cast<T*>(a.conv_state);
  const int n = unit / a.H, h = unit - n * a.H;
  if (tid < D) {
    qv = to_f32(q[base + tid]);
    kv = to_f32(k[base + tid]);
    vv = to_f32(v[base + tid]);
    lav = log_alpha_at(a.log_alpha, a.decay_mode, (size_t)unit, D, tid);
    if constexpr (kConv) {
#pragma unroll
      for (int X = 0; X < 3; ++X) {
        cw[X] = *reinterpret_cast<const float4*>(a.conv_weight +
                                                 (((size_t)X * a.H + h) * D + tid) * 4);
#pragma unroll
        for (int j = 0; j < 3; ++j)
          win[X][j] = cs ? to_f32(cs[(((size_t)n * 9 + X * 3 + j) * a.H + h) * D + tid]) : 0.f;
      }
    }
  }
  if (tid == 0) bv = to_f32(static_cast<const T*>(a.beta)[unit]);
  if (tid < D) {
    if constexpr (kConv) {  // conv over (3 previous rows, this row), then Swish,
      const float raw[3] = {qv, kv, vv};  // held in the data type
      float y[3];
#pragma unroll
      for (int X = 0; X < 3; ++X) {
        y[X] = to_f32(from_f32<T>(conv4_swish(cw[X], win[X][0], win[X][1], win[X][2], raw[X])));
        if (cs) {  // the window that ends with this token
          const size_t wb = ((size_t)n * 9 + X * 3) * a.H + h;
          cs[(wb + 0 * (size_t)a.H) * D + tid] = from_f32<T>(win[X][1]);
          cs[(wb + 1 * (size_t)a.H) * D + tid] = from_f32<T>(win[X][2]);
          cs[(wb + 2 * (size_t)a.H) * D + tid] = from_f32<T>(raw[X]);
        }
      }
      qv = y[0];
      kv = y[1];
      vv = y[2];
    }
    if (a.decay_from_logit)
      lav = log_alpha_from_logit(lav, a.decay_scale, a.decay_bias, h, D, tid, a.g_min);
    sq[tid] = qv;
    sk[tid] = kv;
    sv[tid] = vv;
    sa[tid] = expf(fminf(fmaxf(lav, a.g_min), 0.f));
  }
  __syncthreads();
  if (tid < 32) {
    float ssq = 0.f, ssk = 0.f, skq = 0.f;
    for (int c = tid; c < D; c += 32) {
      ssq += sq[c] * sq[c];
      ssk += sk[c] * sk[c];
      skq += sk[c] * sq[c];
    }
    ssq = warp_sum(ssq);
    ssk = warp_sum(ssk);
    skq = warp_sum(skq);
    if (tid == 0) {
      float b = bv;
      if (a.beta_is_logit) b = sigmoidf_(b);
      float iq = 1.f, ik = 1.f;
      if (a.l2norm_qk) {
        iq = (ssq + a.eps_l2) > 0.f ? 1.0f / sqrtf(ssq + a.eps_l2) : 0.f;
        ik = (ssk + a.eps_l2) > 0.f ? 1.0f / sqrtf(ssk + a.eps_l2) : 0.f;
      }
      misc[0] = iq;
      misc[1] = ik;
      misc[2] = skq * iq * ik;  // k^ . q^
      misc[3] = b;
    }
  }
  __syncthreads();

  // fade, then partial u = S'^T k and r = S'^T q over this thread's rows
  float4 pu = make_float4(0.f, 0.f, 0.f, 0.f), pr = pu;
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    const int row = r0 + p * RPP;
    const float av = sa[row], kr = sk[row], qr = sq[row];
    s[p].x *= av; s[p].y *= av; s[p].z *= av; s[p].w *= av;
    pu.x += s[p].x * kr; pu.y += s[p].y * kr; pu.z += s[p].z * kr; pu.w += s[p].w * kr;
    pr.x += s[p].x * qr; pr.y += s[p].y * qr; pr.z += s[p].z * qr; pr.w += s[p].w * qr;
  }
  *reinterpret_cast<float4*>(&red_u[r0][c4 * 4]) = pu;
  *reinterpret_cast<float4*>(&red_r[r0][c4 * 4]) = pr;
  __syncthreads();
  if (tid < D) {
    float u = 0.f, r = 0.f;
#pragma unroll
    for (int rr = 0; rr < RPP; ++rr) {
      u += red_u[rr][tid];
      r += red_r[rr][tid];
    }
    const float iq = misc[0], ik = misc[1], kq = misc[2], b = misc[3];
    u *= ik;
    r *= iq;
    const float w = b * (sv[tid] - u);
    sw[tid] = w * ik;  // the update adds k^ w^T = k (ik w)^T
    so[tid] = a.q_scale * (r + kq * w);
  }
  __syncthreads();

  // write S_new = S' + k (ik w)^T
#pragma unroll
  for (int p = 0; p < PASSES; ++p) {
    const int row = r0 + p * RPP;
    const float kr = sk[row];
    const float4 w4 = *reinterpret_cast<const float4*>(&sw[c4 * 4]);
    s[p].x += kr * w4.x; s[p].y += kr * w4.y; s[p].z += kr * w4.z; s[p].w += kr * w4.w;
    Sp[(size_t)row * C4 + c4] = s[p];
  }

  // output o (or the gated RMSNorm of it)
  T* o = static_cast<T*>(a.o);
  if (a.gate) {
    if (tid < 32) {
      float ss = 0.f;
      for (int c = tid; c < D; c += 32) ss += so[c] * so[c];
      ss = warp_sum(ss);
      if (tid == 0) misc[4] = rsqrtf(ss / D + a.eps_norm);
    }
    __syncthreads();
    if (tid < D) {
      const T* gate = static_cast<const T*>(a.gate);
      const float nw = a.norm_weight ? a.norm_weight[tid] : 1.f;
      o[base + tid] = from_f32<T>(so[tid] * misc[4] * nw * sigmoidf_(to_f32(gate[base + tid])));
    }
  } else if (tid < D) {
    o[base + tid] = from_f32<T>(so[tid]);
  }
}

// y = o / sqrt(mean(o^2) + eps) * w * sigmoid(gate); one warp per (row, head).
template <int D, typename T>
__global__ void gated_rmsnorm_kernel(const T* o, const T* __restrict__ gate,
                                     const float* __restrict__ w, T* y, long long units,
                                     float eps) {
  constexpr int E = D / 32;
  const long long unit = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (unit >= units) return;
  const size_t base = (size_t)unit * D;
  float x[E];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    x[i] = to_f32(o[base + lane + 32 * i]);
    ss += x[i] * x[i];
  }
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / D + eps);
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int j = lane + 32 * i;
    const float nw = w ? w[j] : 1.f;
    y[base + j] = from_f32<T>(x[i] * inv * nw * sigmoidf_(to_f32(gate[base + j])));
  }
}

template <int D, typename T>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t s) {
  const unsigned grid = (unsigned)a.N * (unsigned)a.H;
  if (a.conv_weight) decode_kernel<D, T, true><<<grid, kDecThreads, 0, s>>>(a);
  else decode_kernel<D, T, false><<<grid, kDecThreads, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_decode_dtype(const DecodeArgs& a, cudaStream_t s) {
  switch (a.d) {
    case 32: return launch_decode_t<32, T>(a, s);
    case 64: return launch_decode_t<64, T>(a, s);
    case 128: return launch_decode_t<128, T>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int D, typename T>
cudaError_t launch_rms_t(const void* o, const void* gate, const float* w, void* y,
                         long long units, float eps, cudaStream_t s) {
  constexpr int kWarps = 8;
  const long long blocks = (units + kWarps - 1) / kWarps;
  if (blocks == 0) return cudaSuccess;
  gated_rmsnorm_kernel<D, T><<<(unsigned)blocks, kWarps * 32, 0, s>>>(
      static_cast<const T*>(o), static_cast<const T*>(gate), w, static_cast<T*>(y), units, eps);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_rms_dtype(const void* o, const void* gate, const float* w, void* y,
                             long long units, int d, float eps, cudaStream_t s) {
  switch (d) {
    case 32: return launch_rms_t<32, T>(o, gate, w, y, units, eps, s);
    case 64: return launch_rms_t<64, T>(o, gate, w, y, units, eps, s);
    case 128: return launch_rms_t<128, T>(o, gate, w, y, units, eps, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, int dtype, cudaStream_t s) {
  if ((long long)a.N * a.H == 0) return cudaSuccess;
  return dtype == KDA_BF16 ? launch_decode_dtype<__nv_bfloat16>(a, s)
                           : launch_decode_dtype<float>(a, s);
}

cudaError_t launch_gated_rmsnorm(const void* o, const void* gate, const float* w, void* y,
                                 long long rows_heads, int d, float eps, int dtype,
                                 cudaStream_t s) {
  return dtype == KDA_BF16
             ? launch_rms_dtype<__nv_bfloat16>(o, gate, w, y, rows_heads, d, eps, s)
             : launch_rms_dtype<float>(o, gate, w, y, rows_heads, d, eps, s);
}

}  // namespace kda
