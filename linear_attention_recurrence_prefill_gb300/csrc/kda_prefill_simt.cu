// kda_prefill_simt.cu -- chunked KDA prefill on CUDA cores, fp32 arithmetic.
//
// One CTA walks one (sequence, head) pair chunk by chunk (16 tokens), keeping
// the d x d state in shared memory.  Inside a chunk the work is parallel; the
// chunks follow one another through the state ("Kimi K3's hybrid block, from
// first principles", section "From linear attention to the delta rule").
//
// Chunk algebra (exactly the token recurrence, regrouped).  With state S at the
// chunk start, g_t the inclusive running sum of the clamped log-decays from the
// chunk start and G_t = exp(g_t) per key channel:
//   K~_t = G_t * k_t,  Q~_t = G_t * q_t,  K-_t = k_t / G_t,  K^_t = (G_C / G_t) * k_t
//   A    = Diag(beta) * strictly_lower(K~ K-^T)
//   T    = (I + A)^-1 Diag(beta),   W = T K~,   U~ = T V
//   U    = U~ - W S                         (the per-token "write errors")
//   O    = Q~ S + incl_lower(Q~ K-^T) U
//   S   <- Diag(G_C) S + K^^T U
// Over 16 tokens g_t >= -80 because log alpha >= -5, so 1/G_t <= e^80 stays
// finite in fp32; this is the floor the pages give for the 16-token tiles
// ("Kimi K3", section "Forgetting different features at different rates").
//
// This path is the fp32 reference implementation on the GPU (tolerance 1e-4
// against the fp64 oracle) and the fallback for shapes the tensor-core path
// does not cover.  It needs no workspace.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kC = 16;
constexpr int kThreads = 256;
static_assert(kC * kC == kThreads, "one thread per entry of the chunk Gram matrix");

template <int D>
struct SimtSmem {  // offsets in floats
  static constexpr int S = 0;               // [D][D]   state
  static constexpr int Qt = S + D * D;      // [C][D]   q -> q^ -> Q~
  static constexpr int Kt = Qt + kC * D;    // [C][D]   k -> k^ -> K~
  static constexpr int Kb = Kt + kC * D;    // [C][D]   K-
  static constexpr int Kh = Kb + kC * D;    // [C][D]   K^
  static constexpr int Vb = Kh + kC * D;    // [C][D]   v
  static constexpr int W = Vb + kC * D;     // [C][D]   W
  static constexpr int Ut = W + kC * D;     // [C][D]   U~, then U
  static constexpr int G = Ut + kC * D;     // [C][D]   running log-decay
  static constexpr int A = G + kC * D;      // [C][C]
  static constexpr int P = A + kC * kC;     // [C][C]
  static constexpr int Tm = P + kC * kC;    // [C][C]
  static constexpr int beta = Tm + kC * kC; // [C]
  static constexpr int gam = beta + kC;     // [D]     G_C
  static constexpr int red = gam + D;       // [warps][C] partial sums of squares
  static constexpr int hist = red + (kThreads / 32) * kC;  // [3][3][D] raw rows before
                                            // the chunk (short convolution), oldest first
  static constexpr int total = hist + 9 * D;
};

template <int D, typename T>
__global__ void __launch_bounds__(kThreads) prefill_simt_kernel(PrefillArgs a) {
  extern __shared__ float4 smem_f4[];
  float* sm = reinterpret_cast<float*>(smem_f4);
  using L = SimtSmem<D>;
  float* S = sm + L::S;
  float* Qt = sm + L::Qt;
  float* Kt = sm + L::Kt;
  float* Kb = sm + L::Kb;
  float* Kh = sm + L::Kh;
  float* Vb = sm + L::Vb;
  float* W = sm + L::W;
  float* Ut = sm + L::Ut;
  float* G = sm + L::G;
  float* sA = sm + L::A;
  float* sP = sm + L::P;
  float* sT = sm + L::Tm;
  float* sbeta = sm + L::beta;
  float* sgam = sm + L::gam;
  float* red = sm + L::red;
  float* hist = sm + L::hist;

  constexpr int RG = kThreads / D;  // row groups in the C x D work split
  constexpr int RPT = kC / RG;      // chunk rows per thread
  constexpr int RS = D / RG;        // state rows per thread in the update

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x % a.H;
  const int n = blockIdx.x / a.H;
  const size_t H = (size_t)a.H;
  int t0, t1;
  seq_range(a.cu_seqlens, a.N, a.T_total, n, t0, t1);
  if (t0 < 0 || t1 < t0 || t1 > a.T_total) {  // malformed cu_seqlens: report, touch nothing
    if (tid == 0) atomicExch(a.status, KDA_ERR_SHAPE);
    return;
  }

  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  const T* beta = static_cast<const T*>(a.beta);
  const T* gate = static_cast<const T*>(a.gate);
  T* o = static_cast<T*>(a.o);

  const size_t sbase = ((size_t)n * H + h) * (size_t)(D * D);
  for (int e = tid; e < D * D; e += kThreads) S[e] = a.S0 ? a.S0[sbase + e] : 0.f;

  const int col = tid % D;
  const int grp = tid / D;

  // short convolution: taps of this thread's column (the same column in every
  // one of its chunk elements, since kThreads is a multiple of D), and the raw
  // rows before the sequence
  constexpr int E = kC * D / kThreads;  // chunk elements per thread
  float4 cw[3];
  if (a.conv_weight) {
    for (int X = 0; X < 3; ++X)
      cw[X] = *reinterpret_cast<const float4*>(a.conv_weight + (((size_t)X * H + h) * D + col) * 4);
    const T* cs = static_cast<const T*>(a.conv_state);
    for (int e = tid; e < 9 * D; e += kThreads) {  // e = (X * 3 + j) * D + c
      const int Xj = e / D, c = e % D;
      hist[e] = cs ? to_f32(cs[(((size_t)n * 9 + Xj) * H + h) * D + c]) : 0.f;
    }
  }

  for (int c0 = t0; c0 < t1; c0 += kC) {
    // 1. load the chunk (tokens past the sequence end are identity steps)
    for (int e = tid; e < kC * D; e += kThreads) {
      const int t = e / D, c = e % D;
      const int tok = c0 + t;
      float qv = 0.f, kv = 0.f, vv = 0.f, la = 0.f;
      if (tok < t1) {
        const size_t gi = ((size_t)tok * H + h) * D + c;
        qv = to_f32(q[gi]);
        kv = to_f32(k[gi]);
        vv = to_f32(v[gi]);
        la = log_alpha_at(a.log_alpha, a.decay_mode, (size_t)tok * H + h, D, c);
        if (a.decay_from_logit)
          la = log_alpha_from_logit(la, a.decay_scale, a.decay_bias, h, D, c, a.g_min);
        la = fminf(fmaxf(la, a.g_min), 0.f);
      }
      Qt[e] = qv;
      Kt[e] = kv;
      Vb[e] = vv;
      G[e] = la;
    }
    if (tid < kC) {
      const int tok = c0 + tid;
      float b = 0.f;
      if (tok < t1) {
        b = to_f32(beta[(size_t)tok * H + h]);
        if (a.beta_is_logit) b = sigmoidf_(b);
      }
      sbeta[tid] = b;
    }
    __syncthreads();

    // 1b. short convolution + Swish of q, k, v over the raw rows (the chunk's
    //     and the three before it), the output held in the data type as a
    //     separate convolution layer would hand it over; rows past the
    //     sequence end stay identity steps whatever their values (beta = 0, no
    //     decay)
    if (a.conv_weight) {
      float out[3][E], raw[3][E];
      float* buf[3] = {Qt, Kt, Vb};
#pragma unroll
      for (int i = 0; i < E; ++i) {
        const int t = (tid + kThreads * i) / D;
#pragma unroll
        for (int X = 0; X < 3; ++X) {
          float x[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = t - 3 + j;
            x[j] = r >= 0 ? buf[X][r * D + col] : hist[(X * 3 + 3 + r) * D + col];
          }
          raw[X][i] = x[3];
          // held in the data type
          out[X][i] = to_f32(from_f32<T>(conv4_swish(cw[X], x[0], x[1], x[2], x[3])));
        }
      }
      __syncthreads();
#pragma unroll
      for (int i = 0; i < E; ++i) {
        const int t = (tid + kThreads * i) / D;
#pragma unroll
        for (int X = 0; X < 3; ++X) {
          buf[X][t * D + col] = out[X][i];
          if (t >= kC - 3) hist[(X * 3 + t - (kC - 3)) * D + col] = raw[X][i];
        }
      }
      __syncthreads();
    }

    // 2. L2 norms of q and k rows (one warp per row), running sum of log-decay
    if (a.l2norm_qk) {
      for (int r = warp; r < 2 * kC; r += kThreads / 32) {
        float* row = (r < kC ? Qt : Kt) + (r % kC) * D;
        float ss = 0.f;
        for (int c = lane; c < D; c += 32) ss += row[c] * row[c];
        ss = warp_sum(ss) + a.eps_l2;
        const float inv = ss > 0.f ? 1.0f / sqrtf(ss) : 0.f;
        for (int c = lane; c < D; c += 32) row[c] *= inv;
      }
    }
    if (tid < D) {
      float g = 0.f;
      for (int t = 0; t < kC; ++t) {
        g += G[t * D + tid];
        G[t * D + tid] = g;
      }
    }
    __syncthreads();

    // 3. decay-rescaled operands
    for (int e = tid; e < kC * D; e += kThreads) {
      const int c = e % D;
      const float g = G[e], gl = G[(kC - 1) * D + c];
      const float kk = Kt[e], qq = Qt[e];
      const float eg = expf(g);
      Kt[e] = kk * eg;
      Qt[e] = qq * eg;
      Kb[e] = kk * expf(-g);
      Kh[e] = kk * expf(gl - g);
    }
    if (tid < D) sgam[tid] = expf(G[(kC - 1) * D + tid]);
    __syncthreads();

    // 4. A = Diag(beta) strictly_lower(K~ K-^T), P = incl_lower(Q~ K-^T)
    {
      const int t = tid / kC, j = tid % kC;
      float dk = 0.f, dq = 0.f;
      for (int cc = 0; cc < D; ++cc) {
        const int c = (cc + j) & (D - 1);  // rotate to spread shared-memory banks
        const float kb = Kb[j * D + c];
        dk += Kt[t * D + c] * kb;
        dq += Qt[t * D + c] * kb;
      }
      sA[tid] = (j < t) ? sbeta[t] * dk : 0.f;
      sP[tid] = (j <= t) ? dq : 0.f;
    }
    __syncthreads();

    // 5. T = (I + A)^-1 Diag(beta), one thread per column, forward substitution
    if (tid < kC) {
      const int j = tid;
      float x[kC];
#pragma unroll
      for (int t = 0; t < kC; ++t) {
        float acc = (t == j) ? 1.f : 0.f;
#pragma unroll
        for (int m = 0; m < t; ++m) acc -= sA[t * kC + m] * x[m];
        x[t] = acc;
      }
      const float bj = sbeta[j];
#pragma unroll
      for (int t = 0; t < kC; ++t) sT[t * kC + j] = x[t] * bj;
    }
    __syncthreads();

    // 6. W = T K~, U~ = T V
    {
      float w[RPT], u[RPT];
#pragma unroll
      for (int r = 0; r < RPT; ++r) w[r] = u[r] = 0.f;
      for (int j = 0; j < kC; ++j) {
        const float kt = Kt[j * D + col], vv = Vb[j * D + col];
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
          const float tm = sT[(grp * RPT + r) * kC + j];
          w[r] += tm * kt;
          u[r] += tm * vv;
        }
      }
#pragma unroll
      for (int r = 0; r < RPT; ++r) {
        W[(grp * RPT + r) * D + col] = w[r];
        Ut[(grp * RPT + r) * D + col] = u[r];
      }
    }
    __syncthreads();

    // 7. U = U~ - W S and O = Q~ S (+ P U below); S is read here, written in 8
    float acc_o[RPT];
    {
      float acc_u[RPT];
#pragma unroll
      for (int r = 0; r < RPT; ++r) {
        acc_u[r] = Ut[(grp * RPT + r) * D + col];
        acc_o[r] = 0.f;
      }
      for (int c = 0; c < D; c += 4) {
        const float s0 = S[(c + 0) * D + col], s1 = S[(c + 1) * D + col];
        const float s2 = S[(c + 2) * D + col], s3 = S[(c + 3) * D + col];
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
          const int t = grp * RPT + r;
          const float4 w4 = *reinterpret_cast<const float4*>(&W[t * D + c]);
          const float4 q4 = *reinterpret_cast<const float4*>(&Qt[t * D + c]);
          acc_u[r] -= w4.x * s0 + w4.y * s1 + w4.z * s2 + w4.w * s3;
          acc_o[r] += q4.x * s0 + q4.y * s1 + q4.z * s2 + q4.w * s3;
        }
      }
#pragma unroll
      for (int r = 0; r < RPT; ++r) Ut[(grp * RPT + r) * D + col] = acc_u[r];
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
      const int t = grp * RPT + r;
      float acc = acc_o[r];
      for (int j = 0; j <= t; ++j) acc += sP[t * kC + j] * Ut[j * D + col];
      acc_o[r] = acc * a.q_scale;
    }

    // 8. S <- Diag(G_C) S + K^^T U
    {
      float uj[kC];
#pragma unroll
      for (int j = 0; j < kC; ++j) uj[j] = Ut[j * D + col];
      for (int rr = 0; rr < RS; ++rr) {
        const int c = grp * RS + rr;
        float s = S[c * D + col] * sgam[c];
#pragma unroll
        for (int j = 0; j < kC; ++j) s += Kh[j * D + c] * uj[j];
        S[c * D + col] = s;
      }
    }

    // 9. write o, or y = RMSNorm(o) * w * sigmoid(gate)
    float inv[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) inv[r] = 1.f;
    if (gate) {
#pragma unroll
      for (int r = 0; r < RPT; ++r) {
        const float ss = warp_sum(acc_o[r] * acc_o[r]);
        if (lane == 0) red[warp * kC + grp * RPT + r] = ss;
      }
      __syncthreads();
#pragma unroll
      for (int r = 0; r < RPT; ++r) {
        const int t = grp * RPT + r;
        float tot = 0.f;
        for (int w2 = 0; w2 < D / 32; ++w2) tot += red[(grp * (D / 32) + w2) * kC + t];
        inv[r] = rsqrtf(tot / D + a.eps_norm);
      }
    }
    const float nw = (gate && a.norm_weight) ? a.norm_weight[col] : 1.f;
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
      const int tok = c0 + grp * RPT + r;
      if (tok < t1) {
        const size_t gi = ((size_t)tok * H + h) * D + col;
        float y = acc_o[r];
        if (gate) y = y * inv[r] * nw * sigmoidf_(to_f32(gate[gi]));
        o[gi] = from_f32<T>(y);
      }
    }
    __syncthreads();
    // state snapshot after a multiple of snapshot_every tokens
    const int m = (c0 + kC <= t1) ? snapshot_slot(a, c0 + kC - t0) : -1;
    if (m >= 0) {
      float* dst = a.snapshots + (((size_t)n * a.snapshot_slots + m) * H + h) * (size_t)(D * D);
      for (int e = tid; e < D * D; e += kThreads) dst[e] = S[e];
    }
  }

  for (int e = tid; e < D * D; e += kThreads) a.S_T[sbase + e] = S[e];
}

template <int D, typename T>
cudaError_t launch_simt(const PrefillArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(float) * SimtSmem<D>::total;
  auto kern = prefill_simt_kernel<D, T>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)a.N * (unsigned)a.H;
  if (grid == 0) return cudaSuccess;
  kern<<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_simt_dtype(const PrefillArgs& a, cudaStream_t s) {
  switch (a.d) {
    case 32: return launch_simt<32, T>(a, s);
    case 64: return launch_simt<64, T>(a, s);
    case 128: return launch_simt<128, T>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs& a, int dtype, cudaStream_t s) {
  return dtype == KDA_BF16 ? launch_simt_dtype<__nv_bfloat16>(a, s)
                           : launch_simt_dtype<float>(a, s);
}

}  // namespace kda
