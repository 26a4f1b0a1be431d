// kda_prefill_tc.cu -- chunked KDA prefill on the tcgen05 tensor cores (sm_103a).
//
// The layer is processed in chunks of C = 64 tokens, each split into four
// 16-token tiles ("KDA trains chunkwise, in parallel inside a chunk and
// recurrently across chunks ... Over a 16-token tile the cumulative log-decay
// stays within (-80, 0), so the rescaling factors fit in BF16's range and every
// tile, including the diagonal ones, runs as dense tensor-core matrix
// multiplies": "Kimi K3's hybrid block, from first principles", section "From
// linear attention to the delta rule").  Three kernels per call:
//
//   1. chunk_base_kernel   prefix sum of chunks per sequence (varlen support).
//   2. prep_kernel         one CTA per (chunk, head), all chunks in parallel:
//                          prologue (L2 norm, beta, log-decay floor and running
//                          sum), the decay-rescaled Gram matrices A and P on the
//                          tensor cores (bf16 hi/lo split, three products, fp32
//                          accumulation in TMEM), the unit-lower-triangular solve
//                          T = (I + A)^-1 Diag(beta) in fp32, then W = T K~ and
//                          U~ = T V on the tensor cores.  Writes one 72.5 KB
//                          block per (chunk, head) to the workspace, already in
//                          the shared-memory operand layout of kernel 3.
//   3. chain_kernel        one CTA per (sequence, head), walking the chunks in
//                          order with the state S^T resident in TMEM (fp32):
//                            U^T  = U~^T - S^T W^T
//                            O^T  = S^T Q~^T + U^T P^T
//                            S^T <- S^T Diag(G_C) + U^T K^
//                          operands S^T and U^T go back into TMEM as fp16, the
//                          chunk blocks stream in by 1-D bulk copies (double
//                          buffered), and the per-head RMSNorm x sigmoid-gate
//                          epilogue is fused into the output store.
//
// Chunk algebra (exactly the token recurrence regrouped), per chunk with start
// state S, inclusive running log-decay g_t and G_t = exp(g_t):
//   A = Diag(beta) strictly_lower(K~ K-^T),  P = incl_lower(Q~ K-^T)   (K~ = G k,
//   K- = k / G, Q~ = G q, K^ = (G_C / G) k), T = (I + A)^-1 Diag(beta),
//   W = T K~, U~ = T V, U = U~ - W S, O = Q~ S + P U, S <- Diag(G_C) S + K^^T U.
// For the Gram matrices the 1/G factors are taken relative to the end of the
// column's own 16-token tile, so every factor is within e^-80 .. e^80.
//
// Precision: the Gram products use a bf16 hi/lo split (hi*hi + hi*lo + lo*hi,
// ~16 significant bits, bf16 keeps the e^+-80 range); every other product uses
// fp16 operands (11 significant bits; all values there are within fp16 range
// or negligibly small) with fp32 accumulation; the state itself stays fp32.
#include <stdio.h>

#include "kda_tc.cuh"
#include "umma.cuh"

namespace kda {
namespace {

using namespace umma;

constexpr int kD = 128;          // head dimension (d_k = d_v)
constexpr int kC = 64;           // chunk length
constexpr int kThreads = 128;    // one thread per TMEM lane / channel
constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kDefaultSpins = 4000000000LL;  // ~2 s of clock cycles

// ---- workspace block per (chunk, head): the chain kernel's operand tiles ----
constexpr uint32_t kWsUt = 0;        // U~^T : A [128 (d_v) x 64 (t)]    fp16 SW128
constexpr uint32_t kWsW = 16384;     // W    : B [64 (t) x 128 (d_k)]    fp16 SW128
constexpr uint32_t kWsQn = 32768;    // -Q~  : B [64 (t) x 128 (d_k)]    fp16 SW128
constexpr uint32_t kWsKh = 49152;    // K^^T : B [128 (d_k) x 64 (t)]    fp16 SW128
constexpr uint32_t kWsP = 65536;     // P    : B [64 (t) x 64 (j)]       fp16 SW128
constexpr uint32_t kWsGam = 73728;   // G_C  : fp32 [128]
constexpr uint32_t kWsBytes = 74240;
constexpr uint32_t kWsStride = 75776;  // 1024-aligned shared-memory buffer stride
constexpr int kWsParts = 6;
__constant__ uint32_t kWsPartOff[kWsParts] = {kWsUt, kWsW, kWsQn, kWsKh, kWsP, kWsGam};
__constant__ uint32_t kWsPartLen[kWsParts] = {16384, 16384, 16384, 16384, 8192, 512};

constexpr uint32_t kIdF16Bf16 = idesc_f16(128, 16, true);   // Gram: M128 N16 bf16
constexpr uint32_t kIdF16N64 = idesc_f16(128, 64, false);   // fp16, N = 64
constexpr uint32_t kIdF16N128 = idesc_f16(128, 128, false); // fp16, N = 128

struct TcArgs {
  PrefillArgs a;
  uint8_t* ws;            // per-(chunk, head) blocks
  int* chunk_base;        // [N + 1]
  int total_chunks_max;   // upper bound of the chunk count (grid of prep)
  long long spins;        // bounded-wait limit
  int debug_timeout;
};

__device__ __forceinline__ void report(int* status, int code) { atomicExch(status, code); }

__device__ __forceinline__ uint8_t* ws_block(const TcArgs& t, int chunk_id, int h) {
  return t.ws + ((size_t)h * (size_t)t.total_chunks_max + (size_t)chunk_id) * kWsBytes;
}

// ============================================================ chunk bases
// base[n] = sum_{m < n} ceil(len_m / C); also checks cu_seqlens.
__global__ void __launch_bounds__(1024) chunk_base_kernel(TcArgs t) {
  __shared__ int warp_tot[32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    carry = 0;
    t.chunk_base[0] = 0;
  }
  __syncthreads();
  for (int n0 = 0; n0 < t.a.N; n0 += 1024) {
    const int n = n0 + tid;
    int cnt = 0;
    if (n < t.a.N) {
      int s0, s1;
      seq_range(t.a.cu_seqlens, t.a.N, t.a.T_total, n, s0, s1);
      if (s0 < 0 || s1 < s0 || s1 > t.a.T_total) {
        report(t.a.status, KDA_ERR_SHAPE);
        s1 = s0;
      }
      cnt = (s1 - s0 + kC - 1) / kC;
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = warp_tot[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_tot[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int before = carry + (warp ? warp_tot[warp - 1] : 0);
    if (n < t.a.N) t.chunk_base[n + 1] = before + incl;
    __syncthreads();
    if (tid == 0) carry += warp_tot[31];
    __syncthreads();
  }
}

// Sequence of a global chunk id (binary search over the chunk bases).
__device__ __forceinline__ int find_seq(const int* base, int N, int gid) {
  int lo = 0, hi = N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (base[mid] <= gid) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// ============================================================ prep kernel
// Shared memory (offsets from a 1024-aligned base):
constexpr uint32_t kPrepAhi = 0;          // gram A operand hi [128 x 128] bf16
constexpr uint32_t kPrepAlo = 32768;      // gram A operand lo
constexpr uint32_t kPrepBhi = 65536;      // gram B operand hi [16 x 128] bf16
constexpr uint32_t kPrepBlo = 69632;      // gram B operand lo
//   after the Gram phase the same 72 KB region holds:
constexpr uint32_t kPrepAmat = 0;         // fp32 [64][64]  Diag(beta) strictly-lower A
constexpr uint32_t kPrepX = 16384;        // fp32 [64][64]  (I + A)^-1
constexpr uint32_t kPrepY = 32768;        // fp32 scratch of the block solve (3 x 256)
constexpr uint32_t kPrepT = 32768;        // T    : B [64 (t) x 64 (j)] fp16 SW128 (after Y)
constexpr uint32_t kPrepKt = 40960;       // K~^T : A [128 (c) x 64 (j)] fp16 SW128
constexpr uint32_t kPrepVt = 57344;       // V^T  : A [128 (c) x 64 (j)] fp16 SW128
constexpr uint32_t kPrepStage = 73728;    // workspace image (74240 B)
constexpr uint32_t kPrepQraw = kPrepStage + kWsStride;  // bf16 [64][128]
constexpr uint32_t kPrepKraw = kPrepQraw + 16384;       // bf16 [64][128]
constexpr uint32_t kPrepSmall = kPrepKraw + 16384;      // inv_q, inv_k, beta [64] fp32
constexpr uint32_t kPrepSmem = kPrepSmall + 3 * 64 * 4 + 1024;  // + alignment slack

__device__ __forceinline__ void st_half(uint8_t* base, uint32_t off, float v) {
  *reinterpret_cast<__half*>(base + off) = __float2half_rn(v);
}

// hi/lo bf16 split of x: x ~= hi + lo with ~16 significant bits together.
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(x);
  lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

__global__ void __launch_bounds__(kThreads, 1) prep_kernel(TcArgs t) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PrefillArgs& a = t.a;

  // ---- which chunk ----
  const int gid = blockIdx.x, h = blockIdx.y;
  const int total = t.chunk_base[a.N];
  if (gid >= total) return;
  const int n = find_seq(t.chunk_base, a.N, gid);
  const int c = gid - t.chunk_base[n];
  int s0, s1;
  seq_range(a.cu_seqlens, a.N, a.T_total, n, s0, s1);
  const int tok0 = s0 + c * kC;
  const int len = min(kC, s1 - tok0);
  if (len <= 0) return;
  const size_t H = (size_t)a.H;

  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(a.v);
  const __nv_bfloat16* beta = static_cast<const __nv_bfloat16*>(a.beta);

  float* s_invq = reinterpret_cast<float*>(sm + kPrepSmall);
  float* s_invk = s_invq + 64;
  float* s_beta = s_invk + 64;
  const __nv_bfloat16* sq = reinterpret_cast<const __nv_bfloat16*>(sm + kPrepQraw);
  const __nv_bfloat16* sk = reinterpret_cast<const __nv_bfloat16*>(sm + kPrepKraw);

  // ---- 1. raw q, k tiles (rows past the sequence end are zero) ----
  for (int e = tid; e < kC * 16; e += kThreads) {
    const int r = e >> 4, ch = e & 15;
    uint4 vq = make_uint4(0, 0, 0, 0), vk = vq;
    if (r < len) {
      const size_t gi = ((size_t)(tok0 + r) * H + h) * kD + ch * 8;
      vq = *reinterpret_cast<const uint4*>(q + gi);
      vk = *reinterpret_cast<const uint4*>(k + gi);
    }
    *reinterpret_cast<uint4*>(sm + kPrepQraw + r * 256 + ch * 16) = vq;
    *reinterpret_cast<uint4*>(sm + kPrepKraw + r * 256 + ch * 16) = vk;
  }
  if (tid < kC) {
    float b = 0.f;
    if (tid < len) {
      b = __bfloat162float(beta[(size_t)(tok0 + tid) * H + h]);
      if (a.beta_is_logit) b = sigmoidf_(b);
    }
    s_beta[tid] = b;
  }
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, 128);
    tmem_relinquish();
  }

  // ---- 2. running log2-decay of channel `tid` (registers) ----
  const int ch = tid;
  float g[kC];
  {
    float run = 0.f;
    const float* la = a.log_alpha + ((size_t)tok0 * H + h) * kD + ch;
#pragma unroll
    for (int r = 0; r < kC; ++r) {
      float x = 0.f;
      if (r < len) x = fminf(fmaxf(la[(size_t)r * H * kD], a.g_min), 0.f) * kLog2e;
      run += x;
      g[r] = run;
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base;

  // L2 norms (warp w: rows w, w+4, ...), q also carries q_scale
  for (int r = warp; r < kC; r += 4) {
    const __nv_bfloat162* rq = reinterpret_cast<const __nv_bfloat162*>(sq + r * kD);
    const __nv_bfloat162* rk = reinterpret_cast<const __nv_bfloat162*>(sk + r * kD);
    float ssq = 0.f, ssk = 0.f;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float2 xq = __bfloat1622float2(rq[lane * 2 + i]);
      const float2 xk = __bfloat1622float2(rk[lane * 2 + i]);
      ssq += xq.x * xq.x + xq.y * xq.y;
      ssk += xk.x * xk.x + xk.y * xk.y;
    }
    ssq = warp_sum(ssq);
    ssk = warp_sum(ssk);
    if (lane == 0) {
      float iq = 1.f, ik = 1.f;
      if (a.l2norm_qk) {
        iq = (ssq + a.eps_l2) > 0.f ? 1.0f / sqrtf(ssq + a.eps_l2) : 0.f;
        ik = (ssk + a.eps_l2) > 0.f ? 1.0f / sqrtf(ssk + a.eps_l2) : 0.f;
      }
      s_invq[r] = iq * a.q_scale;
      s_invk[r] = ik;
    }
  }
  __syncthreads();

  // per-tile log2 values of this channel: end of tile b
  float gend[4];
#pragma unroll
  for (int b = 0; b < 4; ++b) gend[b] = g[16 * b + 15];

  // ---- 3. Gram matrices, one 16-column tile at a time ----
  uint32_t phase = 0;
  bool ok = true;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    if (!ok) continue;
    // B operand: K-^(b)_j = k^_j * 2^(gend_b - g_j), j in tile b   [16 x 128]
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      const int j = 16 * b + jj;
      const float x = __bfloat162float(sk[j * kD + ch]) * s_invk[j] * exp2f(gend[b] - g[j]);
      __nv_bfloat16 hi, lo;
      split_bf16(x, hi, lo);
      const uint32_t off = sw128_offset(jj, ch, 16);
      *reinterpret_cast<__nv_bfloat16*>(sm + kPrepBhi + off) = hi;
      *reinterpret_cast<__nv_bfloat16*>(sm + kPrepBlo + off) = lo;
    }
    // A operand rows r >= 16b: [K~^(b); Q~^(b)] with factor 2^(g_r - gend_b)
#pragma unroll
    for (int r = 16 * b; r < kC; ++r) {
      const float e = exp2f(g[r] - gend[b]);
      const float xk = __bfloat162float(sk[r * kD + ch]) * s_invk[r] * e;
      const float xq = __bfloat162float(sq[r * kD + ch]) * s_invq[r] * e;
      __nv_bfloat16 hk, lk, hq, lq;
      split_bf16(xk, hk, lk);
      split_bf16(xq, hq, lq);
      const uint32_t ok_ = sw128_offset(r, ch, 128), oq = sw128_offset(64 + r, ch, 128);
      *reinterpret_cast<__nv_bfloat16*>(sm + kPrepAhi + ok_) = hk;
      *reinterpret_cast<__nv_bfloat16*>(sm + kPrepAlo + ok_) = lk;
      *reinterpret_cast<__nv_bfloat16*>(sm + kPrepAhi + oq) = hq;
      *reinterpret_cast<__nv_bfloat16*>(sm + kPrepAlo + oq) = lq;
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      fence_after_sync();
      const uint32_t d = tmem + 16 * b;
      const uint32_t ahi = smem_u32(sm + kPrepAhi), alo = smem_u32(sm + kPrepAlo);
      const uint32_t bhi = smem_u32(sm + kPrepBhi), blo = smem_u32(sm + kPrepBlo);
      int first = 1;
      const uint32_t pa[3] = {ahi, ahi, alo}, pb[3] = {bhi, blo, bhi};
      for (int p = 0; p < 3; ++p)
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t kb = ks >> 2, kbyte = (ks & 3) * 32;
          mma_ss(d, desc_k_sw128(pa[p] + kb * 128 * 128, kbyte),
                 desc_k_sw128(pb[p] + kb * 16 * 128, kbyte), kIdF16Bf16, first ? 0u : 1u);
          first = 0;
        }
      mma_commit(&bar);
    }
    ok = mbar_wait(&bar, phase, t.spins);
    phase ^= 1;
    fence_after_sync();
  }
  if (!ok) goto fail;

  {
    // ---- 4. read A (lanes 0..63) and P (lanes 64..127) ----
    float* Amat = reinterpret_cast<float*>(sm + kPrepAmat);
    uint8_t* stage = sm + kPrepStage;
    {
      uint32_t v0[32], v1[32];
      tmem_ld32(taddr(tmem, warp * 32, 0), v0);
      tmem_ld32(taddr(tmem, warp * 32, 32), v1);
      tmem_wait_ld();
      if (tid < kC) {
        const int r = tid;
        const float br = s_beta[r];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          Amat[r * kC + j] = (j < r) ? br * __uint_as_float(v0[j]) : 0.f;
          Amat[r * kC + 32 + j] = (32 + j < r) ? br * __uint_as_float(v1[j]) : 0.f;
        }
      } else {
        const int tr = tid - kC;  // output row t
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int j0 = c8 * 8 + 2 * i;
            const float p0 = (j0 <= tr) ? __uint_as_float(j0 < 32 ? v0[j0] : v1[j0 - 32]) : 0.f;
            const float p1 =
                (j0 + 1 <= tr) ? __uint_as_float(j0 + 1 < 32 ? v0[j0 + 1] : v1[j0 + 1 - 32]) : 0.f;
            w[i] = pack_half2(p0, p1);
          }
          *reinterpret_cast<uint4*>(stage + kWsP + sw128_chunk(tr, c8, 64)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
    fence_before_sync();
    __syncthreads();

    // ---- 5. X = (I + A)^-1 by 16 x 16 blocks, T = X Diag(beta) ----
    float* X = reinterpret_cast<float*>(sm + kPrepX);
    float* Y = reinterpret_cast<float*>(sm + kPrepY);
    for (int e = tid; e < kC * kC; e += kThreads) X[e] = 0.f;
    __syncthreads();
    if (tid < 64) {  // diagonal blocks: thread = (block bi, column cc)
      const int bi = tid >> 4, cc = tid & 15, o = 16 * bi;
      float x[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float acc = (r == cc) ? 1.f : 0.f;
#pragma unroll
        for (int m = 0; m < r; ++m) acc -= Amat[(o + r) * kC + o + m] * x[m];
        x[r] = acc;
      }
#pragma unroll
      for (int r = 0; r < 16; ++r) X[(o + r) * kC + o + cc] = x[r];
    }
    __syncthreads();
    // off-diagonal blocks by distance dd = i - j: X_ij = -X_ii sum_{m=j}^{i-1} A_im X_mj
    for (int dd = 1; dd < 4; ++dd) {
      const int nblk = 4 - dd;
      for (int e = tid; e < nblk * 256; e += kThreads) {
        const int bj = e >> 8, bi = bj + dd, r = (e >> 4) & 15, cc = e & 15;
        float acc = 0.f;
        for (int m = 16 * bj; m < 16 * bi; ++m)
          acc += Amat[(16 * bi + r) * kC + m] * X[m * kC + 16 * bj + cc];
        Y[e] = acc;
      }
      __syncthreads();
      for (int e = tid; e < nblk * 256; e += kThreads) {
        const int bj = e >> 8, bi = bj + dd, r = (e >> 4) & 15, cc = e & 15;
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m)
          acc += X[(16 * bi + r) * kC + 16 * bi + m] * Y[(bj << 8) + m * 16 + cc];
        X[(16 * bi + r) * kC + 16 * bj + cc] = -acc;
      }
      __syncthreads();
    }
    // T tile [N = t][K = j] fp16: thread -> (row t, half of the columns)
    {
      const int tr = tid >> 1, hf = tid & 1;
      uint8_t* T = sm + kPrepT;
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        const int cc8 = hf * 4 + c8;
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int j0 = cc8 * 8 + 2 * i;
          w[i] = pack_half2(X[tr * kC + j0] * s_beta[j0], X[tr * kC + j0 + 1] * s_beta[j0 + 1]);
        }
        *reinterpret_cast<uint4*>(T + sw128_chunk(tr, cc8, 64)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }

    // ---- 6. A operands K~^T and V^T (row = channel) and the W / U~ MMAs ----
    {
      const __nv_bfloat16* vcol = v + ((size_t)tok0 * H + h) * kD + ch;
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        uint32_t wk[4], wv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float kv[2], vv[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int j = c8 * 8 + 2 * i + u;
            kv[u] = __bfloat162float(sk[j * kD + ch]) * s_invk[j] * exp2f(g[j]);
            vv[u] = (j < len) ? __bfloat162float(vcol[(size_t)j * H * kD]) : 0.f;
          }
          wk[i] = pack_half2(kv[0], kv[1]);
          wv[i] = pack_half2(vv[0], vv[1]);
        }
        *reinterpret_cast<uint4*>(sm + kPrepKt + sw128_chunk(ch, c8, 128)) =
            make_uint4(wk[0], wk[1], wk[2], wk[3]);
        *reinterpret_cast<uint4*>(sm + kPrepVt + sw128_chunk(ch, c8, 128)) =
            make_uint4(wv[0], wv[1], wv[2], wv[3]);
      }
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      fence_after_sync();
      const uint32_t T = smem_u32(sm + kPrepT), Kt = smem_u32(sm + kPrepKt);
      const uint32_t Vt = smem_u32(sm + kPrepVt);
      for (int ks = 0; ks < 4; ++ks) {
        const uint32_t kbyte = ks * 32;
        mma_ss(tmem, desc_k_sw128(Kt, kbyte), desc_k_sw128(T, kbyte), kIdF16N64, ks > 0);
        mma_ss(tmem + 64, desc_k_sw128(Vt, kbyte), desc_k_sw128(T, kbyte), kIdF16N64, ks > 0);
      }
      mma_commit(&bar);
    }

    // while the MMAs run: -Q~ (B [t][d_k]), K^^T (B [d_k][t]) and G_C
    {
      const float gl = g[kC - 1];
#pragma unroll
      for (int r = 0; r < kC; ++r) {
        const float e = exp2f(g[r]);
        st_half(stage + kWsQn, sw128_offset(r, ch, 64),
                -__bfloat162float(sq[r * kD + ch]) * s_invq[r] * e);
      }
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r0 = c8 * 8 + 2 * i;
          const float x0 = __bfloat162float(sk[r0 * kD + ch]) * s_invk[r0] * exp2f(gl - g[r0]);
          const float x1 =
              __bfloat162float(sk[(r0 + 1) * kD + ch]) * s_invk[r0 + 1] * exp2f(gl - g[r0 + 1]);
          w[i] = pack_half2(x0, x1);
        }
        *reinterpret_cast<uint4*>(stage + kWsKh + sw128_chunk(ch, c8, 128)) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
      reinterpret_cast<float*>(stage + kWsGam)[ch] = exp2f(gl);
    }
    ok = mbar_wait(&bar, phase, t.spins);
    phase ^= 1;
    fence_after_sync();
    if (!ok) goto fail;

    // ---- 7. W (B [t][d_k], from W^T in lanes = d_k) and U~^T (A [d_v][t]) ----
    {
      uint32_t v0[32], v1[32];
      tmem_ld32(taddr(tmem, warp * 32, 0), v0);
      tmem_ld32(taddr(tmem, warp * 32, 32), v1);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        st_half(stage + kWsW, sw128_offset(j, ch, 64), __uint_as_float(v0[j]));
        st_half(stage + kWsW, sw128_offset(32 + j, ch, 64), __uint_as_float(v1[j]));
      }
      tmem_ld32(taddr(tmem, warp * 32, 64), v0);
      tmem_ld32(taddr(tmem, warp * 32, 96), v1);
      tmem_wait_ld();
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int j0 = c8 * 8 + 2 * i;
          const float x0 = __uint_as_float(j0 < 32 ? v0[j0] : v1[j0 - 32]);
          const float x1 = __uint_as_float(j0 + 1 < 32 ? v0[j0 + 1] : v1[j0 + 1 - 32]);
          w[i] = pack_half2(x0, x1);
        }
        *reinterpret_cast<uint4*>(stage + kWsUt + sw128_chunk(ch, c8, 128)) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      bulk_s2g(ws_block(t, gid, h), stage, kWsBytes);
      bulk_commit();
      bulk_wait_all();
    }
  }
  goto done;
fail:
  // a bounded wait gave up: report, then wait (bounded) for the MMAs this CTA
  // issued, so that TMEM is not released under them
  if (tid == 0) {
    report(a.status, KDA_ERR_TIMEOUT);
    mma_commit(&bar);
    mbar_wait(&bar, phase, t.spins);
  }
done:
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

// ============================================================ chain kernel
constexpr uint32_t kChBuf0 = 0;
constexpr uint32_t kChBuf1 = kWsStride;
constexpr uint32_t kChId = 2 * kWsStride;            // identity B [64 x 64] fp16
constexpr uint32_t kChE = kChId + 8192;              // fp32 [64][kEStride] epilogue
constexpr int kEStride = kD + 4;
constexpr uint32_t kChSmem = kChE + kC * kEStride * 4 + 1024;

// TMEM columns
constexpr uint32_t kTS = 0, kTU = 128, kTO = 192, kTAS = 256, kTAU = 320;

__global__ void __launch_bounds__(kThreads, 1) chain_kernel(TcArgs t) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_full[2], bar_u, bar_s, bar_dbg;
  __shared__ uint32_t tmem_base;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PrefillArgs& a = t.a;
  const int h = blockIdx.x % a.H, n = blockIdx.x / a.H;
  const size_t H = (size_t)a.H;
  int s0, s1;
  seq_range(a.cu_seqlens, a.N, a.T_total, n, s0, s1);
  if (s0 < 0 || s1 < s0 || s1 > a.T_total) return;  // reported by chunk_base_kernel
  const int nchunks = (s1 - s0 + kC - 1) / kC;
  const int cbase = t.chunk_base[n];
  const size_t sbase = ((size_t)n * H + h) * (size_t)(kD * kD);

  if (tid == 0) {
    mbar_init(&bar_full[0], 1);
    mbar_init(&bar_full[1], 1);
    mbar_init(&bar_u, 1);
    mbar_init(&bar_s, 1);
    mbar_init(&bar_dbg, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (t.debug_timeout) {  // test hook: a wait that nothing completes, before any async work
    const bool ok = mbar_wait(&bar_dbg, 0, 1000);
    if (!ok && tid == 0) report(a.status, KDA_ERR_TIMEOUT);
    if (!ok) return;
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  // identity operand for U^T <- U~^T * I
  for (int e = tid; e < kC * 8; e += kThreads) {
    const int r = e >> 3, c8 = e & 7;
    uint32_t w[4] = {0, 0, 0, 0};
    if ((r >> 3) == c8) {
      const int i = (r & 7) >> 1;
      w[i] = (r & 1) ? 0x3C000000u : 0x00003C00u;  // fp16 1.0 in the high / low half
    }
    *reinterpret_cast<uint4*>(sm + kChId + sw128_chunk(r, c8, 64)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  auto issue_load = [&](int i) {
    uint8_t* dst = sm + ((i & 1) ? kChBuf1 : kChBuf0);
    const uint8_t* src = ws_block(t, cbase + i, h);
    mbar_arrive_expect_tx(&bar_full[i & 1], kWsBytes);
    for (int p = 0; p < kWsParts; ++p)
      bulk_g2s(dst + kWsPartOff[p], src + kWsPartOff[p], kWsPartLen[p], &bar_full[i & 1]);
  };
  int issued = 0;  // loads issued (meaningful in thread 0)
  if (tid == 0) {
    for (int i = 0; i < 2 && i < nchunks; ++i) issue_load(i);
    issued = min(2, nchunks);
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base;
  const uint32_t lane_base = taddr(tmem, warp * 32, 0);

  // S0 -> S^T in TMEM (lane = d_v index i, column = d_k index c)
  for (int p = 0; p < 4; ++p) {
    uint32_t r[32];
#pragma unroll
    for (int j = 0; j < 32; ++j)
      r[j] = __float_as_uint(a.S0 ? a.S0[sbase + (size_t)(32 * p + j) * kD + tid] : 0.f);
    tmem_st32(lane_base + kTS + 32 * p, r);
  }
  tmem_wait_st();

  const __nv_bfloat16* gate = static_cast<const __nv_bfloat16*>(a.gate);
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.o);
  float* E = reinterpret_cast<float*>(sm + kChE);
  bool ok = true;
  int consumed = 0;  // chunks whose load has been waited for
  for (int i = 0; i < nchunks && ok; ++i) {
    const uint8_t* buf = sm + ((i & 1) ? kChBuf1 : kChBuf0);
    ok = mbar_wait(&bar_full[i & 1], (i >> 1) & 1, t.spins);
    if (!ok) break;
    consumed = i + 1;
    const float* gam = reinterpret_cast<const float*>(buf + kWsGam);
    // -S^T (fp16) into the A operand, S^T Diag(G_C) back into the accumulator
    for (int p = 0; p < 2; ++p) {
      uint32_t x0[32], x1[32], pk[32];
      tmem_ld32(lane_base + kTS + 64 * p, x0);
      tmem_ld32(lane_base + kTS + 64 * p + 32, x1);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        pk[j] = pack_half2(-__uint_as_float(x0[2 * j]), -__uint_as_float(x0[2 * j + 1]));
        pk[16 + j] = pack_half2(-__uint_as_float(x1[2 * j]), -__uint_as_float(x1[2 * j + 1]));
      }
      tmem_st32(lane_base + kTAS + 32 * p, pk);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        x0[j] = __float_as_uint(__uint_as_float(x0[j]) * gam[64 * p + j]);
        x1[j] = __float_as_uint(__uint_as_float(x1[j]) * gam[64 * p + 32 + j]);
      }
      tmem_st32(lane_base + kTS + 64 * p, x0);
      tmem_st32(lane_base + kTS + 64 * p + 32, x1);
    }
    tmem_wait_st();
    fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      fence_after_sync();
      const uint32_t sb = smem_u32(buf);
      const uint32_t id = smem_u32(sm + kChId);
      for (int ks = 0; ks < 4; ++ks)  // U^T = U~^T I
        mma_ss(tmem + kTU, desc_k_sw128(sb + kWsUt, ks * 32), desc_k_sw128(id, ks * 32), kIdF16N64,
               ks > 0);
      for (int ks = 0; ks < 8; ++ks) {  // U^T += (-S^T) W^T ;  O^T = (-S^T)(-Q~)^T
        const uint32_t kb = ks >> 2, kbyte = (ks & 3) * 32;
        mma_ts(tmem + kTU, tmem + kTAS + 8 * ks, desc_k_sw128(sb + kWsW + kb * 64 * 128, kbyte),
               kIdF16N64, 1);
        mma_ts(tmem + kTO, tmem + kTAS + 8 * ks, desc_k_sw128(sb + kWsQn + kb * 64 * 128, kbyte),
               kIdF16N64, ks > 0);
      }
      mma_commit(&bar_u);
    }
    ok = mbar_wait(&bar_u, i & 1, t.spins);
    fence_after_sync();
    if (!ok) break;
    {  // U^T -> fp16 A operand
      uint32_t x0[32], x1[32], pk[32];
      tmem_ld32(lane_base + kTU, x0);
      tmem_ld32(lane_base + kTU + 32, x1);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        pk[j] = pack_half2(__uint_as_float(x0[2 * j]), __uint_as_float(x0[2 * j + 1]));
        pk[16 + j] = pack_half2(__uint_as_float(x1[2 * j]), __uint_as_float(x1[2 * j + 1]));
      }
      tmem_st32(lane_base + kTAU, pk);
      tmem_wait_st();
    }
    fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      fence_after_sync();
      const uint32_t sb = smem_u32(buf);
      for (int ks = 0; ks < 4; ++ks) {  // O^T += U^T P^T ; S^T += U^T K^
        mma_ts(tmem + kTO, tmem + kTAU + 8 * ks, desc_k_sw128(sb + kWsP, ks * 32), kIdF16N64, 1);
        mma_ts(tmem + kTS, tmem + kTAU + 8 * ks, desc_k_sw128(sb + kWsKh, ks * 32), kIdF16N128, 1);
      }
      mma_commit(&bar_s);
    }
    ok = mbar_wait(&bar_s, i & 1, t.spins);
    fence_after_sync();
    if (!ok) break;
    __syncthreads();
    if (tid == 0 && i + 2 < nchunks) {
      fence_proxy_async();
      issue_load(i + 2);
      issued = i + 3;
    }

    // epilogue: O^T (lane = d_v) -> E[t][d_v] -> rows of y
    {
      uint32_t x0[32], x1[32];
      tmem_ld32(lane_base + kTO, x0);
      tmem_ld32(lane_base + kTO + 32, x1);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        E[j * kEStride + tid] = __uint_as_float(x0[j]);
        E[(32 + j) * kEStride + tid] = __uint_as_float(x1[j]);
      }
    }
    __syncthreads();
    const int tok0 = s0 + i * kC;
    const int len = min(kC, s1 - tok0);
    for (int r = warp; r < len; r += 4) {
      const float4 x = *reinterpret_cast<const float4*>(&E[r * kEStride + 4 * lane]);
      float y[4] = {x.x, x.y, x.z, x.w};
      const size_t gi = ((size_t)(tok0 + r) * H + h) * kD + 4 * lane;
      if (gate) {
        const float ss = warp_sum(y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3]);
        const float inv = rsqrtf(ss / kD + a.eps_norm);
        const uint2 graw = *reinterpret_cast<const uint2*>(gate + gi);
        const float2 g01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&graw.x));
        const float2 g23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&graw.y));
        const float gg[4] = {g01.x, g01.y, g23.x, g23.y};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float nw = a.norm_weight ? a.norm_weight[4 * lane + u] : 1.f;
          y[u] = y[u] * inv * nw * sigmoidf_(gg[u]);
        }
      }
      uint2 out;
      out.x = pack_bf162(y[0], y[1]);
      out.y = pack_bf162(y[2], y[3]);
      *reinterpret_cast<uint2*>(o + gi) = out;
    }
    __syncthreads();
  }
  if (!ok && tid == 0) {
    // a bounded wait gave up: report it, then wait (bounded) for this CTA's
    // own MMAs and bulk copies before releasing TMEM and shared memory
    report(a.status, KDA_ERR_TIMEOUT);
    mma_commit(&bar_dbg);
    mbar_wait(&bar_dbg, 0, t.spins);
    for (int j = consumed; j < issued; ++j) mbar_wait(&bar_full[j & 1], (j >> 1) & 1, t.spins);
  }

  // final state S^T -> S_T[c][i]
  if (ok) {
    for (int p = 0; p < 4; ++p) {
      uint32_t r[32];
      tmem_ld32(lane_base + kTS + 32 * p, r);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) a.S_T[sbase + (size_t)(32 * p + j) * kD + tid] = __uint_as_float(r[j]);
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, 512);
  (void)lane;
}

size_t header_bytes(int N) { return ((size_t)(N + 1) * 4 + 1023) & ~(size_t)1023; }
int chunks_upper(int T_total, int N) { return T_total / kC + N; }

}  // namespace

bool tc_prefill_supported(int d, int dtype, int chunk) {
  return d == kD && dtype == KDA_BF16 && (chunk == 0 || chunk == kC);
}

size_t tc_workspace_bytes(int T_total, int N, int H, int d, const kda_options*) {
  if (d != kD) return 0;
  return header_bytes(N) + (size_t)H * (size_t)chunks_upper(T_total, N) * kWsBytes;
}

int tc_launches(int, int, int, int, const kda_options*) { return 3; }
int tc_chunk(const kda_options*) { return kC; }

cudaError_t launch_prefill_tc(const PrefillArgs& a, const kda_options* opt, cudaStream_t s) {
  TcArgs t;
  t.a = a;
  t.chunk_base = static_cast<int*>(opt->workspace);
  t.ws = static_cast<uint8_t*>(opt->workspace) + header_bytes(a.N);
  t.total_chunks_max = chunks_upper(a.T_total, a.N);
  t.spins = opt->timeout_spins > 0 ? opt->timeout_spins : kDefaultSpins;
  t.debug_timeout = opt->debug_timeout;
  cudaEvent_t const* ev = reinterpret_cast<cudaEvent_t const*>(opt->phase_events);
  cudaError_t e;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    e = cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kPrepSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kChSmem);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  if (ev && (e = cudaEventRecord(ev[0], s)) != cudaSuccess) return e;
  chunk_base_kernel<<<1, 1024, 0, s>>>(t);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (ev && (e = cudaEventRecord(ev[1], s)) != cudaSuccess) return e;
  if (t.total_chunks_max > 0 && !t.debug_timeout) {
    dim3 grid((unsigned)t.total_chunks_max, (unsigned)a.H);
    prep_kernel<<<grid, kThreads, kPrepSmem, s>>>(t);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (ev && (e = cudaEventRecord(ev[2], s)) != cudaSuccess) return e;
  chain_kernel<<<(unsigned)(a.N * a.H), kThreads, kChSmem, s>>>(t);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (ev && (e = cudaEventRecord(ev[3], s)) != cudaSuccess) return e;
  return cudaSuccess;
}

}  // namespace kda
