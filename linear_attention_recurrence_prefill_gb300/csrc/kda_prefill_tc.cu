// kda_prefill_tc.cu -- chunked KDA prefill on the tcgen05 tensor cores (sm_103a).
//
// The layer is processed in chunks of C = 64 tokens.  Inside a chunk all tokens
// are handled at once and the chunks follow one another through the state
// ("Kimi K3's hybrid block, from first principles", section "From linear
// attention to the delta rule").  With log alpha >= -5 the running log-decay
// moves by less than 80 (116 in log2) over 16 tokens, so decay factors taken
// about a row 16 tokens away stay inside the bf16 / fp32 exponent range, and
// every block of the chunk, the diagonal ones included, is a dense tensor-core
// product.  Three kernels per call:
//
//   1. chunk_base_kernel   prefix sum of chunks per sequence (varlen support;
//                          not launched for sequences of one length, whose
//                          chunks follow by arithmetic).
//   2. prep_kernel         persistent, two CTAs per SM walking the (chunk, head)
//                          items, all independent; the inputs of each item
//                          arrive by TMA tensor copies; per item: prologue
//                          (optionally the short convolution and the decay from
//                          its logit, then L2 norm, beta, log-decay floor and
//                          running sum), the decay-rescaled Gram matrices A and P on the
//                          tensor cores (bf16 hi/lo split, three products, fp32
//                          accumulation in TMEM), the unit-lower-triangular solve
//                          T = (I + A)^-1 Diag(beta) (fp32 diagonal blocks, the
//                          lower 32-block as two bf16 hi/lo tensor-core
//                          products), then W = T K~ and U~ = T V on the tensor
//                          cores.  Writes one 72.5 KB
//                          block per (chunk, head) to the workspace, already in
//                          the shared-memory operand layout of kernel 3.
//   3. chain_kernel        one CTA per (sequence, head), launched early
//                          (programmatic dependent launch) so that its set-up
//                          overlaps prep's last items, walking the chunks in
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
// For the Gram matrices both factors are taken about the middle row of the
// row's 32-token span, so every factor is within 2^-116 .. 2^116.
// V, K~ and K^ enter their products as MN-major operands (64-channel blocks of
// token rows), so every one of them is produced row by row, like the inputs.
//
// Precision: the Gram products and the inverse's lower block use a bf16 hi/lo
// split (hi*hi + hi*lo + lo*hi, ~16 significant bits, bf16 keeps the 2^+-116
// range), U~ = T V takes T as a bf16 hi/lo pair against V exact in bf16, and
// every other product uses fp16 operands (11 significant bits; all values there
// are within fp16 range or negligibly small) with fp32 accumulation; the state
// itself stays fp32.
#include <cuda.h>
#include <stdio.h>

#include <mutex>

#include "kda_tc.cuh"
#include "umma.cuh"

namespace kda {
namespace {

using namespace umma;

constexpr int kD = 128;          // head dimension (d_k = d_v)
constexpr int kC = 64;           // chunk length
constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kDefaultSpins = 4000000000LL;  // ~2 s of clock cycles

// ---- workspace block per (chunk, head): the chain kernel's operand tiles ----
constexpr uint32_t kWsUt = 0;        // U~^T : A [128 (d_v) x 64 (t)]    fp16 SW128
constexpr uint32_t kWsWQ = 16384;    // [W; -Q~] : B [128 (t of W, then t of -Q~) x 128 (d_k)]
                                     //            fp16 SW128 (one operand for both products)
constexpr uint32_t kWsKh = 49152;    // K^   : B [128 (d_k) x 64 (t)]    fp16 SW128 MN-major
                                     //        (64 rows t of 128 d_k, 8 KB per 64 d_k)
constexpr uint32_t kWsP = 65536;     // P    : B [64 (t) x 64 (j)]       fp16 SW128
constexpr uint32_t kWsGam = 73728;   // G_C  : fp32 [128]
constexpr uint32_t kWsBytes = 74240;
constexpr uint32_t kWsStride = 75776;  // 1024-aligned shared-memory buffer stride
constexpr int kWsParts = 5;
__constant__ uint32_t kWsPartOff[kWsParts] = {kWsUt, kWsWQ, kWsKh, kWsP, kWsGam};
__constant__ uint32_t kWsPartLen[kWsParts] = {16384, 32768, 16384, 8192, 512};

constexpr uint32_t kIdGram = idesc_f16(128, 96, true);      // Gram: M128 N96 bf16
constexpr uint32_t kIdF16N64 = idesc_f16(128, 64, false);   // fp16, N = 64
constexpr uint32_t kIdKh = idesc_f16(128, 128, false, false, true);  // fp16, N = 128, B MN-major

struct TcArgs {
  PrefillArgs a;
  uint8_t* ws;            // per-(chunk, head) blocks
  int* chunk_base;        // [N + 1]
  int total_chunks_max;   // upper bound of the chunk count (grid of prep)
  long long spins;        // bounded-wait limit
  int debug_timeout;
  // Tensor maps of q, k, v as [T_total][H][128] bf16 (x = channel, y = head,
  // z = token), box 64 channels x 1 head x 64 tokens, 128-byte swizzle: one box
  // is half a chunk's rows of one head, landing as [64 rows][128 B] (the
  // swizzled layout of sw128_chunk with 64 rows).  log alpha likewise as fp32
  // (with one decay per key channel), box 32 channels x 1 x 64 tokens.  Tokens
  // past T_total read 0.
  CUtensorMap tm_q, tm_k, tm_v, tm_la;
};

__device__ __forceinline__ void report(int* status, int code) { atomicExch(status, code); }

__device__ __forceinline__ uint8_t* ws_block(const TcArgs& t, int chunk_id, int h) {
  return t.ws + ((size_t)h * (size_t)t.total_chunks_max + (size_t)chunk_id) * kWsBytes;
}

// ============================================================ chunk bases
// base[n] = sum_{m < n} ceil(len_m / C); also checks cu_seqlens.  Behind the
// bases (at base + N + 1) it writes the order in which the chain grid takes the
// sequences: by descending chunk count (ties by index), so that the longest
// chains start first and the grid's last wave holds short ones; for more than
// kOrderMax sequences the order stays the index order.
constexpr int kOrderMax = 2048;
__global__ void __launch_bounds__(1024) chunk_base_kernel(TcArgs t) {
  __shared__ int warp_tot[32];
  __shared__ int carry;
  __shared__ int s_cnt[kOrderMax];  // chunks per sequence (N <= kOrderMax)
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
    if (n < t.a.N && t.a.N <= kOrderMax) s_cnt[n] = cnt;
    __syncthreads();
    if (tid == 0) carry += warp_tot[31];
    __syncthreads();
  }
  int* order = t.chunk_base + t.a.N + 1;
  for (int n = tid; n < t.a.N; n += 1024) {
    int rank = n;
    if (t.a.N <= kOrderMax) {  // position among the sequences, longest first
      const int c = s_cnt[n];
      rank = 0;
      for (int m = 0; m < t.a.N; ++m) rank += (s_cnt[m] > c || (s_cnt[m] == c && m < n)) ? 1 : 0;
    }
    order[rank] = n;
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
// 256 threads, about 106 KB of shared memory and at most 128 registers per
// thread, so that two CTAs share an SM and hide each other's waits.
// Shared memory (offsets from a 1024-aligned base):
constexpr int kPrepThreads = 256;
constexpr int kPrepHalf = 128;                   // threads per warp group (step 6)
constexpr uint32_t kBarSolve = 2;                // the inverting group's named barrier
constexpr uint32_t kPrepQ = 0;            // q rows, bf16: two 64-channel halves of
                                          // [64 rows][128 B], 128-byte swizzle (TMA)
constexpr uint32_t kPrepK = 16384;        // k rows, the same
constexpr uint32_t kPrepG = 32768;        // log alpha rows, then running log2-decay, fp32:
                                          // four 32-channel slabs of [64 rows][128 B],
                                          // 128-byte swizzle (TMA)
constexpr uint32_t kPrepX = 65536;        // 40 KB region reused by the phases:
//   Gram (per 64-channel half): B = [B_0; B_1] hi and lo, [96 x 64] bf16 K-major
//   SW128 each (B_0: rows 0..31, B_1: rows 32..95)
constexpr uint32_t kPrepBh = kPrepX, kPrepBl = kPrepX + 12288;
//   solve: Diag(beta) strictly_lower(A) and (I + A)^-1, fp32 [64][64] with padded row
//   strides (no bank conflicts between the rows a warp touches), 4 KB scratch
constexpr int kAs = 66, kXs = 68;  // row strides (floats) of A and of the inverse
constexpr uint32_t kPrepAmat = kPrepX, kPrepInv = kPrepX + kC * kAs * 4;
constexpr uint32_t kPrepY = kPrepInv + kC * kXs * 4;
//   W / U~ MMAs: [T; T] [128 (t) x 64 (j)] fp16 K-major over A; V (bf16) and K~
//   (fp16) [64 (j) rows of 128 channels] MN-major over the q and k rows
constexpr uint32_t kPrepTT = kPrepX, kPrepV = kPrepQ, kPrepKt = kPrepK;
//   T as bf16 hi/lo K-major [64 (t)][64 (j)] tiles over the decay rows
constexpr uint32_t kPrepThi = kPrepG, kPrepTlo = kPrepG + 8192;
//   U~^T and W staged for their bulk copies to the workspace
constexpr uint32_t kPrepStU = kPrepX, kPrepStW = kPrepX + 16384;
//   the inverse's 32-level products: B operands A_10^T and -X_00^T as bf16 hi/lo
//   K-major tiles [32 (column) rows][K = 32 in the first 64 B of each 128-byte
//   row], SW128, over the decay rows behind the T tiles (the row pass has
//   finished reading them)
constexpr uint32_t kPrepA10h = kPrepG + 16384, kPrepA10l = kPrepA10h + 4096;
constexpr uint32_t kPrepX00h = kPrepA10h + 8192, kPrepX00l = kPrepA10h + 12288;
// TMEM: the Gram's D = [D_0 | D_1] (32 + 64 columns) and A (hi, lo for each
// channel half: 4 x 32); then U~^T as its T_hi and T_lo parts (2 x 64 columns)
// and W (128)
constexpr uint32_t kPrepTmemCols = 256, kTdD0 = 0, kTdD1 = 32, kTdA = 96;
constexpr uint32_t kTdU = 0, kTdW = 128;
// the inverse (between the two): lanes 0..31 carry rows 32..63; A = X_11 as
// bf16 hi/lo (16 + 16 columns), D = X_11 A_10 (64 columns: hi.hi + lo.hi, then
// hi.lo), A = that product as hi/lo, and D = X_10 (64 columns likewise, over
// X_11's and the first product's, both read by then)
constexpr uint32_t kTdX11 = 128, kTdY = 160, kTdYs = 224, kTdX10 = 128;
static_assert(kTdY + 64 <= kTdYs && kTdYs + 32 <= kPrepTmemCols,
              "the inverse's operands fit the TMEM allocation");
constexpr uint32_t kIdInv32 = idesc_f16(128, 32, true);  // bf16, N = 32
constexpr uint32_t kIdInv64 = idesc_f16(128, 64, true);  // bf16, N = 64
static_assert(kTdA + 128 <= kPrepTmemCols, "Gram accumulators and A fit the TMEM allocation");
static_assert(kTdU + 128 <= kTdW && kTdW + 128 <= kPrepTmemCols, "U~^T and W fit the TMEM allocation");
constexpr uint32_t kIdUt = idesc_f16(128, 128, true, true, false);  // bf16, A MN-major, N = 128
constexpr uint32_t kIdW = idesc_f16(128, 128, false, false, true);  // B MN-major, N = 128
constexpr uint32_t kPrepSmall = kPrepX + 40960;  // inv_q, inv_k, beta [64] fp32
// short convolution: the raw q, k, v rows of the 3 tokens before the chunk,
// bf16 [3 (q, k, v)][3][128] (unswizzled 256-byte rows)
constexpr uint32_t kPrepHalo = kPrepSmall + 3 * 64 * 4;
constexpr uint32_t kPrepSmem = kPrepHalo + 9 * 256 + 1024;  // + alignment slack
static_assert(kPrepY + 4 * 256 * 4 <= kPrepSmall, "solve scratch inside the reused region");
static_assert(kPrepBl + 12288 <= kPrepSmall, "Gram operands inside the reused region");
static_assert(kPrepTT + 2 * kC * 128 <= kPrepInv, "[T; T] tile clear of the inverse");
static_assert(kPrepStW + 16384 <= kPrepSmall, "U~^T and W staging inside the reused region");
static_assert(kPrepTlo + 8192 <= kPrepA10h && kPrepX00l + 4096 <= kPrepX,
              "the inverse's operand tiles clear of the T tiles, inside the decay rows");
static_assert(kPrepInv % 16 == 0 && kPrepY % 16 == 0 && (kXs * 4) % 16 == 0,
              "float4 access to the inverse and the scratch");

__device__ __forceinline__ float ex2f(float x) {  // hardware 2^x (rel. error ~2^-22)
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcpf(float x) {  // hardware 1/x (rel. error ~2^-23)
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// sigmoid(x) from the hardware 2^x and 1/x
__device__ __forceinline__ float sigmoid_fast(float x) { return rcpf(1.f + ex2f(-kLog2e * x)); }

__device__ __forceinline__ void unpack8(const uint4& r, float (&f)[8]) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float2 x = __bfloat1622float2(b[u]);
    f[2 * u] = x.x;
    f[2 * u + 1] = x.y;
  }
}

// The q and k rows in shared memory keep, within each 128-byte half-row, the
// 16-byte chunk c16 (channels 8 c16 .. 8 c16 + 7) of row r at qk_off(r, c16):
// chunk j at position j ^ (r % 8), the tensor copies' 128-byte swizzle, so that
// threads reading the same chunk of eight consecutive rows hit eight different
// bank groups.
__host__ __device__ __forceinline__ uint32_t qk_off(int r, int c16) {
  return sw128_chunk((uint32_t)r, (uint32_t)c16, (uint32_t)kC);
}
// The decay rows: four 32-channel slabs of [64 rows][128 B] with the same
// swizzle.  Float index of channel ch of row r:
__host__ __device__ constexpr int gidx(int r, int ch) {
  return (ch >> 5) * 2048 + r * 32 + ((((ch >> 2) & 7) ^ (r & 7)) << 2) + (ch & 3);
}

// 8-channel group c of decay row r: chunks 2 (c % 4) and 2 (c % 4) + 1 of slab
// c / 4, for accesses where the lanes of a warp read the same group of
// different rows (the row's swizzle keeps those conflict-free).
__device__ __forceinline__ void ld8g_rows(const float* G, int r, int c, float (&f)[8]) {
  const float* row = G + (c >> 2) * 2048 + r * 32;
  const int j = 2 * (c & 3), x = r & 7;
  const float4 a = *reinterpret_cast<const float4*>(row + ((j ^ x) << 2));
  const float4 b = *reinterpret_cast<const float4*>(row + (((j + 1) ^ x) << 2));
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
// The same where the lanes read consecutive groups of one row: odd slabs fetch
// the second chunk first, so that eight consecutive groups (two slabs) read
// eight different bank groups per load.
__device__ __forceinline__ void ld8g(const float* G, int r, int c, float (&f)[8]) {
  const float* row = G + (c >> 2) * 2048 + r * 32;
  const int j = 2 * (c & 3), x = r & 7, odd = (c >> 2) & 1;
  const float4 p = *reinterpret_cast<const float4*>(row + (((j + odd) ^ x) << 2));
  const float4 q = *reinterpret_cast<const float4*>(row + (((j + 1 - odd) ^ x) << 2));
  const float4 a = odd ? q : p, b = odd ? p : q;
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// Packed two-lane fp32 arithmetic (sm_100 family): one instruction per pair.
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
      "sub.rn.f32x2 z, x, y;\n\tmov.b64 {%0, %1}, z;\n\t}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
      "mul.rn.f32x2 z, x, y;\n\tmov.b64 {%0, %1}, z;\n\t}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n\t.reg .b64 x, y, z, w;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
      "mov.b64 z, {%6, %7};\n\tfma.rn.f32x2 w, x, y, z;\n\tmov.b64 {%0, %1}, w;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}
// acc += s * x, four lanes in two packed instructions (each lane one fused
// multiply-add, as the scalar form)
__device__ __forceinline__ void fma4s(float4& acc, float s, const float4& x) {
  const float2 s2 = make_float2(s, s);
  const float2 lo = fma2(s2, make_float2(x.x, x.y), make_float2(acc.x, acc.y));
  const float2 hi = fma2(s2, make_float2(x.z, x.w), make_float2(acc.z, acc.w));
  acc = make_float4(lo.x, lo.y, hi.x, hi.y);
}

// bf16 hi/lo split of a pair: x ~= hi + lo with ~16 significant bits.
__device__ __forceinline__ void split2v(float2 x, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x.x, x.y);
  const uint32_t hb = *reinterpret_cast<const uint32_t*>(&h);
  const float2 hf = make_float2(__uint_as_float(hb << 16), __uint_as_float(hb & 0xFFFF0000u));
  const float2 d = sub2(x, hf);
  const __nv_bfloat162 l = __floats2bfloat162_rn(d.x, d.y);
  hi = hb;
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// One row of the short convolution + Swish for 4 channels: taps w (oldest
// first) over the window of the 3 previous raw rows and the raw row x (4 bf16
// in a uint2); the window moves on by one row.  Returns the 4 outputs as bf16
// pairs (rounded to nearest even: the value stored in the data type).
__device__ __forceinline__ uint2 conv_row4(const float4 (&w)[4], float (&win)[3][4], uint2 raw) {
  const float x[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                      __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
  float y[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    y[c] = conv4_swish(w[c], win[0][c], win[1][c], win[2][c], x[c]);
    win[0][c] = win[1][c];
    win[1][c] = win[2][c];
    win[2][c] = x[c];
  }
  return make_uint2(pack_bf162(y[0], y[1]), pack_bf162(y[2], y[3]));
}

__device__ __forceinline__ void unpack4(uint2 raw, float (&f)[4]) {
  f[0] = __uint_as_float(raw.x << 16);
  f[1] = __uint_as_float(raw.x & 0xFFFF0000u);
  f[2] = __uint_as_float(raw.y << 16);
  f[3] = __uint_as_float(raw.y & 0xFFFF0000u);
}

// taps of channels c0 .. c0 + 3 of tensor X (0 = q, 1 = k, 2 = v), head h
__device__ __forceinline__ void conv_taps4(const float* cw, int X, int H, int h, int c0,
                                           float4 (&w)[4]) {
  const float4* p = reinterpret_cast<const float4*>(cw + (((size_t)X * H + h) * kD + c0) * 4);
#pragma unroll
  for (int c = 0; c < 4; ++c) w[c] = p[c];
}

// kConv: the short convolution runs in the prologue; kLogit: log alpha is
// formed from decay logits.  Separate instantiations, so that the default one
// carries none of their registers.
template <bool kConv, bool kLogit>
__global__ void __launch_bounds__(kPrepThreads, 2) prep_kernel(const __grid_constant__ TcArgs t) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_mma, bar_in, bar_v;  // MMAs; q/k tensor copies; v copies
  __shared__ uint32_t tmem_base;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PrefillArgs& a = t.a;

  // ---- work items: (chunk, head) pairs in the order of `decode` below; a CTA
  //      takes items blockIdx.x, + gridDim.x, ... and streams the next item's
  //      inputs into its buffers while it writes out the current one ----
  // the chain may start its CTAs (set-up only) as SMs free up at this grid's end
  grid_launch_dependents();
  // sequences of one length L (no cu_seqlens) have ceil(L / C) chunks each: the
  // item's tokens follow by arithmetic, without a dependent load
  const int L_eq = a.cu_seqlens ? 0 : a.T_total / a.N;
  const int cps_eq = (L_eq + kC - 1) / kC;
  const int total = a.cu_seqlens ? t.chunk_base[a.N] : a.N * cps_eq;
  const int items = total * a.H;
  if ((int)blockIdx.x >= items) return;
  const size_t H = (size_t)a.H;
  const __nv_bfloat16* beta = static_cast<const __nv_bfloat16*>(a.beta);
  float* s_invq = reinterpret_cast<float*>(sm + kPrepSmall);
  float* s_invk = s_invq + 64;
  float* s_beta = s_invk + 64;
  float* G = reinterpret_cast<float*>(sm + kPrepG);

  if (tid == 0) {
    mbar_init(&bar_mma, 1);
    mbar_init(&bar_in, 1);
    mbar_init(&bar_v, 1);
    mbar_fence_init();
    tma_prefetch_desc(&t.tm_q);
    tma_prefetch_desc(&t.tm_k);
    tma_prefetch_desc(&t.tm_v);
    if (a.decay_mode == KDA_DECAY_CHANNEL) tma_prefetch_desc(&t.tm_la);
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, kPrepTmemCols);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base;

  // Items run chunk position by chunk position, the heads (and sequences) of one
  // position side by side, and the last position first: the CTAs in flight read
  // neighbouring token rows, and the blocks written last (still in L2 when the
  // chain starts) are the ones the chain reads first.
  auto decode = [&](int wi, int& gid_, int& h_, int& tok0_, int& len_, int& n_, int& s0_) {
    const int wr = items - 1 - wi;
    if (!a.cu_seqlens) {  // wr = (position p, sequence n, head h)
      const int nh = a.N * a.H;
      const int p = wr / nh, rem = wr - p * nh;
      n_ = rem / a.H;
      h_ = rem - n_ * a.H;
      gid_ = n_ * cps_eq + p;
      s0_ = n_ * L_eq;
      tok0_ = s0_ + p * kC;
      len_ = min(kC, (n_ + 1) * L_eq - tok0_);
      return;
    }
    gid_ = wr / a.H;  // wr = (chunk, head)
    h_ = wr - gid_ * a.H;
    n_ = find_seq(t.chunk_base, a.N, gid_);
    int s1_;
    seq_range(a.cu_seqlens, a.N, a.T_total, n_, s0_, s1_);
    tok0_ = s0_ + (gid_ - t.chunk_base[n_]) * kC;
    len_ = min(kC, s1_ - tok0_);
  };
  // per-thread values of the item whose copies are in flight: beta of row tid
  // and, with decay logits, the scale and channel tid's bias (global loads whose
  // latency the copies' wait covers)
  // (beta as its raw bf16 bits, widened only when used)
  uint32_t pre_beta = 0u;
  float pre_scale = 1.f, pre_bias = 0.f;
  auto issue_inputs = [&](int h, int tok0, int len, int n, int s0) {
    if (tid < kD) {
      pre_beta = 0u;
      if (tid < len) pre_beta = reinterpret_cast<const uint16_t*>(beta)[(size_t)(tok0 + tid) * H + h];
      if constexpr (kLogit) {
        if (a.decay_scale) pre_scale = a.decay_scale[h];
        if (a.decay_bias) pre_bias = a.decay_bias[(size_t)h * kD + tid];
      }
    }
    // the raw q, k, v rows of the 3 tokens before the chunk (short convolution):
    // from the token arrays inside the sequence, else from the caller's window
    // (zeros without one)
    if (kConv && tid < 144) {
      const int X = tid / 48, j = (tid / 16) % 3, c16 = tid % 16;
      const void* arr = X == 0 ? a.q : (X == 1 ? a.k : a.v);
      const char* src;
      uint32_t nbytes = 16u;
      if (tok0 > s0) {
        src = reinterpret_cast<const char*>(arr) + ((size_t)(tok0 - 3 + j) * H + h) * 256 + c16 * 16;
      } else if (a.conv_state) {
        src = reinterpret_cast<const char*>(a.conv_state) +
              ((((size_t)n * 3 + X) * 3 + j) * H + h) * 256 + c16 * 16;
      } else {
        src = reinterpret_cast<const char*>(arr);
        nbytes = 0u;
      }
      cp_async16(smem_u32(sm + kPrepHalo + (X * 3 + j) * 256 + c16 * 16), src, nbytes);
    }
    // ---- 1. input rows by tensor copies (thread 0): q and k (two boxes each)
    //      and, with one decay per key channel, log alpha (four boxes).  Rows
    //      past the sequence end hold the next tokens (or zeros past T_total):
    //      they are identity steps whatever their q, k, v, since their beta is 0
    //      and the decay scan takes their log alpha as 0.  With one decay per
    //      head (or none) the decay rows are filled by broadcasting the row's
    //      value instead ----
    const bool la_tma = a.decay_mode == KDA_DECAY_CHANNEL;
    if (tid == 0) {
      mbar_arrive_expect_tx(&bar_in, 2 * kC * kD * 2 + (la_tma ? kC * kD * 4 : 0));
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        tma_load_3d(sm + kPrepQ + hf * 8192, &t.tm_q, 64 * hf, h, tok0, &bar_in);
        tma_load_3d(sm + kPrepK + hf * 8192, &t.tm_k, 64 * hf, h, tok0, &bar_in);
      }
      if (la_tma) {
#pragma unroll
        for (int sl = 0; sl < 4; ++sl)
          tma_load_3d(sm + kPrepG + sl * 8192, &t.tm_la, 32 * sl, h, tok0, &bar_in);
      }
    }
    cp_async_commit();
    if (!la_tma) {
      for (int e = tid; e < kC * 32; e += kPrepThreads) {  // 16-byte words of the rows
        const int r = e >> 5, wd = e & 31;
        const float g = (r < len && a.decay_mode == KDA_DECAY_HEAD)
                            ? a.log_alpha[(size_t)(tok0 + r) * H + h] : 0.f;
        *reinterpret_cast<float4*>(sm + kPrepG + (wd >> 3) * 8192 + r * 128 + (wd & 7) * 16) =
            make_float4(g, g, g, g);
      }
    }
  };

  int item = blockIdx.x, gid, h, tok0, len, nseq, sstart;
  decode(item, gid, h, tok0, len, nseq, sstart);
  issue_inputs(h, tok0, len, nseq, sstart);
  uint32_t mma_phase = 0, in_phase = 0, v_phase = 0;
  bool in_pending = true, v_pending = false;  // tensor copies issued, not yet waited on
  bool ok = true;
  for (;;) {
    uint8_t* ws = ws_block(t, gid, h);
    cp_async_wait_all();
    const bool in_ok = mbar_wait(&bar_in, in_phase, t.spins);
    if (tid == 0) bulk_wait_read();  // the previous item's results have left region X
    ok = __syncthreads_and(in_ok);
    if (!ok) goto fail;
    in_phase ^= 1;
    in_pending = false;

    // ---- 1b. short convolution + Swish of the q and k rows, in place: thread =
    //      (tensor, 8-row block rb, 8-channel group c16) streams its rows through
    //      a 3-row window; the 3 rows the next block still reads are written
    //      after a barrier; the output is held in bf16, as a separate
    //      convolution layer would hand it over ----
    if constexpr (kConv) {
      const int c16 = tid & 15, rb = (tid >> 4) & 7, X = tid >> 7;
      uint8_t* rows = sm + (X ? kPrepK : kPrepQ);
      const uint8_t* halo = sm + kPrepHalo + X * 3 * 256;
      uint2 held[2][3];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {  // the two 4-channel halves of the group
        float4 w[4];
        conv_taps4(a.conv_weight, X, a.H, h, 8 * c16 + 4 * hf, w);
        float win[3][4];
#pragma unroll
        for (int j = 0; j < 3; ++j) {
          const int r = 8 * rb - 3 + j;
          const uint8_t* src = r >= 0 ? rows + qk_off(r, c16) : halo + (3 + r) * 256 + c16 * 16;
          unpack4(*reinterpret_cast<const uint2*>(src + 8 * hf), win[j]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = 8 * rb + i;
          uint2* p = reinterpret_cast<uint2*>(rows + qk_off(r, c16) + 8 * hf);
          const uint2 y = conv_row4(w, win, *p);
          if (i < 5) *p = y;
          else held[hf][i - 5] = y;
        }
      }
      __syncthreads();
#pragma unroll
      for (int i = 5; i < 8; ++i) {
        const int r = 8 * rb + i;
        *reinterpret_cast<uint4*>(rows + qk_off(r, c16)) =
            make_uint4(held[0][i - 5].x, held[0][i - 5].y, held[1][i - 5].x, held[1][i - 5].y);
      }
      __syncthreads();
    }

    // ---- 2. running log2-decay per channel (warps 0-3, the channel's 64 rows in
    //      registers); L2 norms of the q, k rows (warps 4-7, one row per thread) ----
    if (tid < kD) {  // thread tid scans channel tid of the rows
      // beta of row tid (stored after the scan) and the decay logits' scale and
      // bias of channel tid: loaded when the item's copies were issued
      const float bt = __uint_as_float(pre_beta << 16), dA = pre_scale, db = pre_bias;
      float x[kC];
#pragma unroll
      for (int r = 0; r < kC; ++r) {
        x[r] = G[gidx(r, tid)];
        if constexpr (kLogit) x[r] = a.g_min * sigmoid_fast(dA * (x[r] + db));  // g_min sigmoid(A (z + b))
        x[r] = fminf(fmaxf(x[r], a.g_min), 0.f);
      }
      if (len < kC) {  // rows past the sequence end: log alpha 0 (identity steps)
#pragma unroll
        for (int r = 0; r < kC; ++r)
          if (r >= len) x[r] = 0.f;
      }
      float run = 0.f;
#pragma unroll
      for (int r = 0; r < kC; ++r) {
        run += x[r] * kLog2e;
        x[r] = run;
      }
#pragma unroll
      for (int r = 0; r < kC; ++r) G[gidx(r, tid)] = x[r];
      if (tid < kC) s_beta[tid] = (a.beta_is_logit && tid < len) ? sigmoidf_(bt) : bt;
    } else {
      // one row per thread (q rows 0..63, then k rows): its sixteen 16-byte chunks
      // (wherever the swizzle put them) in an order rotated by the row, so that a
      // warp's loads hit every bank
      const int rr = tid - kD, r = rr & (kC - 1);
      const uint8_t* src = sm + (rr < kC ? kPrepQ : kPrepK) + r * 128;
      float2 s2[4] = {};  // packed f32x2 sums of squares (even, odd channel of a pair)
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int p = (i + rr) & 15;  // physical chunk: half p / 8, position p % 8
        const uint4 x = *reinterpret_cast<const uint4*>(src + (p >> 3) * 8192 + ((p & 7) << 4));
        const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 v2 = make_float2(__uint_as_float(wv[u] << 16), __uint_as_float(wv[u] & 0xFFFF0000u));
          s2[u] = fma2(v2, v2, s2[u]);
        }
      }
      const float sl = ((s2[0].x + s2[0].y) + (s2[1].x + s2[1].y)) +
                       ((s2[2].x + s2[2].y) + (s2[3].x + s2[3].y)) + a.eps_l2;
      const float inv = a.l2norm_qk ? (sl > 0.f ? rsqrtf(sl) : 0.f) : 1.f;
      if (rr < kC) s_invq[r] = inv * a.q_scale;
      else s_invk[r] = inv;
    }
    __syncthreads();

    // ---- 3. Gram matrices over two 32-token spans sp (rows 32 sp .. 32 sp + 31),
    //   each rescaled about its middle row m = 32 sp + 15: from there the running
    //   log2-decay moves by at most 16 * 5 * log2(e) < 116, so every factor below
    //   lies within 2^-116 .. 2^116 (bf16 range).
    //   A (TMEM, both 64-channel halves): lane r = k^_r 2^(g_r - g_m), lane 64 + r
    //   = q^_r 2^(g_r - g_m), m the middle row of r's span.
    //   B_sp (shared memory, one half at a time, stacked as [B_0; B_1] for one
    //   N = 96 product): rows j < 32 (sp + 1) = k^_j 2^(g_m - g_j).
    //   D_sp = A B_sp^T then holds K~ K-^T and Q~ K-^T on the rows of span sp
    //   (its other rows, and the columns j > r, are never read); bf16 hi/lo,
    //   D += A_hi B_hi + A_hi B_lo + A_lo B_hi.
    fence_after_sync();
    {
      // A: lane 32 (warp % 4) + lane, channel half warp / 4 (the TMEM column of a
      // store is one for the whole warp: every lane takes the same group)
      const int rho = (warp & 3) * 32 + lane, r = rho & (kC - 1), khA = warp >> 2;
      const int mr = 32 * (r >> 5) + 15;
      const uint8_t* xrows = sm + (rho < kC ? kPrepK : kPrepQ);
      const float inv = rho < kC ? s_invk[r] : s_invq[r];
      const float2 inv2 = make_float2(inv, inv);
#pragma unroll 2
      for (int gi = 0; gi < 8; ++gi) {
        const int c = 8 * khA + gi;
        float g8[8], m8[8], xf[8];
        ld8g_rows(G, r, c, g8);
        ld8g_rows(G, mr, c, m8);
        unpack8(*reinterpret_cast<const uint4*>(xrows + qk_off(r, c)), xf);
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 d = sub2(make_float2(g8[2 * u], g8[2 * u + 1]),
                                make_float2(m8[2 * u], m8[2 * u + 1]));
          split2v(mul2(make_float2(xf[2 * u], xf[2 * u + 1]),
                       mul2(make_float2(ex2f(d.x), ex2f(d.y)), inv2)), hi[u], lo[u]);
        }
        // channels 8 gi .. +7 of the half are the bf16 pairs in columns 4 gi .. +3
        const uint32_t col = kTdA + 64 * khA + 4 * gi;
        tmem_st4(taddr(tmem, (warp & 3) * 32, col), hi[0], hi[1], hi[2], hi[3]);
        tmem_st4(taddr(tmem, (warp & 3) * 32, col + 32), lo[0], lo[1], lo[2], lo[3]);
      }
    }
    {
      // B items of half kh: warp w takes the 8-channel group w of the half, lane
      // l the B rows 32 s3 + l (s3 = 0: span 0 row l; s3 = 1, 2: span 1 row
      // 32 (s3 - 1) + l), so that a warp reads one group of 32 rows
      const int c8 = warp;
      uint4 vh[3], vl[3];
      uint32_t vo[3];
      auto b_items = [&](int kh) {
        float m0[8], m1[8];
        ld8g_rows(G, 15, 8 * kh + c8, m0);  // the same for every lane
        ld8g_rows(G, 47, 8 * kh + c8, m1);
#pragma unroll
        for (int s3 = 0; s3 < 3; ++s3) {
          const int j = s3 == 0 ? lane : 32 * (s3 - 1) + lane;
          float g8[8], kf[8];
          ld8g_rows(G, j, 8 * kh + c8, g8);
          unpack8(*reinterpret_cast<const uint4*>(sm + kPrepK + qk_off(j, 8 * kh + c8)), kf);
          const float ik = s_invk[j];
          const float2 ik2 = make_float2(ik, ik);
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float2 m = s3 ? make_float2(m1[2 * u], m1[2 * u + 1])
                                : make_float2(m0[2 * u], m0[2 * u + 1]);
            const float2 d = sub2(m, make_float2(g8[2 * u], g8[2 * u + 1]));
            split2v(mul2(make_float2(kf[2 * u], kf[2 * u + 1]),
                         mul2(make_float2(ex2f(d.x), ex2f(d.y)), ik2)), hi[u], lo[u]);
          }
          vh[s3] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          vl[s3] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          vo[s3] = sw128_chunk(32 * s3 + lane, c8, 96);
        }
      };
      auto b_store = [&]() {
#pragma unroll
        for (int s3 = 0; s3 < 3; ++s3) {
          *reinterpret_cast<uint4*>(sm + kPrepBh + vo[s3]) = vh[s3];
          *reinterpret_cast<uint4*>(sm + kPrepBl + vo[s3]) = vl[s3];
        }
      };
      auto gram_mma = [&](int kh) {
        // one product for both spans: D columns 0..31 (D_0) and 32..95 (D_1)
        const uint64_t dh = desc_k_sw128(smem_u32(sm + kPrepBh), 0);
        const uint64_t dl = desc_k_sw128(smem_u32(sm + kPrepBl), 0);
        // a K-step of 16 channels: 8 TMEM columns of A, 32 bytes (+2 in the
        // descriptor's address field) of each B row
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint32_t ah = tmem + kTdA + 64 * kh + 8 * ks, al = ah + 32;
          mma_ts(tmem + kTdD0, ah, dh + 2 * ks, kIdGram, (kh | ks) ? 1u : 0u);
          mma_ts(tmem + kTdD0, ah, dl + 2 * ks, kIdGram, 1u);
          mma_ts(tmem + kTdD0, al, dh + 2 * ks, kIdGram, 1u);
        }
        mma_commit(&bar_mma);
      };
      b_items(0);
      b_store();
      tmem_wait_st();
      fence_proxy_async();
      fence_before_sync();
      __syncthreads();
      if (tid == 0) {
        fence_after_sync();
        gram_mma(0);
      }
      // half 1's B rows are computed while half 0's products read the tiles
      b_items(1);
      const bool waited = mbar_wait(&bar_mma, mma_phase, t.spins);
      mma_phase ^= 1;
      fence_after_sync();
      b_store();
      fence_proxy_async();
      fence_before_sync();
      ok = __syncthreads_and(waited);
      if (!ok) goto fail;
      if (tid == 0) {
        fence_after_sync();
        gram_mma(1);
      }
    }
    // ---- 5. row pass, while the Gram's last products run: -Q~ rows, K^ rows and
    //      G_C straight to the workspace; K~ (fp16) stays in registers until every
    //      read of the k rows is done.  Item (row r, 8-channel group c16) =
    //      tid + 256 m ----
    uint4 kt4[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int e = tid + kPrepThreads * m, r = e >> 4, c16 = e & 15;
      float g8[8], gl8[8], kf[8], qf[8];
      ld8g(G, r, c16, g8);
      ld8g(G, kC - 1, c16, gl8);
      unpack8(*reinterpret_cast<const uint4*>(sm + kPrepK + qk_off(r, c16)), kf);
      unpack8(*reinterpret_cast<const uint4*>(sm + kPrepQ + qk_off(r, c16)), qf);
      const float ik = s_invk[r], iq = -s_invq[r];
      const float2 ik2 = make_float2(ik, ik), iq2 = make_float2(iq, iq);
      uint32_t wk[4], wq[4], wh[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float2 g2 = make_float2(g8[2 * u], g8[2 * u + 1]);
        const float2 d = sub2(make_float2(gl8[2 * u], gl8[2 * u + 1]), g2);
        const float2 e2 = make_float2(ex2f(g2.x), ex2f(g2.y));
        const float2 f2 = make_float2(ex2f(d.x), ex2f(d.y));
        const float2 k2 = mul2(make_float2(kf[2 * u], kf[2 * u + 1]), ik2);
        const float2 q2 = mul2(make_float2(qf[2 * u], qf[2 * u + 1]), iq2);
        const float2 kt2 = mul2(k2, e2), qt2 = mul2(q2, e2), kh2 = mul2(k2, f2);
        wk[u] = pack_half2(kt2.x, kt2.y);
        wq[u] = pack_half2(qt2.x, qt2.y);
        wh[u] = pack_half2(kh2.x, kh2.y);
      }
      kt4[m] = make_uint4(wk[0], wk[1], wk[2], wk[3]);
      *reinterpret_cast<uint4*>(ws + kWsWQ + sw128_chunk(kC + r, c16, 128)) =
          make_uint4(wq[0], wq[1], wq[2], wq[3]);
      *reinterpret_cast<uint4*>(ws + kWsKh + sw128_chunk(r, c16, kC)) =
          make_uint4(wh[0], wh[1], wh[2], wh[3]);
    }
    if (tid < kD) reinterpret_cast<float*>(ws + kWsGam)[tid] = ex2f(G[gidx(kC - 1, tid)]);
    ok = __syncthreads_and(mbar_wait(&bar_mma, mma_phase, t.spins));
    mma_phase ^= 1;
    if (!ok) goto fail;
    fence_after_sync();
    // every read of the q, k rows is done: they take K~ and the v rows (bf16, by
    // two tensor copies that land during the solve), both MN-major (the q/k row
    // layout is the MN-major operand layout)
    if (tid == 0) {
      mbar_arrive_expect_tx(&bar_v, kC * kD * 2);
      tma_load_3d(sm + kPrepV, &t.tm_v, 0, h, tok0, &bar_v);
      tma_load_3d(sm + kPrepV + 8192, &t.tm_v, 64, h, tok0, &bar_v);
    }
    v_pending = true;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int e = tid + kPrepThreads * m, r = e >> 4, c16 = e & 15;
      *reinterpret_cast<uint4*>(sm + kPrepKt + sw128_chunk(r, c16, kC)) = kt4[m];
    }

    {
      // ---- 4. A (lanes 0..63) to shared memory, P (lanes 64..127) to the workspace ----
      float* Amat = reinterpret_cast<float*>(sm + kPrepAmat);
      {
        const int quarter = warp & 3, chalf = warp >> 2;
        const int r = quarter * 32 + lane;
        // columns j = 32 chalf .. +31 of D_sp, sp = the span of the warp's rows;
        // span 0 has only j < 32 (the rest of its rows' columns are j > r: zero)
        const int sp = quarter & 1;
        uint32_t x[32];
        if (sp || chalf == 0) {
          tmem_ld32(taddr(tmem, quarter * 32, (sp ? kTdD1 : kTdD0) + 32 * chalf), x);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = 0u;
        }
        if (r < kC) {
          const float br = s_beta[r];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int jj = 32 * chalf + j;
            Amat[r * kAs + jj] = (jj < r) ? br * __uint_as_float(x[j]) : 0.f;
          }
        } else {
          const int tr = r - kC;
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            uint32_t w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int j0 = 8 * c8 + 2 * u, jj = 32 * chalf + j0;
              w[u] = pack_half2(jj <= tr ? __uint_as_float(x[j0]) : 0.f,
                                jj + 1 <= tr ? __uint_as_float(x[j0 + 1]) : 0.f);
            }
            *reinterpret_cast<uint4*>(ws + kWsP + sw128_chunk(tr, 4 * chalf + c8, 64)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      fence_before_sync();
      __syncthreads();

      // ---- 6. X = (I + A)^-1: warps 0-1 invert the diagonal 16-blocks (fp32)
      //      while warps 4-7 clear the blocks above the diagonal and lay out the
      //      B operand A_10^T; warps 0-3 then complete the diagonal 32-blocks
      //      (fp32, named barrier), and warp 0 forms the lower 32-block
      //      X_10 = -X_11 A_10 X_00 = (X_11 A_10) (-X_00) by two bf16 hi/lo
      //      products on the tensor cores (as the Gram), while the other warps
      //      write the parts of T that need no X_10 ----
      float* X = reinterpret_cast<float*>(sm + kPrepInv);
      float* Y = reinterpret_cast<float*>(sm + kPrepY);
      // K-major bf16 hi/lo tile of the B operand tile[c][m] = sgn * src[m][c]
      // (m, c = 0..31; src row stride ld): 8 rows m of column c per unit
      auto b_tile = [&](const float* src, int ld, float sgn, uint32_t thi, uint32_t tlo,
                        int c, int m8) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          split2v(make_float2(sgn * src[(8 * m8 + 2 * u) * ld + c],
                              sgn * src[(8 * m8 + 2 * u + 1) * ld + c]), hi[u], lo[u]);
        const uint32_t o = sw128_chunk(c, m8, 32);
        *reinterpret_cast<uint4*>(sm + thi + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(sm + tlo + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      };
      if (tid >= kPrepHalf) {
        for (int e = tid - kPrepHalf; e < 6 * 256; e += kPrepHalf) {
          const int blk = e >> 8, r = (e >> 4) & 15, cc = e & 15;
          const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
          const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
          X[(16 * bi + r) * kXs + 16 * bj + cc] = 0.f;
        }
        // A_10 = A rows 32..63, columns 0..31; unit (column c = lane, 8 rows m8)
        const int u = tid - kPrepHalf;
        b_tile(Amat + 32 * kAs, kAs, 1.f, kPrepA10h, kPrepA10l, u & 31, u >> 5);
        fence_proxy_async();
      } else if (tid < 64) {  // diagonal blocks: thread = (block bi, column cc); right-looking
          const int bi = tid >> 4, cc = tid & 15, o = 16 * bi;  // (x[m] final -> update
          float x[16];                                          // rows below: 15-FMA chain)
#pragma unroll
          for (int r = 0; r < 16; ++r) x[r] = (r == cc) ? 1.f : 0.f;
#pragma unroll
          for (int m = 0; m < 15; ++m) {
#pragma unroll
            for (int r = m + 1; r < 16; ++r) x[r] -= Amat[(o + r) * kAs + o + m] * x[m];
          }
#pragma unroll
          for (int r = 0; r < 16; ++r) X[(o + r) * kXs + o + cc] = x[r];
      }
      __syncthreads();  // the diagonal 16-blocks are complete, the upper blocks clear
      if (tid < kPrepHalf) {
        // 2 x 2 block inverse at 32 x 32: the lower 16 x 16 block of each diagonal
        // 32-block, X_{2p+1,2p} = -X_{2p+1,2p+1} A_{2p+1,2p} X_{2p,2p} (B1, B2).
        // Each unit is 4 adjacent columns of one row (float4 loads), unrolled.
        {  // B1: Y_p = A_{2p+1,2p} X_{2p,2p}; unit (p, r, c4)
          const int p = tid >> 6, r = (tid >> 2) & 15, c4 = (tid & 3) * 4;
          const int i1 = 16 * (2 * p + 1), i0 = 32 * p;
          const float2* arow = reinterpret_cast<const float2*>(Amat + (i1 + r) * kAs + i0);
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int m2 = 0; m2 < 8; ++m2) {
            const float2 am = arow[m2];
            fma4s(acc, am.x, *reinterpret_cast<const float4*>(X + (i0 + 2 * m2) * kXs + i0 + c4));
            fma4s(acc, am.y, *reinterpret_cast<const float4*>(X + (i0 + 2 * m2 + 1) * kXs + i0 + c4));
          }
          *reinterpret_cast<float4*>(Y + (p << 8) + r * 16 + c4) = acc;
        }
        named_sync(kBarSolve, kPrepHalf);
        {  // B2: X_{2p+1,2p} = -X_{2p+1,2p+1} Y_p
          const int p = tid >> 6, r = (tid >> 2) & 15, c4 = (tid & 3) * 4;
          const int i1 = 16 * (2 * p + 1), i0 = 32 * p;
          const float4* xrow = reinterpret_cast<const float4*>(X + (i1 + r) * kXs + i1);
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int m4 = 0; m4 < 4; ++m4) {
            const float4 xm = xrow[m4];
            const float* yb = Y + (p << 8) + 4 * m4 * 16 + c4;
            fma4s(acc, xm.x, *reinterpret_cast<const float4*>(yb));
            fma4s(acc, xm.y, *reinterpret_cast<const float4*>(yb + 16));
            fma4s(acc, xm.z, *reinterpret_cast<const float4*>(yb + 32));
            fma4s(acc, xm.w, *reinterpret_cast<const float4*>(yb + 48));
          }
          *reinterpret_cast<float4*>(X + (i1 + r) * kXs + i0 + c4) =
              make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        }
      }
      __syncthreads();  // the diagonal 32-blocks of X are complete

      // ---- 7. T = X Diag(beta): [T; T] (K-major [t][j] fp16, rows 64..127 repeat
      //      rows 0..63) over A for the W product; T as a bf16 hi/lo pair over the
      //      decay rows for the U~ product (V stays exact in bf16).  Written by
      //      row and 8-column group: the block of X_10 by warp 0 from its
      //      registers, the rest by the other warps while warp 0's products run ----
      // T columns 8 c8 .. 8 c8 + 7 of row tr from the 8 values x of X
      auto t_store = [&](int tr, int c8, const float (&x)[8]) {
        uint32_t w[4], th[4], tl[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j0 = 8 * c8 + 2 * u;
          const float2 t2 = make_float2(x[2 * u] * s_beta[j0], x[2 * u + 1] * s_beta[j0 + 1]);
          w[u] = pack_half2(t2.x, t2.y);
          split2v(t2, th[u], tl[u]);
        }
        const uint4 wt = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(sm + kPrepTT + sw128_chunk(tr, c8, 128)) = wt;
        *reinterpret_cast<uint4*>(sm + kPrepTT + sw128_chunk(kC + tr, c8, 128)) = wt;
        *reinterpret_cast<uint4*>(sm + kPrepThi + sw128_chunk(tr, c8, kC)) =
            make_uint4(th[0], th[1], th[2], th[3]);
        *reinterpret_cast<uint4*>(sm + kPrepTlo + sw128_chunk(tr, c8, kC)) =
            make_uint4(tl[0], tl[1], tl[2], tl[3]);
      };
      // unit e: the rows of T that need no X_10 (rows 0..31, then the columns
      // 32..63 of rows 32..63), 8 columns each
      auto t_unit = [&](int e) {
        const int tr = e < 256 ? e >> 3 : 32 + ((e - 256) >> 2);
        const int c8 = e < 256 ? e & 7 : 4 + (e & 3);
        const float4 a4 = *reinterpret_cast<const float4*>(X + tr * kXs + 8 * c8);
        const float4 b4 = *reinterpret_cast<const float4*>(X + tr * kXs + 8 * c8 + 4);
        const float x[8] = {a4.x, a4.y, a4.z, a4.w, b4.x, b4.y, b4.z, b4.w};
        t_store(tr, c8, x);
      };
      bool solved = true;
      if (warp == 0) {
        // the lower 32-block: A = X_11 (X rows 32..63, columns 32..63) to TMEM lane = row - 32
        {
          const float4* xr = reinterpret_cast<const float4*>(X + (32 + lane) * kXs + 32);
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            const float4 x4 = xr[q4];
            split2v(make_float2(x4.x, x4.y), hi[2 * q4], lo[2 * q4]);
            split2v(make_float2(x4.z, x4.w), hi[2 * q4 + 1], lo[2 * q4 + 1]);
          }
          tmem_st16(taddr(tmem, 0, kTdX11), hi);
          tmem_st16(taddr(tmem, 0, kTdX11 + 16), lo);
        }
        tmem_wait_st();
        fence_before_sync();
        __syncwarp();
        // D = X_11 A_10 (K = 32: two steps of 16 = 8 TMEM columns, 32 bytes of
        // each B row).  The B tile's hi and lo halves are one 64-row tile, so
        // A_hi [B_hi; B_lo]^T is one N = 64 product (columns 0..31: hi.hi, 32..63:
        // hi.lo) and A_lo B_hi^T accumulates into columns 0..31: 4 MMAs, each
        // costing the issuing thread about as much as one of N = 32
        auto inv_mma = [&](uint32_t a_col, uint32_t d_col, uint32_t bh) {
          fence_after_sync();
          const uint64_t dh = desc_k_sw128(smem_u32(sm + bh), 0);
#pragma unroll
          for (int ks = 0; ks < 2; ++ks) {
            const uint32_t ah = tmem + a_col + 8 * ks, al = ah + 16;
            mma_ts(tmem + d_col, ah, dh + 2 * ks, kIdInv64, ks ? 1u : 0u);
            mma_ts(tmem + d_col, al, dh + 2 * ks, kIdInv32, 1u);
          }
          mma_commit(&bar_mma);
        };
        static_assert(kPrepA10l == kPrepA10h + 32 * 128 && kPrepX00l == kPrepX00h + 32 * 128,
                      "each B operand's lo tile follows its hi tile as rows 32..63");
        if (lane == 0) inv_mma(kTdX11, kTdY, kPrepA10h);
        // the B operand -X_00^T while the first product runs: unit (column c =
        // lane, 8 rows m8)
#pragma unroll
        for (int m8 = 0; m8 < 4; ++m8) b_tile(X, kXs, -1.f, kPrepX00h, kPrepX00l, lane, m8);
        fence_proxy_async();
        solved = mbar_wait(&bar_mma, mma_phase, t.spins);
        if (solved) {
          mma_phase ^= 1;
          fence_after_sync();
          uint32_t y[32], y2[32], hi[16], lo[16];
          tmem_ld32(taddr(tmem, 0, kTdY), y);
          tmem_ld32(taddr(tmem, 0, kTdY + 32), y2);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 16; ++u)
            split2v(make_float2(__uint_as_float(y[2 * u]) + __uint_as_float(y2[2 * u]),
                                __uint_as_float(y[2 * u + 1]) + __uint_as_float(y2[2 * u + 1])),
                    hi[u], lo[u]);
          tmem_st16(taddr(tmem, 0, kTdYs), hi);
          tmem_st16(taddr(tmem, 0, kTdYs + 16), lo);
          tmem_wait_st();
          fence_before_sync();
          __syncwarp();
          if (lane == 0) inv_mma(kTdYs, kTdX10, kPrepX00h);
          solved = mbar_wait(&bar_mma, mma_phase, t.spins);
          if (solved) {
            mma_phase ^= 1;
            fence_after_sync();
            // T rows 32..63, columns 0..31 straight from X_10 (lane = row - 32)
            tmem_ld32(taddr(tmem, 0, kTdX10), y);
            tmem_ld32(taddr(tmem, 0, kTdX10 + 32), y2);
            tmem_wait_ld();
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
              float x[8];
#pragma unroll
              for (int j = 0; j < 8; ++j)
                x[j] = __uint_as_float(y[8 * c8 + j]) + __uint_as_float(y2[8 * c8 + j]);
              t_store(32 + lane, c8, x);
            }
          }
        }
        fence_before_sync();
      } else {
        for (int e = tid - 32; e < 32 * 8 + 32 * 4; e += kPrepThreads - 32) t_unit(e);
      }
      ok = __syncthreads_and(solved);  // T is complete
      if (!ok) goto fail;
      // the v rows have landed once bar_v completes; the barrier that checks it
      // is the one before the products (after the convolution's first barrier
      // when the convolution is on)
      const bool vok = mbar_wait(&bar_v, v_phase, t.spins);
      if constexpr (kConv) {
        ok = __syncthreads_and(vok);
        if (!ok) goto fail;
        // ---- 7b. short convolution + Swish of the v rows in place (MN-major
        //      tile): thread = (4-row block, 8-channel group) ----
        const int c16 = tid & 15, rb = tid >> 4;
        const uint8_t* halo = sm + kPrepHalo + 2 * 3 * 256;
        uint2 held[2][3];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          float4 w[4];
          conv_taps4(a.conv_weight, 2, a.H, h, 8 * c16 + 4 * hf, w);
          float win[3][4];
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            const int r = 4 * rb - 3 + j;
            const uint8_t* src = r >= 0 ? sm + kPrepV + sw128_chunk(r, c16, kC) : halo + (3 + r) * 256 + c16 * 16;
            unpack4(*reinterpret_cast<const uint2*>(src + 8 * hf), win[j]);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint2* p = reinterpret_cast<uint2*>(sm + kPrepV + sw128_chunk(4 * rb + i, c16, kC) + 8 * hf);
            const uint2 y = conv_row4(w, win, *p);
            if (i == 0) *p = y;
            else held[hf][i - 1] = y;
          }
        }
        __syncthreads();
#pragma unroll
        for (int i = 1; i < 4; ++i)
          *reinterpret_cast<uint4*>(sm + kPrepV + sw128_chunk(4 * rb + i, c16, kC)) =
              make_uint4(held[0][i - 1].x, held[0][i - 1].y, held[1][i - 1].x, held[1][i - 1].y);
      }
      fence_proxy_async();
      fence_before_sync();
      ok = __syncthreads_and(vok);
      if (!ok) goto fail;
      v_phase ^= 1;
      v_pending = false;

      // ---- 8. U~^T = V^T (T_hi + T_lo)^T (A = V MN-major bf16) and W = [T; T] K~
      //      (B = K~ MN-major fp16) on the tensor cores, then both straight to the
      //      workspace.  The T_hi and T_lo tiles are one 128-row tile, so U~^T is
      //      one N = 128 product per K-step with its hi and lo parts side by side
      //      (summed on the way out): 8 MMAs ----
      static_assert(kPrepTlo == kPrepThi + kC * 128, "T_lo follows T_hi as rows 64..127");
      if (tid == 0) {
        fence_after_sync();
        const uint32_t sT = smem_u32(sm + kPrepTT), sV = smem_u32(sm + kPrepV);
        const uint32_t sKt = smem_u32(sm + kPrepKt);
        const uint32_t sTh = smem_u32(sm + kPrepThi);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          mma_ss(tmem + kTdU, desc_mn_sw128(sV, ks, kC * 128), desc_k_sw128(sTh, 32 * ks),
                 kIdUt, ks > 0);
          mma_ss(tmem + kTdW, desc_k_sw128(sT, 32 * ks), desc_mn_sw128(sKt, ks, kC * 128),
                 kIdW, ks > 0);
        }
        mma_commit(&bar_mma);
      }
      ok = __syncthreads_and(mbar_wait(&bar_mma, mma_phase, t.spins));
      mma_phase ^= 1;
      if (!ok) goto fail;
      fence_after_sync();
      // the products are done with every buffer: the next item's inputs stream in
      // while this one's results leave TMEM
      const int w_next = item + (int)gridDim.x;
      int gid_n = 0, h_n = 0, tok0_n = 0, len_n = 0, n_n = 0, s0_n = 0;
      if (w_next < items) {
        decode(w_next, gid_n, h_n, tok0_n, len_n, n_n, s0_n);
        issue_inputs(h_n, tok0_n, len_n, n_n, s0_n);
        in_pending = true;
      }
      {
        // U~^T and W go to the free region X in the workspace's byte layout (U~^T:
        // 16 KB; W: rows 0..63 of each 128-byte K-block of [W; -Q~], 8 KB each)
        // and leave by three 1-D bulk copies: stored directly, each warp store
        // would touch 32 different 128-byte lines.
        // warp (quarter, chalf): U~^T rows ch = its TMEM lanes, columns t = 32 chalf ..;
        // W rows t = its lanes mod 64 (both copies), 32-column slab 2 chalf + quarter / 2
        const int quarter = warp & 3, chalf = warp >> 2;
        const int lrow = quarter * 32 + lane, slab = 2 * chalf + (quarter >> 1);
        uint32_t x[32], y[32];
        tmem_ld32(taddr(tmem, quarter * 32, kTdU + 32 * chalf), x);
        tmem_ld32(taddr(tmem, quarter * 32, kTdU + 64 + 32 * chalf), y);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j)  // the T_hi and T_lo parts of U~^T
          x[j] = __float_as_uint(__uint_as_float(x[j]) + __uint_as_float(y[j]));
        tmem_ld32(taddr(tmem, quarter * 32, kTdW + 32 * slab), y);
        tmem_wait_ld();
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          uint32_t w[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            w[u] = pack_half2(__uint_as_float(x[8 * c8 + 2 * u]), __uint_as_float(x[8 * c8 + 2 * u + 1]));
          *reinterpret_cast<uint4*>(sm + kPrepStU + sw128_chunk(lrow, 4 * chalf + c8, 128)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
        const int tw = lrow & (kC - 1);
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          uint32_t w[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            w[u] = pack_half2(__uint_as_float(y[8 * c8 + 2 * u]), __uint_as_float(y[8 * c8 + 2 * u + 1]));
          const uint32_t o = sw128_chunk(tw, 4 * slab + c8, 128);  // K-block 1 from 16384
          *reinterpret_cast<uint4*>(sm + kPrepStW + (o < 16384u ? o : o - 8192u)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      fence_proxy_async();
      fence_before_sync();  // the TMEM reads above before the next item's TMEM writes
      __syncthreads();
      if (tid == 0) {
        bulk_s2g(ws + kWsUt, sm + kPrepStU, 16384);
        bulk_s2g(ws + kWsWQ, sm + kPrepStW, 8192);
        bulk_s2g(ws + kWsWQ + 16384, sm + kPrepStW + 8192, 8192);
        bulk_commit();
      }
      if (w_next >= items) break;
      item = w_next;
      gid = gid_n;
      h = h_n;
      tok0 = tok0_n;
      len = len_n;
      nseq = n_n;
      sstart = s0_n;
    }
  }
  goto done;
fail:
  // a bounded wait gave up: report, then wait (bounded) for this CTA's own
  // copies and MMAs before releasing TMEM and shared memory
  if (tid == 0) {
    report(a.status, KDA_ERR_TIMEOUT);
    mma_commit(&bar_mma);
    mbar_wait(&bar_mma, mma_phase, t.spins);
    if (in_pending) mbar_wait(&bar_in, in_phase, t.spins);
    if (v_pending) mbar_wait(&bar_v, v_phase, t.spins);
  }
done:
  if (tid == 0) bulk_wait_all();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, kPrepTmemCols);
}

// ============================================================ chain kernel
// 512 threads.  Warps 0-7 carry the state (conversions split by column half;
// thread 0 also issues the MMAs); warps 8-15 run the epilogue from a
// double-buffered O^T, overlapping the next chunk, and their first thread
// issues the bulk load of chunk i + 2 as soon as chunk i's MMAs are done.  Warp
// w touches TMEM lanes 32*(w%4) .. +31 (lane = d_v index).  Per chunk i:
//   -S^T -> fp16 operand, S^T <- S^T Diag(G_C)   (state warps)
//   D = (-S^T) W^T, then O^T = (-S^T)(-Q~)^T     (8 + 8 MMAs, N = 64; D first)
//   U^T = U~^T + D -> fp16 operand               (state warps, U~^T from the block)
//   S^T += U^T K^ (the critical path), O^T += U^T P^T
//   y rows from O^T                              (epilogue warps)
// Every bounded wait is followed by a vote of the group (reducing barrier), so
// that a timeout makes the whole group leave its loop together.
constexpr int kChThreads = 512;
constexpr int kChState = 256;  // state group: warps 0-7; epilogue group: warps 8-15
constexpr int kChEpi = kChThreads - kChState;
constexpr uint32_t kChBuf0 = 0;
constexpr uint32_t kChBuf1 = kWsStride;
constexpr uint32_t kChE = 2 * kWsStride;             // fp32 [64][kEStride] epilogue
constexpr int kEStride = kD + 4;
constexpr uint32_t kChG = kChE + kC * kEStride * 4;  // gate rows, bf16 [2][64][128]
constexpr uint32_t kChSmem = kChG + 2 * kC * kD * 2 + 1024;
static_assert(kChSmem <= 227 * 1024, "chain kernel shared memory");

// TMEM columns: S^T fp32; [U^T | O^T] fp32 in two buffers; -S^T fp16 operand;
// U^T fp16 operand in two buffers
constexpr uint32_t kTS = 0, kTUO0 = 128, kTAS = 384, kTAU0 = 448;
constexpr uint32_t kBarState = 1, kBarEpi = 2;  // named barriers of the two groups
constexpr int kLoader = kChState;  // epilogue thread that issues the bulk loads


// Hardware tanh (tanh.approx.f32, maximum relative error about 2^-11); the
// gate uses sigmoid(x) = (1 + tanh(x / 2)) / 2, one MUFU operation per value.
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(kChThreads, 1) chain_kernel(TcArgs t) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_full[2], bar_u, bar_s, bar_o[2], bar_oe[2], bar_dbg;
  __shared__ uint32_t tmem_base;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;  // TMEM lane of this thread = d_v index
  const PrefillArgs& a = t.a;
  // packed sequences: CTA b takes head b % H of the sequence at position b / H
  // of the chunk-base kernel's order (longest first)
  const int h = blockIdx.x % a.H;
  const int n = a.cu_seqlens ? t.chunk_base[a.N + 1 + (int)blockIdx.x / a.H] : (int)blockIdx.x / a.H;
  const size_t H = (size_t)a.H;
  int s0, s1;
  seq_range(a.cu_seqlens, a.N, a.T_total, n, s0, s1);
  if (s0 < 0 || s1 < s0 || s1 > a.T_total) return;  // reported by chunk_base_kernel
  const int nchunks = (s1 - s0 + kC - 1) / kC;
  // first chunk of the sequence (equal lengths: by arithmetic; the chunk bases
  // are complete before the prep grid starts)
  const int cbase = a.cu_seqlens ? t.chunk_base[n] : n * nchunks;
  const size_t sbase = ((size_t)n * H + h) * (size_t)(kD * kD);

  if (tid == 0) {
    mbar_init(&bar_full[0], 1);
    mbar_init(&bar_full[1], 1);
    mbar_init(&bar_u, 1);
    mbar_init(&bar_s, 1);
    mbar_init(&bar_o[0], 1);
    mbar_init(&bar_o[1], 1);
    mbar_init(&bar_oe[0], 1);  // O^T of the buffer copied out by the epilogue
    mbar_init(&bar_oe[1], 1);
    mbar_init(&bar_dbg, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (t.debug_timeout) {  // test hook: a wait that nothing completes, before any async work
    const bool ok = __syncthreads_and(mbar_wait(&bar_dbg, 0, 1000));
    if (!ok && tid == 0) report(a.status, KDA_ERR_TIMEOUT);
    if (!ok) return;
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  auto issue_load = [&](int i) {
    uint8_t* dst = sm + ((i & 1) ? kChBuf1 : kChBuf0);
    const uint8_t* src = ws_block(t, cbase + i, h);
    mbar_arrive_expect_tx(&bar_full[i & 1], kWsBytes);
    for (int p = 0; p < kWsParts; ++p)
      bulk_g2s(dst + kWsPartOff[p], src + kWsPartOff[p], kWsPartLen[p], &bar_full[i & 1]);
  };
  int issued = 0;  // loads issued (kLoader)
  if (tid == kLoader) {
    // the chunk blocks are the prep grid's output: everything above overlaps its
    // end when this grid starts early
    grid_wait_prerequisites();
    for (int i = 0; i < 2 && i < nchunks; ++i) issue_load(i);
    issued = min(2, nchunks);
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base;
  const uint32_t lane_base = taddr(tmem, quarter * 32, 0);
  bool ok = true;

  if (tid < kChState) {
    const int chalf = warp >> 2;  // column half of this state warp
    // S0 -> S^T in TMEM (lane = d_v index i, column = d_k index c)
    for (int p = 0; p < 2; ++p) {
      uint32_t r[32];
      const int c0 = 64 * chalf + 32 * p;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        r[j] = __float_as_uint(a.S0 ? a.S0[sbase + (size_t)(c0 + j) * kD + row] : 0.f);
      tmem_st32(lane_base + kTS + c0, r);
    }
    tmem_wait_st();
    for (int i = 0; i < nchunks; ++i) {
      const uint8_t* buf = sm + ((i & 1) ? kChBuf1 : kChBuf0);
      const uint32_t tUO = tmem + kTUO0 + 128 * (i & 1), tAU = kTAU0 + 32 * (i & 1);
      bool w = mbar_wait(&bar_full[i & 1], (i >> 1) & 1, t.spins);
      if (i > 0) w = w && mbar_wait(&bar_s, (i - 1) & 1, t.spins);
      ok = named_sync_and(kBarState, kChState, w);
      if (!ok) break;
      fence_after_sync();
      // -S^T (fp16) into the A operand of the product below
      const float4* gam4 = reinterpret_cast<const float4*>(buf + kWsGam) + 16 * chalf;
      uint32_t x0[32], x1[32];
      tmem_ld32(lane_base + kTS + 64 * chalf, x0);
      tmem_ld32(lane_base + kTS + 64 * chalf + 32, x1);
      tmem_wait_ld();
      if (i > 0) {  // the state after i full chunks, when a snapshot is due there
        const int m = snapshot_slot(a, i * kC);
        if (m >= 0) {
          float* dst = a.snapshots + (((size_t)n * a.snapshot_slots + m) * H + h) * (kD * kD) +
                       (size_t)(64 * chalf) * kD + row;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            dst[(size_t)j * kD] = __uint_as_float(x0[j]);
            dst[(size_t)(32 + j) * kD] = __uint_as_float(x1[j]);
          }
        }
      }
      {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          pk[j] = pack_half2(-__uint_as_float(x0[2 * j]), -__uint_as_float(x0[2 * j + 1]));
        tmem_st16(lane_base + kTAS + 32 * chalf, pk);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          pk[j] = pack_half2(-__uint_as_float(x1[2 * j]), -__uint_as_float(x1[2 * j + 1]));
        tmem_st16(lane_base + kTAS + 32 * chalf + 16, pk);
        tmem_wait_st();
      }
      fence_before_sync();
      named_sync(kBarState, kChState);
      bool woe = true;
      if (tid == 0) {
        fence_after_sync();
        // U^T - U~^T = (-S^T) W^T into columns 0..63 of [U | O] buffer i & 1, the
        // state chain's product, committed on its own; then O^T = (-S^T)(-Q~)^T
        // into columns 64..127, once the epilogue has copied O^T(i - 2) out of
        // them (bar_s below covers it).  B = rows 0..63 (W) or 64..127 (-Q~: +8 KB,
        // +512 in the descriptor's address field) of the tile; K-step: +2 (32
        // bytes); K-block of 64: +1024 (16 KB)
        const uint64_t dWQ = desc_k_sw128(smem_u32(buf) + kWsWQ, 0);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ts(tUO, tmem + kTAS + 8 * ks, dWQ + 1024 * (ks >> 2) + 2 * (ks & 3), kIdF16N64,
                 ks > 0);
        mma_commit(&bar_u);
        if (i >= 2) woe = mbar_wait(&bar_oe[i & 1], ((i - 2) >> 1) & 1, t.spins);
        if (woe) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_ts(tUO + 64, tmem + kTAS + 8 * ks, dWQ + 512 + 1024 * (ks >> 2) + 2 * (ks & 3),
                   kIdF16N64, ks > 0);
        }
      }
      // S^T <- S^T Diag(G_C) while the product runs (only S^T += U^T K^ below
      // reads it; the wait before that barrier covers these stores)
#pragma unroll
      for (int j4 = 0; j4 < 8; ++j4) {
        const float4 g0 = gam4[j4], g1 = gam4[8 + j4];
        x0[4 * j4 + 0] = __float_as_uint(__uint_as_float(x0[4 * j4 + 0]) * g0.x);
        x0[4 * j4 + 1] = __float_as_uint(__uint_as_float(x0[4 * j4 + 1]) * g0.y);
        x0[4 * j4 + 2] = __float_as_uint(__uint_as_float(x0[4 * j4 + 2]) * g0.z);
        x0[4 * j4 + 3] = __float_as_uint(__uint_as_float(x0[4 * j4 + 3]) * g0.w);
        x1[4 * j4 + 0] = __float_as_uint(__uint_as_float(x1[4 * j4 + 0]) * g1.x);
        x1[4 * j4 + 1] = __float_as_uint(__uint_as_float(x1[4 * j4 + 1]) * g1.y);
        x1[4 * j4 + 2] = __float_as_uint(__uint_as_float(x1[4 * j4 + 2]) * g1.z);
        x1[4 * j4 + 3] = __float_as_uint(__uint_as_float(x1[4 * j4 + 3]) * g1.w);
      }
      tmem_st32(lane_base + kTS + 64 * chalf, x0);
      tmem_st32(lane_base + kTS + 64 * chalf + 32, x1);
      // U~^T (this thread's row, its 32 columns) from the chunk block meanwhile
      uint4 ut[4];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        ut[c] = *reinterpret_cast<const uint4*>(buf + kWsUt + sw128_chunk(row, 4 * chalf + c, 128));
      ok = named_sync_and(kBarState, kChState, mbar_wait(&bar_u, i & 1, t.spins) && woe);
      if (!ok) break;
      fence_after_sync();
      {  // U^T = U~^T + the product -> fp16 A operand (column half per warp)
        uint32_t x0[32], pk[16];
        tmem_ld32(lane_base + (tUO - tmem) + 32 * chalf, x0);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t hw = (&ut[j >> 2].x)[j & 3];
          const float2 u2 = __half22float2(*reinterpret_cast<const __half2*>(&hw));
          pk[j] = pack_half2(__uint_as_float(x0[2 * j]) + u2.x, __uint_as_float(x0[2 * j + 1]) + u2.y);
        }
        tmem_st16(lane_base + tAU + 16 * chalf, pk);
        tmem_wait_st();
      }
      fence_before_sync();
      named_sync(kBarState, kChState);
      if (tid == 0) {
        fence_after_sync();
        const uint32_t sb = smem_u32(buf);
        const uint64_t dP = desc_k_sw128(sb + kWsP, 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)  // S^T += U^T K^: the state chain first
          mma_ts(tmem + kTS, tmem + tAU + 8 * ks, desc_mn_sw128(sb + kWsKh, ks, kC * 128),
                 kIdKh, 1);
        mma_commit(&bar_s);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)  // O^T += U^T P^T
          mma_ts(tUO + 64, tmem + tAU + 8 * ks, dP + 2 * ks, kIdF16N64, 1);
        mma_commit(&bar_o[i & 1]);
      }
    }
    if (ok && nchunks > 0)
      ok = named_sync_and(kBarState, kChState, mbar_wait(&bar_s, (nchunks - 1) & 1, t.spins));
    if (ok) {  // final state S^T -> S_T[c][i] (and its snapshot slot, if one is due)
      fence_after_sync();
      const int m = snapshot_slot(a, s1 - s0);
      float* snap = m >= 0 ? a.snapshots + (((size_t)n * a.snapshot_slots + m) * H + h) * (kD * kD)
                           : nullptr;
      for (int p = 0; p < 2; ++p) {
        uint32_t r[32];
        const int c0 = 64 * chalf + 32 * p;
        tmem_ld32(lane_base + kTS + c0, r);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          a.S_T[sbase + (size_t)(c0 + j) * kD + row] = __uint_as_float(r[j]);
          if (snap) snap[(size_t)(c0 + j) * kD + row] = __uint_as_float(r[j]);
        }
      }
    } else if (tid == 0) {
      // a bounded wait gave up: report it, then wait (bounded) for this CTA's
      // own MMAs and bulk copies before TMEM and shared memory are released
      report(a.status, KDA_ERR_TIMEOUT);
      mma_commit(&bar_dbg);
      mbar_wait(&bar_dbg, 0, t.spins);
    }
  } else {
    // ---------------- epilogue warps: O^T (lane = d_v) -> E[t][d_v] -> rows of y.
    // Warp 8 + 4 ehalf + quarter copies columns t = 32 ehalf .. +31 of its lane
    // quarter.  Four threads own one token row: thread (er, eq) takes the
    // 8-channel groups q = eq + 4c, c = 0..3.
    const int et = tid - kChState;            // 0..255
    const int er = et >> 2, eq = et & 3;      // token row, channel-group phase
    const int ehalf = (warp - 8) >> 2;
    const __nv_bfloat16* gate = static_cast<const __nv_bfloat16*>(a.gate);
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.o);
    float* E = reinterpret_cast<float*>(sm + kChE);
    // The gate rows stream into a two-slot ring by 16-byte asynchronous copies,
    // two chunks ahead; each thread copies exactly the 64 bytes it reads later
    // (16-byte group q of row er sits at position (q + 4 (er & 1)) mod 16, so
    // the reads of a warp fall in distinct banks).
    auto gate_slot = [&](int i, int c) -> uint32_t {
      const int q = eq + 4 * c;
      return kChG + (i & 1) * (kC * kD * 2) + er * (kD * 2) + (((q + 4 * (er & 1)) & 15) << 4);
    };
    auto fetch_gate = [&](int i) {
      if (gate && i < nchunks) {
        const int tok0 = s0 + i * kC;
        const bool live = er < min(kC, s1 - tok0);
        const __nv_bfloat16* src = gate + ((size_t)(tok0 + (live ? er : 0)) * H + h) * kD;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          cp_async16(smem_u32(sm + gate_slot(i, c)), src + 8 * (eq + 4 * c), live ? 16u : 0u);
      }
      cp_async_commit();  // one group per chunk, empty or not
    };
    fetch_gate(0);
    fetch_gate(1);
    for (int i = 0; i < nchunks; ++i) {
      const int tok0 = s0 + i * kC;
      const int len = min(kC, s1 - tok0);
      const bool live = er < len;
      const size_t rofs = ((size_t)(tok0 + er) * H + h) * kD;
      ok = named_sync_and(kBarEpi, kChEpi, mbar_wait(&bar_o[i & 1], (i >> 1) & 1, t.spins));
      if (!ok) {
        if (et == 0) report(a.status, KDA_ERR_TIMEOUT);
        break;
      }
      fence_after_sync();
      if (tid == kLoader && i + 2 < nchunks) {  // every MMA of chunk i is done: its
        fence_proxy_async();                    // buffer takes chunk i + 2
        issue_load(i + 2);
        issued = i + 3;
      }
      {
        uint32_t x0[32];
        tmem_ld32(lane_base + kTUO0 + 128 * (i & 1) + 64 + 32 * ehalf, x0);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) E[(32 * ehalf + j) * kEStride + row] = __uint_as_float(x0[j]);
      }
      fence_before_sync();
      named_sync(kBarEpi, kChEpi);
      if (et == 0) mbar_arrive(&bar_oe[i & 1]);  // O^T(i) is out of TMEM: the buffer is free
      // pass 1: sum of squares of the row; pass 2: outputs, 8 channels at a time
      // the row's 32 values of this thread stay in registers for both passes
      const float* erow = E + er * kEStride;
      float4 ev[8];
      float2 ss2 = make_float2(0.f, 0.f);  // packed f32x2 arithmetic: fewer issue slots
#pragma unroll                            // taken from the state warps
      for (int c = 0; c < 4; ++c) {
        const float4 v0 = *reinterpret_cast<const float4*>(erow + 8 * (eq + 4 * c));
        const float4 v1 = *reinterpret_cast<const float4*>(erow + 8 * (eq + 4 * c) + 4);
        ev[2 * c] = v0;
        ev[2 * c + 1] = v1;
        ss2 = fma2(make_float2(v0.x, v0.y), make_float2(v0.x, v0.y), ss2);
        ss2 = fma2(make_float2(v0.z, v0.w), make_float2(v0.z, v0.w), ss2);
        ss2 = fma2(make_float2(v1.x, v1.y), make_float2(v1.x, v1.y), ss2);
        ss2 = fma2(make_float2(v1.z, v1.w), make_float2(v1.z, v1.w), ss2);
      }
      float ss = ss2.x + ss2.y;
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      ss += __shfl_xor_sync(0xffffffffu, ss, 2);
      const float inv = gate ? rsqrtf(ss * (1.0f / kD) + a.eps_norm) : 1.f;
      const float hinv = 0.5f * inv;  // inv * sigmoid(g) = hinv * tanh(g / 2) + hinv
      cp_async_wait_group<1>();       // this thread's gate copies of chunk i have landed
      if (live) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int q = eq + 4 * c;
          const float4 v0 = ev[2 * c], v1 = ev[2 * c + 1];
          float y[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
          if (gate) {
            const uint4 graw = *reinterpret_cast<const uint4*>(sm + gate_slot(i, c));
            const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&graw);
            const float2 hinv2 = make_float2(hinv, hinv);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float2 gh = mul2(__bfloat1622float2(g2[u]), make_float2(0.5f, 0.5f));
              const float2 sg = fma2(make_float2(tanh_approx(gh.x), tanh_approx(gh.y)), hinv2, hinv2);
              const float2 yy = mul2(make_float2(y[2 * u], y[2 * u + 1]), sg);
              y[2 * u] = yy.x;
              y[2 * u + 1] = yy.y;
            }
            if (a.norm_weight) {
              const float4* w4 = reinterpret_cast<const float4*>(a.norm_weight + 8 * q);
              const float4 w0 = w4[0], w1 = w4[1];
              y[0] *= w0.x; y[1] *= w0.y; y[2] *= w0.z; y[3] *= w0.w;
              y[4] *= w1.x; y[5] *= w1.y; y[6] *= w1.z; y[7] *= w1.w;
            }
          }
          uint4 out;
          out.x = pack_bf162(y[0], y[1]);
          out.y = pack_bf162(y[2], y[3]);
          out.z = pack_bf162(y[4], y[5]);
          out.w = pack_bf162(y[6], y[7]);
          *reinterpret_cast<uint4*>(o + rofs + 8 * q) = out;
        }
      }
      fetch_gate(i + 2);  // slot i & 1 is read: it takes chunk i + 2
      named_sync(kBarEpi, kChEpi);  // E is free again
    }
    cp_async_wait_all();  // no copy into shared memory outlives the loop
    if (tid == kLoader && !ok) {
      // a bounded wait gave up: the last two loads may still be in flight; wait
      // (bounded) for them before shared memory is released
      for (int j = max(0, issued - 2); j < issued; ++j)
        mbar_wait(&bar_full[j & 1], (j >> 1) & 1, t.spins);
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// cuTensorMapEncodeTiled, reached through the runtime (no link against the
// driver library).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// Tensor map of a [T][H][128] token array of 2-byte (bf16) or 4-byte (fp32)
// elements: box 128 bytes of channels x 1 head x 64 tokens, 128-byte swizzle
// (base 16-byte aligned, checked by the caller).
bool encode_rows(CUtensorMap* m, const void* base, int T, int H, bool fp32) {
  const EncodeTiledFn fn = encode_tiled();
  if (!fn || T < 1) return false;
  const cuuint64_t esize = fp32 ? 4 : 2;
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)T};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * esize, (cuuint64_t)H * kD * esize};
  const cuuint32_t box[3] = {(cuuint32_t)(128 / esize), 1, (cuuint32_t)kC};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// workspace header: the chunk bases [N + 1] and the chain's sequence order [N]
size_t header_bytes(int N) { return ((size_t)(2 * N + 1) * 4 + 1023) & ~(size_t)1023; }
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
  static int sm_count[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    for (auto kern : {prep_kernel<false, false>, prep_kernel<true, false>,
                      prep_kernel<false, true>, prep_kernel<true, true>}) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kPrepSmem);
      if (e != cudaSuccess) return e;
    }
    e = cudaFuncSetAttribute(chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kChSmem);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  if (ev && (e = cudaEventRecord(ev[0], s)) != cudaSuccess) return e;
  if (a.cu_seqlens) {  // equal lengths need no chunk bases (their interval stays empty)
    chunk_base_kernel<<<1, 1024, 0, s>>>(t);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (ev && (e = cudaEventRecord(ev[1], s)) != cudaSuccess) return e;
  bool prep_launched = false;
  if (a.T_total > 0 && t.total_chunks_max > 0 && !t.debug_timeout) {
    if (!encode_rows(&t.tm_q, a.q, a.T_total, a.H, false) ||
        !encode_rows(&t.tm_k, a.k, a.T_total, a.H, false) ||
        !encode_rows(&t.tm_v, a.v, a.T_total, a.H, false) ||
        (a.decay_mode == KDA_DECAY_CHANNEL &&
         !encode_rows(&t.tm_la, a.log_alpha, a.T_total, a.H, true)))
      return cudaErrorInvalidValue;
    // persistent: two CTAs per SM walk the (chunk, head) items
    const long long items_max = (long long)t.total_chunks_max * a.H;
    const long long resident = 2LL * (dev >= 0 && dev < 64 ? sm_count[dev] : 148);
    const unsigned grid = (unsigned)(items_max < resident ? items_max : resident);
    auto kern = a.conv_weight ? (a.decay_from_logit ? prep_kernel<true, true>
                                                    : prep_kernel<true, false>)
                              : (a.decay_from_logit ? prep_kernel<false, true>
                                                    : prep_kernel<false, false>);
    kern<<<grid, kPrepThreads, kPrepSmem, s>>>(t);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    prep_launched = true;
  }
  if (ev && (e = cudaEventRecord(ev[2], s)) != cudaSuccess) return e;
  // After prep the chain starts early (programmatic dependent launch): its CTAs
  // load S0 and the first gate rows while prep's last items finish, and wait for
  // prep before reading its blocks.  Without prep it launches in order: it reads
  // S0 before that wait, which the kernels before it may have written.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.N * a.H));
  cfg.blockDim = dim3(kChThreads);
  cfg.dynamicSmemBytes = kChSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = prep_launched ? 1 : 0;
  if ((e = cudaLaunchKernelEx(&cfg, chain_kernel, t)) != cudaSuccess) return e;
  if (ev && (e = cudaEventRecord(ev[3], s)) != cudaSuccess) return e;
  return cudaSuccess;
}

}  // namespace kda
