// umma_selftest.cu -- checks of the tensor-core building blocks in
// linear_attention_recurrence_prefill_gb300/csrc/umma.cuh, driven by
// tests/test_umma.py: one tcgen05.mma chain (A from shared memory or from TMEM,
// B from shared memory; each shared-memory operand in the 128-byte-swizzled
// K-major or MN-major layout), TMEM load/store, mbarrier waits with a bound,
// and 1-D bulk copies.
//
// Every wait is bounded; on a timeout the kernel records it and returns.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../linear_attention_recurrence_prefill_gb300/csrc/umma.cuh"

using namespace kda::umma;

namespace {

constexpr long long kLimit = 2000000000LL;  // ~1 s of cycles

// D[128 x N] = A[128 x K] * B[N x K]^T, fp32 accumulate.
// A, B: row-major 16-bit (fp16 or bf16) in global memory.  a_in_tmem: A is
// staged in TMEM (fp16/bf16 pairs per 32-bit column) instead of shared memory.
// a_mn / b_mn: that operand is staged MN-major (64-element M/N blocks of
// K rows of 128 B) instead of K-major.
__global__ void __launch_bounds__(128) mma_kernel(const uint16_t* __restrict__ A,
                                                  const uint16_t* __restrict__ B,
                                                  float* __restrict__ D, int N, int K,
                                                  uint32_t idesc, int a_in_tmem, int a_mn,
                                                  int b_mn, int* status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t* sA = smem_raw + pad;
  uint8_t* sB = sA + 128 * K * 2;
  const int tid = threadIdx.x, warp = tid >> 5;

  // operands into the swizzled K-major or MN-major layout
  for (int e = tid; e < 128 * K; e += 128) {
    const int r = e / K, k = e % K;
    const uint32_t off = a_mn ? sw128_offset(k, r, K) : sw128_offset(r, k, 128);
    *reinterpret_cast<uint16_t*>(sA + off) = A[e];
  }
  for (int e = tid; e < N * K; e += 128) {
    const int r = e / K, k = e % K;
    const uint32_t off = b_mn ? sw128_offset(k, r, K) : sw128_offset(r, k, N);
    *reinterpret_cast<uint16_t*>(sB + off) = B[e];
  }
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, 256);
    tmem_relinquish();
  }
  fence_proxy_async();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tbase = tmem_base;
  const uint32_t d_tmem = tbase;           // columns [0, N)
  const uint32_t a_tmem = tbase + 128;     // columns [128, 128 + K/2)

  if (a_in_tmem) {
    // thread r owns row r = lane r: K/2 packed columns
    const int r = tid;
    for (int c0 = 0; c0 < K / 2; c0 += 32) {
      uint32_t v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int k = 2 * (c0 + j);
        v[j] = (uint32_t)A[r * K + k] | ((uint32_t)A[r * K + k + 1] << 16);
      }
      tmem_st32(taddr(a_tmem, warp * 32, c0), v);
    }
    tmem_wait_st();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();

  if (tid == 0) {
    for (int ks = 0; ks < K / 16; ++ks) {
      const uint32_t kb = ks >> 2, kbyte = (ks & 3) * 32;
      const uint64_t bdesc = b_mn ? desc_mn_sw128(smem_u32(sB), ks, K * 128)
                                  : desc_k_sw128(smem_u32(sB) + kb * N * 128, kbyte);
      if (a_in_tmem) {
        mma_ts(d_tmem, a_tmem + ks * 8, bdesc, idesc, ks > 0);
      } else {
        const uint64_t adesc = a_mn ? desc_mn_sw128(smem_u32(sA), ks, K * 128)
                                    : desc_k_sw128(smem_u32(sA) + kb * 128 * 128, kbyte);
        mma_ss(d_tmem, adesc, bdesc, idesc, ks > 0);
      }
    }
    mma_commit(&bar);
  }
  const bool ok = mbar_wait(&bar, 0, kLimit);
  if (!ok && tid == 0) atomicExch(status, 1);
  fence_after_sync();
  if (ok) {
    for (int c0 = 0; c0 < N; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(taddr(d_tmem, warp * 32, c0), v);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (c0 + j < N) D[tid * N + c0 + j] = __uint_as_float(v[j]);
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, 256);
}

// Round trip global -> shared (several bulk copies on one mbarrier) -> global.
__global__ void bulk_kernel(const uint8_t* src, uint8_t* dst, const int* sizes, int nparts,
                            int* status) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ uint64_t bar;
  int total = 0;
  for (int i = 0; i < nparts; ++i) total += sizes[i];
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bar, (uint32_t)total);
    int off = 0;
    for (int i = 0; i < nparts; ++i) {
      bulk_g2s(sm + off, src + off, (uint32_t)sizes[i], &bar);
      off += sizes[i];
    }
  }
  const bool ok = mbar_wait(&bar, 0, kLimit);
  if (!ok && threadIdx.x == 0) atomicExch(status, 1);
  __syncthreads();
  if (ok && threadIdx.x == 0) {
    fence_proxy_async();
    bulk_s2g(dst, sm, (uint32_t)total);
    bulk_commit();
    bulk_wait_all();
  }
}

}  // namespace

extern "C" {

// Returns 0 on success, 1 if the kernel reported a timeout, -1 on a CUDA error.
int selftest_mma(const void* A, const void* B, float* D, int N, int K, int bf16,
                 int a_in_tmem, int a_mn, int b_mn) {
  if (N % 16 || N < 16 || N > 128 || K % 64 || K < 64 || K > 128) return -2;
  if ((a_mn && a_in_tmem) || (b_mn && N % 64)) return -2;  // MN-major: whole 64-wide blocks
  int* status = nullptr;
  if (cudaMalloc(&status, sizeof(int)) != cudaSuccess) return -1;
  cudaMemset(status, 0, sizeof(int));
  // 64 KB of slack past the operands: any descriptor reads stay inside the allocation
  const size_t smem = 1024 + (size_t)(128 + N) * K * 2 + 65536;
  cudaFuncSetAttribute(mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  mma_kernel<<<1, 128, smem>>>(static_cast<const uint16_t*>(A),
                               static_cast<const uint16_t*>(B), D, N, K,
                               idesc_f16(128, N, bf16 != 0, a_mn != 0, b_mn != 0), a_in_tmem,
                               a_mn, b_mn, status);
  cudaError_t e = cudaDeviceSynchronize();
  int h = 0;
  cudaMemcpy(&h, status, sizeof(int), cudaMemcpyDeviceToHost);
  cudaFree(status);
  if (e != cudaSuccess) return -1;
  return h;
}

int selftest_bulk(const void* src, void* dst, const int* sizes_host, int nparts) {
  int total = 0;
  for (int i = 0; i < nparts; ++i) {
    if (sizes_host[i] % 16) return -2;
    total += sizes_host[i];
  }
  int *status = nullptr, *sizes = nullptr;
  if (cudaMalloc(&status, sizeof(int)) != cudaSuccess) return -1;
  if (cudaMalloc(&sizes, sizeof(int) * nparts) != cudaSuccess) return -1;
  cudaMemset(status, 0, sizeof(int));
  cudaMemcpy(sizes, sizes_host, sizeof(int) * nparts, cudaMemcpyHostToDevice);
  cudaFuncSetAttribute(bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, total);
  bulk_kernel<<<1, 32, total>>>(static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst),
                                sizes, nparts, status);
  cudaError_t e = cudaDeviceSynchronize();
  int h = 0;
  cudaMemcpy(&h, status, sizeof(int), cudaMemcpyDeviceToHost);
  cudaFree(status);
  cudaFree(sizes);
  if (e != cudaSuccess) return -1;
  return h;
}

}  // extern "C"
