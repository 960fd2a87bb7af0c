// kernel_tiny.cu -- SGEMM for tiny products: small C tiles, whole
// K-panels in shared memory (K <= 512).
//
// At 128^3 a product is 4 MFLOP, a few microseconds of one SM: the time
// goes to the launch, to the round trips that bring A and B in, and to how
// many SMs share the work ("Writing a Fast Matmul in CUDA, Step by Step",
// "Size effects": small sizes leave most of the machine idle; the remedy
// is more, smaller pieces of work).  The 128-row tiles of the main kernels
// give 128^3 two CTAs.  Here:
//  * A CTA owns a 32 x 32 tile of C and all of K.  Its A panel (32 x K)
//    and B panel (K x 32) are copied into shared memory at once with
//    cp.async -- 16-byte copies when both operands' rows allow them,
//    coalesced 4-byte copies otherwise (any alignment and leading
//    dimension) -- then one wait: one round trip for the whole panel
//    instead of one per k-slice, and no registers held by the copies.
//  * 256 threads in four k-groups of 64.  Group g takes the k-quads
//    q = g, g + 4, ... (interleaved, so every group has work for any K);
//    a thread of a group holds a 4 x 4 register tile.  Per k-quad: four
//    16-byte reads of A (one per row, four k) and four of B (one per k,
//    four columns), 64 FMAs.
//  * The four groups' partial tiles go to shared memory and every thread
//    finishes four outputs, adding the groups in order 0..3 -- a fixed
//    order, so reruns are bit-identical (k_order=split) -- then alpha*sum
//    (beta == 0, C not read) or fmaf(alpha, sum, beta*C).
//  * Rows past M, columns past N and k past K are zero-filled and never
//    stored.  Strided batches run on grid z.
#include <cuda_runtime.h>
#include <stdint.h>

#include "checked.cuh"
#include "kernels.h"

namespace sgemm {
namespace {

constexpr int kTyT = 32;       // tile rows and columns
constexpr int kTyGroups = 4;   // k-groups
constexpr int kTyGroupThreads = 64;
constexpr int kTyThreads = kTyGroups * kTyGroupThreads;
constexpr int kTyMaxK = 512;

struct TinyParams {
  const float* A;
  const float* B;
  float* C;
  int64_t lda, ldb, ldc;
  int M, N, K;
  float alpha, beta;
  int64_t stride_a, stride_b, stride_c;
  int vec;  // 16-byte copies: A, B 16-byte aligned, lda, ldb, strides multiples of 4
  unsigned int* status;  // per-device status word (checked build: bounds)
};

__host__ __device__ constexpr int tiny_ka(int K) { return ((K + 3) & ~3) + 4; }  // A row stride in smem (floats)
__host__ __device__ constexpr int tiny_kp(int K) { return (K + 3) & ~3; }        // k-rows of B in smem

int tiny_smem_bytes(int K) {
  // As[32][ka], Bs[kp][32], then the groups' partial tiles [4][32 x 32]
  return (kTyT * tiny_ka(K) + tiny_kp(K) * kTyT + kTyGroups * kTyT * kTyT) * static_cast<int>(sizeof(float));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte copy; bytes past src_bytes are zero-filled and not read
__device__ __forceinline__ void cp_async16(float* dst, const float* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void cp_async4(float* dst, const float* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__global__ void __launch_bounds__(kTyThreads) sgemm_tiny_kernel(const TinyParams p) {
  extern __shared__ __align__(16) float ty_smem[];
  const int K = p.K;
  const int ka = tiny_ka(K), kp = tiny_kp(K);
  float* as = ty_smem;                 // [32][ka], row-major
  float* bs = as + kTyT * ka;          // [kp][32]
  float* part = bs + kp * kTyT;        // [4 groups][32][32]
  const int z = blockIdx.z;
  const int m0 = blockIdx.y * kTyT, n0 = blockIdx.x * kTyT;
  const float* A = p.A + z * p.stride_a;
  const float* B = p.B + z * p.stride_b;
  float* C = p.C + z * p.stride_c;
  const int t = threadIdx.x;

  if (p.vec) {
    // A: 32 rows x kp/4 chunks; a warp covers 32 chunks of one or more rows
    const int qa = kp / 4;
    for (int idx = t; idx < kTyT * qa; idx += kTyThreads) {
      const int m = idx / qa, k = 4 * (idx - m * qa);
      const uint32_t bytes = m0 + m < p.M && k < K ? (K - k >= 4 ? 16u : 4u * (K - k)) : 0u;
      if (SG_CHK(SG_IN(m * ka + k + 3, kTyT * ka), p.status))
        cp_async16(as + m * ka + k, bytes ? A + static_cast<int64_t>(m0 + m) * p.lda + k : A, bytes);
    }
    // B: kp rows x 8 chunks of 4 columns
    for (int idx = t; idx < kp * (kTyT / 4); idx += kTyThreads) {
      const int k = idx >> 3, n = 4 * (idx & 7);
      const uint32_t bytes = k < K && n0 + n < p.N ? (p.N - n0 - n >= 4 ? 16u : 4u * (p.N - n0 - n)) : 0u;
      if (SG_CHK(SG_IN(k * kTyT + n + 3, kp * kTyT), p.status))
        cp_async16(bs + k * kTyT + n, bytes ? B + static_cast<int64_t>(k) * p.ldb + n0 + n : B, bytes);
    }
  } else {
    // 4-byte copies along rows (coalesced); zeros outside the matrices
    for (int idx = t; idx < kTyT * kp; idx += kTyThreads) {
      const int m = idx / kp, k = idx - m * kp;
      if (!SG_CHK(SG_IN(m * ka + k, kTyT * ka), p.status)) continue;
      float* d = as + m * ka + k;
      if (m0 + m < p.M && k < K) cp_async4(d, A + static_cast<int64_t>(m0 + m) * p.lda + k);
      else *d = 0.f;
    }
    for (int idx = t; idx < kp * kTyT; idx += kTyThreads) {
      const int k = idx >> 5, n = idx & (kTyT - 1);
      if (!SG_CHK(SG_IN(k * kTyT + n, kp * kTyT), p.status)) continue;
      float* d = bs + k * kTyT + n;
      if (k < K && n0 + n < p.N) cp_async4(d, B + static_cast<int64_t>(k) * p.ldb + n0 + n);
      else *d = 0.f;
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();

  // group g, thread (ty, tx): rows 4 ty .. 4 ty + 3, columns 4 tx .. 4 tx + 3
  const int g = t / kTyGroupThreads, gt = t % kTyGroupThreads;
  const int tx = gt & 7, ty = gt >> 3;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  const float* arow = as + 4 * ty * ka;
  const float* bcol = bs + 4 * tx;
#pragma unroll 2
  for (int q = g; q < kp / 4; q += kTyGroups) {
    if (!SG_CHK(SG_IN(4 * ty * ka + 3 * ka + 4 * q + 3, kTyT * ka) && SG_IN((4 * q + 3) * kTyT + 4 * tx + 3, kp * kTyT),
                p.status))
      break;
    float4 a[4], b[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4*>(arow + i * ka + 4 * q);
#pragma unroll
    for (int j = 0; j < 4; ++j) b[j] = *reinterpret_cast<const float4*>(bcol + (4 * q + j) * kTyT);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const float bv[4] = {kk == 0 ? b[0].x : kk == 1 ? b[1].x : kk == 2 ? b[2].x : b[3].x,
                           kk == 0 ? b[0].y : kk == 1 ? b[1].y : kk == 2 ? b[2].y : b[3].y,
                           kk == 0 ? b[0].z : kk == 1 ? b[1].z : kk == 2 ? b[2].z : b[3].z,
                           kk == 0 ? b[0].w : kk == 1 ? b[1].w : kk == 2 ? b[2].w : b[3].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av, bv[j], acc[i][j]);
      }
    }
  }
  // partial tiles, then each thread adds one float4 of outputs over the groups in order
  float* mine = part + g * kTyT * kTyT;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    *reinterpret_cast<float4*>(mine + (4 * ty + i) * kTyT + 4 * tx) =
        make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  __syncthreads();
  const int r = t >> 3, c = 4 * (t & 7);  // output row r, columns c .. c + 3
  if (!SG_CHK(SG_IN((kTyGroups - 1) * kTyT * kTyT + r * kTyT + c + 3, kTyGroups * kTyT * kTyT), p.status)) return;
  float4 s = *reinterpret_cast<const float4*>(part + r * kTyT + c);
#pragma unroll
  for (int gg = 1; gg < kTyGroups; ++gg) {
    const float4 o = *reinterpret_cast<const float4*>(part + gg * kTyT * kTyT + r * kTyT + c);
    s.x += o.x;
    s.y += o.y;
    s.z += o.z;
    s.w += o.w;
  }
  const int m = m0 + r;
  if (m >= p.M) return;
  float* crow = C + static_cast<int64_t>(m) * p.ldc + n0 + c;
  const float sv[4] = {s.x, s.y, s.z, s.w};
  if (p.beta == 0.f) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (n0 + c + j < p.N) crow[j] = p.alpha * sv[j];
  } else {
    float old[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) old[j] = n0 + c + j < p.N ? crow[j] : 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (n0 + c + j < p.N) crow[j] = fmaf(p.alpha, sv[j], p.beta * old[j]);
  }
}

cudaError_t tiny_prepare() {
  return cudaFuncSetAttribute(sgemm_tiny_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              tiny_smem_bytes(kTyMaxK));
}

cudaError_t tiny_occupancy(int* ctas) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, sgemm_tiny_kernel, kTyThreads, tiny_smem_bytes(kTyMaxK));
}

cudaError_t tiny_launch(const LaunchArgs& a, cudaStream_t stream) {
  TinyParams p;
  p.A = a.A;
  p.B = a.B;
  p.C = a.C;
  p.lda = a.lda;
  p.ldb = a.ldb;
  p.ldc = a.ldc;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.alpha = a.alpha;
  p.beta = a.beta;
  const int batch = a.batch > 1 ? a.batch : 1;
  p.stride_a = batch > 1 ? a.stride_a : 0;
  p.stride_b = batch > 1 ? a.stride_b : 0;
  p.stride_c = batch > 1 ? a.stride_c : 0;
  p.status = a.status;
  p.vec = (reinterpret_cast<uintptr_t>(a.A) & 15) == 0 && (reinterpret_cast<uintptr_t>(a.B) & 15) == 0 &&
          p.lda % 4 == 0 && p.ldb % 4 == 0 && p.stride_a % 4 == 0 && p.stride_b % 4 == 0;
  const dim3 grid((a.N + kTyT - 1) / kTyT, (a.M + kTyT - 1) / kTyT, batch);
  sgemm_tiny_kernel<<<grid, kTyThreads, tiny_smem_bytes(a.K), stream>>>(p);
  return cudaGetLastError();
}

const Variant kTinyVariants[] = {
    // any alignment and leading dimension, K <= 512, strided batches on grid z
    Variant{"tiny_32x32", kKindTiny, kTyT, kTyT, kTyMaxK, 1, 0, kTyThreads, 0, -1, &tiny_prepare, &tiny_occupancy,
            &tiny_launch, 0, 0, 1},
};

}  // namespace

const Variant* tiny_variants(int* count) {
  *count = static_cast<int>(sizeof(kTinyVariants) / sizeof(kTinyVariants[0]));
  return kTinyVariants;
}

}  // namespace sgemm
