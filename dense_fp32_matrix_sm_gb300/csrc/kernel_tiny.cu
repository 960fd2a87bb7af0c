// kernel_tiny.cu -- SGEMM for tiny products: small C tiles, K streamed
// through a shared-memory ring (any K).
//
// At 128^3 a product is 4 MFLOP, a few microseconds of one SM: the time
// goes to the launch, to the round trips that bring A and B in, and to how
// many SMs share the work ("Writing a Fast Matmul in CUDA, Step by Step",
// "Size effects": small sizes leave most of the machine idle; the remedy
// is more, smaller pieces of work).  The 128-row tiles of the main kernels
// give 128^3 two CTAs.  Here:
//  * A CTA owns a 32 x 32 tile of C and all of K.  K goes through a ring
//    of kTyStages chunks of 64 k: the A panel (32 x 64) and the B panel
//    (64 x 32) of a chunk are copied with cp.async -- 16-byte copies when
//    both operands' rows allow them, coalesced 4-byte copies otherwise (any
//    alignment and leading dimension) -- one commit group per chunk, the
//    first kTyStages - 1 chunks before any math, so their round trips
//    overlap each other and the math.  82 KB per CTA: two CTAs per SM, so
//    up to 2 x SMs tiles run in one wave.
//  * 256 threads in four k-groups of 64.  Group g takes the k-quads
//    q = g, g + 4, ... (interleaved, so every group has work for any K);
//    a thread of a group holds 4 rows (ty + 8i) x 4 columns.  Per k-quad:
//    four 16-byte reads of A (one per row, four k) and four of B (one per
//    k, four columns), then 32 FFMA2: a broadcast A element times a pair
//    of adjacent B columns (each half an IEEE fma, so the sums are those
//    of fmaf).  The A rows' smem stride (68 words, 4 mod 8) puts the four
//    rows a warp reads at once in different banks.
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
constexpr int kTyChunk = 64;                 // k per ring stage (16 k-quads: 4 per group)
constexpr int kTyStages = 4;
constexpr int kTyKa = kTyChunk + 4;          // A row stride in a stage (floats), 4 mod 8
constexpr int kTyStageA = kTyT * kTyKa;      // floats
constexpr int kTyStage = kTyStageA + kTyChunk * kTyT;
constexpr int kTySmemFloats = kTyStages * kTyStage + kTyGroups * kTyT * kTyT;
static_assert(kTyKa % 8 == 4 && kTyStageA % 4 == 0 && kTyStage % 4 == 0, "16-byte rows, conflict-free A reads");

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

constexpr int kTySmemBytes = kTySmemFloats * static_cast<int>(sizeof(float));

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

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// this thread's copies of all but the newest n commit groups have landed
template <int n>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(n) : "memory");
}

__global__ void __launch_bounds__(kTyThreads) sgemm_tiny_kernel(const TinyParams p) {
  extern __shared__ __align__(16) float ty_smem[];
  const int K = p.K;
  const int nchunks = (K + kTyChunk - 1) / kTyChunk;
  float* part = ty_smem + kTyStages * kTyStage;  // [4 groups][32][32]
  const int z = blockIdx.z;
  const int m0 = blockIdx.y * kTyT, n0 = blockIdx.x * kTyT;
  const float* A = p.A + z * p.stride_a;
  const float* B = p.B + z * p.stride_b;
  float* C = p.C + z * p.stride_c;
  const int t = threadIdx.x;

  // copy chunk c (k in [64c, 64c + 64)) into its ring stage; zeros outside the matrices
  auto issue = [&](int c) {
    float* as = ty_smem + (c % kTyStages) * kTyStage;  // [32][kTyKa]
    float* bs = as + kTyStageA;                        // [64][32]
    const int c0 = c * kTyChunk;
    if (p.vec) {
#pragma unroll
      for (int u = 0; u < kTyT * kTyChunk / 4 / kTyThreads; ++u) {  // A: 32 rows x 16 quads
        const int idx = t + u * kTyThreads;
        const int m = idx >> 4, kl = 4 * (idx & 15), k = c0 + kl;
        const uint32_t bytes = m0 + m < p.M && k < K ? (K - k >= 4 ? 16u : 4u * (K - k)) : 0u;
        if (SG_CHK(SG_IN((c % kTyStages) * kTyStage + m * kTyKa + kl + 3, kTySmemFloats), p.status))
          cp_async16(as + m * kTyKa + kl, bytes ? A + static_cast<int64_t>(m0 + m) * p.lda + k : A, bytes);
      }
#pragma unroll
      for (int u = 0; u < kTyChunk * kTyT / 4 / kTyThreads; ++u) {  // B: 64 rows x 8 quads of columns
        const int idx = t + u * kTyThreads;
        const int kl = idx >> 3, n = 4 * (idx & 7), k = c0 + kl;
        const uint32_t bytes = k < K && n0 + n < p.N ? (p.N - n0 - n >= 4 ? 16u : 4u * (p.N - n0 - n)) : 0u;
        if (SG_CHK(SG_IN((c % kTyStages) * kTyStage + kTyStageA + kl * kTyT + n + 3, kTySmemFloats), p.status))
          cp_async16(bs + kl * kTyT + n, bytes ? B + static_cast<int64_t>(k) * p.ldb + n0 + n : B, bytes);
      }
    } else {
#pragma unroll 4
      for (int u = 0; u < kTyT * kTyChunk / kTyThreads; ++u) {  // A: along rows (coalesced)
        const int idx = t + u * kTyThreads;
        const int m = idx >> 6, kl = idx & 63, k = c0 + kl;
        if (!SG_CHK(SG_IN((c % kTyStages) * kTyStage + m * kTyKa + kl, kTySmemFloats), p.status)) continue;
        float* d = as + m * kTyKa + kl;
        if (m0 + m < p.M && k < K) cp_async4(d, A + static_cast<int64_t>(m0 + m) * p.lda + k);
        else *d = 0.f;
      }
#pragma unroll 4
      for (int u = 0; u < kTyChunk * kTyT / kTyThreads; ++u) {
        const int idx = t + u * kTyThreads;
        const int kl = idx >> 5, n = idx & (kTyT - 1), k = c0 + kl;
        if (!SG_CHK(SG_IN((c % kTyStages) * kTyStage + kTyStageA + kl * kTyT + n, kTySmemFloats), p.status)) continue;
        float* d = bs + kl * kTyT + n;
        if (k < K && n0 + n < p.N) cp_async4(d, B + static_cast<int64_t>(k) * p.ldb + n0 + n);
        else *d = 0.f;
      }
    }
  };

  // group g, thread (ty, tx): rows ty + 8i, columns 4 tx .. 4 tx + 3 as two pairs
  const int g = t / kTyGroupThreads, gt = t % kTyGroupThreads;
  const int tx = gt & 7, ty = gt >> 3;
  float2 acc[4][2];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = make_float2(0.f, 0.f);

#pragma unroll
  for (int c = 0; c < kTyStages - 1; ++c) {
    if (c < nchunks) issue(c);
    cp_async_commit();  // one group per chunk slot, empty past the last chunk
  }
  for (int c = 0; c < nchunks; ++c) {
    cp_async_wait<kTyStages - 2>();  // chunk c's copies (this thread's) have landed
    __syncthreads();                 // everyone's have; everyone is done with chunk c - 1
    if (c + kTyStages - 1 < nchunks) issue(c + kTyStages - 1);  // into chunk c - 1's stage
    cp_async_commit();
    const float* as = ty_smem + (c % kTyStages) * kTyStage;
    const float* arow = as + ty * kTyKa;
    const float* bcol = as + kTyStageA + 4 * tx;
    // a chunk is 16 k-quads, so group g's quads are q = g, g + 4, g + 8, g + 12 in every chunk
#pragma unroll
    for (int qq = 0; qq < kTyChunk / 4 / kTyGroups; ++qq) {
      const int q = g + kTyGroups * qq;
      if (!SG_CHK(SG_IN((c % kTyStages) * kTyStage + (ty + 24) * kTyKa + 4 * q + 3, kTySmemFloats) &&
                      SG_IN((c % kTyStages) * kTyStage + kTyStageA + (4 * q + 3) * kTyT + 4 * tx + 3, kTySmemFloats),
                  p.status))
        break;
      float4 a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4*>(arow + 8 * i * kTyKa + 4 * q);
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = *reinterpret_cast<const float4*>(bcol + (4 * q + j) * kTyT);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const float4 bk = kk == 0 ? b[0] : kk == 1 ? b[1] : kk == 2 ? b[2] : b[3];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
          acc[i][0] = __ffma2_rn(make_float2(av, av), make_float2(bk.x, bk.y), acc[i][0]);
          acc[i][1] = __ffma2_rn(make_float2(av, av), make_float2(bk.z, bk.w), acc[i][1]);
        }
      }
    }
  }
  cp_async_wait<0>();
  // partial tiles, then each thread adds one float4 of outputs over the groups in order
  float* mine = part + g * kTyT * kTyT;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    *reinterpret_cast<float4*>(mine + (ty + 8 * i) * kTyT + 4 * tx) =
        make_float4(acc[i][0].x, acc[i][0].y, acc[i][1].x, acc[i][1].y);
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
                              kTySmemBytes);
}

cudaError_t tiny_occupancy(int* ctas) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, sgemm_tiny_kernel, kTyThreads, kTySmemBytes);
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
  sgemm_tiny_kernel<<<grid, kTyThreads, kTySmemBytes, stream>>>(p);
  return cudaGetLastError();
}

const Variant kTinyVariants[] = {
    // any alignment, leading dimension and K, strided batches on grid z
    Variant{"tiny_32x32", kKindTiny, kTyT, kTyT, kTyChunk, kTyStages, 1, kTyThreads, kTySmemBytes, -1, &tiny_prepare,
            &tiny_occupancy, &tiny_launch, 0, 0, 1},
};

}  // namespace

const Variant* tiny_variants(int* count) {
  *count = static_cast<int>(sizeof(kTinyVariants) / sizeof(kTinyVariants[0]));
  return kTinyVariants;
}

}  // namespace sgemm
