// kernel_tiny.cu -- SGEMM for tiny and small products: small square C
// tiles, K streamed through a shared-memory ring (any K).
//
// At 128^3 a product is 4 MFLOP, a few microseconds of one SM: the time
// goes to the launch, to the round trips that bring A and B in, and to how
// many SMs share the work ("Writing a Fast Matmul in CUDA, Step by Step",
// "Size effects": small sizes leave most of the machine idle; the remedy
// is more, smaller pieces of work).  The 128-row tiles of the main kernels
// give 128^3 two CTAs.  Here (template on the tile side T = 32 or 64):
//  * A CTA owns a T x T tile of C and all of K.  K goes through a ring of
//    STAGES chunks of 64 k: the A panel (T x 64) and the B panel (64 x T)
//    of a chunk are copied with cp.async -- 16-byte copies when both
//    operands' rows allow them, coalesced 4-byte copies otherwise (any
//    alignment and leading dimension) -- one commit group per chunk, the
//    first STAGES - 1 chunks before any math, so their round trips overlap
//    each other and the math.  One CTA barrier per chunk.
//  * 256 threads in four k-groups of 64.  Group g takes the k-quads
//    q = g, g + 4, ... (interleaved, so every group has work for any K);
//    a thread of a group holds T/8 rows (ty + 8i) x T/8 columns (4 tx + 32h
//    + j), read KSTEP k at a time: per step one KSTEP-wide read of A per
//    row and T/32 16-byte reads of B per k, then FFMA2s, each a broadcast
//    A element times a pair of adjacent B columns (each half an IEEE fma,
//    so the sums are those of fmaf).  The A rows' stride in a
//    stage (68 words, 4 mod 8) puts the four rows a warp reads at once in
//    different banks.
//  * The four groups' partial tiles go to shared memory (over the ring,
//    which is idle by then) and every thread finishes T*T/256 outputs,
//    adding the groups in order 0..3 -- a fixed order, so reruns are
//    bit-identical (k_order=split) -- then alpha*sum (beta == 0, C not
//    read) or fmaf(alpha, sum, beta*C).
//  * Rows past M, columns past N and k past K are zero-filled and never
//    stored.  Strided batches run on grid z.
//  * tiny_32x32: 4 stages, 66 KB, KSTEP 4; small_64x64: 3 stages, 99 KB,
//    KSTEP 2 (so that 64 accumulators and the operands fit 128 registers:
//    two CTAs per SM).
#include <cuda_runtime.h>
#include <stdint.h>

#include "checked.cuh"
#include "kernels.h"

namespace sgemm {
namespace {

constexpr int kTyGroups = 4;  // k-groups
constexpr int kTyGroupThreads = 64;
constexpr int kTyThreads = kTyGroups * kTyGroupThreads;
constexpr int kTyChunk = 64;       // k per ring stage (16 k-quads: 4 per group)
constexpr int kTyKa = kTyChunk + 4;  // A row stride in a stage (floats), 4 mod 8
static_assert(kTyKa % 8 == 4, "conflict-free A reads");

template <int T, int STAGES>
struct TyShape {
  static constexpr int kStageA = T * kTyKa;            // floats
  static constexpr int kStage = kStageA + kTyChunk * T;
  static constexpr int kSmemFloats = STAGES * kStage;
  static constexpr int kSmemBytes = kSmemFloats * static_cast<int>(sizeof(float));
  static_assert(kStageA % 4 == 0 && kStage % 4 == 0, "16-byte rows");
  static_assert(kSmemFloats >= kTyGroups * T * T, "the partial tiles fit over the ring");
};

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

template <int KSTEP>
struct AVec;
template <>
struct AVec<4> {
  using type = float4;
  __device__ static float at(const float4& v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }
};
template <>
struct AVec<2> {
  using type = float2;
  __device__ static float at(const float2& v, int i) { return i == 0 ? v.x : v.y; }
};

template <int T, int STAGES, int KSTEP, int MINB>
__global__ void __launch_bounds__(kTyThreads, MINB) sgemm_tiny_kernel(const TinyParams p) {
  using S = TyShape<T, STAGES>;
  constexpr int RPT = T / 8;   // rows per thread: ty + 8i
  constexpr int HN = T / 32;   // column quads per thread: 4 tx + 32h
  constexpr int TQ = T / 4;    // column quads per tile row
  using AV = typename AVec<KSTEP>::type;
  extern __shared__ __align__(16) float ty_smem[];
  const int K = p.K;
  const int nchunks = (K + kTyChunk - 1) / kTyChunk;
  const int z = blockIdx.z;
  const int m0 = blockIdx.y * T, n0 = blockIdx.x * T;
  const float* A = p.A + z * p.stride_a;
  const float* B = p.B + z * p.stride_b;
  float* C = p.C + z * p.stride_c;
  const int t = threadIdx.x;

  // copy chunk c (k in [64c, 64c + 64)) into its ring stage; zeros outside the matrices
  auto issue = [&](int c) {
    const int so = (c % STAGES) * S::kStage;  // stage offset (floats)
    float* as = ty_smem + so;                 // [T][kTyKa]
    float* bs = as + S::kStageA;              // [64][T]
    const int c0 = c * kTyChunk;
    if (p.vec) {
#pragma unroll
      for (int u = 0; u < T * kTyChunk / 4 / kTyThreads; ++u) {  // A: T rows x 16 quads
        const int idx = t + u * kTyThreads;
        const int m = idx >> 4, kl = 4 * (idx & 15), k = c0 + kl;
        const uint32_t bytes = m0 + m < p.M && k < K ? (K - k >= 4 ? 16u : 4u * (K - k)) : 0u;
        if (SG_CHK(SG_IN(so + m * kTyKa + kl + 3, S::kSmemFloats), p.status))
          cp_async16(as + m * kTyKa + kl, bytes ? A + static_cast<int64_t>(m0 + m) * p.lda + k : A, bytes);
      }
#pragma unroll
      for (int u = 0; u < kTyChunk * T / 4 / kTyThreads; ++u) {  // B: 64 rows x T/4 quads of columns
        const int idx = t + u * kTyThreads;
        const int kl = idx / TQ, n = 4 * (idx % TQ), k = c0 + kl;
        const uint32_t bytes = k < K && n0 + n < p.N ? (p.N - n0 - n >= 4 ? 16u : 4u * (p.N - n0 - n)) : 0u;
        if (SG_CHK(SG_IN(so + S::kStageA + kl * T + n + 3, S::kSmemFloats), p.status))
          cp_async16(bs + kl * T + n, bytes ? B + static_cast<int64_t>(k) * p.ldb + n0 + n : B, bytes);
      }
    } else {
#pragma unroll 4
      for (int u = 0; u < T * kTyChunk / kTyThreads; ++u) {  // A: along rows (coalesced)
        const int idx = t + u * kTyThreads;
        const int m = idx >> 6, kl = idx & 63, k = c0 + kl;
        if (!SG_CHK(SG_IN(so + m * kTyKa + kl, S::kSmemFloats), p.status)) continue;
        float* d = as + m * kTyKa + kl;
        if (m0 + m < p.M && k < K) cp_async4(d, A + static_cast<int64_t>(m0 + m) * p.lda + k);
        else *d = 0.f;
      }
#pragma unroll 4
      for (int u = 0; u < kTyChunk * T / kTyThreads; ++u) {
        const int idx = t + u * kTyThreads;
        const int kl = idx / T, n = idx % T, k = c0 + kl;
        if (!SG_CHK(SG_IN(so + S::kStageA + kl * T + n, S::kSmemFloats), p.status)) continue;
        float* d = bs + kl * T + n;
        if (k < K && n0 + n < p.N) cp_async4(d, B + static_cast<int64_t>(k) * p.ldb + n0 + n);
        else *d = 0.f;
      }
    }
  };

  // group g, thread (ty, tx): rows ty + 8i, columns 4 tx + 32h + j as pairs (j = 0, 1), (2, 3)
  const int g = t / kTyGroupThreads, gt = t % kTyGroupThreads;
  const int tx = gt & 7, ty = gt >> 3;
  float2 acc[RPT][2 * HN];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
#pragma unroll
    for (int h = 0; h < 2 * HN; ++h) acc[i][h] = make_float2(0.f, 0.f);

#pragma unroll
  for (int c = 0; c < STAGES - 1; ++c) {
    if (c < nchunks) issue(c);
    cp_async_commit();  // one group per chunk slot, empty past the last chunk
  }
  for (int c = 0; c < nchunks; ++c) {
    cp_async_wait<STAGES - 2>();  // chunk c's copies (this thread's) have landed
    __syncthreads();              // everyone's have; everyone is done with chunk c - 1
    if (c + STAGES - 1 < nchunks) issue(c + STAGES - 1);  // into chunk c - 1's stage
    cp_async_commit();
    const int so = (c % STAGES) * S::kStage;
    const float* arow = ty_smem + so + ty * kTyKa;
    const float* bcol = ty_smem + so + S::kStageA + 4 * tx;
    // a chunk is 16 k-quads, so group g's quads are q = g, g + 4, g + 8, g + 12 in every chunk
    // (the 64-wide tile keeps one quad's operands live at a time: 128 registers)
    constexpr int kQuadUnroll = T == 64 ? 1 : 4;
#pragma unroll kQuadUnroll
    for (int qq = 0; qq < kTyChunk / 4 / kTyGroups; ++qq) {
      const int q = g + kTyGroups * qq;
#pragma unroll
      for (int st = 0; st < 4 / KSTEP; ++st) {
        const int k0 = 4 * q + KSTEP * st;  // first k of this step within the chunk
        if (!SG_CHK(SG_IN(so + (ty + 8 * (RPT - 1)) * kTyKa + k0 + KSTEP - 1, S::kSmemFloats) &&
                        SG_IN(so + S::kStageA + (k0 + KSTEP - 1) * T + 4 * tx + 32 * (HN - 1) + 3, S::kSmemFloats),
                    p.status))
          break;
        AV a[RPT];
#pragma unroll
        for (int i = 0; i < RPT; ++i) a[i] = *reinterpret_cast<const AV*>(arow + 8 * i * kTyKa + k0);
        float4 b[KSTEP][HN];
#pragma unroll
        for (int kk = 0; kk < KSTEP; ++kk)
#pragma unroll
          for (int h = 0; h < HN; ++h) b[kk][h] = *reinterpret_cast<const float4*>(bcol + (k0 + kk) * T + 32 * h);
#pragma unroll
        for (int kk = 0; kk < KSTEP; ++kk)
#pragma unroll
          for (int i = 0; i < RPT; ++i) {
            const float av = AVec<KSTEP>::at(a[i], kk);
#pragma unroll
            for (int h = 0; h < HN; ++h) {
              acc[i][2 * h] = __ffma2_rn(make_float2(av, av), make_float2(b[kk][h].x, b[kk][h].y), acc[i][2 * h]);
              acc[i][2 * h + 1] =
                  __ffma2_rn(make_float2(av, av), make_float2(b[kk][h].z, b[kk][h].w), acc[i][2 * h + 1]);
            }
          }
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();  // every thread is done with the ring: the partial tiles go over it
  // partial tiles [4 groups][T][T], then each thread adds T*T/256 outputs over the groups in order
  float* part = ty_smem;
  float* mine = part + g * T * T;
#pragma unroll
  for (int i = 0; i < RPT; ++i)
#pragma unroll
    for (int h = 0; h < HN; ++h)
      *reinterpret_cast<float4*>(mine + (ty + 8 * i) * T + 4 * tx + 32 * h) =
          make_float4(acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x, acc[i][2 * h + 1].y);
  __syncthreads();
#pragma unroll
  for (int u = 0; u < T * T / 4 / kTyThreads; ++u) {
    const int idx = t + u * kTyThreads;
    const int r = idx / TQ, c = 4 * (idx % TQ);  // output row r, columns c .. c + 3
    if (!SG_CHK(SG_IN((kTyGroups - 1) * T * T + r * T + c + 3, S::kSmemFloats), p.status)) return;
    float4 s = *reinterpret_cast<const float4*>(part + r * T + c);
#pragma unroll
    for (int gg = 1; gg < kTyGroups; ++gg) {
      const float4 o = *reinterpret_cast<const float4*>(part + gg * T * T + r * T + c);
      s.x += o.x;
      s.y += o.y;
      s.z += o.z;
      s.w += o.w;
    }
    const int m = m0 + r;
    if (m >= p.M) continue;
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
}

template <int T, int STAGES, int KSTEP, int MINB>
struct TinyVariant {
  using S = TyShape<T, STAGES>;
  static constexpr auto kernel = sgemm_tiny_kernel<T, STAGES, KSTEP, MINB>;
  static cudaError_t prepare() {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
  }
  static cudaError_t occupancy(int* ctas) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, kernel, kTyThreads, S::kSmemBytes);
  }
  static cudaError_t launch(const LaunchArgs& a, cudaStream_t stream) {
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
    const dim3 grid((a.N + T - 1) / T, (a.M + T - 1) / T, batch);
    kernel<<<grid, kTyThreads, S::kSmemBytes, stream>>>(p);
    return cudaGetLastError();
  }
  static Variant describe(const char* name) {
    // any alignment, leading dimension and K, strided batches on grid z
    return Variant{name, kKindTiny, T, T, kTyChunk, STAGES, 1, kTyThreads, S::kSmemBytes, -1, &prepare, &occupancy,
                   &launch, 0, 0, 1};
  }
};

const Variant kTinyVariants[] = {
    TinyVariant<32, 4, 4, 1>::describe("tiny_32x32"),
    TinyVariant<64, 3, 2, 2>::describe("small_64x64"),
};

}  // namespace

const Variant* tiny_variants(int* count) {
  *count = static_cast<int>(sizeof(kTinyVariants) / sizeof(kTinyVariants[0]));
  return kTinyVariants;
}

}  // namespace sgemm
