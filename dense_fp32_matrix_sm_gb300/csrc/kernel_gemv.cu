// kernel_gemv.cu -- C = alpha*A*B + beta*C for one to four rows: the
// matrix-vector end of the decode shape.
//
// With M <= 4 every element of B is used at most four times, so the product
// is a stream of B from HBM and nothing else ("Writing a Fast Matmul in
// CUDA, Step by Step", "Why decode doesn't care": a decode-step product
// multiplies each weight a handful of times and sits on the bandwidth
// roof).  There is no reuse for shared memory to capture, so B goes from
// global memory straight into registers, as 16-byte read-only loads with an
// L2 evict-first policy, eight per thread in flight:
//  * B stored K x N (row-major): a CTA of 128 threads owns 512 columns;
//    thread t owns columns 4t .. 4t+3, and a warp reads 512 contiguous bytes
//    of a row of B per k.  Each output is a float32 fma chain in ascending k.
//  * B given transposed (stored N x K, the weight layout of y = x W^T): a
//    warp streams four rows of B^T together (four output columns), its lanes
//    reading 512 contiguous bytes of each per step, so one shared-memory read
//    of A serves four rows; a shuffle tree adds the 32 lane sums.
// K is cut into S chunks of at most 1024 (grid y); the chunk's rows of A are
// staged once per CTA in shared memory.  S is chosen so the CTAs fill whole
// waves of the GPU.  With S > 1 each chunk writes its partial sums to a plan
// workspace and a second kernel adds them in an order fixed by the shape
// (results are identical run to run) and applies alpha and beta; with
// S == 1 the first kernel applies them itself.  beta == 0 never reads C.
// A and B may have any alignment and leading dimension (16-byte loads of B
// where its address and row stride allow them, 4-byte loads otherwise), and
// strided batches run on grid z.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernel_gemv.h"

namespace sgemm {
namespace {

constexpr int kGvThreads = 128;
constexpr int kGvWarps = kGvThreads / 32;
constexpr int kGvCols = 4 * kGvThreads;  // K x N form: columns per CTA
constexpr int kGvRowsPerWarp = 4;        // transposed form: rows of B^T a warp streams together
constexpr int kGvTRows = kGvWarps * kGvRowsPerWarp;
constexpr int kGvMaxRows = 4;
constexpr int kGvMaxChunk = 1024;        // k per chunk: A rows staged, at most 4 x 4 KB
constexpr int kGvMinChunk = 64;

struct GemvParams {
  const float* A;
  const float* B;
  float* C;
  float* ws;  // [batch][S][M][n_pad] partial sums (S > 1)
  int64_t lda, ldb, ldc;
  int M, N, K;
  int S, kc;   // chunks, k per chunk (a multiple of 8)
  int n_pad;   // N rounded up to 4
  int vec_b;   // B's address, row stride and batch stride allow 16-byte loads
  int direct;  // S == 1: apply alpha and beta to C here
  float alpha, beta;
  int64_t stride_a, stride_b, stride_c;
};

// B is read exactly once: non-coherent loads that skip L1 and carry an L2
// evict-first policy, so the stream replaces its own lines in L2 rather than
// whatever else L2 holds (lines still to be written back, the partial sums).
// The loads are volatile so none is moved out of the bounds test guarding it.
__device__ __forceinline__ uint64_t stream_policy() {
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ float4 ldg4(const float* p, uint64_t pol) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
      : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
      : "l"(p), "l"(pol));
  return v;
}

__device__ __forceinline__ float ldg1(const float* p, uint64_t pol) {
  float v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(v) : "l"(p), "l"(pol));
  return v;
}

__device__ __forceinline__ void store_out(const GemvParams& p, int z, int s, int m, int n, float acc) {
  if (p.direct) {
    float* d = p.C + z * p.stride_c + static_cast<int64_t>(m) * p.ldc + n;
    *d = p.beta == 0.f ? p.alpha * acc : fmaf(p.alpha, acc, p.beta * *d);
  } else {
    p.ws[((static_cast<int64_t>(z) * p.S + s) * p.M + m) * p.n_pad + n] = acc;
  }
}

// xs[m][0 .. len) = A[m][k0 .. k0+len) for the CTA's product
template <int MR>
__device__ __forceinline__ int stage_a(const GemvParams& p, float (*xs)[kGvMaxChunk], int z, int k0) {
  const int k1 = k0 + p.kc < p.K ? k0 + p.kc : p.K;
  const int len = k1 - k0;
  const float* A = p.A + z * p.stride_a + k0;
  for (int i = threadIdx.x; i < MR * len; i += kGvThreads) {
    const int m = i / len, k = i - m * len;
    xs[m][k] = A[static_cast<int64_t>(m) * p.lda + k];
  }
  __syncthreads();
  return len;
}

// B stored K x N: thread owns four adjacent columns
template <int MR>
__global__ void __launch_bounds__(kGvThreads) gemv_kn_kernel(const GemvParams p) {
  __shared__ __align__(16) float xs[MR][kGvMaxChunk];
  const int z = blockIdx.z, s = blockIdx.y;
  const int k0 = s * p.kc;
  const int len = stage_a<MR>(p, xs, z, k0);
  const int c = 4 * (blockIdx.x * kGvThreads + threadIdx.x);
  if (c >= p.N) return;
  float acc[MR][4];
#pragma unroll
  for (int m = 0; m < MR; ++m)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[m][j] = 0.f;

  const bool vec = p.vec_b && c + 3 < p.N;
  const float* b = p.B + z * p.stride_b + static_cast<int64_t>(k0) * p.ldb + c;
  const uint64_t pol = stream_policy();
  auto load = [&](int k) -> float4 {
    const float* q = b + static_cast<int64_t>(k) * p.ldb;
    if (vec) return ldg4(q, pol);
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = c + j < p.N ? ldg1(q + j, pol) : 0.f;
    return make_float4(v[0], v[1], v[2], v[3]);
  };
  auto fma_row = [&](const float4 v, int k) {
#pragma unroll
    for (int m = 0; m < MR; ++m) {
      const float x = xs[m][k];
      acc[m][0] = fmaf(x, v.x, acc[m][0]);
      acc[m][1] = fmaf(x, v.y, acc[m][1]);
      acc[m][2] = fmaf(x, v.z, acc[m][2]);
      acc[m][3] = fmaf(x, v.w, acc[m][3]);
    }
  };
  int k = 0;
  for (; k + 8 <= len; k += 8) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = load(k + u);
#pragma unroll
    for (int u = 0; u < 8; ++u) fma_row(v[u], k + u);
  }
  for (; k < len; ++k) fma_row(load(k), k);

  if (!p.direct && vec) {
    // n_pad is a multiple of 4 and c + 3 < n_pad: one 16-byte store per row
    float* w = p.ws + ((static_cast<int64_t>(z) * p.S + s) * p.M) * p.n_pad + c;
#pragma unroll
    for (int m = 0; m < MR; ++m)
      *reinterpret_cast<float4*>(w + static_cast<int64_t>(m) * p.n_pad) =
          make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
    return;
  }
#pragma unroll
  for (int m = 0; m < MR; ++m)
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (c + j < p.N) store_out(p, z, s, m, c + j, acc[m][j]);
}

// B given transposed (stored N x K): a warp streams R rows of B^T at once,
// its lanes splitting k
template <int MR>
__global__ void __launch_bounds__(kGvThreads) gemv_nk_kernel(const GemvParams p) {
  constexpr int R = kGvRowsPerWarp;
  __shared__ __align__(16) float xs[MR][kGvMaxChunk];
  const int z = blockIdx.z, s = blockIdx.y;
  const int k0 = s * p.kc;
  const int len = stage_a<MR>(p, xs, z, k0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = (blockIdx.x * kGvWarps + warp) * R;
  if (n0 >= p.N) return;  // the same for the whole warp; no barrier follows
  // rows past N read row N-1 again (in bounds) and are not stored
  const float* b[R];
#pragma unroll
  for (int r = 0; r < R; ++r)
    b[r] = p.B + z * p.stride_b + static_cast<int64_t>(n0 + r < p.N ? n0 + r : p.N - 1) * p.ldb + k0;
  float acc[R][MR];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < MR; ++m) acc[r][m] = 0.f;
  const uint64_t pol = stream_policy();
  // k0 is a multiple of 8, so a row of B^T is 16-byte aligned from k0 on
  // whenever its start is
  if (p.vec_b) {
    auto step = [&](const float4 (&v)[R], int k) {
#pragma unroll
      for (int m = 0; m < MR; ++m) {
        const float4 x = *reinterpret_cast<const float4*>(&xs[m][k]);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          acc[r][m] = fmaf(x.x, v[r].x, acc[r][m]);
          acc[r][m] = fmaf(x.y, v[r].y, acc[r][m]);
          acc[r][m] = fmaf(x.z, v[r].z, acc[r][m]);
          acc[r][m] = fmaf(x.w, v[r].w, acc[r][m]);
        }
      }
    };
    int k = 4 * lane;
    for (; k + 128 + 3 < len; k += 256) {  // two steps of every row in flight
      float4 v0[R], v1[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        v0[r] = ldg4(b[r] + k, pol);
        v1[r] = ldg4(b[r] + k + 128, pol);
      }
      step(v0, k);
      step(v1, k + 128);
    }
    if (k + 3 < len) {
      float4 v0[R];
#pragma unroll
      for (int r = 0; r < R; ++r) v0[r] = ldg4(b[r] + k, pol);
      step(v0, k);
    }
    const int t = (len & ~3) + lane;  // the last len % 4 elements
    if (t < len) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float v = ldg1(b[r] + t, pol);
#pragma unroll
        for (int m = 0; m < MR; ++m) acc[r][m] = fmaf(xs[m][t], v, acc[r][m]);
      }
    }
  } else {
    for (int k = lane; k < len; k += 32) {
      float v[R];
#pragma unroll
      for (int r = 0; r < R; ++r) v[r] = ldg1(b[r] + k, pol);
#pragma unroll
      for (int m = 0; m < MR; ++m) {
        const float x = xs[m][k];
#pragma unroll
        for (int r = 0; r < R; ++r) acc[r][m] = fmaf(x, v[r], acc[r][m]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < MR; ++m)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[r][m] += __shfl_xor_sync(0xffffffffu, acc[r][m], off);
  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (n0 + r < p.N)
#pragma unroll
        for (int m = 0; m < MR; ++m) store_out(p, z, s, m, n0 + r, acc[r][m]);
  }
}

// C[m][n] = alpha * (sum of the chunk partials) + beta * C.  A block takes
// 32 consecutive outputs of one row; warp w adds chunks w, w+8, w+16, ...
// in that order (coalesced 128-byte loads), and warp 0 adds the eight warp
// sums in warp order: a fixed order for the shape, so reruns agree bit for
// bit.
constexpr int kRedWarps = 8;

__global__ void __launch_bounds__(32 * kRedWarps) gemv_reduce_kernel(const GemvParams p) {
  __shared__ float part[kRedWarps][32];
  const int z = blockIdx.z, m = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * 32 + lane;
  const float* ws = p.ws + (static_cast<int64_t>(z) * p.S * p.M + m) * p.n_pad + (n < p.N ? n : 0);
  const int64_t step = static_cast<int64_t>(p.M) * p.n_pad;  // one chunk to the next
  float sum = 0.f;
  int s = warp;
  for (; s + 3 * kRedWarps < p.S; s += 4 * kRedWarps) {
    float v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldcg(ws + (s + u * kRedWarps) * step);
#pragma unroll
    for (int u = 0; u < 4; ++u) sum += v[u];
  }
  for (; s < p.S; s += kRedWarps) sum += __ldcg(ws + s * step);
  part[warp][lane] = sum;
  __syncthreads();
  if (warp == 0 && n < p.N) {
    float t = part[0][lane];
#pragma unroll
    for (int w = 1; w < kRedWarps; ++w) t += part[w][lane];
    float* d = p.C + z * p.stride_c + static_cast<int64_t>(m) * p.ldc + n;
    *d = p.beta == 0.f ? p.alpha * t : fmaf(p.alpha, t, p.beta * *d);
  }
}

// k per chunk for S chunks: ceil(K / S) rounded up to a multiple of 8
int64_t chunk_len(int64_t K, int64_t S) { return ((K + S - 1) / S + 7) / 8 * 8; }

template <int MR>
void launch_rows(const GemvParams& p, int b_trans, dim3 grid, cudaStream_t stream) {
  if (b_trans)
    gemv_nk_kernel<MR><<<grid, kGvThreads, 0, stream>>>(p);
  else
    gemv_kn_kernel<MR><<<grid, kGvThreads, 0, stream>>>(p);
}

cudaError_t gemv_prepare() { return cudaSuccess; }

// the fewer resident CTAs of the two forms at four rows
cudaError_t gemv_occupancy(int* ctas) {
  int a = 0, b = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, gemv_kn_kernel<kGvMaxRows>, kGvThreads, 0);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, gemv_nk_kernel<kGvMaxRows>, kGvThreads, 0);
  *ctas = a < b ? a : b;
  return e;
}

// a.grid: resident CTA slots of the device; a.split_k: chunks the plan's
// workspace a.ws holds per product; a.b_trans: B given transposed
cudaError_t gemv_launch(const LaunchArgs& a, cudaStream_t stream) {
  const int batch = a.batch > 1 ? a.batch : 1;
  if (a.M < 1 || a.M > kGvMaxRows || a.N < 1 || a.K < 1 || batch > 65535) return cudaErrorInvalidValue;
  const int S = gemv_chunks(a.N, a.K, batch, a.b_trans, a.grid);
  if (S < 1 || S > 65535 || (S > 1 && (S > a.split_k || !a.ws))) return cudaErrorInvalidValue;
  GemvParams p;
  p.A = a.A;
  p.B = a.B;
  p.C = a.C;
  p.ws = a.ws;
  p.lda = a.lda;
  p.ldb = a.ldb;
  p.ldc = a.ldc;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.S = S;
  p.kc = static_cast<int>(chunk_len(a.K, S));
  p.n_pad = (a.N + 3) / 4 * 4;
  p.vec_b = (reinterpret_cast<uintptr_t>(a.B) & 15) == 0 && a.ldb % 4 == 0 && (batch == 1 || a.stride_b % 4 == 0);
  p.direct = S == 1;
  p.alpha = a.alpha;
  p.beta = a.beta;
  p.stride_a = a.stride_a;
  p.stride_b = a.stride_b;
  p.stride_c = a.stride_c;
  const int64_t cols = a.b_trans ? (a.N + kGvTRows - 1) / kGvTRows : (a.N + kGvCols - 1) / kGvCols;
  if (cols > 0x7fffffff) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(cols), S, batch);
  switch (a.M) {
    case 1: launch_rows<1>(p, a.b_trans, grid, stream); break;
    case 2: launch_rows<2>(p, a.b_trans, grid, stream); break;
    case 3: launch_rows<3>(p, a.b_trans, grid, stream); break;
    default: launch_rows<4>(p, a.b_trans, grid, stream); break;
  }
  if (S > 1) {
    const dim3 rgrid(static_cast<unsigned>((a.N + 31) / 32), a.M, batch);
    gemv_reduce_kernel<<<rgrid, 32 * kRedWarps, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

const Variant kGemvVariants[] = {
    // bm = most rows, bn = columns per CTA (K x N form), bk = longest chunk of k
    Variant{"gemv_4x512", kKindGemv, kGvMaxRows, kGvCols, kGvMaxChunk, 1, 0, kGvThreads, 0, -1, &gemv_prepare,
            &gemv_occupancy, &gemv_launch, 0, 0, 1, 1, 0},
};

}  // namespace

int gemv_chunks(int64_t N, int64_t K, int64_t batch, int b_trans, int64_t slots) {
  if (K < 1 || N < 1) return 1;
  if (batch < 1) batch = 1;
  if (slots < 1) slots = 1;
  const int64_t units = batch * (b_trans ? (N + kGvTRows - 1) / kGvTRows : (N + kGvCols - 1) / kGvCols);
  const int64_t s_min = (K + kGvMaxChunk - 1) / kGvMaxChunk;
  int64_t s_max = K / kGvMinChunk;
  if (s_max > 65535) s_max = 65535;
  if (s_max > s_min + 256) s_max = s_min + 256;
  // CTAs of one chunk each do the same work: take the count that fills its
  // last wave best, the fewer chunks unless more fill clearly better
  int64_t best = s_min;
  double best_eff = -1.0;
  for (int64_t s = s_min; s <= s_max || s == s_min; ++s) {
    if ((K + chunk_len(K, s) - 1) / chunk_len(K, s) != s) continue;  // rounding gives fewer chunks
    const int64_t total = units * s;
    const int64_t waves = (total + slots - 1) / slots;
    const double eff = static_cast<double>(total) / static_cast<double>(waves * slots);
    if (eff > best_eff + 0.02) {
      best_eff = eff;
      best = s;
    }
  }
  return static_cast<int>(best);
}

const Variant* gemv_variants(int* count) {
  *count = static_cast<int>(sizeof(kGemvVariants) / sizeof(kGemvVariants[0]));
  return kGemvVariants;
}

}  // namespace sgemm
