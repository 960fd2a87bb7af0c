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
//
// The same stream serves five to sixteen rows (gemv_16x512).  Each element
// of B is then used up to 16 times, so the FMA work (M*N*K FMAs: 53 us at
// 16 x 16384 x 8192 on the whole GPU at 2.07 GHz) must hide under the
// 80 us read of B.  B still goes straight into registers, now with the
// next batch of eight rows in flight while the current one multiplies
// (16 loads of 16 bytes per thread), and the multiply is the paired form
// of the main kernels: one FFMA2 takes a register pair of two rows of A at
// one k and one element of B for both.  A's chunk is staged k-major
// (at[k][16]), so the four 16-byte shared loads of one k give the eight
// pairs.  B given transposed runs the four-rows-per-warp stream of the
// M <= 4 form with FFMA2 over k pairs (even and odd k in the two halves),
// and the lanes' partial sums meet in a halving shuffle exchange.
#include <cuda_runtime.h>
#include <stdint.h>

#include <string.h>

#include <atomic>
#include <type_traits>

#include "checked.cuh"
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
  unsigned int* status;  // per-device status word (checked build: bounds)
  int64_t ws_floats;     // floats the workspace holds (checked build)
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

// A's rows for a chunk are staged by cp.async: every copy of a thread is in
// flight at once, instead of one dependent load-store round trip per
// element (a 16 x 512 chunk took about ten microseconds that way).
__device__ __forceinline__ void cpa4(float* dst, const float* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}

__device__ __forceinline__ void cpa16(float* dst, const float* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}

__device__ __forceinline__ void cpa_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Programmatic dependent launch: a chunk kernel lets its reduce kernel be
// scheduled as soon as every one of its CTAs has started, and the reduce
// kernel waits for the chunk kernel's completion (and its memory) before
// reading the partial sums.  Without the launch attribute the wait returns
// at once, the stream order having done the same.
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// xs[m][0 .. len) = A[m][k0 .. k0+len) for m < MR (zero rows from M on),
// then a CTA barrier.  16-byte copies when A's rows allow them (k0 is a
// multiple of 8), 4-byte copies otherwise.  NT threads, rows XLD floats apart.
template <int MR, int NT, int XLD>
__device__ __forceinline__ void stage_rows(const float* A, int64_t lda, int M, int len, float* xs) {
  const bool vec = (reinterpret_cast<uintptr_t>(A) & 15) == 0 && lda % 4 == 0;
  int done = 0;
  if (vec) {
    const int q4 = len / 4;
    for (int i = threadIdx.x; i < MR * q4; i += NT) {
      const int m = i / q4, q = i - m * q4;
      if (m < M)
        cpa16(xs + m * XLD + 4 * q, A + static_cast<int64_t>(m) * lda + 4 * q);
      else
        *reinterpret_cast<float4*>(xs + m * XLD + 4 * q) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    done = 4 * q4;
  }
  const int rest = len - done;
  for (int i = threadIdx.x; i < MR * rest; i += NT) {
    const int m = i / rest, k = done + (i - m * rest);
    if (m < M)
      cpa4(xs + m * XLD + k, A + static_cast<int64_t>(m) * lda + k);
    else
      xs[m * XLD + k] = 0.f;
  }
  cpa_wait_all();
  __syncthreads();
}

__device__ __forceinline__ void store_out(const GemvParams& p, int z, int s, int m, int n, float acc) {
  if (p.direct) {
    float* d = p.C + z * p.stride_c + static_cast<int64_t>(m) * p.ldc + n;
    *d = p.beta == 0.f ? p.alpha * acc : fmaf(p.alpha, acc, p.beta * *d);
  } else {
    const int64_t wi = ((static_cast<int64_t>(z) * p.S + s) * p.M + m) * p.n_pad + n;
    if (SG_CHK(SG_IN(wi, p.ws_floats), p.status)) p.ws[wi] = acc;
  }
}

// xs[m][0 .. len) = A[m][k0 .. k0+len) for the CTA's product
template <int MR>
__device__ __forceinline__ int stage_a(const GemvParams& p, float (*xs)[kGvMaxChunk], int z, int k0) {
  const int k1 = k0 + p.kc < p.K ? k0 + p.kc : p.K;
  const int len = k1 - k0;
  stage_rows<MR, kGvThreads, kGvMaxChunk>(p.A + z * p.stride_a + k0, p.lda, MR, len, &xs[0][0]);
  return len;
}

// B stored K x N: thread owns four adjacent columns
template <int MR>
__global__ void __launch_bounds__(kGvThreads) gemv_kn_kernel(const GemvParams p) {
  __shared__ __align__(16) float xs[MR][kGvMaxChunk];
  allow_dependents();
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
    if (!SG_CHK(SG_IN(k, kGvMaxChunk), p.status)) return;
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
    const int64_t w0 = ((static_cast<int64_t>(z) * p.S + s) * p.M) * p.n_pad + c;
#pragma unroll
    for (int m = 0; m < MR; ++m)
      if (SG_CHK(SG_IN(w0 + static_cast<int64_t>(m) * p.n_pad + 3, p.ws_floats), p.status))
        *reinterpret_cast<float4*>(p.ws + w0 + static_cast<int64_t>(m) * p.n_pad) =
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
  allow_dependents();
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
      if (!SG_CHK(SG_IN(k + 3, kGvMaxChunk), p.status)) return;
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

// C[m][n] = alpha * (sum of the chunk partials) + beta * C.  Four
// consecutive lanes share one 16-byte group of outputs (row m, columns
// 4g .. 4g+3): lane q adds chunks q, q+4, q+8, ... in ascending order, the
// four sums meet through two xor shuffles as (s0 + s1) + (s2 + s3), the
// same bits in all four lanes, and lane q writes column 4g + q.  The order
// is fixed by the shape, so reruns agree bit for bit.  Every lane issues
// its loads (up to five per round) at once.
constexpr int kRedThreads = 256;

__global__ void __launch_bounds__(kRedThreads) gemv_reduce_kernel(const GemvParams p) {
  const int z = blockIdx.z, m = blockIdx.y;
  const int t = blockIdx.x * kRedThreads + threadIdx.x;
  const int q = t & 3;
  const int n = 4 * (t >> 2);  // the quad's first column
  const bool mine = n + q < p.N;
  const int64_t c_off = z * p.stride_c + static_cast<int64_t>(m) * p.ldc + n + q;
  // The chunk kernel never writes C, and whatever ran before it has
  // finished, so C is read before the wait.
  const float c_old = mine && p.beta != 0.f ? p.C[c_off] : 0.f;
  wait_primary();
  float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
  auto add = [](float4& a, const float4 b) {
    a.x += b.x;
    a.y += b.y;
    a.z += b.z;
    a.w += b.w;
  };
  if (n < p.N) {  // the same for the four lanes of a quad
    const float4* ws =
        reinterpret_cast<const float4*>(p.ws + (static_cast<int64_t>(z) * p.S * p.M + m) * p.n_pad + n);
    const int64_t step = static_cast<int64_t>(p.M) * p.n_pad / 4;  // one chunk to the next, in float4s
    for (int s = q; s < p.S; s += 20) {  // up to five loads in flight (one round for S <= 20)
      float4 v[5];
#pragma unroll
      for (int u = 0; u < 5; ++u)
        if (s + 4 * u < p.S)
          v[u] = SG_CHK(SG_IN((static_cast<int64_t>(z) * p.S * p.M + m) * p.n_pad + n + 4 * (s + 4 * u) * step + 3,
                              p.ws_floats),
                        p.status)
                     ? __ldcg(ws + (s + 4 * u) * step)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < 5; ++u)
        if (s + 4 * u < p.S) add(sum, v[u]);
    }
  }
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    float4 v;
    v.x = __shfl_xor_sync(0xffffffffu, sum.x, o);
    v.y = __shfl_xor_sync(0xffffffffu, sum.y, o);
    v.z = __shfl_xor_sync(0xffffffffu, sum.z, o);
    v.w = __shfl_xor_sync(0xffffffffu, sum.w, o);
    add(sum, v);
  }
  if (mine) {
    const float tot = q == 0 ? sum.x : q == 1 ? sum.y : q == 2 ? sum.z : sum.w;
    p.C[c_off] = p.beta == 0.f ? p.alpha * tot : fmaf(p.alpha, tot, p.beta * c_old);
  }
}

// k per chunk for S chunks: ceil(K / S) rounded up to a multiple of 8
int64_t chunk_len(int64_t K, int64_t S) { return ((K + S - 1) / S + 7) / 8 * 8; }

// ---- five to sixteen rows ----------------------------------------------------

constexpr int kRcThreads = 256;
constexpr int kRcWarps = kRcThreads / 32;
constexpr int kRcCols = 4 * kRcThreads;  // columns per CTA (128 per warp)
constexpr int kRcMaxRows = 16;
constexpr int kRcMaxChunk = 640;         // k per chunk: A staged k-major, at most 640 x 16 floats
constexpr int kRcRing = 16;              // rows of B in flight per warp (512 bytes each)
constexpr int kRcGroup = 4;              // rows per cp.async commit group
constexpr int kRcGroups = kRcRing / kRcGroup;
static_assert(kRcRing % kRcGroup == 0 && (kRcRing & (kRcRing - 1)) == 0, "ring of whole groups, a power of two");

template <int MR>
constexpr int rows_smem_bytes() {
  return (kRcMaxChunk * MR + kRcWarps * kRcRing * 32 * 4) * 4;
}

__device__ __forceinline__ void cpa16_hint(void* dst, const float* src, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "l"(pol)
               : "memory");
}

__device__ __forceinline__ void cpa_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cpa_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// B stored K x N, up to MR rows (8 or 16).  Warp w of a CTA owns 128
// columns, lane l four adjacent ones (c .. c+3) for all MR rows:
// acc[h][j] = {C[2h][c + j], C[2h + 1][c + j]}.  B goes global -> shared
// memory by 16-byte cp.async copies that each lane issues for its own four
// columns, into a ring of kRcRing rows per warp, kRcGroup rows per commit
// group; a lane reads back only what it copied, so no barrier orders the
// ring.  A's chunk is staged k-major (at[k][MR]) once per CTA.
template <int MR>
__global__ void __launch_bounds__(kRcThreads, 2) rows_cp_kernel(const GemvParams p) {
  extern __shared__ __align__(16) float rsm[];
  float* at = rsm;  // [kRcMaxChunk][MR]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float4* const ring = reinterpret_cast<float4*>(rsm + kRcMaxChunk * MR);  // [warps][kRcRing][32]
  float4* slot0 = ring + warp * kRcRing * 32 + lane;
  allow_dependents();
  const int z = blockIdx.z, s = blockIdx.y;
  const int k0 = s * p.kc;
  const int len = p.K - k0 < p.kc ? p.K - k0 : p.kc;
  const int c = 4 * (blockIdx.x * kRcThreads + threadIdx.x);
  const bool live = c < p.N;
  const bool vec = p.vec_b && c + 3 < p.N;
  const float* b = p.B + z * p.stride_b + static_cast<int64_t>(k0) * p.ldb + c;
  const int64_t ldb = p.ldb;
  const uint64_t pol = stream_policy();
  // row q of B (this lane's four columns) into ring slot d; columns past N
  // are zero
  auto fetch = [&](float4* d, const float* q) {
    if (!SG_CHK(SG_IN(d - ring, kRcWarps * kRcRing * 32), p.status)) return;
    if (vec) {
      cpa16_hint(d, q, pol);
    } else {
      float* df = reinterpret_cast<float*>(d);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (c + j < p.N)
          cpa4(df + j, q + j);
        else
          df[j] = 0.f;
      }
    }
  };

  // A's chunk: one commit group, the oldest
  {
    const float* A = p.A + z * p.stride_a + k0;
    for (int i = threadIdx.x; i < MR * len; i += kRcThreads) {
      const int m = i % MR, k = i / MR;
      if (!SG_CHK(SG_IN(k * MR + m, kRcMaxChunk * MR), p.status)) continue;
      if (m < p.M)
        cpa4(at + k * MR + m, A + static_cast<int64_t>(m) * p.lda + k);
      else
        at[k * MR + m] = 0.f;
    }
    cpa_commit();
  }
  // the first kRcGroups groups of B rows (the whole ring)
  {
    const float* q = b;
#pragma unroll
    for (int g = 0; g < kRcGroups; ++g) {
#pragma unroll
      for (int r = 0; r < kRcGroup; ++r) {
        if (live && g * kRcGroup + r < len) fetch(slot0 + (g * kRcGroup + r) * 32, q);
        q += ldb;
      }
      cpa_commit();
    }
  }
  cpa_wait_group<kRcGroups>();  // this thread's copies of A have landed
  __syncthreads();              // and every thread's
  if (!live) return;            // after the CTA's only barrier

  float2 acc[MR / 2][4];
#pragma unroll
  for (int h = 0; h < MR / 2; ++h)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[h][j] = make_float2(0.f, 0.f);
  // one row: A at ap (MR values, k-major), B's four columns in bv
  auto fma_row = [&](const float4 bv, const float* ap) {
    if (!SG_CHK(SG_IN(ap - at + MR - 1, kRcMaxChunk * MR), p.status)) return;
    const float4* a4 = reinterpret_cast<const float4*>(ap);
    const float bb[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
    for (int q = 0; q < MR / 4; ++q) {
      const float4 a = a4[q];  // rows 4q .. 4q+3 at this k (a broadcast read)
      const float2 lo = make_float2(a.x, a.y), hi = make_float2(a.z, a.w);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[2 * q][j] = __ffma2_rn(lo, make_float2(bb[j], bb[j]), acc[2 * q][j]);
        acc[2 * q + 1][j] = __ffma2_rn(hi, make_float2(bb[j], bb[j]), acc[2 * q + 1][j]);
      }
    }
  };
  // Group g (rows 4g .. 4g+3) is the oldest of kRcGroups in flight: wait
  // for it, multiply its rows, then refill its slots with group g + 4 (the
  // chunk's end is checked once per group).  The loop is instantiated for
  // 16-byte and for 4-byte copies, so the hot loop has no branch on them.
  auto run = [&](auto vec_c) {
    constexpr bool V = decltype(vec_c)::value;
    auto put = [&](float4* d, const float* src) {
      if (!SG_CHK(SG_IN(d - ring, kRcWarps * kRcRing * 32), p.status)) return;
      if (V) {
        cpa16_hint(d, src, pol);
      } else {
        float* df = reinterpret_cast<float*>(d);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (c + j < p.N)
            cpa4(df + j, src + j);
          else
            df[j] = 0.f;
        }
      }
    };
    const float* ap = at;
    const float* q = b + kRcRing * ldb;  // the next row to fetch
    const int kfull = len & ~(kRcGroup - 1);
    int k = 0;
#pragma unroll 1
    for (; k < kfull; k += kRcGroup) {
      float4* sg = slot0 + (k & (kRcRing - 1)) * 32;
      cpa_wait_group<kRcGroups - 1>();
      if (!SG_CHK(SG_IN(sg + (kRcGroup - 1) * 32 - ring, kRcWarps * kRcRing * 32), p.status)) break;
      // one row at a time: hoisting every row's shared loads (16 A words
      // and 4 B words per row) would not fit in the registers beside the
      // accumulators
#pragma unroll 1
      for (int r = 0; r < kRcGroup; ++r) fma_row(sg[r * 32], ap + r * MR);
      if (k + kRcRing + kRcGroup <= len) {
#pragma unroll
        for (int r = 0; r < kRcGroup; ++r) {
          put(sg + r * 32, q);
          q += ldb;
        }
      } else {
#pragma unroll
        for (int r = 0; r < kRcGroup; ++r) {
          if (k + kRcRing + r < len) put(sg + r * 32, q);
          q += ldb;
        }
      }
      cpa_commit();
      ap += kRcGroup * MR;
    }
    if (k < len) {  // the last len % 4 rows, already in flight
      float4* sg = slot0 + (k & (kRcRing - 1)) * 32;
      cpa_wait_group<kRcGroups - 1>();
#pragma unroll 1
      for (int r = 0; r < len - k; ++r) fma_row(sg[r * 32], ap + r * MR);
    }
  };
  if (vec)
    run(std::true_type{});
  else
    run(std::false_type{});
  cpa_wait_all();  // nothing real is in flight any more (only empty groups)

  if (!p.direct && vec) {
    // n_pad is a multiple of 4 and c + 3 < n_pad: one 16-byte store per row
    const int64_t w0 = ((static_cast<int64_t>(z) * p.S + s) * p.M) * p.n_pad + c;
    float* wp = p.ws + w0;
#pragma unroll
    for (int h = 0; h < MR / 2; ++h) {
      if (2 * h < p.M && SG_CHK(SG_IN(w0 + static_cast<int64_t>(2 * h) * p.n_pad + 3, p.ws_floats), p.status))
        *reinterpret_cast<float4*>(wp + static_cast<int64_t>(2 * h) * p.n_pad) =
            make_float4(acc[h][0].x, acc[h][1].x, acc[h][2].x, acc[h][3].x);
      if (2 * h + 1 < p.M &&
          SG_CHK(SG_IN(w0 + static_cast<int64_t>(2 * h + 1) * p.n_pad + 3, p.ws_floats), p.status))
        *reinterpret_cast<float4*>(wp + static_cast<int64_t>(2 * h + 1) * p.n_pad) =
            make_float4(acc[h][0].y, acc[h][1].y, acc[h][2].y, acc[h][3].y);
    }
    return;
  }
#pragma unroll
  for (int h = 0; h < MR / 2; ++h)
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (c + j < p.N) {
        if (2 * h < p.M) store_out(p, z, s, 2 * h, c + j, acc[h][j].x);
        if (2 * h + 1 < p.M) store_out(p, z, s, 2 * h + 1, c + j, acc[h][j].y);
      }
}

// Two families share the launch code: gemv_4x512 (one to four rows, B as
// stored or given transposed) and gemv_16x512 (up to sixteen rows, B as
// stored; its kernel instantiated for 8 and 16 rows).
struct Family {
  int max_rows;
  int threads;
  int cols;       // K x N form: columns per CTA
  int trows;      // transposed form: rows of B^T per CTA
  int max_chunk;  // longest k-chunk (the A stage in shared memory)
};
constexpr Family kFamilies[2] = {{kGvMaxRows, kGvThreads, kGvCols, kGvTRows, kGvMaxChunk},
                                 {kRcMaxRows, kRcThreads, kRcCols, kRcCols, kRcMaxChunk}};

int family_of(const Variant* v) { return v->bm > kGvMaxRows ? 1 : 0; }

// The kernel that runs M rows of family f, B as stored or given transposed,
// and its dynamic shared memory.
const void* kernel_for(int f, int M, int b_trans, int* smem) {
  *smem = 0;
  if (f == 1) {
    if (M <= 8) {
      *smem = rows_smem_bytes<8>();
      return reinterpret_cast<const void*>(rows_cp_kernel<8>);
    }
    *smem = rows_smem_bytes<16>();
    return reinterpret_cast<const void*>(rows_cp_kernel<16>);
  }
  switch (M) {
    case 1: return b_trans ? reinterpret_cast<const void*>(gemv_nk_kernel<1>)
                           : reinterpret_cast<const void*>(gemv_kn_kernel<1>);
    case 2: return b_trans ? reinterpret_cast<const void*>(gemv_nk_kernel<2>)
                           : reinterpret_cast<const void*>(gemv_kn_kernel<2>);
    case 3: return b_trans ? reinterpret_cast<const void*>(gemv_nk_kernel<3>)
                           : reinterpret_cast<const void*>(gemv_kn_kernel<3>);
    default: return b_trans ? reinterpret_cast<const void*>(gemv_nk_kernel<4>)
                            : reinterpret_cast<const void*>(gemv_kn_kernel<4>);
  }
}

// Resident CTAs per SM of that kernel on the current device, cached per
// (device, family, rows, form): the chunk count fills waves of the kernel
// that actually runs.  0 on a CUDA error.
constexpr int kMaxDevices = 64;
std::atomic<int> g_resident[kMaxDevices][2][kRcMaxRows + 1][2];

int resident_ctas(int f, int M, int b_trans) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const int m = M < 1 ? 1 : (M > kRcMaxRows ? kRcMaxRows : M);
  std::atomic<int>* slot = dev < kMaxDevices ? &g_resident[dev][f][m][b_trans ? 1 : 0] : nullptr;
  if (slot) {
    const int c = slot->load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int smem = 0;
  const void* kern = kernel_for(f, m, b_trans, &smem);
  if (smem > 0 && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kFamilies[f].threads, smem) != cudaSuccess || n < 1)
    return 0;
  if (slot) slot->store(n, std::memory_order_relaxed);
  return n;
}

// Chunks of K for `slots` resident CTAs, priced in rows of B per CTA:
// every CTA does the same work, chunk_len(K, S) rows, plus a fixed cost of
// about 32 rows (staging its chunk of A, filling and draining its stream,
// writing its partial sums), and the kernel runs waves(S) = ceil(units x
// S / slots) of them; the partial sums add S x M x N floats written and read
// back, S x M x units / slots rows at the same bandwidth.  Take the fewest
// chunks whose cost is within 3% of the cheapest found so far, in ascending
// S.  (Filling waves alone chose 129 chunks of 64 rows for 1 x 16384 x 8192
// at nine CTAs per SM, four waves and 8.5 MB of partial sums, 89.6 us
// against 83.4 us for one wave of 38 chunks.)
int chunks_for(const Family& fam, int64_t M, int64_t N, int64_t K, int64_t batch, int b_trans, int64_t slots) {
  if (K < 1 || N < 1) return 1;
  if (batch < 1) batch = 1;
  if (slots < 1) slots = 1;
  if (M < 1) M = 1;
  const int64_t units = batch * (b_trans ? (N + fam.trows - 1) / fam.trows : (N + fam.cols - 1) / fam.cols);
  const int64_t s_min = (K + fam.max_chunk - 1) / fam.max_chunk;
  int64_t s_max = K / kGvMinChunk;
  if (s_max > 65535) s_max = 65535;
  if (s_max > s_min + 256) s_max = s_min + 256;
  int64_t best = s_min;
  double best_cost = -1.0;
  for (int64_t s = s_min; s <= s_max || s == s_min; ++s) {
    const int64_t kc = chunk_len(K, s);
    if ((K + kc - 1) / kc != s) continue;  // rounding gives fewer chunks
    const int64_t waves = (units * s + slots - 1) / slots;
    const double cost = static_cast<double>(waves) * static_cast<double>(kc + 32) +
                        static_cast<double>(s) * static_cast<double>(M) * static_cast<double>(units) /
                            static_cast<double>(slots);
    if (best_cost < 0.0 || cost < 0.97 * best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return static_cast<int>(best);
}

int plan_chunks(int f, int64_t M, int64_t N, int64_t K, int64_t batch, int b_trans, int sms) {
  const int ctas = resident_ctas(f, static_cast<int>(M), b_trans);
  if (ctas < 1) return -1;
  return chunks_for(kFamilies[f], M, N, K, batch, b_trans, static_cast<int64_t>(sms) * ctas);
}

// set the dynamic shared memory of every instantiation (idempotent)
cudaError_t gemv4_prepare() { return cudaSuccess; }
cudaError_t gemv16_prepare() {
  for (int m : {8, 16})
    if (resident_ctas(1, m, 0) < 1) return cudaErrorInvalidValue;
  return cudaSuccess;
}

// the fewer resident CTAs of the forms at the family's most rows
cudaError_t occupancy_of(int f, int* ctas) {
  const int a = resident_ctas(f, kFamilies[f].max_rows, 0);
  const int b = f == 0 ? resident_ctas(f, kFamilies[f].max_rows, 1) : a;
  if (a < 1 || b < 1) return cudaErrorInvalidValue;
  *ctas = a < b ? a : b;
  return cudaSuccess;
}
cudaError_t gemv4_occupancy(int* ctas) { return occupancy_of(0, ctas); }
cudaError_t gemv16_occupancy(int* ctas) { return occupancy_of(1, ctas); }

// a.grid: the device's SM count; a.split_k: chunks the plan's workspace a.ws
// holds per product; a.b_trans: B given transposed (family 0 only)
cudaError_t launch_family(int f, const LaunchArgs& a, cudaStream_t stream) {
  const Family& fam = kFamilies[f];
  const int batch = a.batch > 1 ? a.batch : 1;
  if (a.M < 1 || a.M > fam.max_rows || a.N < 1 || a.K < 1 || batch > 65535 || (f == 1 && a.b_trans))
    return cudaErrorInvalidValue;
  const int S = plan_chunks(f, a.M, a.N, a.K, batch, a.b_trans, a.grid);
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
  p.status = a.status;
  p.ws_floats = a.ws_slots;
  const int64_t cols = a.b_trans ? (a.N + fam.trows - 1) / fam.trows : (a.N + fam.cols - 1) / fam.cols;
  if (cols > 0x7fffffff) return cudaErrorInvalidValue;
  int smem = 0;
  const void* kern = kernel_for(f, a.M, a.b_trans, &smem);
  void* args[] = {&p};
  cudaError_t e =
      cudaLaunchKernel(kern, dim3(static_cast<unsigned>(cols), S, batch), dim3(fam.threads), args, smem, stream);
  if (e != cudaSuccess) return e;
  if (S > 1) {
    // the reduce kernel, scheduled while the chunk kernel still runs
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>((p.n_pad + kRedThreads - 1) / kRedThreads), a.M, batch);
    cfg.blockDim = dim3(kRedThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gemv_reduce_kernel, p);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}
cudaError_t gemv4_launch(const LaunchArgs& a, cudaStream_t stream) { return launch_family(0, a, stream); }
cudaError_t gemv16_launch(const LaunchArgs& a, cudaStream_t stream) { return launch_family(1, a, stream); }

const Variant kGemvVariants[] = {
    // bm = most rows, bn = columns per CTA (K x N form), bk = longest chunk of k
    Variant{"gemv_4x512", kKindGemv, kGvMaxRows, kGvCols, kGvMaxChunk, 1, 0, kGvThreads, 0, -1, &gemv4_prepare,
            &gemv4_occupancy, &gemv4_launch, 0, 0, 1, 1, 0},
    // B as stored only (b_trans_ok = 0)
    Variant{"gemv_16x1024", kKindGemv, kRcMaxRows, kRcCols, kRcMaxChunk, kRcRing, 1, kRcThreads,
            rows_smem_bytes<16>(), -1, &gemv16_prepare, &gemv16_occupancy, &gemv16_launch, 0, 0, 1, 0, 0},
};

}  // namespace

int gemv_plan_chunks(const Variant* v, int64_t M, int64_t N, int64_t K, int64_t batch, int b_trans, int sms) {
  return plan_chunks(family_of(v), M, N, K, batch, b_trans, sms);
}

bool gemv_takes(const Variant* v, int64_t M, int64_t N, int64_t K, int64_t batch) {
  const Family& fam = kFamilies[family_of(v)];
  return M <= fam.max_rows && N <= (int64_t(1) << 30) && K <= int64_t(65535) * fam.max_chunk && batch <= 65535;
}

const Variant* gemv_variants(int* count) {
  *count = static_cast<int>(sizeof(kGemvVariants) / sizeof(kGemvVariants[0]));
  return kGemvVariants;
}

}  // namespace sgemm
