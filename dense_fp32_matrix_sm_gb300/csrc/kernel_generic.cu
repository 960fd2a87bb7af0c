// kernel_generic.cu -- the any-layout SGEMM kernel, the C = beta*C kernel
// and the wait-limit self-test kernel.
//
// The generic kernel takes any alignment and any leading dimension: every
// global access is a predicated scalar load, so it serves the inputs the
// TMA-fed kernels cannot (unaligned base pointers, lda or ldb not a
// multiple of 4).  It is the pages' shared-memory tiled kernel with 2-D
// register blocking ("Learn: Optimizing GEMM", sections 5 and 6; "Writing a
// Fast Matmul in CUDA, Step by Step", Steps 3 and 4):
//  * a 64 x 64 CTA tile, k-slices of 16 staged in shared memory, A stored
//    transposed (As[k][m], padded by one column so the transposing stores do
//    not collide in a bank) and B as is;
//  * 256 threads, each owning a 4 x 4 thread tile at rows ty + 16i and
//    columns tx + 16j, so a warp's shared reads are broadcasts (A) or 16
//    consecutive words (B);
//  * threadIdx maps to the contiguous dimension of every global load and
//    store ("Learn: Optimizing GEMM", section 4, coalescing);
//  * the next slice is loaded into registers while the current one is
//    multiplied (register-staged double buffering).
// Each output is a chain of fp32 fmas in ascending k, like the TMA kernels.
#include <cuda_runtime.h>
#include <stdint.h>

#include "checked.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace sgemm {
namespace {

constexpr int kGBM = 64, kGBN = 64, kGBK = 16, kGThreads = 256;

struct GenericParams {
  const float* A;
  const float* B;
  float* C;
  int64_t lda, ldb, ldc;
  int M, N, K;
  float alpha, beta;
  int64_t stride_a, stride_b, stride_c;  // batch z = blockIdx.z
  unsigned int* status;                  // per-device status word (checked build: bounds)
};

__global__ void __launch_bounds__(kGThreads) sgemm_generic_kernel(GenericParams p) {
  __shared__ float As[kGBK][kGBM + 1];
  __shared__ float Bs[kGBK][kGBN];
  p.A += blockIdx.z * p.stride_a;
  p.B += blockIdx.z * p.stride_b;
  p.C += blockIdx.z * p.stride_c;

  const int tiles_n = (p.N + kGBN - 1) / kGBN;
  const int tm = blockIdx.x / tiles_n;
  const int tn = blockIdx.x % tiles_n;
  const int m0 = tm * kGBM, n0 = tn * kGBN;
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;

  float ra[4], rb[4];
  auto load_slice = [&](int k0) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int idx = tid + kGThreads * r;
      const int am = idx / kGBK, ak = idx % kGBK;  // consecutive threads: consecutive k of one row
      const int gm = m0 + am, gk = k0 + ak;
      ra[r] = (gm < p.M && gk < p.K) ? p.A[static_cast<int64_t>(gm) * p.lda + gk] : 0.f;
      const int bk = idx / kGBN, bn = idx % kGBN;  // consecutive threads: consecutive n
      const int gkb = k0 + bk, gn = n0 + bn;
      rb[r] = (gkb < p.K && gn < p.N) ? p.B[static_cast<int64_t>(gkb) * p.ldb + gn] : 0.f;
    }
  };
  auto store_slice = [&]() {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int idx = tid + kGThreads * r;
      if (SG_CHK(SG_IN(idx, kGBM * kGBK) && SG_IN(idx, kGBK * kGBN), p.status)) {
        As[idx % kGBK][idx / kGBK] = ra[r];
        Bs[idx / kGBN][idx % kGBN] = rb[r];
      }
    }
  };

  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  load_slice(0);
  for (int k0 = 0; k0 < p.K; k0 += kGBK) {
    store_slice();
    __syncthreads();
    if (k0 + kGBK < p.K) load_slice(k0 + kGBK);
#pragma unroll
    for (int k = 0; k < kGBK; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = SG_CHK(SG_IN(ty + 16 * i, kGBM), p.status) ? As[k][ty + 16 * i] : 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = SG_CHK(SG_IN(tx + 16 * j, kGBN), p.status) ? Bs[k][tx + 16 * j] : 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = m0 + ty + 16 * i;
    if (row >= p.M) continue;
    float* crow = p.C + static_cast<int64_t>(row) * p.ldc;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = n0 + tx + 16 * j;
      if (col < p.N) crow[col] = p.beta == 0.f ? p.alpha * acc[i][j] : fmaf(p.alpha, acc[i][j], p.beta * crow[col]);
    }
  }
}

cudaError_t generic_prepare() { return cudaSuccess; }

cudaError_t generic_occupancy(int* ctas) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, sgemm_generic_kernel, kGThreads, 0);
}

cudaError_t generic_launch(const LaunchArgs& a, cudaStream_t stream) {
  GenericParams p{a.A,       a.B,        a.C,        a.lda,      a.ldb,      a.ldc,      a.M,
                  a.N,       a.K,        a.alpha,    a.beta,     a.stride_a, a.stride_b, a.stride_c,
                  a.status};
  const int64_t tiles = static_cast<int64_t>((a.M + kGBM - 1) / kGBM) * ((a.N + kGBN - 1) / kGBN);
  const int batch = a.batch > 1 ? a.batch : 1;
  if (tiles > 0x7fffffff || batch > 65535) return cudaErrorInvalidConfiguration;
  sgemm_generic_kernel<<<dim3(static_cast<unsigned>(tiles), 1, batch), kGThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

const Variant kGenericVariants[] = {
    Variant{"generic_64x64x16", kKindGeneric, kGBM, kGBN, kGBK, 1, 0, kGThreads, 0, 0, &generic_prepare,
            &generic_occupancy, &generic_launch, 0, 0, 1},
};

// C = beta*C over an M x N window with row stride ldc; beta == 0 writes zeros
// without reading C.
__global__ void scale_kernel(float* C, int64_t ldc, int M, int N, float beta, int64_t stride_c) {
  C += blockIdx.y * stride_c;  // batch
  const int64_t total = static_cast<int64_t>(M) * N;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t i = e / N, j = e % N;
    float* d = C + i * ldc + j;
    *d = beta == 0.f ? 0.f : beta * *d;
  }
}

// One thread waits on phase 0 of a barrier that expects one arrival nobody
// makes; the wait must give up after timeout_ns and record it.
__global__ void wait_selftest_kernel(unsigned int* status, uint64_t timeout_ns) {
  __shared__ __align__(8) unsigned long long bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = ptx::smem_addr(&bar);
  ptx::mbar_init(b, 1);
  ptx::fence_barrier_init();
  if (!ptx::mbar_wait(b, 0, timeout_ns)) atomicOr(status, kStatusTimeoutSelftest);
}

}  // namespace

const Variant* generic_variants(int* count) {
  *count = static_cast<int>(sizeof(kGenericVariants) / sizeof(kGenericVariants[0]));
  return kGenericVariants;
}

cudaError_t launch_scale(float* C, int64_t ldc, int M, int N, float beta, cudaStream_t stream, int batch,
                         int64_t stride_c) {
  const int64_t total = static_cast<int64_t>(M) * N;
  int blocks = static_cast<int>((total + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  if (batch < 1) batch = 1;
  if (batch > 65535) return cudaErrorInvalidConfiguration;
  scale_kernel<<<dim3(blocks, batch), 256, 0, stream>>>(C, ldc, M, N, beta, stride_c);
  return cudaGetLastError();
}

// out (cols x rows, ld_out) = transpose of in (rows x cols, ld_in), through a
// 32 x 33 shared tile so both the reads and the writes are coalesced.  Block
// row blockIdx.y takes row tiles blockIdx.y, + gridDim.y, ... (any row count);
// blockIdx.z is the product of a strided batch (in += z*stride_in, out += z*stride_out).
__global__ void transpose_kernel(const float* __restrict__ in, int64_t ld_in, int rows, int cols,
                                 float* __restrict__ out, int64_t ld_out, int64_t stride_in, int64_t stride_out) {
  __shared__ float t[32][33];
  in += blockIdx.z * stride_in;
  out += blockIdx.z * stride_out;
  const int c0 = blockIdx.x * 32;
  const int row_tiles = (rows + 31) / 32;
  for (int ty = blockIdx.y; ty < row_tiles; ty += gridDim.y) {
    const int r0 = ty * 32;
    for (int j = threadIdx.y; j < 32; j += blockDim.y) {
      const int r = r0 + j, c = c0 + threadIdx.x;
      if (r < rows && c < cols) t[j][threadIdx.x] = in[static_cast<int64_t>(r) * ld_in + c];
    }
    __syncthreads();
    for (int j = threadIdx.y; j < 32; j += blockDim.y) {
      const int c = c0 + j, r = r0 + threadIdx.x;
      if (c < cols && r < rows) out[static_cast<int64_t>(c) * ld_out + r] = t[threadIdx.x][j];
    }
    __syncthreads();  // the tile is refilled by the next row tile
  }
}

cudaError_t launch_transpose(const float* in, int64_t ld_in, int rows, int cols, float* out, int64_t ld_out,
                             cudaStream_t stream, int batch, int64_t stride_in, int64_t stride_out) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  if (batch < 1) batch = 1;
  if (batch > 65535) return cudaErrorInvalidConfiguration;
  const int row_tiles = (rows + 31) / 32;
  const dim3 grid((cols + 31) / 32, row_tiles < 65535 ? row_tiles : 65535, batch);
  transpose_kernel<<<grid, dim3(32, 8), 0, stream>>>(in, ld_in, rows, cols, out, ld_out, stride_in, stride_out);
  return cudaGetLastError();
}

// dst (rows x cols, ldd a multiple of 4, dst 16-byte aligned) = src (rows x
// cols, any lds and alignment): a copy that pads rows to 16-byte multiples.
// Consecutive threads take consecutive float4 columns of a row: coalesced
// scalar loads, one 16-byte store each (the last float4 of a row is
// zero-padded).  Block row blockIdx.y takes rows blockIdx.y, + gridDim.y, ...
__global__ void repack_rows_kernel(const float* __restrict__ src, int64_t lds, int rows, int cols,
                                   float* __restrict__ dst, int64_t ldd) {
  const int c = 4 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (c >= cols) return;
  for (int r = blockIdx.y; r < rows; r += gridDim.y) {
    const float* s = src + static_cast<int64_t>(r) * lds + c;
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = c + i < cols ? s[i] : 0.f;
    *reinterpret_cast<float4*>(dst + static_cast<int64_t>(r) * ldd + c) = make_float4(v[0], v[1], v[2], v[3]);
  }
}

cudaError_t launch_repack(const float* src, int64_t lds, int rows, int cols, float* dst, int64_t ldd,
                          cudaStream_t stream) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const int threads = 128;
  const dim3 grid((cols / 4 + threads) / threads, rows < 8192 ? rows : 8192);
  repack_rows_kernel<<<grid, threads, 0, stream>>>(src, lds, rows, cols, dst, ldd);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(unsigned int* status, uint64_t timeout_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace sgemm
