// tc_tf32x3.cu -- C = alpha*A*B + beta*C in float32 on the 5th-generation
// tensor cores, with each operand split into two TF32 parts ("3xTF32").
//
// The pages name tensor cores as the way past the FP32 FMA pipe ("How a
// Matmul Kernel Gets Fast", "Beyond tiling"; "Writing a Fast Matmul in
// CUDA", "What cuBLAS and CUTLASS add") but compute nothing with them; the
// FP32 result here comes from the split, not from the pages.  This path is
// reported on its own, never as the FFMA figure.
//
// Split: x = hi + lo with hi = tf32(x) (round to nearest) and lo = tf32(x -
// hi); x - hi is exact in float32, so |x - hi - lo| <= 2^-22 |x|.  Then
//   a*b ~= hi_a*hi_b + hi_a*lo_b + lo_a*hi_b,
// dropping lo_a*lo_b (<= 2^-22 |a b|).  Each product of two TF32 values is
// exact in the float32 accumulator, so the error per term is about
// 3 * 2^-22 |a b| plus the accumulator's float32 rounding.
//
// Kernels (all launched by one sgemm_run):
//  * split_rows / split_transpose: A -> A_hi, A_lo (M x kp) and B -> B_hi,
//    B_lo (N x kp), both K-major.  An operand already stored K-major (A as
//    M x K, or B given transposed as N x K) is split row by row; the other
//    layout is transposed through a 32 x 33 shared tile while splitting;
//  * tf32x3_kernel: one 128 x 256 output tile per CTA.  Warp 0 issues TMA
//    copies of the four 32-deep operand slices (128-byte swizzle) into a
//    two-stage ring; warp 1 owns 256 TMEM columns and issues, per slice,
//    12 tcgen05.mma.kind::tf32 of 128 x 256 x 8 (lo*hi, hi*lo, hi*hi for
//    each k-step of 8) into the TMEM accumulator, then commits to the
//    stage's empty barrier; warps 2-5 read the accumulator back with
//    tcgen05.ld (warp w owns TMEM lanes 32*(w%4) .. +31, i.e. those rows)
//    and apply alpha and beta.  Every wait is bounded; the MMA thread
//    always commits to the accumulator barrier, so no MMA is in flight when
//    the epilogue reads TMEM and the CTA frees it.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"
#include "tile_order.cuh"

namespace sgemm {
namespace tc {

constexpr int BM = 128;
constexpr int BK = 32;  // one 128-byte swizzle row of float32
constexpr int kTileA = BM * BK * 4;  // 16 KB
constexpr int kBarBytes = 256;
constexpr int kThreads = 192;

// Tile width BN (the MMA's N and the TMEM columns) and ring depth.
template <int BN, int STAGES>
struct TcShape {
  static constexpr int kTileB = BN * BK * 4;
  static constexpr int kStageBytes = 2 * kTileA + 2 * kTileB;
  static constexpr int kSmemBytes = STAGES * kStageBytes + kBarBytes + 1024;
  static constexpr uint32_t kTmemCols = BN;
  // D float32, A and B TF32, both K-major, M = 128, N = BN
  static constexpr uint32_t kIdesc = (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
                                     (static_cast<uint32_t>(BM >> 4) << 24);
  static_assert(BN == 128 || BN == 256, "UMMA N of 128 or 256");
  static_assert(kTileA % 1024 == 0 && kTileB % 1024 == 0, "swizzle atoms stay 1024-byte aligned");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};

struct TcParams {
  float* C;
  int64_t ldc;
  int M, N, K;
  float alpha, beta;
  int group_m;
  int vec_c;  // C 16-byte aligned with ldc % 4 == 0: float4 epilogue
  unsigned int* status;
  uint64_t timeout_ns;
};

__device__ __forceinline__ float to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// Rows of X (rows x cols, ldx) -> hi, lo (rows x cols, ldh).  Block row
// blockIdx.y covers rows blockIdx.y, + gridDim.y, ...; blockIdx.x a span of
// 4 * blockDim.x columns, read and written as float4 when VEC (X 16-byte
// aligned, ldx and cols multiples of 4; ldh always is).
template <bool VEC>
__global__ void split_rows_kernel(const float* __restrict__ X, int64_t ldx, int rows, int cols, float* __restrict__ hi,
                                  float* __restrict__ lo, int64_t ldh) {
  const int c = 4 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (c >= cols) return;
  for (int r = blockIdx.y; r < rows; r += gridDim.y) {
    const float* x = X + static_cast<int64_t>(r) * ldx + c;
    float v[4];
    if constexpr (VEC) {
      const float4 q = __ldcs(reinterpret_cast<const float4*>(x));
      v[0] = q.x, v[1] = q.y, v[2] = q.z, v[3] = q.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = c + j < cols ? x[j] : 0.f;
    }
    float h[4], l[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      h[j] = to_tf32(v[j]);
      l[j] = to_tf32(v[j] - h[j]);
    }
    float* ho = hi + static_cast<int64_t>(r) * ldh + c;
    float* lo_ = lo + static_cast<int64_t>(r) * ldh + c;
    if constexpr (VEC) {
      *reinterpret_cast<float4*>(ho) = make_float4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<float4*>(lo_) = make_float4(l[0], l[1], l[2], l[3]);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (c + j < cols) {
          ho[j] = h[j];
          lo_[j] = l[j];
        }
    }
  }
}

void launch_split_rows(const float* X, int64_t ldx, int rows, int cols, float* hi, float* lo, int64_t ldh,
                       cudaStream_t stream) {
  const int threads = 128;
  const int gx = (cols + 4 * threads - 1) / (4 * threads);
  const int gy = rows < 4096 ? rows : 4096;
  const bool vec = (reinterpret_cast<uintptr_t>(X) & 15) == 0 && ldx % 4 == 0 && cols % 4 == 0;
  if (vec) {
    split_rows_kernel<true><<<dim3(gx, gy), threads, 0, stream>>>(X, ldx, rows, cols, hi, lo, ldh);
  } else {
    split_rows_kernel<false><<<dim3(gx, gy), threads, 0, stream>>>(X, ldx, rows, cols, hi, lo, ldh);
  }
}

// X (rows x cols, ldx) -> hi, lo transposed (cols x rows, ldh).
__global__ void split_transpose_kernel(const float* __restrict__ X, int64_t ldx, int rows, int cols,
                                       float* __restrict__ hi, float* __restrict__ lo, int64_t ldh) {
  __shared__ float t[32][33];
  const int c0 = blockIdx.x * 32;
  const int r0 = blockIdx.y * 32;
  for (int j = threadIdx.y; j < 32; j += blockDim.y) {
    const int r = r0 + j, c = c0 + threadIdx.x;
    t[j][threadIdx.x] = (r < rows && c < cols) ? X[static_cast<int64_t>(r) * ldx + c] : 0.f;
  }
  __syncthreads();
  for (int j = threadIdx.y; j < 32; j += blockDim.y) {
    const int c = c0 + j, r = r0 + threadIdx.x;  // output row c, column r
    if (c < cols && r < rows) {
      const float x = t[threadIdx.x][j];
      const float h = to_tf32(x);
      hi[static_cast<int64_t>(c) * ldh + r] = h;
      lo[static_cast<int64_t>(c) * ldh + r] = to_tf32(x - h);
    }
  }
}

// Shared-memory matrix descriptor: K-major operand, rows of 128 bytes with
// the 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);  // start address
  d |= static_cast<uint64_t>(1) << 16;                          // leading offset (unused when swizzled K-major)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;                  // stride offset between 8-row groups
  d |= static_cast<uint64_t>(1) << 46;                          // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                          // 128-byte swizzle
  return d;
}

__device__ __forceinline__ void mma_tf32(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 32 columns of 32-bit words: thread t of the warp gets lane
// (taddr lane + t), columns taddr col .. +31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    tf32x3_kernel(const __grid_constant__ CUtensorMap tmAh, const __grid_constant__ CUtensorMap tmAl,
                  const __grid_constant__ CUtensorMap tmBh, const __grid_constant__ CUtensorMap tmBl,
                  const TcParams p) {
  using S = TcShape<BN, STAGES>;
  constexpr int kTileB = S::kTileB;
  constexpr int kStageBytes = S::kStageBytes;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_base = ptx::smem_addr(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
  const uint32_t smem_base = ptx::smem_addr(smem);
  const uint32_t bar_base = smem_base + STAGES * kStageBytes;
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  const uint32_t accum_bar = bar_base + 8u * (2 * STAGES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + STAGES * kStageBytes + 8 * (2 * STAGES + 1));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_m = (p.M + BM - 1) / BM;
  const int tiles_n = (p.N + BN - 1) / BN;
  int tm, tn;
  tile_coords(blockIdx.x, tiles_m, tiles_n, p.group_m, tm, tn);
  const int KT = (p.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    ptx::mbar_init(accum_bar, 1);
    ptx::fence_barrier_init();
    ptx::prefetch_tensormap(&tmAh);
    ptx::prefetch_tensormap(&tmAl);
    ptx::prefetch_tensormap(&tmBh);
    ptx::prefetch_tensormap(&tmBl);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(ptx::smem_addr(tmem_slot)),
                 "r"(S::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  if (warp == 0 && lane == 0) {
    // ---- producer: four TMA copies per slice ----
    int issued = 0;
    for (int kb = 0; kb < KT; ++kb) {
      const int s = kb % STAGES;
      if (kb >= STAGES && !ptx::mbar_wait(empty_bar(s), ((kb / STAGES) - 1) & 1, p.timeout_ns)) {
        atomicOr(p.status, kStatusTimeoutEmpty);
        break;
      }
      const uint32_t st = smem_base + s * kStageBytes;
      ptx::mbar_arrive_expect_tx(full_bar(s), kStageBytes);
      ptx::tma_load_2d(st, &tmAh, kb * BK, tm * BM, full_bar(s));
      ptx::tma_load_2d(st + kTileA, &tmAl, kb * BK, tm * BM, full_bar(s));
      ptx::tma_load_2d(st + 2 * kTileA, &tmBh, kb * BK, tn * BN, full_bar(s));
      ptx::tma_load_2d(st + 2 * kTileA + kTileB, &tmBl, kb * BK, tn * BN, full_bar(s));
      issued = kb + 1;
    }
    // Before leaving, every copy this thread started has landed (bounded):
    // the last STAGES slices are the only ones possibly still in flight.
    for (int kb = issued > STAGES ? issued - STAGES : 0; kb < issued; ++kb)
      ptx::mbar_wait(full_bar(kb % STAGES), (kb / STAGES) & 1, p.timeout_ns);
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ----
    for (int kb = 0; kb < KT; ++kb) {
      const int s = kb % STAGES;
      if (!ptx::mbar_wait(full_bar(s), (kb / STAGES) & 1, p.timeout_ns)) {
        atomicOr(p.status, kStatusTimeoutFull);
        break;
      }
      tc_fence_after();
      const uint32_t st = smem_base + s * kStageBytes;
#pragma unroll
      for (int kk = 0; kk < BK / 8; ++kk) {  // 8 TF32 = 32 bytes per MMA along K
        const uint64_t ah = smem_desc_sw128(st + 32 * kk);
        const uint64_t al = smem_desc_sw128(st + kTileA + 32 * kk);
        const uint64_t bh = smem_desc_sw128(st + 2 * kTileA + 32 * kk);
        const uint64_t bl = smem_desc_sw128(st + 2 * kTileA + kTileB + 32 * kk);
        mma_tf32(tmem, al, bh, S::kIdesc, (kb | kk) != 0 ? 1u : 0u);
        mma_tf32(tmem, ah, bl, S::kIdesc, 1u);
        mma_tf32(tmem, ah, bh, S::kIdesc, 1u);
      }
      mma_commit(empty_bar(s));  // the stage is free once these MMAs have read it
    }
    mma_commit(accum_bar);  // arrives when every MMA issued above has completed
  } else if (warp >= 2) {
    // ---- epilogue: TMEM -> registers -> alpha, beta -> C ----
    const bool ok = ptx::mbar_wait(accum_bar, 0, p.timeout_ns);
    if (!ok) atomicOr(p.status, kStatusTimeoutFull);
    tc_fence_after();
    const int lane_base = 32 * (warp & 3);
    const int row = tm * BM + lane_base + lane;
#pragma unroll 1
    for (int cc = 0; cc < BN; cc += 32) {
      uint32_t r[32];
      tmem_ld32(tmem + (static_cast<uint32_t>(lane_base) << 16) + static_cast<uint32_t>(cc), r);
      if (!ok || row >= p.M) continue;
      float* crow = p.C + static_cast<int64_t>(row) * p.ldc;
      const int col0 = tn * BN + cc;
      if (p.vec_c && col0 + 32 <= p.N) {  // this thread's 32 columns as eight float4
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          float4* d = reinterpret_cast<float4*>(crow + col0 + j);
          const float4 v = make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]), __uint_as_float(r[j + 2]),
                                       __uint_as_float(r[j + 3]));
          if (p.beta == 0.f) {
            *d = make_float4(p.alpha * v.x, p.alpha * v.y, p.alpha * v.z, p.alpha * v.w);
          } else {
            const float4 o = *d;
            *d = make_float4(fmaf(p.alpha, v.x, p.beta * o.x), fmaf(p.alpha, v.y, p.beta * o.y),
                             fmaf(p.alpha, v.z, p.beta * o.z), fmaf(p.alpha, v.w, p.beta * o.w));
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int col = col0 + j;
          if (col < p.N) {
            const float v = __uint_as_float(r[j]);
            crow[col] = p.beta == 0.f ? p.alpha * v : fmaf(p.alpha, v, p.beta * crow[col]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(S::kTmemCols) : "memory");
  }
}

// Operand split for one run: A_hi, A_lo (M x kp), then B_hi, B_lo (N x kp),
// both K-major, in a.split; the tensor maps in a (tmA, tmA2, tmB, tmB2)
// describe those four buffers.
void launch_split(const LaunchArgs& a, cudaStream_t stream) {
  const int64_t kp = a.split_ld;
  float* ah = a.split;
  float* al = ah + static_cast<int64_t>(a.M) * kp;
  float* bh = al + static_cast<int64_t>(a.M) * kp;
  float* bl = bh + static_cast<int64_t>(a.N) * kp;
  // both operands end K-major: A as M x kp, B as N x kp
  if (a.a_trans) {  // A stored K x M
    split_transpose_kernel<<<dim3((a.M + 31) / 32, (a.K + 31) / 32), dim3(32, 8), 0, stream>>>(a.A, a.lda, a.K, a.M,
                                                                                            ah, al, kp);
  } else {
    launch_split_rows(a.A, a.lda, a.M, a.K, ah, al, kp, stream);
  }
  if (a.b_trans) {  // B stored N x K: already K-major
    launch_split_rows(a.B, a.ldb, a.N, a.K, bh, bl, kp, stream);
  } else {
    split_transpose_kernel<<<dim3((a.N + 31) / 32, (a.K + 31) / 32), dim3(32, 8), 0, stream>>>(a.B, a.ldb, a.K, a.N,
                                                                                            bh, bl, kp);
  }
}

template <int BN, int STAGES>
struct TcVariant {
  using S = TcShape<BN, STAGES>;
  static constexpr auto kernel = tf32x3_kernel<BN, STAGES>;
  static cudaError_t prepare() {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
  }
  static cudaError_t occupancy(int* ctas) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, kernel, kThreads, S::kSmemBytes);
  }
  static cudaError_t launch(const LaunchArgs& a, cudaStream_t stream) {
    launch_split(a, stream);
    TcParams p;
    p.C = a.C;
    p.ldc = a.ldc;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.alpha = a.alpha;
    p.beta = a.beta;
    p.group_m = 8;
    p.vec_c = (reinterpret_cast<uintptr_t>(a.C) & 15) == 0 && a.ldc % 4 == 0;
    p.status = a.status;
    p.timeout_ns = a.timeout_ns;
    kernel<<<a.grid, kThreads, S::kSmemBytes, stream>>>(a.tmA, a.tmA2, a.tmB, a.tmB2, p);
    return cudaGetLastError();
  }
  static Variant describe(const char* name) {
    return Variant{name, kKindTc, BM, BN, BK, STAGES, 0, kThreads, S::kSmemBytes, 128, &prepare, &occupancy,
                   &launch, 0, 0};
  }
};

const Variant kVariants[] = {
    TcVariant<256, 2>::describe("tf32x3_128x256x32_s2"),
    TcVariant<128, 3>::describe("tf32x3_128x128x32_s3"),
};

}  // namespace tc

const Variant* tc_variants(int* count) {
  *count = static_cast<int>(sizeof(tc::kVariants) / sizeof(tc::kVariants[0]));
  return tc::kVariants;
}

}  // namespace sgemm
