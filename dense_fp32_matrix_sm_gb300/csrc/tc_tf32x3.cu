// tc_tf32x3.cu -- C = alpha*A*B + beta*C in float32 on the 5th-generation
// tensor cores, with each operand split into two TF32 parts ("3xTF32").
//
// The pages name tensor cores as the way past the FP32 FMA pipe ("CUDA
// Matrix Multiplication Optimization: From Naive to Near-cuBLAS", "Beyond
// Tiling: Async, Tensor Cores, and Scheduling"; "Writing a Fast Matmul in
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

// X (rows x cols, ldx) -> hi, lo transposed (cols x rows, ldh; ldh a
// multiple of 4, hi and lo 16-byte aligned).  A block of 32 x 8 threads
// moves 32 x 32 tiles through shared memory: coalesced 128-byte row reads,
// then each thread writes one float4 of four consecutive rows to each
// output (a warp covers four output rows; the column reads hit 32 distinct
// banks).  Block row blockIdx.y takes row tiles blockIdx.y, + gridDim.y,
// ... (any row count).
__global__ void split_transpose_kernel(const float* __restrict__ X, int64_t ldx, int rows, int cols,
                                       float* __restrict__ hi, float* __restrict__ lo, int64_t ldh) {
  __shared__ float t[32][33];
  const int c0 = blockIdx.x * 32;
  const int row_tiles = (rows + 31) / 32;
  const int tid = threadIdx.y * 32 + threadIdx.x;
  const int oc = tid >> 3;  // output row c0 + oc
  const int q = tid & 7;    // output columns r0 + 4q .. + 3
  for (int ty = blockIdx.y; ty < row_tiles; ty += gridDim.y) {
    const int r0 = ty * 32;
    for (int j = threadIdx.y; j < 32; j += blockDim.y) {
      const int r = r0 + j, c = c0 + threadIdx.x;
      t[j][threadIdx.x] = (r < rows && c < cols) ? X[static_cast<int64_t>(r) * ldx + c] : 0.f;
    }
    __syncthreads();
    const int c = c0 + oc;
    const int r = r0 + 4 * q;
    if (c < cols && r < rows) {
      float h[4], l[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float x = t[4 * q + i][oc];
        h[i] = to_tf32(x);
        l[i] = to_tf32(x - h[i]);
      }
      float* ho = hi + static_cast<int64_t>(c) * ldh + r;
      float* lo_ = lo + static_cast<int64_t>(c) * ldh + r;
      if (r + 3 < rows) {
        *reinterpret_cast<float4*>(ho) = make_float4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<float4*>(lo_) = make_float4(l[0], l[1], l[2], l[3]);
      } else {
        for (int i = 0; i < 4 && r + i < rows; ++i) {
          ho[i] = h[i];
          lo_[i] = l[i];
        }
      }
    }
    __syncthreads();  // the tile is refilled by the next row tile
  }
}

void launch_split_transpose(const float* X, int64_t ldx, int rows, int cols, float* hi, float* lo, int64_t ldh,
                            cudaStream_t stream) {
  const int row_tiles = (rows + 31) / 32;
  const dim3 grid((cols + 31) / 32, row_tiles < 65535 ? row_tiles : 65535);
  split_transpose_kernel<<<grid, dim3(32, 8), 0, stream>>>(X, ldx, rows, cols, hi, lo, ldh);
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
    ptx::drain_ring(full_bar(0), 8u, static_cast<uint32_t>(issued), STAGES, p.timeout_ns);
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
    launch_split_transpose(a.A, a.lda, a.K, a.M, ah, al, kp, stream);
  } else {
    launch_split_rows(a.A, a.lda, a.M, a.K, ah, al, kp, stream);
  }
  if (a.b_trans) {  // B stored N x K: already K-major
    launch_split_rows(a.B, a.ldb, a.N, a.K, bh, bl, kp, stream);
  } else {
    launch_split_transpose(a.B, a.ldb, a.K, a.N, bh, bl, kp, stream);
  }
}

// ---------------------------------------------------------------------------
// Persistent form: one CTA per SM walks tiles (grouped order) with the same
// split operands and ring, and two TMEM accumulators of BN columns.  The MMA
// warp fills one accumulator while warps 2-5 drain the other: after reading
// a chunk of it they store it, and once the whole accumulator is read they
// release it (one arrival per warp) for the tile after next.  A role that
// gives up sets a shared abort flag, so the others stop waiting at once.
template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    tf32x3_persistent_kernel(const __grid_constant__ CUtensorMap tmAh, const __grid_constant__ CUtensorMap tmAl,
                             const __grid_constant__ CUtensorMap tmBh, const __grid_constant__ CUtensorMap tmBl,
                             const TcParams p) {
  using S = TcShape<BN, STAGES>;
  constexpr int kTileB = S::kTileB;
  constexpr int kStageBytes = S::kStageBytes;
  constexpr uint32_t kCols = 2 * S::kTmemCols;  // two accumulators
  static_assert(kCols <= 512, "TMEM holds 512 columns");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ int s_abort;
  const uint32_t raw_base = ptx::smem_addr(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
  const uint32_t smem_base = ptx::smem_addr(smem);
  const uint32_t bar_base = smem_base + STAGES * kStageBytes;
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  auto acc_full = [&](int b) { return bar_base + 8u * (2 * STAGES + b); };
  auto acc_empty = [&](int b) { return bar_base + 8u * (2 * STAGES + 2 + b); };
  const uint32_t mma_done = bar_base + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + STAGES * kStageBytes + 8 * (2 * STAGES + 5));
  const volatile int* abort_flag = &s_abort;
  auto fail = [&](unsigned int bit) {
    atomicOr(p.status, bit);
    *reinterpret_cast<volatile int*>(&s_abort) = 1;
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_m = (p.M + BM - 1) / BM;
  const int tiles_n = (p.N + BN - 1) / BN;
  const int num_tiles = tiles_m * tiles_n;
  const int G = static_cast<int>(gridDim.x);
  const int my_tiles = static_cast<int>(blockIdx.x) < num_tiles ? (num_tiles - 1 - static_cast<int>(blockIdx.x)) / G + 1 : 0;
  const int KT = (p.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(acc_full(b), 1);
      ptx::mbar_init(acc_empty(b), 4);  // one arrival per epilogue warp
    }
    ptx::mbar_init(mma_done, 1);
    ptx::fence_barrier_init();
    ptx::prefetch_tensormap(&tmAh);
    ptx::prefetch_tensormap(&tmAl);
    ptx::prefetch_tensormap(&tmBh);
    ptx::prefetch_tensormap(&tmBl);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(ptx::smem_addr(tmem_slot)),
                 "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  if (warp == 0 && lane == 0) {
    // ---- producer: slices of every tile, one ring across tiles ----
    uint32_t g = 0;
    for (int i = 0; i < my_tiles && !*abort_flag; ++i) {
      int tm, tn;
      tile_coords(static_cast<int>(blockIdx.x) + i * G, tiles_m, tiles_n, p.group_m, tm, tn);
      for (int kb = 0; kb < KT; ++kb, ++g) {
        const int s = static_cast<int>(g % STAGES);
        const uint32_t use = g / STAGES;
        if (g >= STAGES && !ptx::mbar_wait_or_abort(empty_bar(s), (use - 1) & 1u, p.timeout_ns, abort_flag)) {
          if (!*abort_flag) fail(kStatusTimeoutEmpty);
          i = my_tiles;
          break;
        }
        const uint32_t st = smem_base + s * kStageBytes;
        ptx::mbar_arrive_expect_tx(full_bar(s), kStageBytes);
        ptx::tma_load_2d(st, &tmAh, kb * BK, tm * BM, full_bar(s));
        ptx::tma_load_2d(st + kTileA, &tmAl, kb * BK, tm * BM, full_bar(s));
        ptx::tma_load_2d(st + 2 * kTileA, &tmBh, kb * BK, tn * BN, full_bar(s));
        ptx::tma_load_2d(st + 2 * kTileA + kTileB, &tmBl, kb * BK, tn * BN, full_bar(s));
      }
    }
    // every copy started here has landed before the CTA can leave
    ptx::drain_ring(full_bar(0), 8u, g, STAGES, p.timeout_ns);
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ----
    uint32_t g = 0;
    bool ok = true;
    for (int i = 0; i < my_tiles && ok; ++i) {
      const int b = i & 1;
      if (i >= 2 && !ptx::mbar_wait_or_abort(acc_empty(b), ((i >> 1) - 1) & 1, p.timeout_ns, abort_flag)) {
        if (!*abort_flag) fail(kStatusTimeoutEmpty);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem + static_cast<uint32_t>(b) * S::kTmemCols;
      for (int kb = 0; kb < KT; ++kb, ++g) {
        const int s = static_cast<int>(g % STAGES);
        if (!ptx::mbar_wait_or_abort(full_bar(s), (g / STAGES) & 1u, p.timeout_ns, abort_flag)) {
          if (!*abort_flag) fail(kStatusTimeoutFull);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t st = smem_base + s * kStageBytes;
#pragma unroll
        for (int kk = 0; kk < BK / 8; ++kk) {
          const uint64_t ah = smem_desc_sw128(st + 32 * kk);
          const uint64_t al = smem_desc_sw128(st + kTileA + 32 * kk);
          const uint64_t bh = smem_desc_sw128(st + 2 * kTileA + 32 * kk);
          const uint64_t bl = smem_desc_sw128(st + 2 * kTileA + kTileB + 32 * kk);
          mma_tf32(d, al, bh, S::kIdesc, (kb | kk) != 0 ? 1u : 0u);
          mma_tf32(d, ah, bl, S::kIdesc, 1u);
          mma_tf32(d, ah, bh, S::kIdesc, 1u);
        }
        mma_commit(empty_bar(s));
      }
      if (ok) mma_commit(acc_full(b));
    }
    mma_commit(mma_done);  // arrives when every MMA issued above has completed
  } else if (warp >= 2) {
    // ---- epilogue: TMEM -> registers -> alpha, beta -> C, tile after tile ----
    const int lane_base = 32 * (warp & 3);
    for (int i = 0; i < my_tiles; ++i) {
      const int b = i & 1;
      if (!ptx::mbar_wait_or_abort(acc_full(b), (i >> 1) & 1, p.timeout_ns, abort_flag)) {
        if (!*abort_flag) fail(kStatusTimeoutFull);
        break;
      }
      tc_fence_after();
      int tm, tn;
      tile_coords(static_cast<int>(blockIdx.x) + i * G, tiles_m, tiles_n, p.group_m, tm, tn);
      const int row = tm * BM + lane_base + lane;
      float* crow = p.C + static_cast<int64_t>(row) * p.ldc;
#pragma unroll 1
      for (int cc = 0; cc < BN; cc += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(lane_base) << 16) + static_cast<uint32_t>(b * BN + cc), r);
        if (row >= p.M) continue;
        const int col0 = tn * BN + cc;
        if (p.vec_c && col0 + 32 <= p.N) {
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            float4* dst = reinterpret_cast<float4*>(crow + col0 + j);
            const float4 v = make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]), __uint_as_float(r[j + 2]),
                                         __uint_as_float(r[j + 3]));
            if (p.beta == 0.f) {
              *dst = make_float4(p.alpha * v.x, p.alpha * v.y, p.alpha * v.z, p.alpha * v.w);
            } else {
              const float4 o = *dst;
              *dst = make_float4(fmaf(p.alpha, v.x, p.beta * o.x), fmaf(p.alpha, v.y, p.beta * o.y),
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
      // this warp has read its lanes of accumulator b: release it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(acc_empty(b));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) ptx::mbar_wait(mma_done, 0, p.timeout_ns);  // no MMA may still write TMEM
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols) : "memory");
  }
}

template <int BN, int STAGES, bool PERSIST = false>
struct TcVariant {
  using S = TcShape<BN, STAGES>;
  static constexpr auto kernel = PERSIST ? tf32x3_persistent_kernel<BN, STAGES> : tf32x3_kernel<BN, STAGES>;
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
                   &launch, PERSIST ? 1 : 0, 0};
  }
};

// ---------------------------------------------------------------------------
// Fused form: the split happens inside the GEMM kernel.
//  * Warp 0 copies the raw float32 slices of A and B (32 deep, 128 rows
//    each) by TMA into a 3-deep raw ring, hiding the copy latency.
//  * Eight converter warps turn raw slot r into the hi and lo parts of both
//    operands in slot h of a 2-deep split ring: K-major tiles in the layout
//    the MMA reads (128-byte rows, 16-byte chunk q of row r at position
//    q ^ (r % 8), the layout TMA's 128-byte swizzle gives).  A K-major
//    source (A as stored, B given transposed) arrives with that swizzle and
//    converts chunk by chunk; an MN-major source (B as stored, A given
//    transposed) arrives unswizzled as [32 k][128 rows] and is transposed
//    while converting.  They fence the async proxy, then release the raw
//    slot and publish the split slot.
//  * Warp 1 issues the MMAs on split slots as they are published.
//  * The converter warps run the epilogue after the last slice.
constexpr int kFBN = 128;
constexpr int kFRawStages = 3;
constexpr int kFSplitStages = 2;
constexpr int kFThreads = 320;                    // warp 0 TMA, warp 1 MMA, warps 2-9 convert + epilogue
constexpr int kFConv = 256;                       // converter threads
constexpr int kFTile = BM * BK * 4;               // 16 KB: one 128-row x 32-k operand slice
constexpr int kFRawBytes = kFRawStages * 2 * kFTile;      // raw A, raw B per slot
constexpr int kFSplitBytes = kFSplitStages * 4 * kFTile;  // A_hi, A_lo, B_hi, B_lo per slot
constexpr int kFSmemBytes = kFRawBytes + kFSplitBytes + kBarBytes + 1024;
static_assert(kFSmemBytes <= 227 * 1024, "shared memory per CTA");
constexpr uint32_t kFIdesc = TcShape<kFBN, 1>::kIdesc;

// Converter thread t (0..255) takes half of one 128-row x 32-k slice:
// raw -> hi, lo (both K-major, swizzled).  MN_MAJOR: raw is [32 k][128 rows]
// (512-byte rows, no swizzle); else raw is already K-major and swizzled.
template <bool MN_MAJOR>
__device__ __forceinline__ void convert_half(const unsigned char* raw, unsigned char* hi, unsigned char* lo, int t) {
  if constexpr (MN_MAJOR) {
    // row t % 128, chunks q of half t / 128: 4 k values per chunk, one from
    // each raw row (consecutive threads read consecutive words), stored as
    // one 16-byte chunk
    const float* r = reinterpret_cast<const float*>(raw);
    const int row = t & 127;
    const int q0 = 4 * (t >> 7);
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
      const int q = q0 + qq;
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = r[(4 * q + j) * BM + row];
      float h[4], l[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        h[j] = to_tf32(v[j]);
        l[j] = to_tf32(v[j] - h[j]);
      }
      const int off = row * 128 + ((q ^ (row & 7)) << 4);
      *reinterpret_cast<float4*>(hi + off) = make_float4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<float4*>(lo + off) = make_float4(l[0], l[1], l[2], l[3]);
    }
  } else {
    // 1024 chunks of 16 bytes, 4 per thread; the swizzle is the same in all three tiles
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int off = (t + kFConv * i) << 4;
      const float4 v = *reinterpret_cast<const float4*>(raw + off);
      const float x[4] = {v.x, v.y, v.z, v.w};
      float h[4], l[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        h[j] = to_tf32(x[j]);
        l[j] = to_tf32(x[j] - h[j]);
      }
      *reinterpret_cast<float4*>(hi + off) = make_float4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<float4*>(lo + off) = make_float4(l[0], l[1], l[2], l[3]);
    }
  }
}

// TA: A given transposed (stored K x M); TB: B given transposed (stored N x K).
template <bool TA, bool TB>
__global__ void __launch_bounds__(kFThreads, 1)
    tf32x3_fused_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const TcParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_base = ptx::smem_addr(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
  const uint32_t smem_base = ptx::smem_addr(smem);
  // raw slot r: A at raw_off(r, 0), B at raw_off(r, 1); split slot h: part i
  // (0 A_hi, 1 A_lo, 2 B_hi, 3 B_lo) at split_off(h, i)
  auto raw_off = [](int r, int i) { return (2 * r + i) * kFTile; };
  auto split_off = [](int h, int i) { return kFRawBytes + (4 * h + i) * kFTile; };
  const uint32_t bar_base = smem_base + kFRawBytes + kFSplitBytes;
  auto raw_full = [&](int r) { return bar_base + 8u * r; };
  auto raw_empty = [&](int r) { return bar_base + 8u * (kFRawStages + r); };
  auto split_full = [&](int h) { return bar_base + 8u * (2 * kFRawStages + h); };
  auto split_empty = [&](int h) { return bar_base + 8u * (2 * kFRawStages + kFSplitStages + h); };
  const uint32_t accum_bar = bar_base + 8u * (2 * kFRawStages + 2 * kFSplitStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kFRawBytes + kFSplitBytes +
                                                    8 * (2 * kFRawStages + 2 * kFSplitStages + 1));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_m = (p.M + BM - 1) / BM;
  const int tiles_n = (p.N + kFBN - 1) / kFBN;
  int tm, tn;
  tile_coords(blockIdx.x, tiles_m, tiles_n, p.group_m, tm, tn);
  const int KT = (p.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int r = 0; r < kFRawStages; ++r) {
      ptx::mbar_init(raw_full(r), 1);
      ptx::mbar_init(raw_empty(r), kFConv);
    }
    for (int h = 0; h < kFSplitStages; ++h) {
      ptx::mbar_init(split_full(h), kFConv);
      ptx::mbar_init(split_empty(h), 1);
    }
    ptx::mbar_init(accum_bar, 1);
    ptx::fence_barrier_init();
    ptx::prefetch_tensormap(&tmA);
    ptx::prefetch_tensormap(&tmB);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(ptx::smem_addr(tmem_slot)),
                 "r"(static_cast<uint32_t>(kFBN))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  if (warp == 0 && lane == 0) {
    // ---- producer: raw slices of A and B ----
    int issued = 0;
    for (int kb = 0; kb < KT; ++kb) {
      const int r = kb % kFRawStages;
      if (kb >= kFRawStages && !ptx::mbar_wait(raw_empty(r), ((kb / kFRawStages) - 1) & 1, p.timeout_ns)) {
        atomicOr(p.status, kStatusTimeoutEmpty);
        break;
      }
      ptx::mbar_arrive_expect_tx(raw_full(r), 2 * kFTile);
      if constexpr (TA) {
        ptx::tma_load_2d(smem_base + raw_off(r, 0), &tmA, tm * BM, kb * BK, raw_full(r));
      } else {
        ptx::tma_load_2d(smem_base + raw_off(r, 0), &tmA, kb * BK, tm * BM, raw_full(r));
      }
      if constexpr (TB) {
        ptx::tma_load_2d(smem_base + raw_off(r, 1), &tmB, kb * BK, tn * kFBN, raw_full(r));
      } else {
        ptx::tma_load_2d(smem_base + raw_off(r, 1), &tmB, tn * kFBN, kb * BK, raw_full(r));
      }
      issued = kb + 1;
    }
    // every copy started here has landed before the CTA can leave
    ptx::drain_ring(raw_full(0), 8u, static_cast<uint32_t>(issued), kFRawStages, p.timeout_ns);
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ----
    for (int kb = 0; kb < KT; ++kb) {
      const int h = kb % kFSplitStages;
      if (!ptx::mbar_wait(split_full(h), (kb / kFSplitStages) & 1, p.timeout_ns)) {
        atomicOr(p.status, kStatusTimeoutFull);
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < BK / 8; ++kk) {
        const uint64_t ah = smem_desc_sw128(smem_base + split_off(h, 0) + 32 * kk);
        const uint64_t al = smem_desc_sw128(smem_base + split_off(h, 1) + 32 * kk);
        const uint64_t bh = smem_desc_sw128(smem_base + split_off(h, 2) + 32 * kk);
        const uint64_t bl = smem_desc_sw128(smem_base + split_off(h, 3) + 32 * kk);
        mma_tf32(tmem, al, bh, kFIdesc, (kb | kk) != 0 ? 1u : 0u);
        mma_tf32(tmem, ah, bl, kFIdesc, 1u);
        mma_tf32(tmem, ah, bh, kFIdesc, 1u);
      }
      mma_commit(split_empty(h));  // the split slot is free once these MMAs have read it
    }
    mma_commit(accum_bar);  // arrives when every MMA issued above has completed
  } else if (warp >= 2) {
    // ---- converters ----
    const int t = threadIdx.x - 64;
    bool ok = true;
    for (int kb = 0; kb < KT; ++kb) {
      const int r = kb % kFRawStages, h = kb % kFSplitStages;
      if (!ptx::mbar_wait(raw_full(r), (kb / kFRawStages) & 1, p.timeout_ns) ||
          (kb >= kFSplitStages && !ptx::mbar_wait(split_empty(h), ((kb / kFSplitStages) - 1) & 1, p.timeout_ns))) {
        atomicOr(p.status, kStatusTimeoutFull);
        ok = false;
        break;
      }
      convert_half<TA>(smem + raw_off(r, 0), smem + split_off(h, 0), smem + split_off(h, 1), t);
      convert_half<!TB>(smem + raw_off(r, 1), smem + split_off(h, 2), smem + split_off(h, 3), t);
      ptx::fence_proxy_async_smem();  // the MMA reads the split tiles through the async proxy
      ptx::mbar_arrive(split_full(h));
      ptx::mbar_arrive(raw_empty(r));
    }
    // ---- epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 (its rows),
    //      columns 64 ((w - 2) / 4) .. +63 ----
    const bool done = ptx::mbar_wait(accum_bar, 0, p.timeout_ns);
    if (!done) atomicOr(p.status, kStatusTimeoutFull);
    tc_fence_after();
    const int lane_base = 32 * (warp & 3);
    const int col_half = (warp - 2) >> 2;
    const int row = tm * BM + lane_base + lane;
#pragma unroll 1
    for (int cc = 64 * col_half; cc < 64 * col_half + 64; cc += 32) {
      uint32_t rr[32];
      tmem_ld32(tmem + (static_cast<uint32_t>(lane_base) << 16) + static_cast<uint32_t>(cc), rr);
      if (!done || !ok || row >= p.M) continue;
      float* crow = p.C + static_cast<int64_t>(row) * p.ldc;
      const int col0 = tn * kFBN + cc;
      if (p.vec_c && col0 + 32 <= p.N) {
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          float4* d = reinterpret_cast<float4*>(crow + col0 + j);
          const float4 v = make_float4(__uint_as_float(rr[j]), __uint_as_float(rr[j + 1]),
                                       __uint_as_float(rr[j + 2]), __uint_as_float(rr[j + 3]));
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
            const float v = __uint_as_float(rr[j]);
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
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(static_cast<uint32_t>(kFBN))
                 : "memory");
  }
}

struct TcFusedVariant {
  static constexpr auto k00 = tf32x3_fused_kernel<false, false>;
  static constexpr auto k01 = tf32x3_fused_kernel<false, true>;
  static constexpr auto k10 = tf32x3_fused_kernel<true, false>;
  static constexpr auto k11 = tf32x3_fused_kernel<true, true>;
  static cudaError_t prepare() {
    for (auto k : {k00, k01, k10, k11}) {
      const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kFSmemBytes);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  static cudaError_t occupancy(int* ctas) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, k00, kFThreads, kFSmemBytes);
  }
  // a.tmA / a.tmB: maps over A and B as stored (see the split-TF32 fused
  // branch of the plan code): K-major sources with the 128-byte swizzle and
  // 32 x 128 boxes, MN-major ones unswizzled with 128 x 32 boxes
  static cudaError_t launch(const LaunchArgs& a, cudaStream_t stream) {
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
    const auto k = a.a_trans ? (a.b_trans ? k11 : k10) : (a.b_trans ? k01 : k00);
    k<<<a.grid, kFThreads, kFSmemBytes, stream>>>(a.tmA, a.tmB, p);
    return cudaGetLastError();
  }
  static Variant describe(const char* name) {
    return Variant{name, kKindTcFused, BM, kFBN, BK, kFRawStages, 0, kFThreads, kFSmemBytes, 128, &prepare, &occupancy,
                   &launch, 0, 0};
  }
};

const Variant kVariants[] = {
    TcVariant<256, 2>::describe("tf32x3_128x256x32_s2"),
    TcVariant<128, 3>::describe("tf32x3_128x128x32_s3"),
    TcVariant<128, 3, true>::describe("tf32x3p_128x128x32_s3"),
    TcVariant<256, 2, true>::describe("tf32x3p_128x256x32_s2"),
    TcFusedVariant::describe("tf32x3f_128x128x32_s3"),
};

}  // namespace tc

const Variant* tc_variants(int* count) {
  *count = static_cast<int>(sizeof(tc::kVariants) / sizeof(tc::kVariants[0]));
  return tc::kVariants;
}

}  // namespace sgemm
