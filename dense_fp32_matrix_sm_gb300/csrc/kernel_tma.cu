// kernel_tma.cu -- the main FP32 SGEMM kernel family for sm_103a.
//
// C = alpha*A*B + beta*C, row-major float32, computed with single-rounding
// fp32 FMAs on the CUDA cores in ascending k for every output.
//
// Structure (each level is a tile of the one above it -- "Learn: Optimizing
// GEMM", section 8 and the warp-tiling rung; "How a Matmul Kernel Gets Fast",
// section 13 "Kernel 10: warptiling"):
//
//  * Persistent CTAs walk the BM x BN output tiles in a grouped (L2-aware)
//    order: consecutive tile ids cover GROUP_M tile-rows before moving right,
//    so CTAs running at the same time share A and B tiles in L2 ("Writing a
//    Fast Matmul in CUDA, Step by Step", "What cuBLAS and CUTLASS add":
//    threadblock rasterization).
//  * A STAGES-deep shared-memory ring is filled by TMA bulk tensor copies
//    (A tile BM x BK, B tile BK x BN) signalled on per-stage "full"
//    mbarriers; each warp releases a stage on its "empty" mbarrier when it
//    has read it.  Thread 0 issues every copy: after its own warp finishes
//    slice `it` it refills the stage released at slice it-1 (all warps are
//    normally past it by then) with slice it-1+STAGES.  So loads of later
//    k-slices overlap the math on the current one -- the pages' double
//    buffering ("Writing a Fast Matmul in CUDA", "Bank conflicts and double
//    buffering") generalised to a ring, with no register staging and no CTA
//    barrier in the main loop.  No warp is set aside for copies: with 8
//    warps per CTA each thread may hold up to 255 registers (a ninth warp
//    would put three warps on one SM sub-partition and cap them at 168).
//    Out-of-range rows/columns/k of edge tiles are zero-filled by the TMA
//    unit, so the main loop needs no predicates.
//  * Eight warps, each owning a 64 x 32 warp tile; each lane owns an
//    8 x 8 thread tile (rows g + 8i, columns 4c + j and 16 + 4c + j, lane =
//    4g + c).  Per k step a lane reads 8 values of A and 8 of B and does the
//    64-FMA outer product ("Learn: Optimizing GEMM", section 6, 2D register
//    blocking; "Writing a Fast Matmul in CUDA", Step 4).
//  * Shared-memory layout: TMA cannot transpose 4-byte elements, so A stays
//    k-contiguous ([BM][BK], 128-byte rows) and is read four k at a time
//    with 128-bit loads; the TMA 128-byte swizzle (16-byte chunk q of row r
//    stored at chunk q ^ (r & 7)) puts the rows a half-warp reads in
//    different banks.  B stays n-contiguous ([BK][BN]); a half-warp reads
//    64 contiguous bytes.  Both are the pages' conflict-free-read goal
//    ("Writing a Fast Matmul in CUDA", kernel 7) met without the transpose.
//  * With FFMA2 the 64 FMAs of a k step issue as 32 paired fp32 FMAs
//    (sm_100+ packed fp32), halving the issue slots the FMAs take -- the
//    pages' limit for an FP32 kernel is issue slots ("Writing a Fast Matmul
//    in CUDA", "Why 70% and not 100%").  Each half is an IEEE fp32 fma, so
//    the results are bit-identical to the scalar form.
//  * Epilogue: out = alpha*acc (beta == 0, C not read) or
//    fmaf(alpha, acc, beta*C), 128-bit stores where aligned, predicated at
//    the M/N edges.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"

namespace sgemm {
namespace {

struct TmaParams {
  float* C;
  int64_t ldc;
  int M, N, K;
  float alpha, beta;
  int vec_c;  // C 16-byte aligned and ldc % 4 == 0
  int group_m;
  unsigned int* status;
  uint64_t timeout_ns;
};

template <int BM, int BN, int BK, int STAGES, bool FFMA2>
struct TmaShape {
  static_assert(BK == 32, "A tile rows are exactly one 128-byte swizzle span");
  static_assert(BM % 64 == 0 && BN % 32 == 0, "warp tile is 64 x 32");
  static constexpr int kWarpsM = BM / 64;
  static constexpr int kWarpsN = BN / 32;
  static constexpr int kConsumerWarps = kWarpsM * kWarpsN;
  static constexpr int kThreads = kConsumerWarps * 32;
  static constexpr int kStageA = BM * BK * 4;
  static constexpr int kStageB = BK * BN * 4;
  static constexpr int kStageBytes = kStageA + kStageB;
  static_assert(kStageA % 1024 == 0 && kStageB % 1024 == 0, "stages keep 1024-byte alignment");
  static constexpr int kBarrierBytes = 2 * STAGES * 8;
  // 1024 bytes of slack to align the ring for the 128-byte swizzle
  static constexpr int kSmemBytes = STAGES * kStageBytes + kBarrierBytes + 1024;
};

__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int group_m, int& tm,
                                            int& tn) {
  const int per_group = group_m * tiles_n;
  const int group = tile / per_group;
  const int first_m = group * group_m;
  const int rows = min(tiles_m - first_m, group_m);
  const int in_group = tile - group * per_group;
  tm = first_m + in_group % rows;
  tn = in_group / rows;
}

template <int BM, int BN, int BK, int STAGES, bool FFMA2>
__global__ void __launch_bounds__(TmaShape<BM, BN, BK, STAGES, FFMA2>::kThreads, 1)
    sgemm_tma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const TmaParams p) {
  using S = TmaShape<BM, BN, BK, STAGES, FFMA2>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t smem_base = ptx::smem_addr(smem);
  const uint32_t bar_full = smem_base + STAGES * S::kStageBytes;  // STAGES x 8 bytes
  const uint32_t bar_empty = bar_full + STAGES * 8;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int tiles_m = (p.M + BM - 1) / BM;
  const int tiles_n = (p.N + BN - 1) / BN;
  const int num_tiles = tiles_m * tiles_n;
  const int KT = (p.K + BK - 1) / BK;

  // this CTA's tiles are blockIdx.x, blockIdx.x + gridDim.x, ...; its k-slices
  // are numbered it = local_tile * KT + kt across all of them
  const int my_tiles = blockIdx.x < num_tiles ? (num_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const uint32_t total_it = static_cast<uint32_t>(my_tiles) * static_cast<uint32_t>(KT);

  // Issue the TMA copies of k-slice `j` into its ring stage (thread 0 only).
  auto issue = [&](uint32_t j) {
    const uint32_t s = j % STAGES;
    const int lt = static_cast<int>(j / KT);
    const int kt = static_cast<int>(j % KT);
    int tm, tn;
    tile_coords(blockIdx.x + lt * gridDim.x, tiles_m, tiles_n, p.group_m, tm, tn);
    const uint32_t dst = smem_base + s * S::kStageBytes;
    ptx::mbar_arrive_expect_tx(bar_full + 8 * s, S::kStageBytes);
    ptx::tma_load_2d(dst, &tmA, kt * BK, tm * BM, bar_full + 8 * s);
    ptx::tma_load_2d(dst + S::kStageA, &tmB, tn * BN, kt * BK, bar_full + 8 * s);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(bar_full + 8 * s, 1);
      ptx::mbar_init(bar_empty + 8 * s, S::kConsumerWarps);
    }
    ptx::fence_barrier_init();
    ptx::prefetch_tensormap(&tmA);
    ptx::prefetch_tensormap(&tmB);
    for (uint32_t j = 0; j < STAGES && j < total_it; ++j) issue(j);
  }
  __syncthreads();

  // ---------------- consumers ----------------
  const int wm = warp / S::kWarpsN;
  const int wn = warp % S::kWarpsN;
  const int g = lane >> 2;  // row group: rows g + 8i of the warp tile
  const int c = lane & 3;   // column group: columns 4c + j and 16 + 4c + j

  uint32_t it = 0;
  for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
    int tm, tn;
    tile_coords(tile, tiles_m, tiles_n, p.group_m, tm, tn);

    float2 acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.f, 0.f);

    for (int kt = 0; kt < KT; ++kt, ++it) {
      const uint32_t s = it % STAGES;
      const uint32_t phase = (it / STAGES) & 1u;
      if (!ptx::mbar_wait(bar_full + 8 * s, phase, p.timeout_ns)) {
        atomicOr(p.status, kStatusTimeoutFull);
        return;
      }
      const unsigned char* stage = smem + s * S::kStageBytes;
      // A rows of this lane: (wm*64 + g + 8i), 128 bytes each, swizzled chunks.
      const float4* As4 = reinterpret_cast<const float4*>(stage) + (wm * 64 + g) * (BK / 4);
      const float4* Bs4 = reinterpret_cast<const float4*>(stage + S::kStageA) + (wn * 32 + c * 4) / 4;

#pragma unroll
      for (int q = 0; q < BK / 4; ++q) {
        float4 a[8];
        const int chunk = q ^ g;
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = As4[i * 8 * (BK / 4) + chunk];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int k = q * 4 + kk;
          const float4 b0 = Bs4[k * (BN / 4)];
          const float4 b1 = Bs4[k * (BN / 4) + 4];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float ai = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
            if constexpr (FFMA2) {
              const float2 aa = make_float2(ai, ai);
              acc[i][0] = __ffma2_rn(aa, make_float2(b0.x, b0.y), acc[i][0]);
              acc[i][1] = __ffma2_rn(aa, make_float2(b0.z, b0.w), acc[i][1]);
              acc[i][2] = __ffma2_rn(aa, make_float2(b1.x, b1.y), acc[i][2]);
              acc[i][3] = __ffma2_rn(aa, make_float2(b1.z, b1.w), acc[i][3]);
            } else {
              acc[i][0].x = fmaf(ai, b0.x, acc[i][0].x);
              acc[i][0].y = fmaf(ai, b0.y, acc[i][0].y);
              acc[i][1].x = fmaf(ai, b0.z, acc[i][1].x);
              acc[i][1].y = fmaf(ai, b0.w, acc[i][1].y);
              acc[i][2].x = fmaf(ai, b1.x, acc[i][2].x);
              acc[i][2].y = fmaf(ai, b1.y, acc[i][2].y);
              acc[i][3].x = fmaf(ai, b1.z, acc[i][3].x);
              acc[i][3].y = fmaf(ai, b1.w, acc[i][3].y);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_empty + 8 * s);
      // Thread 0 refills the stage released one slice ago (by now every warp
      // is normally past it) with the slice STAGES ahead of that one.
      if (threadIdx.x == 0 && it >= 1 && it - 1 + STAGES < total_it) {
        const uint32_t r = it - 1;
        if (!ptx::mbar_wait(bar_empty + 8 * (r % STAGES), (r / STAGES) & 1u, p.timeout_ns)) {
          atomicOr(p.status, kStatusTimeoutEmpty);
          return;
        }
        issue(r + STAGES);
      }
    }

    // ---------------- epilogue ----------------
    const int row0 = tm * BM + wm * 64 + g;
    const int col0 = tn * BN + wn * 32 + c * 4;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = row0 + 8 * i;
      if (row >= p.M) break;
      float* crow = p.C + static_cast<int64_t>(row) * p.ldc;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int col = col0 + 16 * h;
        float v[4] = {acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x, acc[i][2 * h + 1].y};
        if (p.vec_c && col + 3 < p.N) {
          float4* dst = reinterpret_cast<float4*>(crow + col);
          float4 o;
          if (p.beta == 0.f) {
            o = make_float4(p.alpha * v[0], p.alpha * v[1], p.alpha * v[2], p.alpha * v[3]);
          } else {
            const float4 old = *dst;
            o = make_float4(fmaf(p.alpha, v[0], p.beta * old.x), fmaf(p.alpha, v[1], p.beta * old.y),
                            fmaf(p.alpha, v[2], p.beta * old.z), fmaf(p.alpha, v[3], p.beta * old.w));
          }
          *dst = o;
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (col + j < p.N) {
              float* d = crow + col + j;
              *d = p.beta == 0.f ? p.alpha * v[j] : fmaf(p.alpha, v[j], p.beta * *d);
            }
          }
        }
      }
    }
  }
}

template <int BM, int BN, int BK, int STAGES, bool FFMA2>
struct TmaVariant {
  using S = TmaShape<BM, BN, BK, STAGES, FFMA2>;
  static cudaError_t prepare() {
    return cudaFuncSetAttribute(sgemm_tma_kernel<BM, BN, BK, STAGES, FFMA2>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
  }
  static cudaError_t occupancy(int* ctas) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, sgemm_tma_kernel<BM, BN, BK, STAGES, FFMA2>,
                                                         S::kThreads, S::kSmemBytes);
  }
  static cudaError_t launch(const LaunchArgs& a, cudaStream_t stream) {
    TmaParams p;
    p.C = a.C;
    p.ldc = a.ldc;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.alpha = a.alpha;
    p.beta = a.beta;
    p.vec_c = ((reinterpret_cast<uintptr_t>(a.C) & 15) == 0) && (a.ldc % 4 == 0);
    p.group_m = 8;
    p.status = a.status;
    p.timeout_ns = a.timeout_ns;
    sgemm_tma_kernel<BM, BN, BK, STAGES, FFMA2><<<a.grid, S::kThreads, S::kSmemBytes, stream>>>(a.tmA, a.tmB, p);
    return cudaGetLastError();
  }
  static Variant describe(const char* name) {
    return Variant{name, kKindTma, BM, BN, BK, STAGES, FFMA2 ? 1 : 0, S::kThreads, S::kSmemBytes, 128,
                   &prepare, &occupancy, &launch};
  }
};

const Variant kTmaVariants[] = {
    TmaVariant<128, 128, 32, 4, true>::describe("tma_128x128x32_s4_ffma2"),
    TmaVariant<128, 128, 32, 4, false>::describe("tma_128x128x32_s4_ffma"),
    TmaVariant<128, 128, 32, 6, true>::describe("tma_128x128x32_s6_ffma2"),
    TmaVariant<128, 64, 32, 4, true>::describe("tma_128x64x32_s4_ffma2"),
};

}  // namespace

const Variant* tma_variants(int* count) {
  *count = static_cast<int>(sizeof(kTmaVariants) / sizeof(kTmaVariants[0]));
  return kTmaVariants;
}

}  // namespace sgemm
