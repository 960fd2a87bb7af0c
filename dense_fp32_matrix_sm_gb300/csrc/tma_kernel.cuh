// tma_kernel.cuh -- the main FP32 SGEMM kernel family for sm_103a (template;
// instantiated by the tma_variants_*.cu translation units).
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
//    mbarriers.  When a warp has read a stage it bumps that stage's release
//    counter; the warp whose bump completes the set issues the refill with
//    the slice STAGES ahead, so a stage is reloaded the moment the last
//    reader leaves it and no warp ever waits for another.  Each warp probes
//    the next stage's barrier (non-blocking) before its FMAs, so the answer
//    is back by the time it is needed.  Loads of later k-slices overlap the
//    math on the current one -- the pages' double buffering ("Writing a
//    Fast Matmul in CUDA", "Bank conflicts and double buffering")
//    generalised to a ring, with no register staging and no CTA barrier in
//    the main loop.  No warp is set aside for copies, so every warp
//    computes and the register budget is not split.  Out-of-range
//    rows/columns/k of edge tiles are zero-filled by the TMA unit, so the
//    main loop needs no predicates.
//  * Warps own WM x WN warp tiles; a warp's lanes form an 8 x 4 grid
//    (lane = 4g + c) and lane (g, c) owns a TM x TN thread tile, TM = WM/8,
//    TN = WN/4, at rows g + 8i and columns 4c + 16h + j (j < 4).  Per k step a
//    lane reads TM values of A and TN of B and does the TM*TN-FMA outer
//    product ("Learn: Optimizing GEMM", section 6, 2D register blocking;
//    "Writing a Fast Matmul in CUDA", Step 4).
//  * Shared-memory layout: TMA cannot transpose 4-byte elements, so A stays
//    k-contiguous ([BM][BK], BK*4-byte rows) under the TMA swizzle that
//    matches the row length (BK 32: 128-byte swizzle, chunk q of row r at
//    q ^ (r & 7); BK 16: 64-byte swizzle, chunk q of row r at
//    q ^ ((r >> 1) & 3)).  The rows one load instruction touches then sit in
//    different banks.  AMODE kQuad reads A four k at a time with 128-bit
//    loads into TM*4 registers; AMODE kScalar reads the TM values of one k
//    with 32-bit loads, using fewer registers so more warps fit on an SM.
//    B stays n-contiguous ([BK][BN]); each quarter-warp's 128-bit B load is
//    64 contiguous bytes.  Both meet the pages' conflict-free-read goal
//    ("Writing a Fast Matmul in CUDA", kernel 7) without a transpose.
//  * With FFMA2 the FMAs of a k step issue as paired fp32 FMAs (sm_100+
//    packed fp32), halving the issue slots the FMAs take -- the pages'
//    limit for an FP32 kernel is issue slots ("Writing a Fast Matmul in
//    CUDA", "Why 70% and not 100%").  Each half is an IEEE fp32 fma, so the
//    results are bit-identical to the scalar form.
//  * Epilogue: out = alpha*acc (beta == 0, C not read) or
//    fmaf(alpha, acc, beta*C), 128-bit stores where aligned, predicated at
//    the M/N edges.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"
#include "tile_order.cuh"

namespace sgemm {
namespace tma {

enum AMode : int { kQuad = 0, kScalar = 1 };

struct Params {
  float* C;
  int64_t ldc;
  int M, N, K;
  float alpha, beta;
  int vec_c;  // C 16-byte aligned and ldc % 4 == 0
  int group_m;
  unsigned int* status;
  uint64_t timeout_ns;
};

template <int BM, int BN, int BK, int WM, int WN, int STAGES>
struct Shape {
  static_assert(BK == 32 || BK == 16, "A rows must be one 128- or 64-byte swizzle span");
  static_assert(WM % 8 == 0 && WN % 16 == 0, "lane grid is 8 x 4, columns in 16-wide groups");
  static_assert(BM % WM == 0 && BN % WN == 0, "warp tiles cover the CTA tile");
  static constexpr int kTM = WM / 8;
  static constexpr int kTN = WN / 4;
  static constexpr int kTN4 = kTN / 4;  // float4 column groups per lane
  static constexpr int kWarpsM = BM / WM;
  static constexpr int kWarpsN = BN / WN;
  static constexpr int kWarps = kWarpsM * kWarpsN;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kStageA = BM * BK * 4;
  static constexpr int kStageB = BK * BN * 4;
  static constexpr int kStageBytes = kStageA + kStageB;
  static_assert(kStageA % 1024 == 0 && kStageB % 1024 == 0, "stages keep 1024-byte alignment");
  // per stage: one "full" mbarrier (8 bytes) and one release counter (4 bytes, padded to 8)
  static constexpr int kBarrierBytes = 2 * STAGES * 8;
  // 1024 bytes of slack to align the ring for the swizzle pattern
  static constexpr int kSmemBytes = STAGES * kStageBytes + kBarrierBytes + 1024;
};

// The TMA swizzle of a [BM][BK] A tile moves 16-byte chunk q of row r to
// chunk q ^ x(r), with x(r) = r & 7 for 128-byte rows (BK 32) and
// (r >> 1) & 3 for 64-byte rows (BK 16).  A lane's rows r0 + 8i all share
// x(r0), so the XOR is one per-lane constant.
template <int BK>
__device__ __forceinline__ int a_swizzle(int r0) {
  if constexpr (BK == 32) {
    return r0 & 7;
  } else {
    return (r0 >> 1) & 3;
  }
}

template <int BM, int BN, int BK, int WM, int WN, int STAGES, int AMODE, int MINB, bool FFMA2>
__global__ void __launch_bounds__(Shape<BM, BN, BK, WM, WN, STAGES>::kThreads, MINB)
    sgemm_tma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const Params p) {
  using S = Shape<BM, BN, BK, WM, WN, STAGES>;
  constexpr int TM = S::kTM;
  constexpr int TN4 = S::kTN4;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // Align the ring to 1024 bytes (the swizzle pattern's period) by offsetting
  // from the __shared__ array itself, so the compiler keeps every operand read
  // in the shared state space (an integer round trip would turn them into
  // generic loads).
  const uint32_t raw_base = ptx::smem_addr(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
  const uint32_t smem_base = ptx::smem_addr(smem);
  const uint32_t bar_full = smem_base + STAGES * S::kStageBytes;  // STAGES x 8 bytes
  // per-stage count of warps that have finished reading it (monotonic; the
  // warp whose increment completes a multiple of kWarps refills the stage)
  unsigned int* released = reinterpret_cast<unsigned int*>(smem + STAGES * S::kStageBytes + STAGES * 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int tiles_m = (p.M + BM - 1) / BM;
  const int tiles_n = (p.N + BN - 1) / BN;
  const int num_tiles = tiles_m * tiles_n;
  const int KT = (p.K + BK - 1) / BK;

  // this CTA's tiles are blockIdx.x, blockIdx.x + gridDim.x, ...; its k-slices
  // are numbered it = local_tile * KT + kt across all of them
  const int my_tiles = static_cast<int>(blockIdx.x) < num_tiles
                           ? (num_tiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                           : 0;
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
      released[s] = 0u;
    }

    ptx::fence_barrier_init();
    ptx::prefetch_tensormap(&tmA);
    ptx::prefetch_tensormap(&tmB);
    for (uint32_t j = 0; j < STAGES && j < total_it; ++j) issue(j);
  }
  __syncthreads();

  const int wm = warp / S::kWarpsN;
  const int wn = warp % S::kWarpsN;
  const int g = lane >> 2;  // row group: rows g + 8i of the warp tile
  const int c = lane & 3;   // column group: columns 4c + 16h + j
  const int row_base = wm * WM + g;
  const int a_swz = a_swizzle<BK>(row_base);

  uint32_t it = 0;
  bool ready = false;  // the stage of slice `it` is known to be full
  for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
    int tm, tn;
    tile_coords(tile, tiles_m, tiles_n, p.group_m, tm, tn);

    // acc[i][2h + e] holds columns 4c + 16h + 2e, +1 of row g + 8i
    float2 acc[TM][2 * TN4];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < 2 * TN4; ++j) acc[i][j] = make_float2(0.f, 0.f);

    for (int kt = 0; kt < KT; ++kt, ++it) {
      const uint32_t s = it % STAGES;
      const uint32_t phase = (it / STAGES) & 1u;
      if (!ready && !ptx::mbar_wait(bar_full + 8 * s, phase, p.timeout_ns)) {
        atomicOr(p.status, kStatusTimeoutFull);
        // copies still in flight land before this thread leaves; a copy issued
        // later is waited on by the thread that issued it or by its consumers
        ptx::drain_ring_released(bar_full, 8, released, S::kWarps, STAGES, total_it, p.timeout_ns);
        return;
      }
      // Probe the next slice's stage now; the answer arrives while this
      // slice's FMAs run, so a ready stage costs no wait at the next step.
      if (it + 1 < total_it) {
        ready = ptx::mbar_test_wait(bar_full + 8 * ((it + 1) % STAGES), ((it + 1) / STAGES) & 1u);
      }
      const float* As = reinterpret_cast<const float*>(smem + s * S::kStageBytes) + row_base * BK;
      const float4* Bs4 = reinterpret_cast<const float4*>(smem + s * S::kStageBytes + S::kStageA) +
                          (wn * WN + c * 4) / 4;

      auto fma_step = [&](const float (&a)[TM], const float4 (&b)[TN4]) {
#pragma unroll
        for (int i = 0; i < TM; ++i) {
#pragma unroll
          for (int h = 0; h < TN4; ++h) {
            if constexpr (FFMA2) {
              const float2 aa = make_float2(a[i], a[i]);
              acc[i][2 * h] = __ffma2_rn(aa, make_float2(b[h].x, b[h].y), acc[i][2 * h]);
              acc[i][2 * h + 1] = __ffma2_rn(aa, make_float2(b[h].z, b[h].w), acc[i][2 * h + 1]);
            } else {
              acc[i][2 * h].x = fmaf(a[i], b[h].x, acc[i][2 * h].x);
              acc[i][2 * h].y = fmaf(a[i], b[h].y, acc[i][2 * h].y);
              acc[i][2 * h + 1].x = fmaf(a[i], b[h].z, acc[i][2 * h + 1].x);
              acc[i][2 * h + 1].y = fmaf(a[i], b[h].w, acc[i][2 * h + 1].y);
            }
          }
        }
      };

      if constexpr (AMODE == kQuad) {
#pragma unroll
        for (int q = 0; q < BK / 4; ++q) {
          float4 a4[TM];
#pragma unroll
          for (int i = 0; i < TM; ++i)
            a4[i] = *reinterpret_cast<const float4*>(As + 8 * BK * i + ((q ^ a_swz) << 2));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            float a[TM];
            float4 b[TN4];
#pragma unroll
            for (int i = 0; i < TM; ++i)
              a[i] = kk == 0 ? a4[i].x : kk == 1 ? a4[i].y : kk == 2 ? a4[i].z : a4[i].w;
#pragma unroll
            for (int h = 0; h < TN4; ++h) b[h] = Bs4[(4 * q + kk) * (BN / 4) + 4 * h];
            fma_step(a, b);
          }
        }
      } else {
#pragma unroll 2
        for (int q = 0; q < BK / 4; ++q) {
          const float* Aq = As + ((q ^ a_swz) << 2);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            float a[TM];
            float4 b[TN4];
#pragma unroll
            for (int i = 0; i < TM; ++i) a[i] = Aq[8 * BK * i + kk];
#pragma unroll
            for (int h = 0; h < TN4; ++h) b[h] = Bs4[(4 * q + kk) * (BN / 4) + 4 * h];
            fma_step(a, b);
          }
        }
      }
      // Release the stage.  The warp whose release completes the set refills
      // it at once with the slice STAGES ahead (no warp waits for another).
      __syncwarp();
      if (lane == 0) {
        const unsigned int before = ptx::atom_add_acq_rel_cta(&released[s], 1u);
        if ((before + 1u) % S::kWarps == 0u && it + STAGES < total_it) {
          ptx::fence_proxy_async_smem();
          issue(it + STAGES);
        }
      }
    }

    // ---------------- epilogue ----------------
    const int row0 = tm * BM + row_base;
    const int col0 = tn * BN + wn * WN + c * 4;
#pragma unroll
    for (int i = 0; i < TM; ++i) {
      const int row = row0 + 8 * i;
      if (row >= p.M) break;
      float* crow = p.C + static_cast<int64_t>(row) * p.ldc;
#pragma unroll
      for (int h = 0; h < TN4; ++h) {
        const int col = col0 + 16 * h;
        const float v[4] = {acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x, acc[i][2 * h + 1].y};
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

template <int BM, int BN, int BK, int WM, int WN, int STAGES, int AMODE, int MINB, bool FFMA2>
struct Variant_ {
  using S = Shape<BM, BN, BK, WM, WN, STAGES>;
  static constexpr auto kernel = sgemm_tma_kernel<BM, BN, BK, WM, WN, STAGES, AMODE, MINB, FFMA2>;
  static cudaError_t prepare() {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
  }
  static cudaError_t occupancy(int* ctas) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, kernel, S::kThreads, S::kSmemBytes);
  }
  static cudaError_t launch(const LaunchArgs& a, cudaStream_t stream) {
    Params p;
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
    kernel<<<a.grid, S::kThreads, S::kSmemBytes, stream>>>(a.tmA, a.tmB, p);
    return cudaGetLastError();
  }
  static Variant describe(const char* name) {
    return Variant{name,           kKindTma,       BM, BN, BK, STAGES, FFMA2 ? 1 : 0, S::kThreads, S::kSmemBytes,
                   BK == 32 ? 128 : 64, &prepare, &occupancy, &launch};
  }
};

}  // namespace tma
}  // namespace sgemm
