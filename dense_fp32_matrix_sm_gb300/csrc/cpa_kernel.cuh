// cpa_kernel.cuh -- the FP32 SGEMM kernel family with A staged transposed
// (template; instantiated by cpa_variants_*.cu).
//
// C = alpha*A*B + beta*C, row-major float32, single-rounding fp32 FMAs in
// ascending k for every output (bit-identical to the float32 fma chain).
//
// What differs from tma_kernel.cuh is the operand form of the inner loop.
// Each paired-FP32 FMA (FFMA2) takes one register PAIR and one BROADCAST
// scalar.  Measured on GB300 with identical data in registers, the paired
// FMAs keep the FP32 pipe ~87% busy when the pair holds two rows of A
// (m, m+1) and the broadcast is one element of B, against ~81% the other
// way round.  Two rows of A at one k are adjacent only in a transposed
// tile, and TMA cannot transpose 4-byte elements, so:
//
//  * A is copied into shared memory transposed, At[k][m], by 4-byte
//    cp.async copies issued by every thread ("Learn: Optimizing GEMM",
//    section 7 and "Writing a Fast Matmul in CUDA", Step 5: A stored
//    transposed as it is loaded, so the inner loop reads contiguous m).
//    The 32 lanes of one copy instruction cover a KW (k) x 32/KW (m)
//    patch, and the XOR swizzle m ^ (32/KW)*(k mod KW) puts the 32
//    shared-memory writes in 32 banks while keeping pairs (m, m+1)
//    adjacent.  Small KW writes few At rows per instruction (cheaper
//    shared writes), large KW reads whole 32-byte sectors of A.  Each thread's copies complete on the
//    stage's "full" mbarrier (cp.async.mbarrier.arrive.noinc), so no
//    wait_group or CTA barrier is needed for them.  Out-of-range rows or k
//    are zero-filled (source size 0), so A needs no alignment at all.
//  * B is copied by TMA ([BK][BN], n contiguous) onto the same barrier.
//  * A stage is refilled once every warp has released it (a per-stage
//    "empty" mbarrier).  All threads refill the stage released one slice
//    earlier, at the top of each slice, then wait for the current one.
//  * Warps own 64 x 32 warp tiles; lane (g, c) (lane = 4g + c) owns rows
//    16i + 2g + e (i < 4, e < 2) and columns 4c + 16h + j (h < 2, j < 4):
//    per k it loads four A pairs (64-bit, from At) and eight B values
//    (two 128-bit loads) and issues 32 FFMA2 (pair of A rows x one B
//    element).  Lanes of one quad share their A addresses, so an A pair
//    load is one shared-memory wavefront.
//  * Persistent CTAs over tiles in grouped order (GROUP_M = 8), bounded
//    waits with a status word, epilogue out = alpha*acc (beta == 0, C not
//    read) or fmaf(alpha, acc, beta*C) with 128-bit stores where aligned.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"
#include "tile_order.cuh"

namespace sgemm {
namespace cpa {

struct Params {
  const float* A;
  int64_t lda;
  float* C;
  int64_t ldc;
  int M, N, K;
  float alpha, beta;
  int vec_c;
  int group_m;
  unsigned int* status;
  uint64_t timeout_ns;
};

__device__ __forceinline__ void cp_async_4(uint32_t dst, const float* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(valid ? 4 : 0) : "memory");
}

__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// KW: k-width of one copy instruction's patch (KW k x 32/KW m).
template <int BM, int BN, int STAGES, int KW>
struct Shape {
  static constexpr int BK = 32;
  static_assert(KW == 2 || KW == 4 || KW == 8, "copy patch is KW (k) x 32/KW (m)");
  static constexpr int MW = 32 / KW;
  static constexpr int kWarpsM = BM / 64;
  static constexpr int kWarpsN = BN / 32;
  static constexpr int kWarps = kWarpsM * kWarpsN;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kStageA = BK * BM * 4;
  static constexpr int kStageB = BK * BN * 4;
  static constexpr int kStageBytes = kStageA + kStageB;
  static_assert(BM % 64 == 0 && BN % 32 == 0, "warp tile is 64 x 32");
  static_assert(kStageA % 1024 == 0 && kStageB % 1024 == 0, "stages keep 1024-byte alignment");
  // A copy patches: KW k x MW m per warp instruction
  static constexpr int kPatches = (BK / KW) * (BM / MW);
  static_assert(kPatches % kWarps == 0, "patches split evenly over warps");
  static constexpr int kCopiesPerThread = kPatches / kWarps;
  static constexpr int kSmemBytes = STAGES * kStageBytes + STAGES * 16 + 1024;
};

template <int BM, int BN, int STAGES, int KW, int MINB>
__global__ void __launch_bounds__(Shape<BM, BN, STAGES, KW>::kThreads, MINB)
    sgemm_cpa_kernel(const __grid_constant__ CUtensorMap tmB, const Params p) {
  using S = Shape<BM, BN, STAGES, KW>;
  constexpr int MW = S::MW;
  constexpr int BK = S::BK;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_base = ptx::smem_addr(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
  const uint32_t smem_base = ptx::smem_addr(smem);
  const uint32_t bar_full = smem_base + STAGES * S::kStageBytes;
  const uint32_t bar_empty = bar_full + STAGES * 8;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_m = (p.M + BM - 1) / BM;
  const int tiles_n = (p.N + BN - 1) / BN;
  const int num_tiles = tiles_m * tiles_n;
  const int KT = (p.K + BK - 1) / BK;
  const int my_tiles = static_cast<int>(blockIdx.x) < num_tiles
                           ? (num_tiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                           : 0;
  const uint32_t total_it = static_cast<uint32_t>(my_tiles) * static_cast<uint32_t>(KT);

  // This thread's A copies: lane -> (k_off = lane % KW, m_off = lane / KW).
  // Copy r (r < kCopiesPerThread) of warp w covers patch P = w*kCopies + r
  // with m-block mb = P / (BK/KW) and k-block kb = P % (BK/KW); since
  // kCopies is a multiple of BK/KW, the thread touches kRows =
  // kCopies/(BK/KW) rows, row t = MW*(w*kRows + t) + m_off, each at
  // k = KW*kb + k_off.  Element (k, m) is stored at At[k][m ^ MW*(k % KW)]:
  // the 32 lanes of a patch land in 32 banks, pairs (m, m+1) stay adjacent.
  constexpr int kKB = BK / KW;
  constexpr int kRows = S::kCopiesPerThread / kKB;
  static_assert(S::kCopiesPerThread % kKB == 0, "each copied row spans the whole k-slice");
  const int k_off = lane % KW;
  const int m_off = lane / KW;
  // shared-memory offset (bytes, within a stage) of copy (t, kb = 0)
  uint32_t a_dst[kRows];
#pragma unroll
  for (int t = 0; t < kRows; ++t) {
    const int m = MW * (warp * kRows + t) + m_off;
    a_dst[t] = static_cast<uint32_t>((k_off * BM + (m ^ (MW * k_off))) * 4);
  }

  // Producer state for the next slice to issue (slices are issued in order).
  struct Cursor {
    int lt, kt, tm, tn;
  } cur{0, 0, 0, 0};
  const float* a_row[kRows];  // this thread's rows of the current tile (k_off folded in)
  bool row_ok[kRows];
  auto load_tile_rows = [&]() {
    tile_coords(blockIdx.x + cur.lt * gridDim.x, tiles_m, tiles_n, p.group_m, cur.tm, cur.tn);
#pragma unroll
    for (int t = 0; t < kRows; ++t) {
      const int m = cur.tm * BM + MW * (warp * kRows + t) + m_off;
      row_ok[t] = m < p.M;
      a_row[t] = p.A + static_cast<int64_t>(row_ok[t] ? m : 0) * p.lda + k_off;
    }
  };

  uint32_t issued = 0;  // slices this thread has issued
  auto issue = [&](uint32_t j) {
    issued = j + 1;
    const uint32_t s = j % STAGES;
    const uint32_t a_stage = smem_base + s * S::kStageBytes;
    const int k0 = cur.kt * BK;
    if (k0 + BK <= p.K) {  // interior slice: only rows can fall outside
#pragma unroll
      for (int t = 0; t < kRows; ++t)
#pragma unroll
        for (int kb = 0; kb < kKB; ++kb)
          cp_async_4(a_stage + a_dst[t] + kb * KW * BM * 4, a_row[t] + k0 + KW * kb, row_ok[t]);
    } else {
#pragma unroll
      for (int t = 0; t < kRows; ++t)
#pragma unroll
        for (int kb = 0; kb < kKB; ++kb) {
          const bool ok = row_ok[t] && (k0 + KW * kb + k_off < p.K);
          cp_async_4(a_stage + a_dst[t] + kb * KW * BM * 4, ok ? a_row[t] + k0 + KW * kb : p.A, ok);
        }
    }
    cp_async_arrive_noinc(bar_full + 8 * s);
    if (threadIdx.x == 0) {
      ptx::mbar_arrive_expect_tx(bar_full + 8 * s, S::kStageB);
      ptx::tma_load_2d(a_stage + S::kStageA, &tmB, cur.tn * BN, k0, bar_full + 8 * s);
    }
    if (++cur.kt == KT) {  // advance to the next tile of this CTA
      cur.kt = 0;
      ++cur.lt;
      if (j + 1 < total_it) load_tile_rows();
    }
  };
  if (total_it > 0) load_tile_rows();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // one arrival per thread (its cp.async copies) plus thread 0's expect_tx
      ptx::mbar_init(bar_full + 8 * s, S::kThreads + 1);
      ptx::mbar_init(bar_empty + 8 * s, S::kWarps);
    }
    ptx::fence_barrier_init();
    ptx::prefetch_tensormap(&tmB);
  }
  __syncthreads();
  // prologue: the first STAGES slices
  for (uint32_t j = 0; j < STAGES && j < total_it; ++j) issue(j);

  const int wm = warp / S::kWarpsN;
  const int wn = warp % S::kWarpsN;
  const int g = lane >> 2;
  const int c = lane & 3;
  // A pair i of this lane starts at m = wm*64 + 16i + 2g, stored at
  // m ^ f(k), f(k) = MW*(k % KW) < 32:  (16i + 2g) ^ f = 16*(i ^ (f >> 4)) + (2g ^ (f & 15)).
  int a_off[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) a_off[t] = wm * 64 + ((2 * g) ^ (4 * t));  // f & 15 is a multiple of 4

  uint32_t it = 0;
  bool failed = false;
  for (int tile = blockIdx.x; tile < num_tiles && !failed; tile += gridDim.x) {
    int tm, tn;
    tile_coords(tile, tiles_m, tiles_n, p.group_m, tm, tn);

    // acc[i][j] = {C[row 16i+2g][col j], C[row 16i+2g+1][col j]}, col j = 4c + 16(j/4) + j%4
    float2 acc[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = make_float2(0.f, 0.f);

    for (int kt = 0; kt < KT; ++kt, ++it) {
      // refill the stage released at slice it-1 with slice it-1+STAGES
      if (it >= 1 && it - 1 + STAGES < total_it) {
        const uint32_t r = it - 1;
        if (!ptx::mbar_wait(bar_empty + 8 * (r % STAGES), (r / STAGES) & 1u, p.timeout_ns)) {
          atomicOr(p.status, kStatusTimeoutEmpty);
          failed = true;
          break;
        }
        issue(r + STAGES);
      }
      const uint32_t s = it % STAGES;
      if (!ptx::mbar_wait(bar_full + 8 * s, (it / STAGES) & 1u, p.timeout_ns)) {
        atomicOr(p.status, kStatusTimeoutFull);
        failed = true;
        break;
      }
      const float* At = reinterpret_cast<const float*>(smem + s * S::kStageBytes);
      const float4* Bs4 = reinterpret_cast<const float4*>(smem + s * S::kStageBytes + S::kStageA) + (wn * 32 + 4 * c) / 4;
#pragma unroll
      for (int k = 0; k < BK; ++k) {
        const float* Ak = At + k * BM;
        float2 ap[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int f = MW * (k % KW);
          ap[i] = *reinterpret_cast<const float2*>(Ak + a_off[(f & 15) >> 2] + 16 * (i ^ (f >> 4)));
        }
        const float4 b0 = Bs4[k * (BN / 4)];
        const float4 b1 = Bs4[k * (BN / 4) + 4];
        const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = __ffma2_rn(ap[i], make_float2(bb[j], bb[j]), acc[i][j]);
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_empty + 8 * s);
    }
    if (failed) break;

    // ---------------- epilogue ----------------
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int row = tm * BM + wm * 64 + 16 * i + 2 * g + e;
        if (row >= p.M) continue;
        float* crow = p.C + static_cast<int64_t>(row) * p.ldc;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int col = tn * BN + wn * 32 + 4 * c + 16 * h;
          float v[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) v[q] = e ? acc[i][4 * h + q].y : acc[i][4 * h + q].x;
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
            for (int q = 0; q < 4; ++q) {
              if (col + q < p.N) {
                float* d = crow + col + q;
                *d = p.beta == 0.f ? p.alpha * v[q] : fmaf(p.alpha, v[q], p.beta * *d);
              }
            }
          }
        }
      }
    }
  }
  // After a failed wait: this thread's cp.async copies, and thread 0's TMA
  // copies (bounded), land before the CTA's shared memory is released.
  if (failed) {
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (threadIdx.x == 0) ptx::drain_ring(bar_full, 8, issued, STAGES, p.timeout_ns);
  }
}

template <int BM, int BN, int STAGES, int KW, int MINB>
struct Variant_ {
  using S = Shape<BM, BN, STAGES, KW>;
  static constexpr auto kernel = sgemm_cpa_kernel<BM, BN, STAGES, KW, MINB>;
  static cudaError_t prepare() {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
  }
  static cudaError_t occupancy(int* ctas) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, kernel, S::kThreads, S::kSmemBytes);
  }
  static cudaError_t launch(const LaunchArgs& a, cudaStream_t stream) {
    Params p;
    p.A = a.A;
    p.lda = a.lda;
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
    kernel<<<a.grid, S::kThreads, S::kSmemBytes, stream>>>(a.tmB, p);
    return cudaGetLastError();
  }
  static Variant describe(const char* name) {
    return Variant{name, kKindCpa, BM, BN, S::BK, STAGES, 1, S::kThreads, S::kSmemBytes, 0,
                   &prepare, &occupancy, &launch};
  }
};

}  // namespace cpa
}  // namespace sgemm
