// tmat_kernel.cuh -- FP32 SGEMM with both operands fed by TMA and A
// transposed inside shared memory (template; instantiated by
// tmat_variants.cu).
//
// C = alpha*A*B + beta*C, row-major float32, single-rounding fp32 FMAs in
// ascending k for every output of a data-parallel tile (bit-identical to
// the float32 fma chain); tiles of a stream-K tail add fixed-order partial
// sums instead (see below).
//
// The inner loop is the fast paired-FMA form: each FFMA2 multiplies a
// register PAIR holding two rows of A at one k, (A[m][k], A[m+1][k]), by
// one BROADCAST element of B; on GB300 this keeps the FP32 pipe ~87% busy
// against ~81% for the mirrored form (pair of B columns, broadcast A).  It
// needs A k-major in shared memory (At[k][m]).  TMA cannot transpose
// 4-byte elements, so:
//
//  * TMA copies the A slice [BM][BK] (128-byte swizzle) and the B slice
//    [BK][BN] into a STAGES-deep ring signalled by mbarriers, as in
//    tma_kernel.cuh.
//  * While the math runs on slice j, all threads transpose the A slice j+1
//    into a double-buffered At[BK][BM]: with T = threads/BM (1, 2 or 4)
//    threads per row, thread t reads row t/T, k-part t%T (BK/T k, 128-bit
//    loads) and writes At[k][m ^ (32/T)*(k / (BK/T))].  The XOR puts the T
//    k-parts of a warp's 32/T rows in different bank groups (conflict-free
//    writes) and keeps pairs (m, m+1) adjacent.  The copy sits at a fixed
//    step of the unrolled k loop (TA), or in two halves (TA, TB), so its
//    wait and its load-to-store latency hide behind FFMA2s; placed before
//    the loop instead it cost 3.5% at 4096^3 (measured on GB300).
//  * A given transposed (AT: stored K x M) needs no transpose: TMA copies
//    [BK][BM] boxes, which the k loop reads from the ring stage directly.
//    ("Learn: Optimizing GEMM", section 7, and "Writing a Fast Matmul in
//    CUDA", Step 5: A stored transposed so the inner loop reads contiguous
//    m -- here the transpose runs on the on-chip copy instead of on the
//    global loads.)
//  * One plain CTA barrier per slice: after it the next transposed slice is
//    complete and the current ring stage is free; thread 0 then refills
//    that stage with the slice STAGES ahead.  A wait that runs out sets a
//    shared flag before the barrier, so every thread leaves together.
//  * Or (SPLIT) the barrier's two jobs go to two pairs of mbarriers, so
//    warps may drift apart by most of a slice: "slice j+1 transposed"
//    (arrived after the copy, waited before slice j+1) and "slice j done"
//    (arrived after the k loop, waited before the copy in slice j+1, which
//    overwrites At[j & 1]; thread 0 then refills slice j's stage).  Waits
//    stop early once any thread has failed, and the threads agree on
//    failure with one CTA barrier per segment.
//  * Warps own 64 x 32 tiles; lane (g, c) owns rows 16i + 2g + e and
//    columns 4c + 16h + j; per k: four 64-bit A-pair loads, two 128-bit B
//    loads, 32 FFMA2.
//  * Persistent CTAs in grouped tile order, bounded waits with a status
//    word, epilogue out = alpha*acc (beta == 0, C not read) or
//    fmaf(alpha, acc, beta*C).
//  * Stream-K tail (when the tile count is not a multiple of the grid):
//    full waves of tiles run data-parallel; the k-slices of the remaining
//    tiles are split evenly over all CTAs, partial tiles go through a
//    per-CTA workspace slot and a release/acquire flag, and the CTA that
//    owns a tile's last slice adds them to its own in CTA order (so results
//    are reproducible, though not the single ascending-k chain).  This
//    removes the idle SMs of the last partial wave ("Writing a Fast Matmul
//    in CUDA", "Size effects": a partial last wave; split-K as the remedy
//    in "What cuBLAS and CUTLASS add").
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "checked.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tile_order.cuh"

namespace sgemm {
namespace tmat {

struct Params {
  float* C;
  int64_t ldc;
  int M, N, K;
  float alpha, beta;
  int vec_c;
  int group_m;
  unsigned int* status;
  uint64_t timeout_ns;
  // stream-K tail (sk_iters == 0: every tile data-parallel)
  int dp_waves;          // tiles [0, dp_waves*grid) are data-parallel, tile b + i*grid for CTA b
  int64_t sk_iters;      // k-slices of tiles [dp_waves*grid, tiles), split evenly over the CTAs
  float* ws;             // one partial tile per CTA
  unsigned int* flags;   // flags[b] == epoch: CTA b's partial tile is published
  int64_t ws_slots;      // partial tiles (and flags) the workspace holds (checked build)
  unsigned int epoch;
  // strided batch: tiles are numbered batch-outermost; A and B come through
  // 3-D tensor maps (batch = the third coordinate), C is offset by stride_c
  int batch;
  int64_t stride_c;
  int a_batched, b_batched;  // 0: the operand is shared by every product (read at batch 0)
};

template <int BM_, int BN, int STAGES>
struct Shape {
  static constexpr int BM = BM_;
  static constexpr int BK = 32;
  static constexpr int kWarpsM = BM / 64;
  static constexpr int kWarpsN = BN / 32;
  static constexpr int kWarps = kWarpsM * kWarpsN;
  static constexpr int kThreads = kWarps * 32;
  // transpose mapping: kTPR threads per A row, each taking BK/kTPR k
  static constexpr int kTPR = kThreads / BM;
  static_assert(kThreads % BM == 0 && (kTPR == 1 || kTPR == 2 || kTPR == 4), "1, 2 or 4 threads per A row");
  static constexpr int kKPart = BK / kTPR;       // k per thread
  static constexpr int kSwz = 32 / kTPR;         // At[k][m ^ kSwz*(k / kKPart)]
  static constexpr int kStageA = BM * BK * 4;
  static constexpr int kStageB = BK * BN * 4;
  static constexpr int kStageBytes = kStageA + kStageB;
  static constexpr int kAtBytes = BK * BM * 4;
  static_assert(kStageA % 1024 == 0 && kStageB % 1024 == 0, "stages keep 1024-byte alignment");
  static constexpr int kSmemBytes = STAGES * kStageBytes + 2 * kAtBytes + STAGES * 8 + 1024;
};

// The next slice is transposed at step k == TA of the current one's k loop
// (all of it when TB < 0, else the first half, the second at k == TB).
// SPLIT: split-phase slice synchronisation through mbarriers instead of one
// CTA barrier per slice: every thread arrives on at_full[(j+1) & 1] after its
// part of slice j+1's transpose and on slice_done[j & 1] after slice j; it
// waits on at_full[j & 1] before slice j and on slice_done[(j-1) & 1] before
// overwriting At[(j+1) & 1], where thread 0 also refills stage (j-1) % STAGES.
// AT: A given transposed (stored K x M, M contiguous).  TMA then copies
// [BK][BM] boxes that already are At, and the k loop reads them from the
// ring stage: no on-chip transpose (and, with SPLIT, no "transposed"
// barriers; the slice's full barrier is waited on at its start).
template <int BM_, int BN, int STAGES, int MINB, bool BATCHED, int TA, int TB, bool SPLIT, bool AT = false>
__global__ void __launch_bounds__(Shape<BM_, BN, STAGES>::kThreads, MINB)
    sgemm_tmat_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const Params p) {
  using S = Shape<BM_, BN, STAGES>;
  constexpr int BM = S::BM;
  constexpr int BK = S::BK;
  static_assert(TA >= 0 && TA < BK && TB < BK && (TB < 0 || TB > TA), "transpose steps inside the k loop");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ int s_fail;
  __shared__ __align__(8) unsigned long long s_sync[4];  // SPLIT: at_full[2], slice_done[2]
  const uint32_t raw_base = ptx::smem_addr(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
  const uint32_t smem_base = ptx::smem_addr(smem);
  float* at_buf = reinterpret_cast<float*>(smem + STAGES * S::kStageBytes);  // [2][BK][BM]
  const uint32_t bar_full = smem_base + STAGES * S::kStageBytes + 2 * S::kAtBytes;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_m = (p.M + BM - 1) / BM;
  const int tiles_n = (p.N + BN - 1) / BN;
  const int tiles_per_batch = tiles_m * tiles_n;
  const int num_tiles = BATCHED ? tiles_per_batch * p.batch : tiles_per_batch;
  // tile -> (batch z, tile row, tile column), grouped order within a batch
  auto decode = [&](int tile, int& z, int& tm, int& tn) {
    if constexpr (BATCHED) {
      z = tile / tiles_per_batch;
      tile_coords(tile - z * tiles_per_batch, tiles_m, tiles_n, p.group_m, tm, tn);
    } else {
      z = 0;
      tile_coords(tile, tiles_m, tiles_n, p.group_m, tm, tn);
    }
  };
  const int KT = (p.K + BK - 1) / BK;
  // ---- this CTA's schedule: up to two stream-K segments first, then data-parallel tiles ----
  // Stream-K: the k-slices of the tail tiles are numbered x = 0 .. sk_iters-1
  // (tile-major) and CTA b takes x in [b*I/G, (b+1)*I/G).  Fewer tail tiles
  // than CTAs means a range spans at most two tiles: the head of the later
  // one (this CTA is a contributor: it publishes a partial tile) and the
  // tail of the earlier one (this CTA owns the tile's last slice: it waits
  // for the contributors, adds their partials in CTA order, and writes C).
  // The contributor segment runs first, so nobody waits on a CTA that is
  // itself waiting.
  const int G = static_cast<int>(gridDim.x);
  const int b = static_cast<int>(blockIdx.x);
  const int sk_tile0 = p.sk_iters > 0 ? p.dp_waves * G : num_tiles;
  int n_sk = 0;
  int sk_tile_a = 0, sk_k0_a = 0, sk_k1_a = 0;  // first stream-K segment
  int sk_tile_b = 0, sk_k0_b = 0, sk_k1_b = 0;  // second
  if (p.sk_iters > 0) {
    const int64_t s0 = (static_cast<int64_t>(b) * p.sk_iters) / G;
    const int64_t e0 = (static_cast<int64_t>(b + 1) * p.sk_iters) / G;
    if (s0 < e0) {
      const int t_first = static_cast<int>(s0 / KT);
      const int t_last = static_cast<int>((e0 - 1) / KT);
      if (t_last != t_first) {  // head of t_last (contributor) first, then tail of t_first
        sk_tile_a = sk_tile0 + t_last;
        sk_k0_a = 0;
        sk_k1_a = static_cast<int>(e0 - static_cast<int64_t>(t_last) * KT);
        sk_tile_b = sk_tile0 + t_first;
        sk_k0_b = static_cast<int>(s0 - static_cast<int64_t>(t_first) * KT);
        sk_k1_b = KT;
        n_sk = 2;
      } else {
        sk_tile_a = sk_tile0 + t_first;
        sk_k0_a = static_cast<int>(s0 - static_cast<int64_t>(t_first) * KT);
        sk_k1_a = static_cast<int>(e0 - static_cast<int64_t>(t_first) * KT);
        n_sk = 1;
      }
    }
  }
  const int dp_count = p.sk_iters > 0 ? p.dp_waves
                                      : (b < num_tiles ? (num_tiles - 1 - b) / G + 1 : 0);
  const int nseg = n_sk + dp_count;
  auto segment = [&](int i, int& tile, int& k0, int& k1) {
    if (i == 0 && n_sk > 0) {
      tile = sk_tile_a;
      k0 = sk_k0_a;
      k1 = sk_k1_a;
    } else if (i == 1 && n_sk > 1) {
      tile = sk_tile_b;
      k0 = sk_k0_b;
      k1 = sk_k1_b;
    } else {
      tile = b + (i - n_sk) * G;
      k0 = 0;
      k1 = KT;
    }
  };
  uint32_t total_it = static_cast<uint32_t>(dp_count) * static_cast<uint32_t>(KT);
  if (n_sk > 0) total_it += static_cast<uint32_t>(sk_k1_a - sk_k0_a);
  if (n_sk > 1) total_it += static_cast<uint32_t>(sk_k1_b - sk_k0_b);

  // producer cursor (thread 0): slices are issued in schedule order
  int c_seg = 0, c_kt = 0, c_k1 = 0, c_tm = 0, c_tn = 0, c_z = 0;
  uint32_t c_issued = 0;  // slices issued so far
  auto issue = [&](uint32_t j) {
    c_issued = j + 1;
    if (c_kt == c_k1) {  // enter the next segment
      int tile, k0;
      segment(c_seg++, tile, k0, c_k1);
      c_kt = k0;
      decode(tile, c_z, c_tm, c_tn);
    }
    const uint32_t s = j % STAGES;
    const uint32_t dst = smem_base + s * S::kStageBytes;
    ptx::mbar_arrive_expect_tx(bar_full + 8 * s, S::kStageBytes);
    if constexpr (BATCHED) {
      if constexpr (AT)
        ptx::tma_load_3d(dst, &tmA, c_tm * BM, c_kt * BK, c_z * p.a_batched, bar_full + 8 * s);
      else
        ptx::tma_load_3d(dst, &tmA, c_kt * BK, c_tm * BM, c_z * p.a_batched, bar_full + 8 * s);
      ptx::tma_load_3d(dst + S::kStageA, &tmB, c_tn * BN, c_kt * BK, c_z * p.b_batched, bar_full + 8 * s);
    } else {
      if constexpr (AT)
        ptx::tma_load_2d(dst, &tmA, c_tm * BM, c_kt * BK, bar_full + 8 * s);
      else
        ptx::tma_load_2d(dst, &tmA, c_kt * BK, c_tm * BM, bar_full + 8 * s);
      ptx::tma_load_2d(dst + S::kStageA, &tmB, c_tn * BN, c_kt * BK, bar_full + 8 * s);
    }
    ++c_kt;
  };

  if (threadIdx.x == 0) {
    s_fail = 0;
    for (int s = 0; s < STAGES; ++s) ptx::mbar_init(bar_full + 8 * s, 1);
    if constexpr (SPLIT)
      for (int i = 0; i < 4; ++i) ptx::mbar_init(ptx::smem_addr(&s_sync[i]), S::kThreads);
    ptx::fence_barrier_init();
    ptx::prefetch_tensormap(&tmA);
    ptx::prefetch_tensormap(&tmB);
    for (uint32_t j = 0; j < STAGES && j < total_it; ++j) issue(j);
  }
  __syncthreads();

  // transpose mapping: row tr = t / kTPR, k-part th = t % kTPR (kKPart k)
  const int tr = threadIdx.x / S::kTPR;
  const int th = threadIdx.x % S::kTPR;
  const int at_col = tr ^ (S::kSwz * th);  // k / kKPart == th for every k this thread writes
  bool failed;
  // Transpose A of slice j (ring stage j % STAGES) into at_buf[j & 1].
  // chunks [q0, q1) of this thread's part; `wait` first waits for the slice
  auto transpose_part = [&](uint32_t j, int q0, int q1, bool wait) -> bool {
    const uint32_t s = j % STAGES;
    if (wait && !ptx::mbar_wait(bar_full + 8 * s, (j / STAGES) & 1u, p.timeout_ns)) {
      atomicOr(p.status, kStatusTimeoutFull);
      return false;
    }
    const float* As = reinterpret_cast<const float*>(smem + s * S::kStageBytes) + tr * BK;
    float* At = at_buf + (j & 1) * (BK * BM);
#pragma unroll
    for (int q = q0; q < q1; ++q) {
      const int chunk = (S::kKPart / 4) * th + q;  // k = 4*chunk .. +3
      const int src = tr * BK + ((chunk ^ (tr & 7)) << 2);
      const float4 v = SG_CHK(SG_IN(src + 3, BM * BK), p.status) ? *reinterpret_cast<const float4*>(As - tr * BK + src)
                                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
      const float e4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (SG_CHK(SG_IN((4 * chunk + u) * BM + at_col, BK * BM), p.status)) At[(4 * chunk + u) * BM + at_col] = e4[u];
    }
    return true;
  };
  auto transpose = [&](uint32_t j) -> bool { return transpose_part(j, 0, S::kKPart / 4, true); };

  const int wm = warp / S::kWarpsN;
  const int wn = warp % S::kWarpsN;
  const int g = lane >> 2;
  const int c = lane & 3;
  // A pair i of this lane starts at m = wm*64 + 16i + 2g and is stored at
  // m ^ f(k), f(k) = kSwz * (k / kKPart) < 32:
  // (16i + 2g) ^ f = 16*(i ^ (f >> 4)) + (2g ^ (f & 15)); f & 15 is 0 or 8.
  const int a_lo0 = wm * 64 + (2 * g);
  const int a_lo8 = wm * 64 + ((2 * g) ^ 8);

  // failures are made CTA-uniform through the barrier, so every thread
  // leaves the loop at the same slice and no barrier is left waiting
  failed = __syncthreads_or(!AT && total_it > 0 && !transpose(0)) != 0;

  uint32_t it = 0;
  for (int seg = 0; seg < nseg && !failed; ++seg) {
    int tile, seg_k0, seg_k1;
    segment(seg, tile, seg_k0, seg_k1);
    int tz, tm, tn;
    decode(tile, tz, tm, tn);
    float* const Cz = BATCHED ? p.C + tz * p.stride_c : p.C;

    // acc[i][j] = {C[row 16i+2g][col j], C[row 16i+2g+1][col j]}, col j = 4c + 16(j/4) + j%4
    float2 acc[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = make_float2(0.f, 0.f);

    const uint32_t at_full0 = ptx::smem_addr(&s_sync[0]);
    const uint32_t done0 = ptx::smem_addr(&s_sync[2]);
    // SPLIT: a bounded wait that gives up as soon as another thread failed; warp-uniform result
    auto split_wait = [&](uint32_t bar, uint32_t parity) -> bool {
      const bool ok = ptx::mbar_wait_or_abort(bar, parity, p.timeout_ns, &s_fail);
      if (!ok) {
        atomicOr(p.status, kStatusTimeoutFull);
        *reinterpret_cast<volatile int*>(&s_fail) = 1;
      }
      return __all_sync(0xffffffffu, ok);
    };
    for (int kt = seg_k0; kt < seg_k1; ++kt, ++it) {
      // the next slice's A is transposed during this one (its buffer was last read one slice ago)
      bool bad = false;
      const uint32_t s = it % STAGES;
      if constexpr (AT) {
        // this slice's At and B are in stage s once its full barrier completes
        if constexpr (SPLIT) {
          if (!split_wait(bar_full + 8 * s, (it / STAGES) & 1u)) {
            failed = true;
            break;
          }
        } else {
          bad = !ptx::mbar_wait(bar_full + 8 * s, (it / STAGES) & 1u, p.timeout_ns);
          if (bad) atomicOr(p.status, kStatusTimeoutFull);  // the barrier below makes the failure CTA-wide
        }
      } else if constexpr (SPLIT) {
        // At[it & 1] is complete once every thread has transposed its part (slice 0: the prologue barrier)
        if (it >= 1 && !split_wait(at_full0 + 8 * (it & 1), ((it - 1) >> 1) & 1u)) {
          failed = true;
          break;
        }
      }
      const float* At = AT ? reinterpret_cast<const float*>(smem + s * S::kStageBytes)
                           : at_buf + (it & 1) * (BK * BM);
      const float4* Bs4 = reinterpret_cast<const float4*>(smem + s * S::kStageBytes + S::kStageA) + (wn * 32 + 4 * c) / 4;
      // operands of step k+1 are loaded while step k multiplies (register double buffer)
      auto load_ops = [&](int k, float2 (&ap)[4], float4& b0, float4& b1) {
        const int f = S::kSwz * (k / S::kKPart);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int ai = AT ? k * BM + a_lo0 + 16 * i : k * BM + ((f & 15) ? a_lo8 : a_lo0) + 16 * (i ^ (f >> 4));
          ap[i] = SG_CHK(SG_IN(ai + 1, BK * BM), p.status) ? *reinterpret_cast<const float2*>(At + ai)
                                                           : make_float2(0.f, 0.f);
        }
        const int bi = k * (BN / 4) + (wn * 32 + 4 * c) / 4;  // Bs4 starts at float4 (wn * 32 + 4c) / 4
        b0 = SG_CHK(SG_IN(bi, BK * BN / 4), p.status) ? Bs4[k * (BN / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
        b1 = SG_CHK(SG_IN(bi + 4, BK * BN / 4), p.status) ? Bs4[k * (BN / 4) + 4] : make_float4(0.f, 0.f, 0.f, 0.f);
      };
      float2 apn[4];
      float4 b0n, b1n;
      load_ops(0, apn, b0n, b1n);
#pragma unroll
      for (int k = 0; k < BK; ++k) {
        constexpr int kNq = S::kKPart / 4;
        if constexpr (SPLIT) {
          if (k == TA && it >= 1) {
            // every thread is done with slice it-1: At[(it+1) & 1] and stage (it-1) % STAGES are free
            bad = !split_wait(done0 + 8 * ((it - 1) & 1), ((it - 1) >> 1) & 1u);
            if (!bad && threadIdx.x == 0 && it - 1 + STAGES < total_it) {
              ptx::fence_proxy_async_smem();
              issue(it - 1 + STAGES);
            }
          }
        }
        if constexpr (AT) {
        } else if constexpr (TB >= 0) {  // in two halves
          if (k == TA && !bad) bad = it + 1 < total_it && !transpose_part(it + 1, 0, kNq / 2, true);
          if (k == TB && it + 1 < total_it && !bad) transpose_part(it + 1, kNq / 2, kNq, false);
        } else {
          if (k == TA && !bad) bad = it + 1 < total_it && !transpose(it + 1);
        }
        if constexpr (SPLIT && !AT) {
          if (k == (TB >= 0 ? TB : TA) && !bad && it + 1 < total_it) ptx::mbar_arrive(at_full0 + 8 * ((it + 1) & 1));
        }
        float2 ap[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) ap[i] = apn[i];
        const float bb[8] = {b0n.x, b0n.y, b0n.z, b0n.w, b1n.x, b1n.y, b1n.z, b1n.w};
        if (k + 1 < BK) load_ops(k + 1, apn, b0n, b1n);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = __ffma2_rn(ap[i], make_float2(bb[j], bb[j]), acc[i][j]);
      }
      if constexpr (SPLIT) {
        if (__any_sync(0xffffffffu, bad)) {
          *reinterpret_cast<volatile int*>(&s_fail) = 1;
          failed = true;
          break;
        }
        ptx::mbar_arrive(done0 + 8 * (it & 1));  // this thread is done with slice it
      } else {
        // every warp is done with stage s and At[it & 1]; At[(it+1) & 1] is complete
        if (bad) *reinterpret_cast<volatile int*>(&s_fail) = 1;
        __syncthreads();
        failed = *reinterpret_cast<volatile int*>(&s_fail) != 0;
        if (failed) break;
        if (threadIdx.x == 0 && it + STAGES < total_it) {
          ptx::fence_proxy_async_smem();
          issue(it + STAGES);
        }
      }
    }
    // SPLIT: warps leave a failed segment at different slices; agree before going on
    if constexpr (SPLIT) failed = __syncthreads_or(failed) != 0;
    if (failed) break;

    // ---------------- stream-K: publish, or gather the partial tiles ----------------
    constexpr int kQ = 16;  // float4s per thread: acc[4][8] float2 = 64 floats
    float4* ws4 = reinterpret_cast<float4*>(p.ws);
    if (seg_k1 < KT) {  // contributor: partial tile to this CTA's slot, then the flag
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        const int i = q >> 2, j2 = 2 * (q & 3);
        const int64_t wi = (static_cast<int64_t>(b) * kQ + q) * S::kThreads + threadIdx.x;
        if (SG_CHK(SG_IN(wi, p.ws_slots * (BM * BN / 4)), p.status))
          ws4[wi] = make_float4(acc[i][j2].x, acc[i][j2].y, acc[i][j2 + 1].x, acc[i][j2 + 1].y);
      }
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0 && SG_CHK(SG_IN(b, p.ws_slots), p.status)) ptx::st_release_gpu(p.flags + b, p.epoch);
      continue;
    }
    if (seg_k0 > 0) {  // finisher of a shared tile: wait for the contributors, add them in CTA order
      const int64_t x0 = static_cast<int64_t>(tile - sk_tile0) * KT;  // first slice of this tile
      const int c_first = static_cast<int>(((x0 + 1) * G - 1) / p.sk_iters);
      bool timed_out = false;
      if (threadIdx.x == 0) {
        for (int c = c_first; c < b && !timed_out; ++c) {
          if (!SG_CHK(SG_IN(c, p.ws_slots), p.status)) continue;
          if (ptx::ld_acquire_gpu(p.flags + c) == p.epoch) continue;
          const uint64_t t0 = ptx::globaltimer_ns();
          while (ptx::ld_acquire_gpu(p.flags + c) != p.epoch) {
            if (ptx::globaltimer_ns() - t0 > p.timeout_ns) {
              atomicOr(p.status, kStatusTimeoutFull);
              timed_out = true;
              break;
            }
          }
        }
      }
      failed = __syncthreads_or(timed_out) != 0;
      if (failed) break;
      // own slices (the tile's last) first, then the contributors' in CTA order
#pragma unroll 1
      for (int c = c_first; c < b; ++c) {
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
          const int i = q >> 2, j2 = 2 * (q & 3);
          const int64_t wi = (static_cast<int64_t>(c) * kQ + q) * S::kThreads + threadIdx.x;
          const float4 v = SG_CHK(SG_IN(wi, p.ws_slots * (BM * BN / 4)), p.status) ? __ldcg(&ws4[wi])
                                                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
          acc[i][j2].x += v.x;
          acc[i][j2].y += v.y;
          acc[i][j2 + 1].x += v.z;
          acc[i][j2 + 1].y += v.w;
        }
      }
      // every thread has read the partials: clear their flags, so each run
      // (a replayed graph included, whose epoch is fixed) starts from zero
      __syncthreads();
      if (threadIdx.x == 0)
        for (int c = c_first; c < b; ++c)
          if (SG_CHK(SG_IN(c, p.ws_slots), p.status)) *reinterpret_cast<volatile unsigned int*>(p.flags + c) = 0u;
    }

    // ---------------- epilogue ----------------
    if (p.beta == 0.f) {  // C is not read
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int row = tm * BM + wm * 64 + 16 * i + 2 * g + e;
          if (row >= p.M) continue;
          float* crow = Cz + static_cast<int64_t>(row) * p.ldc;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int col = tn * BN + wn * 32 + 4 * c + 16 * h;
            float v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) v[q] = e ? acc[i][4 * h + q].y : acc[i][4 * h + q].x;
            if (p.vec_c && col + 3 < p.N) {
              *reinterpret_cast<float4*>(crow + col) =
                  make_float4(p.alpha * v[0], p.alpha * v[1], p.alpha * v[2], p.alpha * v[3]);
            } else {
#pragma unroll
              for (int q = 0; q < 4; ++q)
                if (col + q < p.N) crow[col + q] = p.alpha * v[q];
            }
          }
        }
      }
    } else {
      // The four C reads of a row pair (i) are all issued before any of its
      // writes: the compiler cannot move a read of C above a write to
      // another row of C, so in the plain order each read waited out the
      // previous write's round trip.
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float4 old[2][2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int row = tm * BM + wm * 64 + 16 * i + 2 * g + e;
          const float* crow = Cz + static_cast<int64_t>(row) * p.ldc;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int col = tn * BN + wn * 32 + 4 * c + 16 * h;
            old[e][h] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (row >= p.M) continue;
            if (p.vec_c && col + 3 < p.N) {
              old[e][h] = *reinterpret_cast<const float4*>(crow + col);
            } else {
              if (col < p.N) old[e][h].x = crow[col];
              if (col + 1 < p.N) old[e][h].y = crow[col + 1];
              if (col + 2 < p.N) old[e][h].z = crow[col + 2];
              if (col + 3 < p.N) old[e][h].w = crow[col + 3];
            }
          }
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int row = tm * BM + wm * 64 + 16 * i + 2 * g + e;
          if (row >= p.M) continue;
          float* crow = Cz + static_cast<int64_t>(row) * p.ldc;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int col = tn * BN + wn * 32 + 4 * c + 16 * h;
            float v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) v[q] = e ? acc[i][4 * h + q].y : acc[i][4 * h + q].x;
            const float oo[4] = {old[e][h].x, old[e][h].y, old[e][h].z, old[e][h].w};
            float r[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) r[q] = fmaf(p.alpha, v[q], p.beta * oo[q]);
            if (p.vec_c && col + 3 < p.N) {
              *reinterpret_cast<float4*>(crow + col) = make_float4(r[0], r[1], r[2], r[3]);
            } else {
#pragma unroll
              for (int q = 0; q < 4; ++q)
                if (col + q < p.N) crow[col + q] = r[q];
            }
          }
        }
      }
    }
  }
  // after a failure, copies still in flight land before the CTA's shared memory is released
  if (failed && threadIdx.x == 0) ptx::drain_ring(bar_full, 8, c_issued, STAGES, p.timeout_ns);
}

template <int BM_, int BN, int STAGES, int MINB, int TA, int TB = -1, bool SPLIT = false>
struct Variant_ {
  using S = Shape<BM_, BN, STAGES>;
  // a single product runs the plain 2-D kernel (or, A given transposed, its
  // AT form); strided batches their own instantiations
  static constexpr auto kernel = sgemm_tmat_kernel<BM_, BN, STAGES, MINB, false, TA, TB, SPLIT>;
  static constexpr auto kernel_at = sgemm_tmat_kernel<BM_, BN, STAGES, MINB, false, TA, TB, SPLIT, true>;
  static constexpr auto kernel_batched = sgemm_tmat_kernel<BM_, BN, STAGES, MINB, true, TA, TB, SPLIT>;
  static constexpr auto kernel_at_batched = sgemm_tmat_kernel<BM_, BN, STAGES, MINB, true, TA, TB, SPLIT, true>;
  static cudaError_t prepare() {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel_at, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kernel_at_batched, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
    return e != cudaSuccess ? e
                            : cudaFuncSetAttribute(kernel_batched, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   S::kSmemBytes);
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
    p.vec_c = ((reinterpret_cast<uintptr_t>(a.C) & 15) == 0) && (a.ldc % 4 == 0) &&
              (a.batch <= 1 || a.stride_c % 4 == 0);
    p.group_m = 8;
    p.status = a.status;
    p.timeout_ns = a.timeout_ns;
    p.dp_waves = a.dp_waves;
    p.sk_iters = a.sk_iters;
    p.ws = a.ws;
    p.flags = a.flags;
    p.ws_slots = a.ws_slots;
    p.epoch = a.epoch;
    p.batch = a.batch > 1 ? a.batch : 1;
    p.stride_c = a.stride_c;
    p.a_batched = a.batch > 1 && a.stride_a != 0;
    p.b_batched = a.batch > 1 && a.stride_b != 0;
    if (p.batch > 1 && a.a_trans) {
      kernel_at_batched<<<a.grid, S::kThreads, S::kSmemBytes, stream>>>(a.tmA, a.tmB, p);
    } else if (p.batch > 1) {
      kernel_batched<<<a.grid, S::kThreads, S::kSmemBytes, stream>>>(a.tmA, a.tmB, p);
    } else if (a.a_trans) {
      kernel_at<<<a.grid, S::kThreads, S::kSmemBytes, stream>>>(a.tmA, a.tmB, p);
    } else {
      kernel<<<a.grid, S::kThreads, S::kSmemBytes, stream>>>(a.tmA, a.tmB, p);
    }
    return cudaGetLastError();
  }
  static Variant describe(const char* name) {
    Variant v{name, kKindTma, S::BM, BN, S::BK, STAGES, 1, S::kThreads, S::kSmemBytes, 128,
              &prepare, &occupancy, &launch, 0, 1, 1};
    v.a_trans_ok = 1;  // reads A given transposed (K x M) by TMA itself
    return v;
  }
};

}  // namespace tmat
}  // namespace sgemm
