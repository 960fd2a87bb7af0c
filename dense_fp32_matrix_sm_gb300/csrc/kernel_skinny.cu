// kernel_skinny.cu -- SGEMM for few rows (M <= 16): the decode-shaped case.
//
// With M <= 16 every element of B is used at most 16 times, so the product
// is bound by streaming B from HBM, not by the FMA pipe ("Writing a Fast
// Matmul in CUDA, Step by Step", "Why decode doesn't care": a decode-step
// matrix product multiplies each weight a handful of times, so it sits on
// the bandwidth roof).  What matters is keeping enough bytes of B in
// flight on every SM and spending no FMAs on padding rows.
//
//  * CTA tile: all 16 rows x BN columns (BN a multiple of 128), over one
//    contiguous k-range.  Each 128-column group has GW (4 or 8) warps; warp
//    w of a group multiplies k-quads w, w + GW, ... of every 32-deep
//    k-slice, and
//    lane l owns columns 4l .. 4l + 3 of its group for all 16 rows (a
//    16 x 4 thread tile).  Wider tiles read longer contiguous runs of each
//    B row (BN * 4 bytes) per DRAM access.  The _ef variants load B with an
//    L2 evict-first hint: it is read exactly once, so it should not push A
//    (read by every CTA) out of L2.  A TMA ring (A slice 16 x 32 with the 128-byte
//    swizzle, B slice 32 x 128) feeds it exactly like the main kernel, with
//    the same stage-release counters and bounded waits.
//  * Cluster c walks column slabs c, c + #clusters, ...  With one slab per
//    cluster (the default grid) clusters come and go independently; the
//    _persist variant launches only as many clusters as fit on the GPU at
//    once and keeps each TMA ring running across slab boundaries (measured
//    slower on the 16 x 16384 x 8192 decode shape: lock-stepped clusters).
//  * Split-K without scratch memory ("How a Matmul Kernel Gets Fast",
//    section 14, and "Writing a Fast Matmul in CUDA", "What cuBLAS and
//    CUTLASS add": split the k loop across blocks and add the pieces):
//    the S CTAs that share a column slab form one thread-block cluster and
//    take consecutive k-ranges.  Each CTA first adds, per column group, its GW warps'
//    partial tiles into one shared tile (warp order 0..GW-1), then the cluster
//    synchronises and CTA r finalises 1/S of the 16 x 128 outputs by
//    reading the S partial tiles through distributed shared memory in rank
//    order 0..S-1.  The reduction order is fixed, so results are
//    reproducible run to run; it is not the ascending-k chain of the
//    single-pass kernels (the plan reports k_order=split).
//  * _pa variants multiply in the paired form the main kernels found
//    fastest on GB300: each warp transposes its own 16 x 4 k-quad of A into
//    a small per-warp buffer (no CTA barrier), then each FFMA2 multiplies a
//    register pair of two A rows by one broadcast element of B.
//  * Epilogue: out = alpha*sum (beta == 0, C not read) or
//    fmaf(alpha, sum, beta*C), predicated on m < M and n < N.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "checked.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace sgemm {
namespace {

constexpr int kSBM = 16;
constexpr int kSBK = 32;

struct SkinnyParams {
  float* C;
  int64_t ldc;
  int M, N, K;
  float alpha, beta;
  unsigned int* status;
  uint64_t timeout_ns;
};

// BN columns per CTA (a warp spans 128), GW warps per 128-column group
// splitting each k-slice's eight quads.
template <int BN, int GW, int STAGES>
struct SkinnyShape {
  static constexpr int kAtwBytes = 4 * 32 * 4;  // per warp: one transposed k-quad, rows padded to 32
  static_assert(GW == 4 || GW == 8, "each warp takes 8 / GW quads of a 32-deep slice");
  static constexpr int kQuadsPerWarp = (kSBK / 4) / GW;
  static_assert(BN % 128 == 0 && BN <= 256, "a warp spans 128 columns (32 lanes x 4); one TMA box spans <= 256");
  static constexpr int kGroups = BN / 128;
  static constexpr int kWarps = GW * kGroups;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kStageA = kSBM * kSBK * 4;  // 2 KB
  static constexpr int kStageB = kSBK * BN * 4;    // 16 KB
  static constexpr int kStageBytes = kStageA + kStageB;
  static_assert(kStageA % 1024 == 0 && kStageB % 1024 == 0, "stages keep 1024-byte alignment");
  static constexpr int kRingBytes = STAGES * kStageBytes;
  static constexpr int kPartialBytes = kSBM * BN * 4;
  static constexpr int kSmemBytes = kRingBytes + kPartialBytes + kWarps * kAtwBytes + STAGES * 16 + 1024;
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

// All threads of all CTAs of the cluster; orders shared-memory writes
// before the peers' reads.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ float ld_peer(const float* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(ptx::smem_addr(local)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

// One 32-deep slice in the paired form: this warp's k-quads q = gw, gw + GW,
// ... of the stage (A at As, B at Bs4 = this lane's float4 column of its
// group), accumulated into accp[p][j] = {C[2p][4l + j], C[2p + 1][4l + j]}.
template <int BN, int GW>
__device__ __forceinline__ void pa_slice(const float* As, const float4* Bs4, float* atw, int gw, int lane,
                                         float2 (&accp)[kSBM / 2][4], unsigned int* status) {
#pragma unroll
  for (int qq = 0; qq < (kSBK / 4) / GW; ++qq) {
    // Transpose this warp's k-quad of A (16 rows x 4 k) into atw[k][m]:
    // lane takes row l/2, k pair 2*(l%2); rows are 32 floats apart and
    // k = 2, 3 sit 16 floats further in, so the 32 writes hit 32 banks.
    const int q = gw + GW * qq;
    {
      const int m = lane >> 1, h = lane & 1;
      const int ai = m * kSBK + ((q ^ (m & 7)) << 2) + 2 * h;
      const float2 v = SG_CHK(SG_IN(ai + 1, kSBM * kSBK) && SG_IN((2 * h + 1) * 32 + 16 * h + m, 128), status)
                           ? *reinterpret_cast<const float2*>(As + ai)
                           : make_float2(0.f, 0.f);
      atw[(2 * h) * 32 + 16 * h + m] = v.x;
      atw[(2 * h + 1) * 32 + 16 * h + m] = v.y;
    }
    __syncwarp();
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const float4 b = SG_CHK(SG_IN(4 * q + kk, kSBK), status) ? Bs4[(4 * q + kk) * (BN / 4)]
                                                               : make_float4(0.f, 0.f, 0.f, 0.f);
      const float bb[4] = {b.x, b.y, b.z, b.w};
      const float* ak = atw + kk * 32 + 16 * ((kk >> 1) & 1);
#pragma unroll
      for (int pp = 0; pp < kSBM / 2; ++pp) {
        const float2 ap = *reinterpret_cast<const float2*>(ak + 2 * pp);  // rows 2pp, 2pp+1
#pragma unroll
        for (int j = 0; j < 4; ++j) accp[pp][j] = __ffma2_rn(ap, make_float2(bb[j], bb[j]), accp[pp][j]);
      }
    }
    __syncwarp();  // the next quad overwrites atw
  }
}

// As pa_slice, with B given transposed (stored N x K): the stage holds
// Bt[n][k], rows of 32 k (128 bytes) with the 128-byte swizzle (16-byte
// chunk q of row n at position q ^ (n % 8)).  Lane l of column group g owns
// columns n = 128 g + l + 32 j (j = 0..3): per k-quad it reads one float4
// of 4 k from each of its 4 rows; accp[p][j] = {C[2p][n_j], C[2p+1][n_j]}.
template <int BN, int GW>
__device__ __forceinline__ void pa_slice_bt(const float* As, const float* Bt, float* atw, int gw, int lane, int group,
                                            float2 (&accp)[kSBM / 2][4], unsigned int* status) {
#pragma unroll
  for (int qq = 0; qq < (kSBK / 4) / GW; ++qq) {
    const int q = gw + GW * qq;
    {
      const int m = lane >> 1, h = lane & 1;
      const int ai = m * kSBK + ((q ^ (m & 7)) << 2) + 2 * h;
      const float2 v = SG_CHK(SG_IN(ai + 1, kSBM * kSBK) && SG_IN((2 * h + 1) * 32 + 16 * h + m, 128), status)
                           ? *reinterpret_cast<const float2*>(As + ai)
                           : make_float2(0.f, 0.f);
      atw[(2 * h) * 32 + 16 * h + m] = v.x;
      atw[(2 * h + 1) * 32 + 16 * h + m] = v.y;
    }
    float4 bq[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = 128 * group + lane + 32 * j;
      const int bi = n * kSBK + ((q ^ (n & 7)) << 2);
      bq[j] = SG_CHK(SG_IN(bi + 3, BN * kSBK), status) ? *reinterpret_cast<const float4*>(Bt + bi)
                                                       : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncwarp();
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const float* ak = atw + kk * 32 + 16 * ((kk >> 1) & 1);
#pragma unroll
      for (int pp = 0; pp < kSBM / 2; ++pp) {
        const float2 ap = *reinterpret_cast<const float2*>(ak + 2 * pp);  // rows 2pp, 2pp+1
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float b = kk == 0 ? bq[j].x : kk == 1 ? bq[j].y : kk == 2 ? bq[j].z : bq[j].w;
          accp[pp][j] = __ffma2_rn(ap, make_float2(b, b), accp[pp][j]);
        }
      }
    }
    __syncwarp();  // the next quad overwrites atw
  }
}

template <int BN, int GW, int STAGES, int MINB, bool EVICT_FIRST, bool PAIRA>
__global__ void __launch_bounds__(SkinnyShape<BN, GW, STAGES>::kThreads, MINB)
    sgemm_skinny_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const SkinnyParams p) {
  using S = SkinnyShape<BN, GW, STAGES>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ int s_failed;  // set when any wait of this CTA ran out; later waits are skipped
  const uint32_t raw_base = ptx::smem_addr(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
  const uint32_t smem_base = ptx::smem_addr(smem);
  float* partial = reinterpret_cast<float*>(smem + S::kRingBytes);  // [16][BN], read by cluster peers
  constexpr int kBarOff = S::kRingBytes + S::kPartialBytes + S::kWarps * S::kAtwBytes;
  float* atw = reinterpret_cast<float*>(smem + S::kRingBytes + S::kPartialBytes) + (threadIdx.x >> 5) * (S::kAtwBytes / 4);
  const uint32_t bar_full = smem_base + kBarOff;
  unsigned int* released = reinterpret_cast<unsigned int*>(smem + kBarOff + STAGES * 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int group = warp / GW;  // columns 128*group .. +127 of the tile
  const int gw = warp % GW;     // k-quads gw, gw + GW, ... of each slice
  const uint32_t rank = cluster_rank();
  const uint32_t nsplit = cluster_size();
  // Persistent clusters: cluster cid walks column slabs cid, cid + ncl, ...;
  // its S CTAs take the same consecutive k-ranges of every slab.
  const int cid = static_cast<int>(blockIdx.x / nsplit);
  const int ncl = static_cast<int>(gridDim.x / nsplit);
  const int nslabs = (p.N + BN - 1) / BN;
  const int my_slabs = cid < nslabs ? (nslabs - 1 - cid) / ncl + 1 : 0;
  const int KT = (p.K + kSBK - 1) / kSBK;
  const int kt_begin = static_cast<int>((static_cast<int64_t>(KT) * rank) / nsplit);
  const int kt_end = static_cast<int>((static_cast<int64_t>(KT) * (rank + 1)) / nsplit);
  const uint32_t nkt = static_cast<uint32_t>(kt_end - kt_begin);
  const uint32_t total_it = static_cast<uint32_t>(my_slabs) * nkt;

  // slices are numbered j = local_slab * nkt + (kt - kt_begin) over all of this CTA's slabs
  auto issue = [&](uint32_t j) {
    const uint32_t s = j % STAGES;
    const int kt = kt_begin + static_cast<int>(j % nkt);
    const int n0 = (cid + static_cast<int>(j / nkt) * ncl) * BN;
    const uint32_t dst = smem_base + s * S::kStageBytes;
    ptx::mbar_arrive_expect_tx(bar_full + 8 * s, S::kStageBytes);
    ptx::tma_load_2d(dst, &tmA, kt * kSBK, 0, bar_full + 8 * s);
    if constexpr (EVICT_FIRST) {
      ptx::tma_load_2d_hint(dst + S::kStageA, &tmB, n0, kt * kSBK, bar_full + 8 * s, ptx::l2_policy_evict_first());
    } else {
      ptx::tma_load_2d(dst + S::kStageA, &tmB, n0, kt * kSBK, bar_full + 8 * s);
    }
  };

  if (threadIdx.x == 0) {
    s_failed = 0;
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

  uint32_t it = 0;
  bool ready = false;
  for (int ls = 0; ls < my_slabs; ++ls) {
    const int n0 = (cid + ls * ncl) * BN;
    // row-major form: acc[m][0] = columns 4l, 4l+1 of row m; acc[m][1] = columns 4l+2, 4l+3.
    // pair form (PAIRA): accp[p][j] = {C[2p][4l + j], C[2p+1][4l + j]}.
    float2 acc[kSBM][2];
    float2 accp[kSBM / 2][4];
#pragma unroll
    for (int m = 0; m < kSBM; ++m) acc[m][0] = acc[m][1] = make_float2(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < kSBM / 2; ++q)
#pragma unroll
      for (int j = 0; j < 4; ++j) accp[q][j] = make_float2(0.f, 0.f);

    for (uint32_t kk_it = 0; kk_it < nkt; ++kk_it, ++it) {
      if (*reinterpret_cast<volatile int*>(&s_failed)) continue;
      const uint32_t s = it % STAGES;
      if (!ready && !ptx::mbar_wait(bar_full + 8 * s, (it / STAGES) & 1u, p.timeout_ns)) {
        atomicOr(p.status, kStatusTimeoutFull);
        *reinterpret_cast<volatile int*>(&s_failed) = 1;
        continue;  // keep step with the CTA and cluster barriers below
      }
      ready = it + 1 < total_it &&
              ptx::mbar_test_wait(bar_full + 8 * ((it + 1) % STAGES), ((it + 1) / STAGES) & 1u);
      const float* As = reinterpret_cast<const float*>(smem + s * S::kStageBytes);
      const float4* Bs4 = reinterpret_cast<const float4*>(smem + s * S::kStageBytes + S::kStageA) + group * 32 + lane;
      if constexpr (PAIRA) pa_slice<BN, GW>(As, Bs4, atw, gw, lane, accp, p.status);
#pragma unroll
      for (int qq = 0; qq < S::kQuadsPerWarp && !PAIRA; ++qq) {
        const int q = gw + GW * qq;
        float4 a4[kSBM];
#pragma unroll
        for (int m = 0; m < kSBM; ++m)
          a4[m] = *reinterpret_cast<const float4*>(As + m * kSBK + ((q ^ (m & 7)) << 2));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const float4 b = Bs4[(4 * q + kk) * (BN / 4)];
          const float2 b01 = make_float2(b.x, b.y);
          const float2 b23 = make_float2(b.z, b.w);
#pragma unroll
          for (int m = 0; m < kSBM; ++m) {
            const float a = kk == 0 ? a4[m].x : kk == 1 ? a4[m].y : kk == 2 ? a4[m].z : a4[m].w;
            const float2 aa = make_float2(a, a);
            acc[m][0] = __ffma2_rn(aa, b01, acc[m][0]);
            acc[m][1] = __ffma2_rn(aa, b23, acc[m][1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        const unsigned int before = ptx::atom_add_acq_rel_cta(&released[s], 1u);
        if ((before + 1u) % S::kWarps == 0u && it + STAGES < total_it) {
          ptx::fence_proxy_async_smem();
          issue(it + STAGES);
        }
      }
    }

    // ---- this slab: add each column group's GW warp partials into `partial` (warp order) ----
    // The ring keeps streaming the next slab meanwhile.
#pragma unroll 1
    for (int w = 0; w < GW; ++w) {
      if (gw == w) {
        float4* part4 = reinterpret_cast<float4*>(partial);
#pragma unroll
        for (int m = 0; m < kSBM; ++m) {
          float4 v;
          if constexpr (PAIRA) {
            const int pp = m >> 1;
            v = (m & 1) ? make_float4(accp[pp][0].y, accp[pp][1].y, accp[pp][2].y, accp[pp][3].y)
                        : make_float4(accp[pp][0].x, accp[pp][1].x, accp[pp][2].x, accp[pp][3].x);
          } else {
            v = make_float4(acc[m][0].x, acc[m][0].y, acc[m][1].x, acc[m][1].y);
          }
          float4* d = part4 + m * (BN / 4) + group * 32 + lane;
          if (w == 0) {
            *d = v;
          } else {
            const float4 o = *d;
            *d = make_float4(o.x + v.x, o.y + v.y, o.z + v.z, o.w + v.w);
          }
        }
      }
      __syncthreads();
    }

    // ---- reduce the cluster's partial tiles (rank order) and write C ----
    cluster_sync();
    constexpr int kTile = kSBM * BN;
    const int begin = static_cast<int>((static_cast<int64_t>(kTile) * rank) / nsplit);
    const int end = static_cast<int>((static_cast<int64_t>(kTile) * (rank + 1)) / nsplit);
    for (int idx = begin + static_cast<int>(threadIdx.x); idx < end; idx += S::kThreads) {
      const int m = idx / BN;
      const int n = n0 + idx % BN;
      float sum = 0.f;
      for (uint32_t r = 0; r < nsplit; ++r) sum += ld_peer(partial + idx, r);
      if (m < p.M && n < p.N) {
        float* d = p.C + static_cast<int64_t>(m) * p.ldc + n;
        *d = p.beta == 0.f ? p.alpha * sum : fmaf(p.alpha, sum, p.beta * *d);
      }
    }
    cluster_sync();  // peers may still be reading this CTA's partial tile
  }
  // After a failed wait, copies still in flight land before the CTA's shared
  // memory is released.  Every warp that sees the failure drains what has been
  // issued so far; a copy issued later is drained by the warp that issued it
  // (or was waited on by every warp, when no warp saw the failure).
  if (lane == 0 && *reinterpret_cast<volatile int*>(&s_failed))
    ptx::drain_ring_released(bar_full, 8, released, S::kWarps, STAGES, total_it, p.timeout_ns);
}

// ---------------------------------------------------------------------------
// Stream-K form: one resident wave, no clusters.  The work units are
// (column slab, 32-deep k-slice) pairs numbered slab-major, U in all; CTA b
// of G streams units [b*U/G, (b+1)*U/G) through one TMA ring without
// draining between slabs.  Its range covers the tail of slab s_first, any
// whole slabs, and the head of slab s_last; it runs the head first.
//  * a whole slab is written straight to C;
//  * a head (or a piece inside one slab) is a contributor: its 16 x BN
//    partial tile goes to workspace slot b, then flags[b] = epoch (release);
//  * the tail of s_first is the finisher: it waits (acquire, bounded) for
//    the flags of the CTAs c_first .. b-1 that hold the slab's earlier
//    slices, adds their partials in CTA order after its own, and writes C.
// Every contributor piece is its CTA's first piece, so a finisher never
// waits on a CTA that is itself waiting.  The sum order is fixed (results
// are reproducible run to run; k_order=split).
struct SkinnySkParams {
  float* C;
  int64_t ldc;
  int M, N, K;
  float alpha, beta;
  unsigned int* status;
  uint64_t timeout_ns;
  float* ws;             // kSBM x BN floats per CTA
  unsigned int* flags;   // one per CTA
  unsigned int epoch;
  int64_t ws_slots;      // partial tiles (and flags) the workspace holds (checked build)
  // strided batch (BATCHED): slabs are numbered product-major over all
  // products; A and B come through 3-D tensor maps (batch = third
  // coordinate, 0 for an operand every product shares), C is offset by stride_c
  int batch;
  int64_t stride_c;
  int a_batched, b_batched;
};

// BT: B given transposed (stored N x K), loaded as swizzled [n][k] boxes.
// BATCHED: a strided batch of products (B as stored, or given transposed).
template <int BN, int GW, int STAGES, int MINB, bool EVICT_FIRST, bool BT, bool BATCHED = false>
__global__ void __launch_bounds__(SkinnyShape<BN, GW, STAGES>::kThreads, MINB)
    sgemm_skinny_sk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                           const SkinnySkParams p) {
  using S = SkinnyShape<BN, GW, STAGES>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ int s_failed;
  const uint32_t raw_base = ptx::smem_addr(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
  const uint32_t smem_base = ptx::smem_addr(smem);
  float* partial = reinterpret_cast<float*>(smem + S::kRingBytes);  // [16][BN]
  constexpr int kBarOff = S::kRingBytes + S::kPartialBytes + S::kWarps * S::kAtwBytes;
  float* atw = reinterpret_cast<float*>(smem + S::kRingBytes + S::kPartialBytes) + (threadIdx.x >> 5) * (S::kAtwBytes / 4);
  const uint32_t bar_full = smem_base + kBarOff;
  unsigned int* released = reinterpret_cast<unsigned int*>(smem + kBarOff + STAGES * 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int group = warp / GW;
  const int gw = warp % GW;
  const int G = static_cast<int>(gridDim.x);
  const int b = static_cast<int>(blockIdx.x);
  const int KT = (p.K + kSBK - 1) / kSBK;
  const int nslabs = (p.N + BN - 1) / BN;  // per product
  // slabs over every product: gs = z * nslabs + slab of product z
  const int64_t U = static_cast<int64_t>(nslabs) * (BATCHED ? p.batch : 1) * KT;
  const int64_t s0 = (static_cast<int64_t>(b) * U) / G;
  const int64_t e0 = (static_cast<int64_t>(b + 1) * U) / G;
  const uint32_t total_it = static_cast<uint32_t>(e0 - s0);
  const int s_first = total_it ? static_cast<int>(s0 / KT) : 0;
  const int s_last = total_it ? static_cast<int>((e0 - 1) / KT) : 0;
  const int64_t head_begin = static_cast<int64_t>(s_last) * KT;
  // the head of s_last runs first when the range spans several slabs
  const uint32_t head_len = s_last > s_first ? static_cast<uint32_t>(e0 - head_begin) : 0u;
  const int npieces = total_it ? s_last - s_first + 1 : 0;

  auto unit_of = [&](uint32_t j) -> int64_t { return j < head_len ? head_begin + j : s0 + (j - head_len); };
  auto issue = [&](uint32_t j) {
    const uint32_t s = j % STAGES;
    const int64_t u = unit_of(j);
    const int kt = static_cast<int>(u % KT);
    const int gs = static_cast<int>(u / KT);
    const uint32_t dst = smem_base + s * S::kStageBytes;
    ptx::mbar_arrive_expect_tx(bar_full + 8 * s, S::kStageBytes);
    if constexpr (BATCHED) {
      const int z = gs / nslabs;
      const int n0 = (gs - z * nslabs) * BN;
      ptx::tma_load_3d(dst, &tmA, kt * kSBK, 0, z * p.a_batched, bar_full + 8 * s);
      const int bx = BT ? kt * kSBK : n0, by = BT ? n0 : kt * kSBK;  // B as [k][n], or Bt as [n][k]
      if constexpr (EVICT_FIRST)
        ptx::tma_load_3d_hint(dst + S::kStageA, &tmB, bx, by, z * p.b_batched, bar_full + 8 * s,
                              ptx::l2_policy_evict_first());
      else
        ptx::tma_load_3d(dst + S::kStageA, &tmB, bx, by, z * p.b_batched, bar_full + 8 * s);
      return;
    }
    const int n0 = gs * BN;
    ptx::tma_load_2d(dst, &tmA, kt * kSBK, 0, bar_full + 8 * s);
    const int bx = BT ? kt * kSBK : n0, by = BT ? n0 : kt * kSBK;  // B as [k][n], or Bt as [n][k]
    if constexpr (EVICT_FIRST) {
      ptx::tma_load_2d_hint(dst + S::kStageA, &tmB, bx, by, bar_full + 8 * s, ptx::l2_policy_evict_first());
    } else {
      ptx::tma_load_2d(dst + S::kStageA, &tmB, bx, by, bar_full + 8 * s);
    }
  };

  if (threadIdx.x == 0) {
    s_failed = 0;
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

  uint32_t it = 0;
  bool ready = false;
#pragma unroll 1
  for (int pc = 0; pc < npieces; ++pc) {
    int slab, k0, k1;
    if (head_len > 0 && pc == 0) {
      slab = s_last;
      k0 = 0;
      k1 = static_cast<int>(head_len);
    } else {
      slab = s_first + (head_len > 0 ? pc - 1 : pc);
      const int64_t lo = static_cast<int64_t>(slab) * KT;
      k0 = static_cast<int>((s0 > lo ? s0 : lo) - lo);
      k1 = static_cast<int>((e0 < lo + KT ? e0 : lo + KT) - lo);
    }
    // slab is numbered over every product (BATCHED): product z, its column slab
    const int z = BATCHED ? slab / nslabs : 0;
    const int n0 = (slab - z * nslabs) * BN;
    float* const Cz = BATCHED ? p.C + z * p.stride_c : p.C;
    float2 accp[kSBM / 2][4];
#pragma unroll
    for (int q = 0; q < kSBM / 2; ++q)
#pragma unroll
      for (int j = 0; j < 4; ++j) accp[q][j] = make_float2(0.f, 0.f);

#pragma unroll 1
    for (int kt = k0; kt < k1; ++kt, ++it) {
      if (*reinterpret_cast<volatile int*>(&s_failed)) continue;
      const uint32_t s = it % STAGES;
      if (!ready && !ptx::mbar_wait(bar_full + 8 * s, (it / STAGES) & 1u, p.timeout_ns)) {
        atomicOr(p.status, kStatusTimeoutFull);
        *reinterpret_cast<volatile int*>(&s_failed) = 1;
        continue;
      }
      ready = it + 1 < total_it &&
              ptx::mbar_test_wait(bar_full + 8 * ((it + 1) % STAGES), ((it + 1) / STAGES) & 1u);
      const float* As = reinterpret_cast<const float*>(smem + s * S::kStageBytes);
      if constexpr (BT) {
        pa_slice_bt<BN, GW>(As, reinterpret_cast<const float*>(smem + s * S::kStageBytes + S::kStageA), atw, gw, lane,
                            group, accp, p.status);
      } else {
        const float4* Bs4 = reinterpret_cast<const float4*>(smem + s * S::kStageBytes + S::kStageA) + group * 32 + lane;
        pa_slice<BN, GW>(As, Bs4, atw, gw, lane, accp, p.status);
      }
      __syncwarp();
      if (lane == 0) {
        const unsigned int before = ptx::atom_add_acq_rel_cta(&released[s], 1u);
        if ((before + 1u) % S::kWarps == 0u && it + STAGES < total_it) {
          ptx::fence_proxy_async_smem();
          issue(it + STAGES);
        }
      }
    }

    // this piece's GW warp partials into `partial`, in warp order
#pragma unroll 1
    for (int w = 0; w < GW; ++w) {
      if (gw == w) {
        float4* part4 = reinterpret_cast<float4*>(partial);
#pragma unroll
        for (int m = 0; m < kSBM; ++m) {
          const int pp = m >> 1;
          const float4 v = (m & 1) ? make_float4(accp[pp][0].y, accp[pp][1].y, accp[pp][2].y, accp[pp][3].y)
                                   : make_float4(accp[pp][0].x, accp[pp][1].x, accp[pp][2].x, accp[pp][3].x);
          if constexpr (BT) {  // lane's columns l + 32 j of the group
            float* d = partial + m * BN + 128 * group + lane;
            const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) d[32 * j] = w == 0 ? vv[j] : d[32 * j] + vv[j];
          } else {  // lane's columns 4 l .. 4 l + 3 of the group
            float4* d = part4 + m * (BN / 4) + group * 32 + lane;
            if (w == 0) {
              *d = v;
            } else {
              const float4 o = *d;
              *d = make_float4(o.x + v.x, o.y + v.y, o.z + v.z, o.w + v.w);
            }
          }
        }
      }
      __syncthreads();
    }

    constexpr int kTile4 = kSBM * BN / 4;  // float4s in a partial tile
    const float4* part4 = reinterpret_cast<const float4*>(partial);
    float4* ws4 = reinterpret_cast<float4*>(p.ws);
    if (k1 < KT) {  // contributor: partial tile to slot b, then the flag
      for (int i = threadIdx.x; i < kTile4; i += S::kThreads)
        if (SG_CHK(SG_IN(static_cast<int64_t>(b) * kTile4 + i, p.ws_slots * kTile4), p.status))
          ws4[static_cast<int64_t>(b) * kTile4 + i] = part4[i];
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0 && SG_CHK(SG_IN(b, p.ws_slots), p.status)) ptx::st_release_gpu(p.flags + b, p.epoch);
      continue;
    }
    int c_first = b;
    if (k0 > 0) {  // finisher: wait for the CTAs holding this slab's earlier slices
      const int64_t x0 = static_cast<int64_t>(slab) * KT;
      c_first = static_cast<int>(((x0 + 1) * G - 1) / U);
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
      if (__syncthreads_or(timed_out)) c_first = b;  // give up on the partials; the status word says why
    }
    // own partial, then the contributors' in CTA order; then the epilogue
    if constexpr (BT || BATCHED) {
      // one output float4 at a time: holding every output's reads at once
      // spills registers in these forms and measured slower
      for (int i = threadIdx.x; i < kTile4; i += S::kThreads) {
        float4 v = part4[i];
        for (int c = c_first; c < b; ++c) {
          const float4 o = SG_CHK(SG_IN(static_cast<int64_t>(c) * kTile4 + i, p.ws_slots * kTile4), p.status)
                               ? __ldcg(&ws4[static_cast<int64_t>(c) * kTile4 + i])
                               : make_float4(0.f, 0.f, 0.f, 0.f);
          v.x += o.x;
          v.y += o.y;
          v.z += o.z;
          v.w += o.w;
        }
        const int m = (4 * i) / BN;
        const int n = n0 + (4 * i) % BN;
        if (m < p.M) {
          float* crow = Cz + static_cast<int64_t>(m) * p.ldc;
          const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (n + j < p.N) crow[n + j] = p.beta == 0.f ? p.alpha * vv[j] : fmaf(p.alpha, vv[j], p.beta * crow[n + j]);
          }
        }
      }
      __syncthreads();  // the next piece rewrites `partial`
      if (threadIdx.x == 0)
        for (int c = c_first; c < b; ++c)
          if (SG_CHK(SG_IN(c, p.ws_slots), p.status)) *reinterpret_cast<volatile unsigned int*>(p.flags + c) = 0u;
      continue;
    }
    // Every global read (a contributor's partials, then C) is issued for all
    // of this thread's outputs before any is used or C is written, so the
    // fixup costs one round trip per contributor and one for C (measured at
    // 16 x 16384 x 8192, beta 1: 0.1071 ms against 0.1092).
    constexpr int kIt = kTile4 / S::kThreads;
    static_assert(kTile4 % S::kThreads == 0, "whole float4s per thread");
    float4 v[kIt];
#pragma unroll
    for (int t = 0; t < kIt; ++t) v[t] = part4[threadIdx.x + t * S::kThreads];
    for (int c = c_first; c < b; ++c) {
      float4 o[kIt];
#pragma unroll
      for (int t = 0; t < kIt; ++t)
        o[t] = SG_CHK(SG_IN(static_cast<int64_t>(c) * kTile4 + threadIdx.x + t * S::kThreads, p.ws_slots * kTile4),
                      p.status)
                   ? __ldcg(&ws4[static_cast<int64_t>(c) * kTile4 + threadIdx.x + t * S::kThreads])
                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int t = 0; t < kIt; ++t) {
        v[t].x += o[t].x;
        v[t].y += o[t].y;
        v[t].z += o[t].z;
        v[t].w += o[t].w;
      }
    }
    const bool vec_c = (reinterpret_cast<uintptr_t>(Cz) & 15) == 0 && (p.ldc & 3) == 0;
    float4 old[kIt];
    if (p.beta != 0.f) {
#pragma unroll
      for (int t = 0; t < kIt; ++t) {
        const int i = threadIdx.x + t * S::kThreads;
        const int m = (4 * i) / BN;
        const int n = n0 + (4 * i) % BN;
        old[t] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (m < p.M) {
          const float* crow = Cz + static_cast<int64_t>(m) * p.ldc + n;
          if (vec_c && n + 3 < p.N) {
            old[t] = *reinterpret_cast<const float4*>(crow);
          } else {
            if (n < p.N) old[t].x = crow[0];
            if (n + 1 < p.N) old[t].y = crow[1];
            if (n + 2 < p.N) old[t].z = crow[2];
            if (n + 3 < p.N) old[t].w = crow[3];
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kIt; ++t) {
      const int i = threadIdx.x + t * S::kThreads;
      const int m = (4 * i) / BN;
      const int n = n0 + (4 * i) % BN;
      if (m < p.M) {
        float* crow = Cz + static_cast<int64_t>(m) * p.ldc + n;
        const float vv[4] = {v[t].x, v[t].y, v[t].z, v[t].w};
        const float oo[4] = {old[t].x, old[t].y, old[t].z, old[t].w};
        float r[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) r[j] = p.beta == 0.f ? p.alpha * vv[j] : fmaf(p.alpha, vv[j], p.beta * oo[j]);
        if (vec_c && n + 3 < p.N) {
          *reinterpret_cast<float4*>(crow) = make_float4(r[0], r[1], r[2], r[3]);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (n + j < p.N) crow[j] = r[j];
        }
      }
    }
    __syncthreads();  // the next piece rewrites `partial`
    // every thread has read the contributors' partials: clear their flags, so
    // each run (a replayed graph included, whose epoch is fixed) starts from zero
    if (threadIdx.x == 0)
      for (int c = c_first; c < b; ++c)
          if (SG_CHK(SG_IN(c, p.ws_slots), p.status)) *reinterpret_cast<volatile unsigned int*>(p.flags + c) = 0u;
  }
  // After a failed wait, copies still in flight land before the CTA's shared
  // memory is released.  Every warp that sees the failure drains what has been
  // issued so far; a copy issued later is drained by the warp that issued it
  // (or was waited on by every warp, when no warp saw the failure).
  if (lane == 0 && *reinterpret_cast<volatile int*>(&s_failed))
    ptx::drain_ring_released(bar_full, 8, released, S::kWarps, STAGES, total_it, p.timeout_ns);
}

template <int BN, int GW, int STAGES, int MINB, bool EVICT_FIRST>
struct SkinnySkVariant {
  using S = SkinnyShape<BN, GW, STAGES>;
  static constexpr auto kernel = sgemm_skinny_sk_kernel<BN, GW, STAGES, MINB, EVICT_FIRST, false>;
  static constexpr auto kernel_bt = sgemm_skinny_sk_kernel<BN, GW, STAGES, MINB, EVICT_FIRST, true>;
  static constexpr auto kernel_batched = sgemm_skinny_sk_kernel<BN, GW, STAGES, MINB, EVICT_FIRST, false, true>;
  static constexpr auto kernel_bt_batched = sgemm_skinny_sk_kernel<BN, GW, STAGES, MINB, EVICT_FIRST, true, true>;
  static cudaError_t prepare() {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel_bt, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kernel_batched, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kernel_bt_batched, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
    return e;
  }
  static cudaError_t occupancy(int* ctas) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, kernel, S::kThreads, S::kSmemBytes);
  }
  static cudaError_t launch(const LaunchArgs& a, cudaStream_t stream) {
    SkinnySkParams p;
    p.C = a.C;
    p.ldc = a.ldc;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.alpha = a.alpha;
    p.beta = a.beta;
    p.status = a.status;
    p.timeout_ns = a.timeout_ns;
    p.ws = a.ws;
    p.flags = a.flags;
    p.ws_slots = a.ws_slots;
    p.epoch = a.epoch;
    p.batch = a.batch > 1 ? a.batch : 1;
    p.stride_c = a.stride_c;
    p.a_batched = a.batch > 1 && a.stride_a != 0;
    p.b_batched = a.batch > 1 && a.stride_b != 0;
    if (p.batch > 1 && a.b_trans) {
      kernel_bt_batched<<<a.grid, S::kThreads, S::kSmemBytes, stream>>>(a.tmA, a.tmB, p);
    } else if (p.batch > 1) {
      kernel_batched<<<a.grid, S::kThreads, S::kSmemBytes, stream>>>(a.tmA, a.tmB, p);
    } else if (a.b_trans) {
      kernel_bt<<<a.grid, S::kThreads, S::kSmemBytes, stream>>>(a.tmA, a.tmB, p);
    } else {
      kernel<<<a.grid, S::kThreads, S::kSmemBytes, stream>>>(a.tmA, a.tmB, p);
    }
    return cudaGetLastError();
  }
  static Variant describe(const char* name) {
    Variant v{name, kKindSkinny, kSBM, BN, kSBK, STAGES, 1, S::kThreads, S::kSmemBytes, 128, &prepare, &occupancy,
              &launch, 0, 1, 1};  // stream-K, strided batches
    v.b_trans_ok = 1;  // reads B given transposed (N x K) itself
    return v;
  }
};

template <int BN, int GW, int STAGES, int MINB, bool EVICT_FIRST, bool PAIRA = false, int PERSIST = 0>
struct SkinnyVariant {
  using S = SkinnyShape<BN, GW, STAGES>;
  static constexpr auto kernel = sgemm_skinny_kernel<BN, GW, STAGES, MINB, EVICT_FIRST, PAIRA>;
  static cudaError_t prepare() {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
  }
  static cudaError_t occupancy(int* ctas) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, kernel, S::kThreads, S::kSmemBytes);
  }
  static cudaError_t launch(const LaunchArgs& a, cudaStream_t stream) {
    SkinnyParams p;
    p.C = a.C;
    p.ldc = a.ldc;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.alpha = a.alpha;
    p.beta = a.beta;
    p.status = a.status;
    p.timeout_ns = a.timeout_ns;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.grid), 1, 1);
    cfg.blockDim = dim3(S::kThreads, 1, 1);
    cfg.dynamicSmemBytes = S::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(a.split_k);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, a.tmA, a.tmB, p);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  static Variant describe(const char* name) {
    return Variant{name, kKindSkinny, kSBM, BN, kSBK, STAGES, 1, S::kThreads, S::kSmemBytes, 128, &prepare, &occupancy,
                   &launch, PERSIST};
  }
};

const Variant kSkinnyVariants[] = {
    SkinnyVariant<128, 4, 3, 3, true, true>::describe("skinny_16x128x32_w4_s3_b3_ef_pa"),
    SkinnySkVariant<128, 4, 3, 3, true>::describe("skinny_sk_16x128x32_w4_s3_b3_ef"),
    SkinnySkVariant<128, 4, 4, 3, true>::describe("skinny_sk_16x128x32_w4_s4_b3_ef"),
    SkinnySkVariant<128, 4, 3, 3, false>::describe("skinny_sk_16x128x32_w4_s3_b3"),
    SkinnyVariant<128, 4, 3, 3, true, false>::describe("skinny_16x128x32_w4_s3_b3_ef"),
    SkinnyVariant<128, 4, 3, 3, true, true, 1>::describe("skinny_16x128x32_w4_s3_b3_ef_pa_persist"),
    SkinnyVariant<128, 4, 3, 3, false, true>::describe("skinny_16x128x32_w4_s3_b3_pa"),
};

}  // namespace

const Variant* skinny_variants(int* count) {
  *count = static_cast<int>(sizeof(kSkinnyVariants) / sizeof(kSkinnyVariants[0]));
  return kSkinnyVariants;
}

}  // namespace sgemm
