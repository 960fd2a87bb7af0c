// kernels.h -- host-side interface between the C-ABI layer (sgemm_api.cu)
// and the kernel translation units.  Internal; not installed.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sgemm {

enum VariantKind : int {
  kKindGeneric = 0,  // scalar predicated loads, any alignment / leading dimension
  kKindTma = 1,      // TMA-fed multi-stage pipeline, needs 16-byte aligned A/B rows
  kKindSkinny = 2,   // small-M streaming kernel, needs 16-byte aligned A/B rows
  kKindCpa = 3,      // A by cp.async (transposed, any alignment), B by TMA (16-byte aligned rows)
  kKindTc = 4,       // tensor cores, operands split into two TF32 parts (any alignment; plan workspace)
  kKindTcFused = 5,  // tensor cores, the split inside the GEMM kernel (A and B read by TMA as stored)
  // 6 is kKindGemv, the M <= 4 kernels (kernel_gemv.h)
  kKindTiny = 7,     // small C tiles, whole K-panels in shared memory (any alignment; K <= bk)
};

// Everything one launch needs.  Tensor maps are encoded by the caller per
// run (they hold the A/B addresses) and passed by value to the kernel.
struct LaunchArgs {
  const float* A;
  const float* B;
  float* C;
  int64_t lda, ldb, ldc;
  int M, N, K;
  float alpha, beta;
  CUtensorMap tmA;       // used by TMA-fed variants only
  CUtensorMap tmB;
  int grid;              // CTAs to launch (persistent variants: <= tiles)
  int split_k;           // skinny variant: CTAs per cluster along K
  // stream-K tail (variants with streamk = 1; sk_iters == 0 disables it)
  int dp_waves;
  int64_t sk_iters;
  float* ws;
  unsigned int* flags;
  unsigned int epoch;
  int64_t ws_slots;      // stream-K: partial tiles (and flags) ws holds; gemv: floats ws holds
  unsigned int* status;  // per-device status word (error bits)
  uint64_t timeout_ns;   // limit for every in-kernel wait
  // split-TF32 tensor-core variants: A_hi, A_lo (M x split_ld), then B_hi,
  // B_lo transposed (N x split_ld) in one plan-owned buffer, described by
  // tmA (A_hi), tmA2 (A_lo), tmB (B_hi), tmB2 (B_lo)
  float* split;
  int64_t split_ld;
  CUtensorMap tmA2;
  CUtensorMap tmB2;
  // split-TF32 variants read A and B themselves: a_trans = 1 means A is
  // stored K x M (row-major, lda), b_trans = 1 means B is stored N x K
  int a_trans;
  int b_trans;
  // strided batch (variants with batched = 1): product z reads A + z*stride_a,
  // B + z*stride_b and writes C + z*stride_c, z = 0 .. batch-1
  int batch;
  int64_t stride_a, stride_b, stride_c;
};

struct Variant {
  const char* name;
  int kind;
  int bm, bn, bk;        // CTA tile (bk: k-slice per pipeline stage)
  int stages;            // shared-memory pipeline depth (1 = register-staged)
  int ffma2;             // 1: inner product issued as paired fp32 FMAs
  int threads;           // threads per CTA
  int smem_bytes;        // dynamic shared memory per CTA
  int tma_swizzle_a;     // 0 none, 64/128: A tile swizzle; -1: the variant takes no tensor maps
  // set kernel attributes for the current device (idempotent)
  cudaError_t (*prepare)();
  // resident CTAs per SM for this variant on the current device
  cudaError_t (*occupancy)(int* ctas_per_sm);
  cudaError_t (*launch)(const LaunchArgs& args, cudaStream_t stream);
  int persistent;        // few-row kernels: 1 = clusters walk several column slabs
  int streamk;           // 1: the kernel can split its tail tiles along K (workspace per plan)
  int batched;           // 1: runs strided batches (TMA variants: 3-D tensor maps, batch outermost)
  int b_trans_ok;        // 1: reads B given transposed (stored N x K) itself, LaunchArgs::b_trans = 1
  int a_trans_ok;        // 1: reads A given transposed (stored K x M) itself, LaunchArgs::a_trans = 1
};

// Variant tables, one per kernel translation unit.
const Variant* generic_variants(int* count);
const Variant* tma_variants_a(int* count);
const Variant* tma_variants_b(int* count);
const Variant* tma_variants_c(int* count);
const Variant* skinny_variants(int* count);
const Variant* cpa_variants(int* count);
const Variant* tmat_variants(int* count);
const Variant* tc_variants(int* count);
const Variant* tiny_variants(int* count);

// C = beta * C (K == 0 or alpha == 0), any leading dimension; `batch`
// matrices stride_c apart.
cudaError_t launch_scale(float* C, int64_t ldc, int M, int N, float beta, cudaStream_t stream, int batch = 1,
                         int64_t stride_c = 0);

// out (cols x rows, ld_out) = in (rows x cols, ld_in) transposed, for
// `batch` products stride_in / stride_out apart.
cudaError_t launch_transpose(const float* in, int64_t ld_in, int rows, int cols, float* out, int64_t ld_out,
                             cudaStream_t stream, int batch = 1, int64_t stride_in = 0, int64_t stride_out = 0);
// dst = src with rows padded to 16-byte multiples (ldd % 4 == 0, dst 16-byte
// aligned); src may have any leading dimension and alignment.
cudaError_t launch_repack(const float* src, int64_t lds, int rows, int cols, float* dst, int64_t ldd,
                          cudaStream_t stream);

// One-thread kernel that waits on a barrier phase nothing completes.
cudaError_t launch_wait_selftest(unsigned int* status, uint64_t timeout_ns, cudaStream_t stream);

// Status bits written by kernels.
enum : unsigned int {
  kStatusTimeoutFull = 1u,    // a consumer gave up waiting for a filled stage
  kStatusTimeoutEmpty = 2u,   // the producer gave up waiting for a free stage
  kStatusTimeoutSelftest = 4u,
  kStatusTimeoutCluster = 8u,
};

}  // namespace sgemm
