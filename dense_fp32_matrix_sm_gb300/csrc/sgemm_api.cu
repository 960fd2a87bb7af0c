// sgemm_api.cu -- the C ABI declared in include/sgemm.h: argument checks,
// the per-shape config table, TMA descriptor encoding, launches, the
// per-device status word.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <atomic>
#include <map>
#include <tuple>
#include <mutex>
#include <new>
#include <vector>

#include "api_internal.h"
#include "kernel_gemv.h"
#include "checked.cuh"
#include "kernels.h"
#include "sgemm.h"

using namespace sgemm;

static_assert(kKindGemv != kKindGeneric && kKindGemv != kKindTma && kKindGemv != kKindSkinny &&
                  kKindGemv != kKindCpa && kKindGemv != kKindTc && kKindGemv != kKindTcFused && kKindGemv != kKindTiny,
              "every variant kind is distinct");

struct sgemm_plan_s {
  int64_t M, N, K, lda, ldb, ldc;
  int64_t batch, stride_a, stride_b, stride_c;  // strided batch (batch 1: a single product)
  int device;
  int num_sms;
  int config_id;
  int generic_id;   // scalar-load variant used when A or B is not 16-byte aligned
  int ctas_per_sm;
  int grid;
  int split;        // CTAs per cluster along K (skinny variants), else 1
  uint64_t wait_floor_ns;  // the plan's work-based floor for in-kernel wait limits
  int64_t tiles;
  // stream-K tail (tmat variants): dp_waves full waves, then sk_iters k-slices
  // split over the grid; ws/flags are device memory owned by the plan.
  int dp_waves;
  int64_t sk_iters;
  float* ws;
  unsigned int* flags;
  int64_t ws_slots;  // what ws holds: partial tiles (and flags) for stream-K, floats for gemv
  std::atomic<unsigned int> epoch;
  // split-TF32 tensor-core variants: operand buffer and its four tensor maps
  float* tc_split;
  int64_t tc_split_ld;
  CUtensorMap tc_maps[4];
  // sgemm_plan_ex: the problem as given, reduced to row-major (after the
  // column-major swap of A and B); ta / tb: that operand is stored
  // transposed (A as K x M, B as N x K) with leading dimension ex_lda /
  // ex_ldb.  ex_wa / ex_wb: plan-owned buffers the run transposes it into
  // (none for the split-TF32 variants, which read both layouts).
  int ex_order;
  int ex_swap;
  int ex_ta, ex_tb;
  int64_t ex_lda, ex_ldb;
  float* ex_wa;
  float* ex_wb;
  int ex_native_tb;  // the variant reads B given transposed (N x K) itself: no ex_wb
  int ex_native_ta;  // the variant reads A given transposed (K x M) itself: no ex_wa
  // the caller's batch strides of the stored operands (after the swap); the
  // kernels' own (stride_a / stride_b) differ when an operand goes through ex_wa / ex_wb
  int64_t ex_stride_a, ex_stride_b;
  // An untransposed operand whose rows are not 16-byte multiples (lda or ldb
  // not a multiple of 4) is copied each run into rp_a / rp_b, rows padded
  // to lda / ldb (the kernels' view); ex_lda / ex_ldb keep the caller's.
  float* rp_a;
  float* rp_b;
  // sgemm_run_host_pipelined: copy streams (host to device, device to host)
  // and, per buffer set b, events loaded / computed / stored; made on first use
  std::mutex pipe_mutex;
  bool pipe_ready;
  cudaStream_t pipe_h2d, pipe_d2h;
  cudaEvent_t pipe_ev[2][3];
};

// Per-device status word written by kernels (timeouts).  Its device address
// is looked up once per device with that device current.
__device__ unsigned int g_sgemm_status_word;

namespace sgemm {
// the 64-row instantiations of the transposed-A kernel (tmat_variants_rows.cu)
const Variant* tmat_rows_variants(int* count);
}  // namespace sgemm

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 4000000000ull;

std::atomic<uint64_t> g_timeout_ns{kDefaultTimeoutNs};

// A launch's waits may legitimately last as long as the launch itself: a
// stream-K finisher waits for contributors that run a K-range of their own
// after their data-parallel tiles.  So the limit never goes below the time
// the whole product would take at kFloorFlopsPerSm FLOP/s per SM, about
// 1/45 of what the FFMA kernels sustain on GB300 (450 GFLOP/s per SM).
constexpr double kFloorFlopsPerSm = 1e10;

uint64_t work_floor_ns(int64_t M, int64_t N, int64_t K, int64_t batch, int sms) {
  if (M <= 0 || N <= 0 || K <= 0 || sms <= 0) return 0;
  const double flops = 2.0 * static_cast<double>(M) * static_cast<double>(N) * static_cast<double>(K) *
                       static_cast<double>(batch > 1 ? batch : 1);
  const double ns = flops / (static_cast<double>(sms) * kFloorFlopsPerSm) * 1e9;
  return ns >= 1.8e19 ? UINT64_C(18000000000000000000) : static_cast<uint64_t>(ns);
}

uint64_t wait_limit_ns(uint64_t floor_ns) {
  const uint64_t t = g_timeout_ns.load(std::memory_order_relaxed);
  return t > floor_ns ? t : floor_ns;
}
std::mutex g_status_mutex;
unsigned int* g_status_addr[kMaxDevices] = {};

struct Registry {
  std::vector<const Variant*> all;
  int first_generic = -1;
  Registry() {
    int n = 0;
    const Variant* v = generic_variants(&n);
    first_generic = static_cast<int>(all.size());
    for (int i = 0; i < n; ++i) all.push_back(&v[i]);
    for (auto fn : {&tma_variants_a, &tma_variants_b, &tma_variants_c}) {
      v = fn(&n);
      for (int i = 0; i < n; ++i) all.push_back(&v[i]);
    }
    v = skinny_variants(&n);
    for (int i = 0; i < n; ++i) all.push_back(&v[i]);
    v = cpa_variants(&n);
    for (int i = 0; i < n; ++i) all.push_back(&v[i]);
    v = tmat_variants(&n);
    for (int i = 0; i < n; ++i) all.push_back(&v[i]);
    v = tmat_rows_variants(&n);
    for (int i = 0; i < n; ++i) all.push_back(&v[i]);
    v = tc_variants(&n);
    for (int i = 0; i < n; ++i) all.push_back(&v[i]);
    v = gemv_variants(&n);
    for (int i = 0; i < n; ++i) all.push_back(&v[i]);
    v = tiny_variants(&n);
    for (int i = 0; i < n; ++i) all.push_back(&v[i]);
  }
};

const Registry& registry() {
  static Registry r;
  return r;
}

int find_variant(const char* name) {
  const Registry& r = registry();
  for (size_t i = 0; i < r.all.size(); ++i)
    if (strcmp(r.all[i]->name, name) == 0) return static_cast<int>(i);
  return -1;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

sgemm_status_t status_addr(int device, unsigned int** out) {
  if (device < 0 || device >= kMaxDevices) return SGEMM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_status_mutex);
  if (!g_status_addr[device]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sgemm_status_word) != cudaSuccess) return SGEMM_ERR_CUDA;
    g_status_addr[device] = static_cast<unsigned int*>(p);
  }
  *out = g_status_addr[device];
  return SGEMM_OK;
}

// Elements from the first to the last element of a stored matrix of `outer`
// lines of `inner` elements, `ld` apart (0 when it is empty).  Computed in
// double so that no argument overflows it.
double span_elems(int64_t outer, int64_t inner, int64_t ld) {
  return outer > 0 && inner > 0 ? static_cast<double>(outer - 1) * static_cast<double>(ld) + static_cast<double>(inner)
                                : 0.0;
}

// The largest span a stored matrix (or a strided batch of them) may cover:
// 2^40 elements, 4 TiB of floats, beyond any device memory.  Larger
// arguments cannot describe real buffers; refusing them keeps every element
// offset, workspace size and address computed from them far inside int64.
constexpr double kMaxSpan = 1099511627776.0;

sgemm_status_t check_dims(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc) {
  if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_ARG;
  if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1)) return SGEMM_ERR_INVALID_ARG;
  const int64_t lim = 0x7fffffff;
  if (M > lim || N > lim || K > lim) return SGEMM_ERR_UNSUPPORTED;
  // element offsets must fit in int64 with room to spare
  if (lda > (int64_t(1) << 40) || ldb > (int64_t(1) << 40) || ldc > (int64_t(1) << 40)) return SGEMM_ERR_UNSUPPORTED;
  if (span_elems(M, K, lda) > kMaxSpan || span_elems(K, N, ldb) > kMaxSpan || span_elems(M, N, ldc) > kMaxSpan)
    return SGEMM_ERR_UNSUPPORTED;
  return SGEMM_OK;
}

// A strided batch of `batch` matrices of span `one`, `stride` apart.
double batch_span(int64_t batch, int64_t stride, double one) {
  return batch > 1 ? static_cast<double>(batch - 1) * static_cast<double>(stride) + one : one;
}

// Products the M <= 4 kernels take: one to four rows (any alignment, any
// leading dimension or batch stride), K in at most 65535 chunks of 1024, and
// column indexes with room to spare in 32 bits.
bool gemv_shape(int64_t M, int64_t N, int64_t K, int64_t batch) {
  return M <= 4 && N <= (int64_t(1) << 30) && K <= int64_t(65535) * 1024 && batch <= 65535;
}

// Products the table sends to the five-to-sixteen-row matrix-vector kernel
// (gemv_16x1024): B as stored, at least 16 MB of B over the batch (a stream
// worth keeping at full bandwidth), any alignment, leading dimension or
// batch stride.  Measured against the few-row stream-K kernel (L2 clean,
// median of 30-40): 16 x 16384 x 8192 0.090 ms against 0.102; 8 x 16384 x
// 8192 0.084 against 0.105; 12 x 8192 x 4096 0.037 against 0.039; 16 x 4096
// x 4096 0.027 against 0.029; batches 8 x (16 x 8192 x 4096) 0.181 against
// 0.284, 32 x (16 x 4096 x 1024) 0.115 against 0.125, 16 x (8 x 16384 x
// 2048) 0.323 against 0.414, 64 x (12 x 4096 x 1024) 0.209 against 0.216.
bool rows_shape(int64_t M, int64_t N, int64_t K, int64_t batch, int b_trans) {
  return !b_trans && M > 4 && M <= 16 && std::max<int64_t>(batch, 1) * N * K >= (int64_t(1) << 22) &&
         N <= (int64_t(1) << 30) && K <= int64_t(65535) * 640 && batch <= 65535;
}

// Products the tiny kernel takes from the table: more than 16 rows (fewer
// go to the few-row kernels, which do not fill 32-row tiles with padding),
// and either K <= 512 with at most two of its 32 x 32 tiles per SM (over
// the whole batch: one wave), or at most 32 rows with rows that allow its
// 16-byte copies (`rows16`: lda, ldb multiples of 4) and at least 3/4 of a
// tile per SM (it does not split K).  Measured against the 128-row kernels
// and cuBLAS (TFLOP/s, L2 flushed): 128^3 0.54 (cuBLAS 0.41), 256^3 4.1
// (2.7), 384^3 11.1 (7.5), 512^3 18.8 (14.4), 512 x 512 x 128 8.2 (6.3),
// 608 x 512 x 512 22.2 (16.9), 200 x 130 x 100 with odd ldb 0.64 (0.59);
// 32 x 4096 x 4096 21.9 (128 x 128 tiles 11.6, cuBLAS 16.6), 24 x 8192 x
// 4096 21.3 (10.9, 15.7), 32 x 9728 x 1024 26.0 (12.3, 20.8).
bool tiny_shape(int64_t M, int64_t N, int64_t K, int64_t batch, int num_sms, bool rows16) {
  const int64_t tiles = std::max<int64_t>(batch, 1) * ((M + 31) / 32) * ((N + 31) / 32);
  if (M <= 16) return false;
  if (K <= 512) return tiles <= 2 * static_cast<int64_t>(num_sms);
  return rows16 && M <= 32 && 4 * tiles >= 3 * static_cast<int64_t>(num_sms);
}

// Products the 64 x 64 form of the tiny kernel takes from the table: more
// than 16 rows, K <= 512 and at most two of its tiles per SM over the whole
// batch (one wave, no split along K), when the tiny kernel's rule does not
// apply; and either at most one tile per SM, a k loop of at most 256, or
// at least 0.9 of the two-per-SM slots filled (between those the SMs that
// get two tiles set the time).  Measured (TFLOP/s, L2 flushed; the 128-row
// choice and cuBLAS in brackets): 768 x 768 x 512 29.5 (25.8, 31.9), 768 x
// 768 x 256 21.2 (16.0, 22.7), 1024 x 512 x 512 26.3 (23.4, 26.3), 1024 x
// 1024 x 256 26.3 (23.8, 29.1), 2048 x 512 x 256 26.3 (23.4, 29.0), 1088 x
// 1088 x 448 34.6 (32.0, 39.5), 1536 x 768 x 384 34.1 (33.1, 39.5); left
// to the 128-row tiles: 1024 x 1024 x 512 (32.8 against 34.4), 896 x 896 x
// 512 (25.1 against 32.8), 960 x 960 x 384 (26.7 against 28.2).
bool small_shape(int64_t M, int64_t N, int64_t K, int64_t batch, int num_sms) {
  const int64_t tiles = std::max<int64_t>(batch, 1) * ((M + 63) / 64) * ((N + 63) / 64);
  const int64_t sms = num_sms;
  return M > 16 && K <= 512 && tiles <= 2 * sms && (tiles <= sms || K <= 256 || 5 * tiles >= 9 * sms);
}

// a_span / b_span: elements one stored A / B spans (-1: M*lda / K*ldb, an
// operand stored as the kernels read it)
bool variant_supports(const Variant* v, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                      int64_t batch = 1, int64_t stride_a = 0, int64_t stride_b = 0, int64_t a_span = -1,
                      int64_t b_span = -1) {
  if (v->kind == kKindGemv) return gemv_takes(v, M, N, K, batch);
  // K streamed through a shared-memory ring; tiles on grid x (columns) and y (rows)
  if (v->kind == kKindTiny) return batch <= 65535 && (M + v->bm - 1) / v->bm <= 65535;
  if (batch > 1) {
    if (!v->batched) return false;
    if (v->kind == kKindGeneric) return batch <= 65535;
    // 3-D tensor maps: 16-byte batch strides that do not overlap the matrices,
    // or 0 for an operand shared by every product
    if (a_span < 0) a_span = M * lda;
    if (b_span < 0) b_span = K * ldb;
    if (stride_a % 4 != 0 || stride_b % 4 != 0 || (stride_a != 0 && stride_a < a_span) ||
        (stride_b != 0 && stride_b < b_span))
      return false;
  }
  if (v->kind == kKindGeneric) return true;
  // split-TF32: the split kernels read A and B with plain loads (any layout).
  // The split leaves ~3 * 2^-22 |a b| per product; K >= 16 keeps that well
  // inside the acceptance bound 4 K 2^-24 |A||B|.
  if (v->kind == kKindTc) return K >= 16;
  // the fused form reads A and B by TMA as stored: 16-byte rows (the stored
  // leading dimensions are checked again by sgemm_plan_ex)
  if (v->kind == kKindTcFused) return K >= 16 && lda % 4 == 0 && ldb % 4 == 0;
  if (ldb % 4 != 0) return false;  // TMA row strides must be multiples of 16 bytes
  if (v->kind == kKindCpa) return true;  // A is copied 4 bytes at a time: any lda
  if (lda % 4 != 0) return false;
  if (v->kind == kKindSkinny) {
    // the register-streaming form reads whole float4s of B: N must be a multiple of 4
    return M <= v->bm && (v->tma_swizzle_a >= 0 || N % 4 == 0);
  }
  return true;
}

// Tile width for the transposed-A family, over `batch` products of M x N x K.
// Measured on GB300 with stream-K (which removes the partial-wave loss once
// there is at least one full wave, and with fewer tiles than CTA slots
// splits every tile along K once every CTA gets a k-slice):
//  * 128 x 256 tiles from a third of a wave of them on (with stream-K
//    splitting the tiles that do not fill a wave), K >= 256: 66.3-69.6
//    TFLOP/s from 2560^3 up, 1-2% above 128 x 128; below a wave (measured
//    against 128 x 128): 1280^3 53.9 vs 52.5, 1536^3 59.0 vs 58.0, 1792^3
//    62.4 vs 58.5, 2048^3 65.5 vs 61.2, 2048 x 1024 x 2048 61.6 vs 59.1,
//    2048 x 2048 x 512 53.8 vs 52.4; 1024 x 2048 x 1024 53.1 vs 53.8 and
//    1152^3 (45 tiles) 42.7 vs 48.2 stay on the other side of the line;
//  * 128 x 128 tiles down to half a wave (1536^3: 61.2 vs 56.2 for 128 x 64),
//    or below that when every tile can be split along K: 1024^3 45.8 vs
//    43.6, 512 x 512 x 8192 52.3 vs 49.8, 2048 x 640 x 2048 58.1 vs 53.4;
//  * otherwise 128 x 64 tiles two to an SM (384^3: 4.4 vs 3.1);
//  * never a tile more than twice as wide as N: 64 x (512 x 64 x 512) ran
//    14.5 TFLOP/s on 256-wide tiles, three quarters of each tile empty.
const char* tmat_choice(int64_t M, int64_t N, int64_t K, int64_t batch, int num_sms) {
  const int64_t wide_tiles = batch * ((M + 127) / 128) * ((N + 255) / 256);
  const int64_t square_tiles = batch * ((M + 127) / 128) * ((N + 127) / 128);
  const int64_t narrow_tiles = batch * ((M + 127) / 128) * ((N + 63) / 64);
  const int64_t KT = (K + 31) / 32;
  // up to 64 rows: 64-row tiles, so at most half of a tile is padding (the
  // 128-row tiles' is three quarters at 32 rows).  Measured (TFLOP/s, L2
  // flushed; 128-row table choice, cuBLAS): 64 x 16384 x 8192 62.6 (33.7,
  // 55.9), 64 x 4096 x 4096 41.6 (23.3, 21.0), 48 x 4096 x 4096 31.2 (17.4,
  // 15.7), 64 x 9728 x 2048 47.5 (27.5, 41.5), 64 x 8192 x 8192 51.0 (30.6,
  // 37.8).  Up to 32 rows with enough 32-column tiles the tiny kernel's
  // rule comes first (32 x 16384 x 8192: 30.4 there, 31.4 here).
  if (M <= 64) return "tmat_64x256x32_s3_b1";
  // 128 x 256 tiles from 0.3 of a wave on (20 wide tiles per 6 SMs), unless
  // the last column of tiles would be mostly empty below N = 4096 (1408^3:
  // 51.4 TFLOP/s against 55.6 on 128 x 128), or a 256-deep k loop with less
  // than 3/4 of a wave (1536 x 1536 x 256: 34.3 against 39.3; 2048 x 1024 x
  // 256: 30.2 against 36.7; 2048^2 x 256 with a whole wave: 45.6 against 43.7)
  const bool wide_fits = N % 256 == 0 || N % 256 > 128 || N >= 4096;
  if (N > 128 && wide_fits && 20 * wide_tiles >= 6 * num_sms && K >= 256 &&
      (K >= 512 || 4 * wide_tiles >= 3 * num_sms))
    return "tmat_128x256x32_s3_b1";
  // few tiles and a short k loop: 128 x 64 tiles split into three or more
  // pieces along K each (api_streamk_schedule) beat 128 x 128 tiles, whose
  // finishers add twice the bytes per contributor (512^3: 14.2 TFLOP/s
  // against 12.7; 640^3: 22.9 against 21.0; 256 x 256 x 2048: 10.7 against
  // 8.6); with a long k loop the larger tile wins (512 x 512 x 8192: 49.0
  // against 38.7)
  if (KT >= 2 && KT <= 64 && 3 * narrow_tiles <= num_sms) return "tmat_128x64x32_s3_b2";
  if (N > 64 && (2 * square_tiles >= static_cast<int64_t>(num_sms) ||
                 (KT >= 8 && square_tiles * KT >= static_cast<int64_t>(num_sms))))
    return "tmat_128x128x32_s4_b1";
  return "tmat_128x64x32_s3_b2";
}

// The per-shape config table.  Keys are shape classes; values are variant
// names.  The entries come from the measured sweeps on GB300.
const char* table_choice(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int num_sms, int64_t batch = 1,
                         int64_t stride_a = 0, int64_t stride_b = 0, int64_t a_span = -1, int64_t b_span = -1,
                         int b_trans = 0) {
  // one to four rows: B streamed once by plain loads, any layout
  if (gemv_shape(M, N, K, batch)) return "gemv_4x512";
  // five to sixteen rows of one product, B as stored: B streamed once
  // through per-warp cp.async rings, any layout
  if (rows_shape(M, N, K, batch, b_trans)) return "gemv_16x1024";
  // tiny products, and long-K products of 17 to 32 rows: 32 x 32 tiles, any layout
  if (tiny_shape(M, N, K, batch, num_sms, lda % 4 == 0 && ldb % 4 == 0)) return "tiny_32x32";
  // a short k loop and at most two 64 x 64 tiles per SM: the same ring with 64 x 64 tiles
  if (small_shape(M, N, K, batch, num_sms)) return "small_64x64";
  if (batch > 1) {
    // Strided batches run on the batched variants only: the transposed-A
    // family when TMA can take the layout (tile counts over the whole batch),
    // else the scalar-load kernel.
    if (a_span < 0) a_span = M * lda;
    if (b_span < 0) b_span = K * ldb;
    if (ldb % 4 != 0 || lda % 4 != 0 || stride_a % 4 != 0 || stride_b % 4 != 0 ||
        (stride_a != 0 && stride_a < a_span) || (stride_b != 0 && stride_b < b_span))
      return "generic_64x64x16";
    // few rows: the stream-K few-row kernel over (product, slab, k-slice)
    // units, instead of 128-row tiles that are 7/8 empty
    if (M <= 16) return "skinny_sk_16x128x32_w4_s3_b3_ef";
    return tmat_choice(M, N, K, batch, num_sms);
  }
  if (ldb % 4 != 0) return "generic_64x64x16";
  if (M <= 16 && lda % 4 == 0) {
    // Few rows: the stream-K form once there are enough (128-column slab,
    // 32-deep k-slice) units to keep one resident wave streaming and enough
    // slabs that each finisher adds only a few partial tiles.  Measured:
    // 16 x 16384 x 8192 0.109 ms against 0.124 for the cluster form;
    // 16 x 8192 x 4096 0.044 against 0.047; but 16 x 4096 x 8192 (32 slabs)
    // 0.046 against 0.039 and 16 x 4096 x 4096 0.036 against 0.026.
    const int64_t slabs = (N + 127) / 128;
    const int64_t units = slabs * ((K + 31) / 32);
    return slabs >= 64 && units >= 48 * static_cast<int64_t>(num_sms) ? "skinny_sk_16x128x32_w4_s3_b3_ef"
                                                                       : "skinny_16x128x32_w4_s3_b3_ef_pa";
  }
  if (lda % 4 != 0) return "cpa_128x128x32_s3_k8_b2";  // A copied 4 bytes at a time: any lda
  return tmat_choice(M, N, K, 1, num_sms);
}

// The table's variant for a product on `sms` SMs, after the padding-copy
// rule: TMA needs rows that are 16-byte multiples.  From 256^3 of work on,
// an operand without them is copied each run into a plan buffer with padded
// rows, so the table's TMA kernels can read it (measured at 4096^3, lda =
// 4097 ran 54.6 TFLOP/s on the cp.async kernel and ldb = 4097 29.8 on the
// scalar-load kernel, against 68.8 aligned).  *lda / *ldb become the padded
// leading dimensions when *rp_a / *rp_b are set.  Pure host arithmetic.
const char* plan_table_choice(int64_t M, int64_t N, int64_t K, int64_t* lda, int64_t* ldb, int sms, int64_t batch,
                              int64_t stride_a, int64_t stride_b, int64_t a_span, int64_t b_span, int b_trans,
                              bool* rp_a, bool* rp_b) {
  *rp_a = *rp_b = false;
  if (batch <= 1 && K > 0 && !gemv_shape(M, N, K, batch) &&
      !tiny_shape(M, N, K, batch, sms, *lda % 4 == 0 && *ldb % 4 == 0) && !rows_shape(M, N, K, batch, b_trans) &&
      static_cast<double>(M) * static_cast<double>(N) * static_cast<double>(K) >= 16777216.0) {
    *rp_a = *lda % 4 != 0;
    *rp_b = *ldb % 4 != 0;
    if (*rp_a) *lda = (K + 3) / 4 * 4;
    if (*rp_b) *ldb = (N + 3) / 4 * 4;
  }
  return table_choice(M, N, K, *lda, *ldb, sms, batch, stride_a, stride_b, a_span, b_span, b_trans);
}

// b_trans: the caller's B is stored transposed and a transpose buffer will
// hold it unless the chosen kernel reads it as stored (the table then
// prefers a kernel that does).
sgemm_status_t make_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int config_id,
                         sgemm_plan_t* out, int64_t batch = 1, int64_t stride_a = 0, int64_t stride_b = 0,
                         int64_t stride_c = 0, int64_t a_span = -1, int64_t b_span = -1, int b_trans = 0) {
  if (!out) return SGEMM_ERR_INVALID_ARG;
  sgemm_status_t st = check_dims(M, N, K, lda, ldb, ldc);
  if (st != SGEMM_OK) return st;
  const Registry& reg = registry();
  if (config_id >= static_cast<int>(reg.all.size())) return SGEMM_ERR_INVALID_ARG;

  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return SGEMM_ERR_CUDA;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return SGEMM_ERR_CUDA;

  const int64_t lda_caller = lda, ldb_caller = ldb;
  bool rp_a = false, rp_b = false;
  if (config_id < 0) {
    const char* forced = getenv("SGEMM_FORCE_CONFIG");
    if (forced && *forced) {
      config_id = find_variant(forced);
      if (config_id < 0) return SGEMM_ERR_INVALID_ARG;
    } else {
      config_id = find_variant(
          plan_table_choice(M, N, K, &lda, &ldb, sms, batch, stride_a, stride_b, a_span, b_span, b_trans, &rp_a, &rp_b));
      if (config_id < 0) config_id = reg.first_generic;
    }
  }
  const Variant* v = reg.all[config_id];
  if (!variant_supports(v, M, N, K, lda, ldb, batch, stride_a, stride_b, a_span, b_span))
    return SGEMM_ERR_UNSUPPORTED;
  if (v->kind != kKindGeneric && v->tma_swizzle_a >= 0 && !encode_fn()) return SGEMM_ERR_CUDA;

  unsigned int* status = nullptr;
  st = status_addr(device, &status);
  if (st != SGEMM_OK) return st;

  if (v->prepare() != cudaSuccess) return SGEMM_ERR_CUDA;
  int ctas = 0;
  if (v->occupancy(&ctas) != cudaSuccess || ctas < 1) return SGEMM_ERR_CUDA;
  const Variant* gv = reg.all[reg.first_generic];
  if (gv->prepare() != cudaSuccess) return SGEMM_ERR_CUDA;

  sgemm_plan_s* p = new (std::nothrow) sgemm_plan_s;
  if (!p) return SGEMM_ERR_NOMEM;
  p->M = M;
  p->N = N;
  p->K = K;
  p->lda = lda;
  p->ldb = ldb;
  p->ldc = ldc;
  p->batch = batch;
  p->stride_a = stride_a;
  p->stride_b = stride_b;
  p->ex_stride_a = stride_a;
  p->ex_stride_b = stride_b;
  p->stride_c = stride_c;
  p->device = device;
  p->num_sms = sms;
  p->config_id = config_id;
  p->generic_id = reg.first_generic;
  p->ctas_per_sm = ctas;
  p->tiles = ((M + v->bm - 1) / v->bm) * ((N + v->bn - 1) / v->bn) * batch;
  int64_t grid = p->tiles;
  p->split = 1;
  p->wait_floor_ns = work_floor_ns(M, N, K, batch, sms);
  p->dp_waves = 0;
  p->sk_iters = 0;
  p->ws = nullptr;
  p->ws_slots = 0;
  p->flags = nullptr;
  p->epoch.store(0);
  p->tc_split = nullptr;
  p->tc_split_ld = 0;
  p->ex_order = SGEMM_ROW_MAJOR;
  p->ex_swap = 0;
  p->ex_ta = p->ex_tb = 0;
  p->ex_lda = lda_caller;
  p->ex_ldb = ldb_caller;
  p->ex_wa = nullptr;
  p->ex_wb = nullptr;
  p->ex_native_tb = 0;
  p->ex_native_ta = 0;
  p->rp_a = nullptr;
  p->rp_b = nullptr;
  p->pipe_ready = false;
  // From here on every device buffer is stored in the plan as soon as it is
  // allocated, and a failure frees them all through sgemm_plan_destroy.
  auto fail = [&](sgemm_status_t e) {
    sgemm_plan_destroy(p);
    return e;
  };
  if ((rp_a && cudaMalloc(reinterpret_cast<void**>(&p->rp_a), sizeof(float) * M * lda) != cudaSuccess) ||
      (rp_b && cudaMalloc(reinterpret_cast<void**>(&p->rp_b), sizeof(float) * K * ldb) != cudaSuccess))
    return fail(SGEMM_ERR_CUDA);
  if (v->kind == kKindTma || v->kind == kKindCpa) {
    const int64_t slots = static_cast<int64_t>(sms) * ctas;
    const StreamKSchedule sk = api_streamk_schedule(p->tiles, (K + v->bk - 1) / v->bk, sms, ctas,
                                                    v->streamk && getenv("SGEMM_NO_STREAMK") == nullptr);
    grid = sk.grid;
    if (sk.sk_iters > 0) {
      p->dp_waves = sk.dp_waves;
      p->sk_iters = sk.sk_iters;
      const size_t ws_bytes = static_cast<size_t>(slots) * v->bm * v->bn * sizeof(float);
      p->ws_slots = slots;
      if (cudaMalloc(reinterpret_cast<void**>(&p->ws), ws_bytes) != cudaSuccess ||
          cudaMalloc(reinterpret_cast<void**>(&p->flags), static_cast<size_t>(slots) * sizeof(unsigned int)) !=
              cudaSuccess ||
          cudaMemset(p->flags, 0, static_cast<size_t>(slots) * sizeof(unsigned int)) != cudaSuccess)
        return fail(SGEMM_ERR_CUDA);
    }
  } else if (v->kind == kKindSkinny && v->streamk) {
    // Stream-K few-row kernel: one resident wave over (slab, k-slice) units;
    // every CTA gets at least one unit.  Empty problems and K == 0 never
    // launch it and need no workspace.
    const int64_t KT = (K + v->bk - 1) / v->bk;
    const int64_t units = p->tiles * KT;
    const int64_t slots = static_cast<int64_t>(sms) * ctas;
    grid = units < slots ? units : slots;
    if (units > 0) {
      p->sk_iters = units;
      const size_t ws_bytes = static_cast<size_t>(grid) * v->bm * v->bn * sizeof(float);
      p->ws_slots = grid;
      if (cudaMalloc(reinterpret_cast<void**>(&p->ws), ws_bytes) != cudaSuccess ||
          cudaMalloc(reinterpret_cast<void**>(&p->flags), static_cast<size_t>(grid) * sizeof(unsigned int)) !=
              cudaSuccess ||
          cudaMemset(p->flags, 0, static_cast<size_t>(grid) * sizeof(unsigned int)) != cudaSuccess)
        return fail(SGEMM_ERR_CUDA);
    }
  } else if (v->kind == kKindGemv) {
    // The kernels cut K into chunks that fill whole waves of resident CTAs
    // (more chunks when there are few column blocks); the workspace holds
    // the partial sums of the larger count of the two forms (B as stored,
    // B given transposed).  One chunk needs none.
    grid = sms;
    const int s_kn = gemv_plan_chunks(v, M, N, K, batch, 0, sms), s_nk = gemv_plan_chunks(v, M, N, K, batch, 1, sms);
    if (s_kn < 1 || s_nk < 1) return fail(SGEMM_ERR_CUDA);
    p->split = std::max(s_kn, s_nk);
    if (p->split > 1 && M > 0 && N > 0 && K > 0) {
      const double floats = static_cast<double>(std::max<int64_t>(batch, 1)) * p->split * M * ((N + 3) / 4 * 4);
      if (floats > kMaxSpan) return fail(SGEMM_ERR_UNSUPPORTED);
      const size_t ws_bytes =
          static_cast<size_t>(std::max<int64_t>(batch, 1)) * p->split * M * ((N + 3) / 4 * 4) * sizeof(float);
      p->ws_slots = static_cast<int64_t>(ws_bytes / sizeof(float));
      if (cudaMalloc(reinterpret_cast<void**>(&p->ws), ws_bytes) != cudaSuccess) return fail(SGEMM_ERR_CUDA);
    }
  } else if (v->kind == kKindTc) {
    // persistent forms: one CTA per SM walks the tiles
    if (v->persistent) grid = std::min<int64_t>(grid, static_cast<int64_t>(sms) * ctas);
    // One tile per CTA (or per step of a persistent CTA).  The plan owns the split operands
    // (A_hi, A_lo: M x kp; B_hi, B_lo transposed: N x kp) and encodes their
    // four tensor maps once: 32-float (128-byte, swizzled) k-slices of 128
    // rows of A and 256 rows of B.
    if (p->tiles > 0 && K > 0) {
      const int64_t kp = (K + 3) / 4 * 4;  // 16-byte row stride for TMA
      const size_t bytes = static_cast<size_t>(2 * (M + N) * kp) * sizeof(float);
      if (cudaMalloc(reinterpret_cast<void**>(&p->tc_split), bytes) != cudaSuccess) return fail(SGEMM_ERR_CUDA);
      p->tc_split_ld = kp;
      float* parts[4] = {p->tc_split, p->tc_split + M * kp, p->tc_split + 2 * M * kp,
                         p->tc_split + (2 * M + N) * kp};
      const int64_t rows[4] = {M, M, N, N};
      const cuuint32_t box_rows[4] = {static_cast<cuuint32_t>(v->bm), static_cast<cuuint32_t>(v->bm),
                                      static_cast<cuuint32_t>(v->bn), static_cast<cuuint32_t>(v->bn)};
      EncodeTiledFn enc = encode_fn();
      for (int i = 0; i < 4; ++i) {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows[i])};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kp) * 4};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(v->bk), box_rows[i]};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&p->tc_maps[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, parts[i], dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
          return fail(SGEMM_ERR_CUDA);
      }
    }
  } else if (v->kind == kKindSkinny) {
    // Persistent clusters of S CTAs (S <= 8, the portable cluster size)
    // split K; each cluster walks column slabs.  Pick S and the cluster
    // count so the slabs divide evenly over clusters that all fit on the
    // GPU at once: efficiency = slabs / (clusters * rounds) * (resident
    // CTAs used / CTA slots); ties go to the larger S.
    const int64_t KT = (K + v->bk - 1) / v->bk;
    const int64_t slots = static_cast<int64_t>(sms) * ctas;
    double best = -1.0;
    int64_t best_ncl = 1;
    for (int s = 1; s <= 8 && s <= KT; ++s) {
      // one slab per cluster unless the variant keeps clusters resident
      const int64_t ncl = v->persistent ? std::min<int64_t>(p->tiles, std::max<int64_t>(1, slots / s)) : p->tiles;
      double eff;
      if (v->persistent) {
        const int64_t rounds = (p->tiles + ncl - 1) / ncl;
        eff = static_cast<double>(p->tiles) / static_cast<double>(ncl * rounds) *
              std::min(1.0, static_cast<double>(ncl * s) / static_cast<double>(slots));
      } else {
        // CTAs spread over SMs: (CTAs per SM) / ceil(CTAs per SM), times the filled fraction of slots
        const double total = static_cast<double>(ncl) * s;
        const double per_sm = total / sms;
        eff = per_sm / static_cast<double>(static_cast<int64_t>(per_sm + 0.999999)) *
              std::min(1.0, total / static_cast<double>(slots));
      }
      if (eff >= best - 1e-9) {
        best = eff;
        p->split = s;
        best_ncl = ncl;
      }
    }
    grid = best_ncl * p->split;
  }

  p->grid = static_cast<int>(grid > 0x7fffffff ? 0x7fffffff : grid);
  *out = p;
  return SGEMM_OK;
}

sgemm_status_t encode_maps(const Variant* v, const sgemm_plan_s* p, const float* A, const float* B,
                           LaunchArgs* a) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return SGEMM_ERR_CUDA;
  // batched variants take 3-D maps, the batch outermost (a single product is a batch of one)
  const cuuint32_t rank = v->batched && p->batch > 1 ? 3 : 2;
  // an operand shared by every product (stride 0) is a batch of one
  const cuuint64_t nb_a = static_cast<cuuint64_t>(p->batch > 1 && p->stride_a != 0 ? p->batch : 1);
  const cuuint64_t nb_b = static_cast<cuuint64_t>(p->batch > 1 && p->stride_b != 0 ? p->batch : 1);
  if (a->a_trans) {  // A given transposed (K x M): [bk][bm] boxes, M innermost, unswizzled
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(p->M), static_cast<cuuint64_t>(p->K), nb_a};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(p->ex_lda) * 4,
                                   static_cast<cuuint64_t>(nb_a > 1 ? p->stride_a : p->K * p->ex_lda) * 4};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(v->bm), static_cast<cuuint32_t>(v->bk), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(&a->tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank, const_cast<float*>(A), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return SGEMM_ERR_CUDA;
  } else if (v->kind != kKindCpa) {  // the transposed-A kernels copy A themselves
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(p->K), static_cast<cuuint64_t>(p->M), nb_a};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(p->lda) * 4,
                                   static_cast<cuuint64_t>(nb_a > 1 ? p->stride_a : p->M * p->lda) * 4};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(v->bk), static_cast<cuuint32_t>(v->bm), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(&a->tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank, const_cast<float*>(A), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     v->tma_swizzle_a == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                     : v->tma_swizzle_a == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return SGEMM_ERR_CUDA;
  }
  if (a->b_trans) {  // B given transposed (N x K): K-major boxes of 32 k x bn rows, 128-byte swizzle
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(p->K), static_cast<cuuint64_t>(p->N), nb_b};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(p->ex_ldb) * 4,
                                   static_cast<cuuint64_t>(nb_b > 1 ? p->stride_b : p->N * p->ex_ldb) * 4};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(v->bk), static_cast<cuuint32_t>(v->bn), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(&a->tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank, const_cast<float*>(B), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return SGEMM_ERR_CUDA;
  } else {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(p->N), static_cast<cuuint64_t>(p->K), nb_b};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(p->ldb) * 4,
                                   static_cast<cuuint64_t>(nb_b > 1 ? p->stride_b : p->K * p->ldb) * 4};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(v->bn), static_cast<cuuint32_t>(v->bk), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(&a->tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank, const_cast<float*>(B), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return SGEMM_ERR_CUDA;
  }
  return SGEMM_OK;
}

// Tensor maps for the fused split-TF32 kernel over A and B as stored: a
// K-major operand (A as M x K, B given as N x K) with the 128-byte swizzle
// and 32 (k) x 128 (rows) boxes; an MN-major one (B as K x N, A given as
// K x M) unswizzled with 128 (rows) x 32 (k) boxes.
sgemm_status_t encode_maps_tcf(const Variant* v, const sgemm_plan_s* p, const float* A, const float* B,
                               LaunchArgs* a) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return SGEMM_ERR_CUDA;
  auto one = [&](CUtensorMap* map, const float* base, bool k_major, int64_t rows, int64_t ld, int box_rows) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(k_major ? p->K : rows),
                                static_cast<cuuint64_t>(k_major ? rows : p->K)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(k_major ? v->bk : box_rows),
                               static_cast<cuuint32_t>(k_major ? box_rows : v->bk)};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, k_major ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  if (!one(&a->tmA, A, !p->ex_ta, p->M, p->ex_lda, v->bm) || !one(&a->tmB, B, p->ex_tb != 0, p->N, p->ex_ldb, v->bn))
    return SGEMM_ERR_CUDA;
  a->a_trans = p->ex_ta;
  a->b_trans = p->ex_tb;
  return SGEMM_OK;
}

// Autotuning cache: (device, shape, leading dimensions, tensor cores
// allowed) -> the fastest variant measured by sgemm_plan_autotune.
struct TuneKey {
  int device;
  int64_t M, N, K, lda, ldb, ldc;
  bool tensor;
  bool operator<(const TuneKey& o) const {
    return std::tie(device, M, N, K, lda, ldb, ldc, tensor) <
           std::tie(o.device, o.M, o.N, o.K, o.lda, o.ldb, o.ldc, o.tensor);
  }
};
std::mutex g_tune_mutex;
std::map<TuneKey, int> g_tune_cache;

// Whether the address span of C, [C, C + (M-1) ldc + N + (batch-1) stride_c),
// meets that of operand A (is_a) or B as the caller stores it.
bool spans_overlap(const sgemm_plan_s* p, const float* C, const float* X, bool is_a) {
  // stored shapes in row-major terms (a column-major plan holds A and B swapped)
  const bool internal_a = p->ex_swap ? !is_a : is_a;
  const int64_t rows = internal_a ? (p->ex_ta ? p->K : p->M) : (p->ex_tb ? p->N : p->K);
  const int64_t cols = internal_a ? (p->ex_ta ? p->M : p->K) : (p->ex_tb ? p->K : p->N);
  const int64_t ld = internal_a ? p->ex_lda : p->ex_ldb;
  const int64_t nb = p->batch > 1 ? p->batch : 1;
  const int64_t stride = internal_a ? p->ex_stride_a : p->ex_stride_b;
  const uintptr_t x0 = reinterpret_cast<uintptr_t>(X);
  const uintptr_t x1 = x0 + static_cast<uintptr_t>(((rows - 1) * ld + cols + (nb - 1) * stride) * 4);
  const uintptr_t c0 = reinterpret_cast<uintptr_t>(C);
  const uintptr_t c1 = c0 + static_cast<uintptr_t>(((p->M - 1) * p->ldc + p->N + (nb - 1) * p->stride_c) * 4);
  return x0 < c1 && c0 < x1;
}

// Host-to-device copies of one product's inputs (A and B when there is a
// product, C when beta != 0) with their stored shapes, one 2-D copy per
// matrix of a batch; and the device-to-host copy of its result.
sgemm_status_t copy_inputs(const sgemm_plan_s* p, bool product, float beta, const float* hA, const float* hB,
                           const float* hC, float* dA, float* dB, float* dC, cudaStream_t stream) {
  const size_t fs = sizeof(float);
  const int64_t nb = p->batch > 1 ? p->batch : 1;
  if (product) {
    // stored shapes in row-major terms (a column-major plan holds them swapped)
    const int64_t ra = p->ex_ta ? p->K : p->M, ca = p->ex_ta ? p->M : p->K;
    const int64_t rb = p->ex_tb ? p->N : p->K, cb = p->ex_tb ? p->K : p->N;
    const int64_t ra_u = p->ex_swap ? rb : ra, ca_u = p->ex_swap ? cb : ca, lda_u = p->ex_swap ? p->ex_ldb : p->ex_lda;
    const int64_t rb_u = p->ex_swap ? ra : rb, cb_u = p->ex_swap ? ca : cb, ldb_u = p->ex_swap ? p->ex_lda : p->ex_ldb;
    for (int64_t z = 0; z < nb; ++z) {
      const int64_t sa_u = p->ex_swap ? p->ex_stride_b : p->ex_stride_a, sb_u = p->ex_swap ? p->ex_stride_a : p->ex_stride_b;
      if (cudaMemcpy2DAsync(dA + z * sa_u, lda_u * fs, hA + z * sa_u, lda_u * fs, ca_u * fs, ra_u,
                            cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return SGEMM_ERR_CUDA;
      if (cudaMemcpy2DAsync(dB + z * sb_u, ldb_u * fs, hB + z * sb_u, ldb_u * fs, cb_u * fs, rb_u,
                            cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return SGEMM_ERR_CUDA;
    }
  }
  if (beta != 0.f) {
    for (int64_t z = 0; z < nb; ++z)
      if (cudaMemcpy2DAsync(dC + z * p->stride_c, p->ldc * fs, hC + z * p->stride_c, p->ldc * fs, p->N * fs, p->M,
                            cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return SGEMM_ERR_CUDA;
  }
  return SGEMM_OK;
}

sgemm_status_t copy_output(const sgemm_plan_s* p, float* hC, const float* dC, cudaStream_t stream) {
  const size_t fs = sizeof(float);
  const int64_t nb = p->batch > 1 ? p->batch : 1;
  for (int64_t z = 0; z < nb; ++z)
    if (cudaMemcpy2DAsync(hC + z * p->stride_c, p->ldc * fs, dC + z * p->stride_c, p->ldc * fs, p->N * fs, p->M,
                          cudaMemcpyDeviceToHost, stream) != cudaSuccess)
      return SGEMM_ERR_CUDA;
  return SGEMM_OK;
}

// sgemm_plan_ex and sgemm_plan_ex_batched: storage order and transposed
// operands, for one product (batch 1) or a strided batch.
sgemm_status_t make_plan_ex(int order, int transa, int transb, int64_t M, int64_t N, int64_t K, int64_t lda,
                            int64_t ldb, int64_t ldc, int config_id, sgemm_plan_t* out, int64_t batch = 1,
                            int64_t stride_a = 0, int64_t stride_b = 0, int64_t stride_c = 0) {
  if (!out) return SGEMM_ERR_INVALID_ARG;
  if ((order != SGEMM_ROW_MAJOR && order != SGEMM_COL_MAJOR) || (transa != SGEMM_NO_TRANS && transa != SGEMM_TRANS) ||
      (transb != SGEMM_NO_TRANS && transb != SGEMM_TRANS))
    return SGEMM_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_ARG;
  // leading dimensions of the stored matrices, in the given order
  const int64_t a_rows = transa ? K : M, a_cols = transa ? M : K;
  const int64_t b_rows = transb ? N : K, b_cols = transb ? K : N;
  const bool row = order == SGEMM_ROW_MAJOR;
  if (lda < std::max<int64_t>(1, row ? a_cols : a_rows) || ldb < std::max<int64_t>(1, row ? b_cols : b_rows) ||
      ldc < std::max<int64_t>(1, row ? N : M))
    return SGEMM_ERR_INVALID_ARG;
  // the stored matrices (one product, or the whole strided batch)
  const int64_t nb = batch > 1 ? batch : 1;
  if (batch_span(nb, stride_a, row ? span_elems(a_rows, a_cols, lda) : span_elems(a_cols, a_rows, lda)) > kMaxSpan ||
      batch_span(nb, stride_b, row ? span_elems(b_rows, b_cols, ldb) : span_elems(b_cols, b_rows, ldb)) > kMaxSpan ||
      batch_span(nb, stride_c, row ? span_elems(M, N, ldc) : span_elems(N, M, ldc)) > kMaxSpan)
    return SGEMM_ERR_UNSUPPORTED;
  // Column-major C = op(A) op(B) is the row-major C^T = op(B)^T op(A)^T over
  // the same memory: swap the operands, their transpose flags and strides.
  const int swap = row ? 0 : 1;
  const int64_t M2 = swap ? N : M, N2 = swap ? M : N;
  const int ta = swap ? transb : transa, tb = swap ? transa : transb;
  const int64_t lda2 = swap ? ldb : lda, ldb2 = swap ? lda : ldb;
  const int64_t sa2 = swap ? stride_b : stride_a, sb2 = swap ? stride_a : stride_b;
  if (M2 > 0x7fffffff || N2 > 0x7fffffff || K > 0x7fffffff) return SGEMM_ERR_UNSUPPORTED;
  const bool batched = batch > 1;

  const Registry& reg = registry();
  if (config_id >= static_cast<int>(reg.all.size())) return SGEMM_ERR_INVALID_ARG;
  int forced = config_id;
  if (forced < 0) {
    const char* env = getenv("SGEMM_FORCE_CONFIG");
    if (env && *env) forced = find_variant(env);
  }
  const bool native = forced >= 0 && (reg.all[forced]->kind == kKindTc ||
                                      reg.all[forced]->kind == kKindTcFused);  // reads either layout itself
  if (native && reg.all[forced]->kind == kKindTcFused && (lda2 % 4 != 0 || ldb2 % 4 != 0))
    return SGEMM_ERR_UNSUPPORTED;
  // the row-major, untransposed operands the other kernels read: a
  // transposed operand goes through a plan buffer with a 16-byte row stride
  const int64_t lda_eff = ta && !native ? std::max<int64_t>(4, (K + 3) / 4 * 4) : (ta ? (K + 3) / 4 * 4 : lda2);
  const int64_t ldb_eff = tb && !native ? std::max<int64_t>(4, (N2 + 3) / 4 * 4) : (tb ? (N2 + 3) / 4 * 4 : ldb2);
  // A batch decides up front which transposed operand the kernel reads as
  // stored (its batch stride and extent are then the caller's), using the
  // table's rule: few rows read B given transposed, the transposed-A kernels
  // A given transposed; a forced variant says for itself.  If the plan then
  // gets a kernel that cannot (the table fell back to the scalar-load
  // kernel, say), it is made again with both operands through buffers.
  bool nat_a = false, nat_b = false;
  if (batched) {
    nat_a = ta && lda2 % 4 == 0 && (forced >= 0 ? reg.all[forced]->a_trans_ok != 0 : M2 > 16);
    // (the M <= 4 kernels read B^T with plain loads: any row stride)
    const bool any_ldb = forced >= 0 ? reg.all[forced]->kind == kKindGemv : gemv_shape(M2, N2, K, batch);
    nat_b = tb && (ldb2 % 4 == 0 || any_ldb) && (forced >= 0 ? reg.all[forced]->b_trans_ok != 0 : M2 <= 16);
  }
  sgemm_plan_t p = nullptr;
  sgemm_status_t st = SGEMM_OK;
  for (int attempt = 0; attempt < 2; ++attempt) {
    // the kernels' batch strides and the extent of one stored operand
    const int64_t ka_stride = ta && !nat_a ? (sa2 == 0 ? 0 : M2 * lda_eff) : sa2;
    const int64_t kb_stride = tb && !nat_b ? (sb2 == 0 ? 0 : K * ldb_eff) : sb2;
    const int64_t a_span = nat_a ? K * lda2 : -1;
    const int64_t b_span = nat_b ? N2 * ldb2 : -1;
    st = batched ? make_plan(M2, N2, K, lda_eff, ldb_eff, ldc, config_id, &p, batch, ka_stride, kb_stride, stride_c,
                             a_span, b_span, tb && !native ? 1 : 0)
                 : make_plan(M2, N2, K, lda_eff, ldb_eff, ldc, config_id, &p, 1, 0, 0, 0, -1, -1, tb && !native ? 1 : 0);
    if (!batched || (!nat_a && !nat_b)) break;
    const Variant* got = st == SGEMM_OK ? registry().all[p->config_id] : nullptr;
    if (got && (!nat_a || got->a_trans_ok) && (!nat_b || got->b_trans_ok)) break;
    if (st == SGEMM_OK) sgemm_plan_destroy(p);
    p = nullptr;
    nat_a = nat_b = false;
  }
  if (st != SGEMM_OK) return st;
  p->ex_order = order;
  p->ex_swap = swap;
  p->ex_ta = ta;
  p->ex_tb = tb;
  p->ex_lda = lda2;
  p->ex_ldb = ldb2;
  p->ex_stride_a = batched ? sa2 : 0;
  p->ex_stride_b = batched ? sb2 : 0;
  const Variant* chosen = registry().all[p->config_id];
  const int kind = chosen->kind;
  if (batched) {
    if (kind == kKindTc || kind == kKindTcFused) {  // not batched (make_plan refuses them too)
      sgemm_plan_destroy(p);
      return SGEMM_ERR_UNSUPPORTED;
    }
    p->ex_native_ta = nat_a ? 1 : 0;
    p->ex_native_tb = nat_b ? 1 : 0;
  } else {
    // a few-row kernel reads B given transposed (N x K, K contiguous) by TMA itself
    if (tb && !native && chosen->b_trans_ok && (ldb2 % 4 == 0 || kind == kKindGemv)) p->ex_native_tb = 1;
    // the transposed-A kernels read A given transposed (K x M, M contiguous) by TMA themselves
    if (ta && !native && chosen->a_trans_ok && lda2 % 4 == 0) p->ex_native_ta = 1;
  }
  if (!native && kind != kKindTc && kind != kKindTcFused) {
    // transposed operands the kernel does not read as stored: plan buffers,
    // one per product of a batch (one for a shared operand)
    const int64_t nba = batched && sa2 != 0 ? batch : 1, nbb = batched && sb2 != 0 ? batch : 1;
    if (ta && !p->ex_native_ta && M2 > 0 && K > 0 &&
        cudaMalloc(reinterpret_cast<void**>(&p->ex_wa), sizeof(float) * nba * M2 * lda_eff) != cudaSuccess) {
      sgemm_plan_destroy(p);
      return SGEMM_ERR_CUDA;
    }
    if (tb && !p->ex_native_tb && N2 > 0 && K > 0 &&
        cudaMalloc(reinterpret_cast<void**>(&p->ex_wb), sizeof(float) * nbb * K * ldb_eff) != cudaSuccess) {
      sgemm_plan_destroy(p);
      return SGEMM_ERR_CUDA;
    }
  }
  *out = p;
  return SGEMM_OK;
}

}  // namespace

extern "C" {

sgemm_status_t sgemm_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                          sgemm_plan_t* out) {
  return make_plan(M, N, K, lda, ldb, ldc, -1, out);
}

sgemm_status_t sgemm_plan_with_config(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                      int config_id, sgemm_plan_t* out) {
  if (config_id < 0) return SGEMM_ERR_INVALID_ARG;
  return make_plan(M, N, K, lda, ldb, ldc, config_id, out);
}

sgemm_status_t sgemm_plan_autotune(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                   const float* A, const float* B, float* C, int flags, void* stream_,
                                   double* times_ms, sgemm_plan_t* out) {
  if (!out) return SGEMM_ERR_INVALID_ARG;
  sgemm_status_t st = check_dims(M, N, K, lda, ldb, ldc);
  if (st != SGEMM_OK) return st;
  if ((flags & ~SGEMM_TUNE_TENSOR_CORES) != 0) return SGEMM_ERR_INVALID_ARG;
  const Registry& reg = registry();
  const int nv = static_cast<int>(reg.all.size());
  if (times_ms)
    for (int i = 0; i < nv; ++i) times_ms[i] = -1.0;
  if (M == 0 || N == 0 || K == 0) return make_plan(M, N, K, lda, ldb, ldc, -1, out);  // nothing to time
  if (!A || !B || !C) return SGEMM_ERR_INVALID_ARG;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return SGEMM_ERR_CUDA;
  const bool tensor = (flags & SGEMM_TUNE_TENSOR_CORES) != 0;
  const TuneKey key{device, M, N, K, lda, ldb, ldc, tensor};
  {
    std::lock_guard<std::mutex> lock(g_tune_mutex);
    auto it = g_tune_cache.find(key);
    if (it != g_tune_cache.end() && !times_ms) return make_plan(M, N, K, lda, ldb, ldc, it->second, out);
  }
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
    if (e0) cudaEventDestroy(e0);
    return SGEMM_ERR_CUDA;
  }
  constexpr int kReps = 5;
  int best = -1;
  double best_ms = 0.0;
  st = SGEMM_OK;
  for (int id = 0; id < nv && st == SGEMM_OK; ++id) {
    const Variant* v = reg.all[id];
    if (!tensor && (v->kind == kKindTc || v->kind == kKindTcFused)) continue;
    sgemm_plan_t p = nullptr;
    if (make_plan(M, N, K, lda, ldb, ldc, id, &p) != SGEMM_OK) continue;  // this variant does not take the shape
    // one warm run (kernel attributes, modules, TMA descriptors), then kReps timed back to back
    if (sgemm_run(p, 1.0f, A, B, 0.0f, C, stream_) != SGEMM_OK) {
      sgemm_plan_destroy(p);
      continue;  // e.g. the fused form refuses unaligned buffers
    }
    float ms = 0.f;
    bool ok = cudaEventRecord(e0, stream) == cudaSuccess;
    for (int r = 0; r < kReps && ok; ++r) ok = sgemm_run(p, 1.0f, A, B, 0.0f, C, stream_) == SGEMM_OK;
    ok = ok && cudaEventRecord(e1, stream) == cudaSuccess && cudaEventSynchronize(e1) == cudaSuccess &&
         cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess;
    sgemm_plan_destroy(p);
    if (!ok) {
      st = SGEMM_ERR_CUDA;
      break;
    }
    const double per = static_cast<double>(ms) / kReps;
    if (times_ms) times_ms[id] = per;
    if (best < 0 || per < best_ms) {
      best = id;
      best_ms = per;
    }
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (st != SGEMM_OK) return st;
  if (best < 0) return SGEMM_ERR_UNSUPPORTED;
  {
    std::lock_guard<std::mutex> lock(g_tune_mutex);
    g_tune_cache[key] = best;
  }
  return make_plan(M, N, K, lda, ldb, ldc, best, out);
}

sgemm_status_t sgemm_plan_batched(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                  int64_t batch, int64_t stride_a, int64_t stride_b, int64_t stride_c, int config_id,
                                  sgemm_plan_t* out) {
  if (!out) return SGEMM_ERR_INVALID_ARG;
  if (batch < 0 || stride_a < 0 || stride_b < 0 || stride_c < 0) return SGEMM_ERR_INVALID_ARG;
  if (batch_span(batch, stride_a, span_elems(M, K, lda)) > kMaxSpan ||
      batch_span(batch, stride_b, span_elems(K, N, ldb)) > kMaxSpan ||
      batch_span(batch, stride_c, span_elems(M, N, ldc)) > kMaxSpan)
    return SGEMM_ERR_UNSUPPORTED;
  // the products' C matrices must not overlap (A and B may be shared: stride 0)
  if (batch > 1 && static_cast<double>(stride_c) < span_elems(M, N, ldc)) return SGEMM_ERR_INVALID_ARG;
  if (batch > 65535) return SGEMM_ERR_UNSUPPORTED;
  if (config_id < -1) return SGEMM_ERR_INVALID_ARG;
  return make_plan(M, N, K, lda, ldb, ldc, config_id, out, batch, stride_a, stride_b, stride_c);
}

sgemm_status_t sgemm_plan_ex(int order, int transa, int transb, int64_t M, int64_t N, int64_t K, int64_t lda,
                             int64_t ldb, int64_t ldc, int config_id, sgemm_plan_t* out) {
  return make_plan_ex(order, transa, transb, M, N, K, lda, ldb, ldc, config_id, out);
}

sgemm_status_t sgemm_plan_ex_batched(int order, int transa, int transb, int64_t M, int64_t N, int64_t K, int64_t lda,
                                     int64_t ldb, int64_t ldc, int64_t batch, int64_t stride_a, int64_t stride_b,
                                     int64_t stride_c, int config_id, sgemm_plan_t* out) {
  if (!out) return SGEMM_ERR_INVALID_ARG;
  if (batch < 0 || stride_a < 0 || stride_b < 0 || stride_c < 0 || config_id < -1) return SGEMM_ERR_INVALID_ARG;
  // the products' C matrices must not overlap (A and B may be shared: stride 0)
  const bool row = order == SGEMM_ROW_MAJOR;
  if (batch_span(batch, stride_c, row ? span_elems(M, N, ldc) : span_elems(N, M, ldc)) > kMaxSpan)
    return SGEMM_ERR_UNSUPPORTED;
  if (batch > 1 && static_cast<double>(stride_c) < (row ? span_elems(M, N, ldc) : span_elems(N, M, ldc)))
    return SGEMM_ERR_INVALID_ARG;
  if (batch > 65535) return SGEMM_ERR_UNSUPPORTED;
  return make_plan_ex(order, transa, transb, M, N, K, lda, ldb, ldc, config_id, out, batch, stride_a, stride_b,
                      stride_c);
}

sgemm_status_t sgemm_run(sgemm_plan_t plan, float alpha, const float* A, const float* B, float beta, float* C,
                         void* stream_) {
  if (!plan) return SGEMM_ERR_INVALID_ARG;
  const sgemm_plan_s* p = plan;
  if (p->M == 0 || p->N == 0 || p->batch == 0) return SGEMM_OK;
  if (!C) return SGEMM_ERR_INVALID_ARG;
  const bool product = p->K > 0 && alpha != 0.f;
  if (product && (!A || !B)) return SGEMM_ERR_INVALID_ARG;
  // C may not share its address span with A or B (the kernels read A and B
  // while other CTAs write C): a conservative span test, rows included
  if (product && (spans_overlap(p, C, A, true) || spans_overlap(p, C, B, false))) return SGEMM_ERR_UNSUPPORTED;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) return SGEMM_ERR_CUDA;
  if (device != p->device) return SGEMM_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);

  if (!product) {
    return launch_scale(C, p->ldc, static_cast<int>(p->M), static_cast<int>(p->N), beta, stream,
                        static_cast<int>(p->batch), p->stride_c) == cudaSuccess
               ? SGEMM_OK
               : SGEMM_ERR_CUDA;
  }

  const Registry& reg = registry();
  const Variant* v = reg.all[p->config_id];
  // sgemm_plan_ex: column-major runs the row-major product of the swapped
  // operands; a transposed operand is first transposed into the plan's
  // buffer (the split-TF32 variants read it as stored instead)
  if (p->ex_swap) std::swap(A, B);
  // operands whose rows are not 16-byte multiples: padded copies first
  if (p->rp_a) {
    if (launch_repack(A, p->ex_lda, static_cast<int>(p->M), static_cast<int>(p->K), p->rp_a, p->lda, stream) !=
        cudaSuccess)
      return SGEMM_ERR_CUDA;
    A = p->rp_a;
  }
  if (p->rp_b) {
    if (launch_repack(B, p->ex_ldb, static_cast<int>(p->K), static_cast<int>(p->N), p->rp_b, p->ldb, stream) !=
        cudaSuccess)
      return SGEMM_ERR_CUDA;
    B = p->rp_b;
  }
  // (a strided batch transposes every product's operand; a shared one once)
  if (p->ex_wa) {
    const int nb = p->batch > 1 && p->ex_stride_a != 0 ? static_cast<int>(p->batch) : 1;
    if (launch_transpose(A, p->ex_lda, static_cast<int>(p->K), static_cast<int>(p->M), p->ex_wa, p->lda, stream, nb,
                         p->ex_stride_a, p->stride_a) != cudaSuccess)
      return SGEMM_ERR_CUDA;
    A = p->ex_wa;
  }
  if (p->ex_wb) {
    const int nb = p->batch > 1 && p->ex_stride_b != 0 ? static_cast<int>(p->batch) : 1;
    if (launch_transpose(B, p->ex_ldb, static_cast<int>(p->N), static_cast<int>(p->K), p->ex_wb, p->ldb, stream, nb,
                         p->ex_stride_b, p->stride_b) != cudaSuccess)
      return SGEMM_ERR_CUDA;
    B = p->ex_wb;
  }
  int grid = p->grid;
  const bool a_needs_16 = v->kind == kKindTma || v->kind == kKindSkinny;
  if (v->kind == kKindTcFused &&
      ((reinterpret_cast<uintptr_t>(A) & 15) != 0 || (reinterpret_cast<uintptr_t>(B) & 15) != 0))
    return SGEMM_ERR_UNSUPPORTED;  // TMA needs 16-byte aligned bases; the scalar kernel cannot read every layout
  if (p->ex_native_tb && v->kind != kKindGemv &&
      ((reinterpret_cast<uintptr_t>(B) & 15) != 0 || (reinterpret_cast<uintptr_t>(A) & 15) != 0))
    return SGEMM_ERR_UNSUPPORTED;  // B given transposed is read by TMA; the scalar kernel cannot take it
  if (p->ex_native_ta && ((reinterpret_cast<uintptr_t>(A) & 15) != 0 || (reinterpret_cast<uintptr_t>(B) & 15) != 0))
    return SGEMM_ERR_UNSUPPORTED;  // A given transposed is read by TMA; the scalar kernel cannot take it
  if (v->kind != kKindGeneric && v->kind != kKindTc && v->kind != kKindTcFused && v->kind != kKindGemv &&
      v->kind != kKindTiny &&
      ((a_needs_16 && (reinterpret_cast<uintptr_t>(A) & 15) != 0) || (reinterpret_cast<uintptr_t>(B) & 15) != 0)) {
    v = reg.all[p->generic_id];
    grid = 0;
  }

  LaunchArgs a;
  memset(&a, 0, sizeof(a));
  a.A = A;
  a.B = B;
  a.C = C;
  a.lda = p->lda;
  a.ldb = p->ldb;
  a.ldc = p->ldc;
  a.M = static_cast<int>(p->M);
  a.N = static_cast<int>(p->N);
  a.K = static_cast<int>(p->K);
  a.alpha = alpha;
  a.beta = beta;
  a.grid = grid;
  a.split_k = v->kind == kKindSkinny || v->kind == kKindGemv ? p->split : 1;
  a.batch = static_cast<int>(p->batch);
  a.b_trans = p->ex_native_tb;
  a.a_trans = p->ex_native_ta;
  a.stride_a = p->stride_a;
  a.stride_b = p->stride_b;
  a.stride_c = p->stride_c;
  if (v->kind == kKindGemv) {
    a.ws = p->ws;
    a.ws_slots = p->ws_slots;
    if (p->ex_native_tb) a.ldb = p->ex_ldb;  // read as stored (N x K)
  }
  if (v == reg.all[p->config_id] && p->sk_iters > 0) {
    a.dp_waves = p->dp_waves;
    a.sk_iters = p->sk_iters;
    a.ws = p->ws;
    a.flags = p->flags;
    a.ws_slots = p->ws_slots;
    // each run publishes under a new epoch, so flags need no reset --
    // except when the counter wraps: then a flag may hold any earlier
    // value, so clear them all and start again from 1
    sgemm_plan_s* mp = const_cast<sgemm_plan_s*>(p);
    unsigned int e = mp->epoch.fetch_add(1u) + 1u;
    if (e == 0u) {
      if (cudaMemsetAsync(p->flags, 0, static_cast<size_t>(p->grid) * sizeof(unsigned int), stream) != cudaSuccess)
        return SGEMM_ERR_CUDA;
      mp->epoch.store(1u);
      e = 1u;
    }
    a.epoch = e;
  }
  a.timeout_ns = wait_limit_ns(p->wait_floor_ns);
  sgemm_status_t st = status_addr(device, &a.status);
  if (st != SGEMM_OK) return st;
  if (v->kind == kKindTc) {
    a.split = p->tc_split;
    a.split_ld = p->tc_split_ld;
    a.a_trans = p->ex_ta;
    a.b_trans = p->ex_tb;
    a.lda = p->ex_lda;
    a.ldb = p->ex_ldb;
    a.tmA = p->tc_maps[0];
    a.tmA2 = p->tc_maps[1];
    a.tmB = p->tc_maps[2];
    a.tmB2 = p->tc_maps[3];
  } else if (v->kind == kKindTcFused) {
    st = encode_maps_tcf(v, p, A, B, &a);
    if (st != SGEMM_OK) return st;
  } else if (v->kind != kKindGeneric && v->tma_swizzle_a >= 0) {
    st = encode_maps(v, p, A, B, &a);
    if (st != SGEMM_OK) return st;
  }
  return v->launch(a, stream) == cudaSuccess ? SGEMM_OK : SGEMM_ERR_CUDA;
}

sgemm_status_t sgemm_run_host(sgemm_plan_t plan, float alpha, const float* hA, const float* hB, float beta,
                              float* hC, float* dA, float* dB, float* dC, void* stream_) {
  if (!plan) return SGEMM_ERR_INVALID_ARG;
  const sgemm_plan_s* p = plan;
  if (p->M == 0 || p->N == 0 || p->batch == 0) return SGEMM_OK;
  if (!hC || !dC) return SGEMM_ERR_INVALID_ARG;
  const bool product = p->K > 0 && alpha != 0.f;
  if (product && (!hA || !hB || !dA || !dB)) return SGEMM_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  sgemm_status_t st = copy_inputs(p, product, beta, hA, hB, hC, dA, dB, dC, stream);
  if (st != SGEMM_OK) return st;
  st = sgemm_run(plan, alpha, dA, dB, beta, dC, stream_);
  if (st != SGEMM_OK) return st;
  return copy_output(p, hC, dC, stream);
}

sgemm_status_t sgemm_run_host_pipelined(sgemm_plan_t plan, int count, float alpha, const float* const* hA,
                                        const float* const* hB, float beta, float* const* hC, float* const* dA,
                                        float* const* dB, float* const* dC, void* stream_) {
  if (!plan || count < 0) return SGEMM_ERR_INVALID_ARG;
  sgemm_plan_s* p = plan;
  if (count == 0 || p->M == 0 || p->N == 0 || p->batch == 0) return SGEMM_OK;
  const bool product = p->K > 0 && alpha != 0.f;
  if (!hC || !dC || !dC[0] || !dC[1]) return SGEMM_ERR_INVALID_ARG;
  if (product && (!hA || !hB || !dA || !dB || !dA[0] || !dA[1] || !dB[0] || !dB[1])) return SGEMM_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i)
    if (!hC[i] || (product && (!hA[i] || !hB[i]))) return SGEMM_ERR_INVALID_ARG;
  {
    std::lock_guard<std::mutex> lock(p->pipe_mutex);
    if (!p->pipe_ready) {
      // create everything or nothing: a failure destroys what was made
      cudaStream_t s[2] = {nullptr, nullptr};
      cudaEvent_t ev[2][3] = {{nullptr, nullptr, nullptr}, {nullptr, nullptr, nullptr}};
      bool ok = cudaStreamCreateWithFlags(&s[0], cudaStreamNonBlocking) == cudaSuccess &&
                cudaStreamCreateWithFlags(&s[1], cudaStreamNonBlocking) == cudaSuccess;
      for (int b = 0; b < 2 && ok; ++b)
        for (int e = 0; e < 3 && ok; ++e) ok = cudaEventCreateWithFlags(&ev[b][e], cudaEventDisableTiming) == cudaSuccess;
      if (!ok) {
        for (int b = 0; b < 2; ++b)
          for (int e = 0; e < 3; ++e)
            if (ev[b][e]) cudaEventDestroy(ev[b][e]);
        for (int i = 0; i < 2; ++i)
          if (s[i]) cudaStreamDestroy(s[i]);
        return SGEMM_ERR_CUDA;
      }
      p->pipe_h2d = s[0];
      p->pipe_d2h = s[1];
      for (int b = 0; b < 2; ++b)
        for (int e = 0; e < 3; ++e) p->pipe_ev[b][e] = ev[b][e];
      p->pipe_ready = true;
    }
  }
  cudaStream_t compute = static_cast<cudaStream_t>(stream_);
  enum { kLoaded = 0, kComputed = 1, kStored = 2 };
  // Work already on the caller's stream (earlier writes to the buffers or
  // the host arrays) comes first: both copy streams wait for it.
  if (cudaEventRecord(p->pipe_ev[0][kComputed], compute) != cudaSuccess ||
      cudaStreamWaitEvent(p->pipe_h2d, p->pipe_ev[0][kComputed], 0) != cudaSuccess ||
      cudaStreamWaitEvent(p->pipe_d2h, p->pipe_ev[0][kComputed], 0) != cudaSuccess)
    return SGEMM_ERR_CUDA;
  for (int i = 0; i < count; ++i) {
    const int b = i & 1;
    cudaEvent_t* ev = p->pipe_ev[b];
    if (i >= 2) {
      // buffer set b is free once product i-2 has been computed (A, B read)
      // and its result copied out (C)
      if (cudaStreamWaitEvent(p->pipe_h2d, ev[kComputed], 0) != cudaSuccess ||
          cudaStreamWaitEvent(p->pipe_h2d, ev[kStored], 0) != cudaSuccess)
        return SGEMM_ERR_CUDA;
    }
    sgemm_status_t st = copy_inputs(p, product, beta, product ? hA[i] : nullptr, product ? hB[i] : nullptr, hC[i],
                                    product ? dA[b] : nullptr, product ? dB[b] : nullptr, dC[b], p->pipe_h2d);
    if (st != SGEMM_OK) return st;
    if (cudaEventRecord(ev[kLoaded], p->pipe_h2d) != cudaSuccess ||
        cudaStreamWaitEvent(compute, ev[kLoaded], 0) != cudaSuccess)
      return SGEMM_ERR_CUDA;
    st = sgemm_run(plan, alpha, product ? dA[b] : nullptr, product ? dB[b] : nullptr, beta, dC[b], compute);
    if (st != SGEMM_OK) return st;
    if (cudaEventRecord(ev[kComputed], compute) != cudaSuccess ||
        cudaStreamWaitEvent(p->pipe_d2h, ev[kComputed], 0) != cudaSuccess)
      return SGEMM_ERR_CUDA;
    st = copy_output(p, hC[i], dC[b], p->pipe_d2h);
    if (st != SGEMM_OK) return st;
    if (cudaEventRecord(ev[kStored], p->pipe_d2h) != cudaSuccess) return SGEMM_ERR_CUDA;
  }
  // the caller's stream reaches this point once every result is in host memory
  for (int b = 0; b < (count > 1 ? 2 : 1); ++b)
    if (cudaStreamWaitEvent(compute, p->pipe_ev[b][kStored], 0) != cudaSuccess) return SGEMM_ERR_CUDA;
  return SGEMM_OK;
}

sgemm_status_t sgemm_plan_destroy(sgemm_plan_t plan) {
  if (!plan) return SGEMM_OK;
  sgemm_status_t st = SGEMM_OK;
  if (plan->ws && cudaFree(plan->ws) != cudaSuccess) st = SGEMM_ERR_CUDA;
  if (plan->flags && cudaFree(plan->flags) != cudaSuccess) st = SGEMM_ERR_CUDA;
  if (plan->tc_split && cudaFree(plan->tc_split) != cudaSuccess) st = SGEMM_ERR_CUDA;
  if (plan->ex_wa && cudaFree(plan->ex_wa) != cudaSuccess) st = SGEMM_ERR_CUDA;
  if (plan->ex_wb && cudaFree(plan->ex_wb) != cudaSuccess) st = SGEMM_ERR_CUDA;
  if (plan->rp_a && cudaFree(plan->rp_a) != cudaSuccess) st = SGEMM_ERR_CUDA;
  if (plan->rp_b && cudaFree(plan->rp_b) != cudaSuccess) st = SGEMM_ERR_CUDA;
  if (plan->pipe_ready) {
    if (cudaStreamSynchronize(plan->pipe_h2d) != cudaSuccess || cudaStreamSynchronize(plan->pipe_d2h) != cudaSuccess)
      st = SGEMM_ERR_CUDA;
    for (int b = 0; b < 2; ++b)
      for (int e = 0; e < 3; ++e) cudaEventDestroy(plan->pipe_ev[b][e]);
    cudaStreamDestroy(plan->pipe_h2d);
    cudaStreamDestroy(plan->pipe_d2h);
  }
  delete plan;
  return st;
}

sgemm_status_t sgemm_plan_describe(sgemm_plan_t plan, char* buf, size_t n) {
  if (!plan || !buf || n == 0) return SGEMM_ERR_INVALID_ARG;
  const Variant* v = registry().all[plan->config_id];
  snprintf(buf, n,
           "variant=%s kind=%s tile=%dx%dx%d stages=%d ffma2=%d threads=%d smem=%d grid=%d ctas_per_sm=%d "
           "tiles=%lld sms=%d split=%d streamk=%d dp_waves=%d sk_tiles=%lld k_order=%s M=%lld N=%lld K=%lld "
           "order=%s op=%c%c batch=%lld repack=%d",
           v->name, v->kind == kKindGeneric ? "generic" : v->kind == kKindTma ? "tma" : v->kind == kKindCpa ? "cpa" : v->kind == kKindTc ? "tc" : v->kind == kKindTcFused ? "tcf" : v->kind == kKindGemv ? "gemv" : v->kind == kKindTiny ? "tiny" : "skinny", v->bm, v->bn,
           v->bk, v->stages, v->ffma2, v->threads, v->smem_bytes, plan->grid, plan->ctas_per_sm,
           static_cast<long long>(plan->tiles), plan->num_sms, plan->split, plan->sk_iters > 0 ? 1 : 0, plan->dp_waves,
           static_cast<long long>(plan->sk_iters > 0 ? plan->tiles - static_cast<int64_t>(plan->dp_waves) * plan->grid : 0),
           (v->kind == kKindTc || v->kind == kKindTcFused) ? "tf32x3"
           : (plan->split > 1 || v->kind == kKindSkinny || v->kind == kKindTiny || plan->sk_iters > 0) ? "split"
                                                                                                     : "sequential",
           static_cast<long long>(plan->ex_swap ? plan->N : plan->M),
           static_cast<long long>(plan->ex_swap ? plan->M : plan->N), static_cast<long long>(plan->K),
           plan->ex_order == SGEMM_COL_MAJOR ? "col" : "row",
           (plan->ex_swap ? plan->ex_tb : plan->ex_ta) ? 'T' : 'N', (plan->ex_swap ? plan->ex_ta : plan->ex_tb) ? 'T' : 'N',
           static_cast<long long>(plan->batch),
           // padded copies of the caller's A (1) and B (2), in the caller's terms
           ((plan->ex_swap ? plan->rp_b : plan->rp_a) ? 1 : 0) | ((plan->ex_swap ? plan->rp_a : plan->rp_b) ? 2 : 0));
  return SGEMM_OK;
}

sgemm_status_t sgemm_plan_launches(sgemm_plan_t plan, int* out) {
  if (!plan || !out) return SGEMM_ERR_INVALID_ARG;
  // the split-TF32 variants launch two operand-split kernels before the GEMM
  const Variant* v = registry().all[plan->config_id];
  *out = (plan->M == 0 || plan->N == 0 || plan->batch == 0) ? 0 : v->kind == kKindTc && plan->K > 0 ? 3 : 1;
  // the M <= 4 kernels add their chunks' partial sums in a second kernel
  if (*out > 0 && v->kind == kKindGemv && plan->K > 0 &&
      gemv_plan_chunks(v, plan->M, plan->N, plan->K, plan->batch, plan->ex_native_tb, plan->num_sms) > 1)
    *out = 2;
  if (*out > 0 && plan->K > 0)
    *out += (plan->ex_wa ? 1 : 0) + (plan->ex_wb ? 1 : 0) + (plan->rp_a ? 1 : 0) + (plan->rp_b ? 1 : 0);
  return SGEMM_OK;
}

sgemm_status_t sgemm_plan_config_id(sgemm_plan_t plan, int* out) {
  if (!plan || !out) return SGEMM_ERR_INVALID_ARG;
  *out = plan->config_id;
  return SGEMM_OK;
}

int sgemm_num_configs(void) { return static_cast<int>(registry().all.size()); }

const char* sgemm_config_name(int config_id) {
  const Registry& r = registry();
  if (config_id < 0 || config_id >= static_cast<int>(r.all.size())) return nullptr;
  return r.all[config_id]->name;
}

const char* sgemm_status_string(sgemm_status_t s) {
  switch (s) {
    case SGEMM_OK: return "SGEMM_OK";
    case SGEMM_ERR_INVALID_ARG: return "SGEMM_ERR_INVALID_ARG: bad dimension, leading dimension, pointer or id";
    case SGEMM_ERR_UNSUPPORTED: return "SGEMM_ERR_UNSUPPORTED: valid but not handled by this build";
    case SGEMM_ERR_CUDA: return "SGEMM_ERR_CUDA: a CUDA call failed";
    case SGEMM_ERR_TIMEOUT: return "SGEMM_ERR_TIMEOUT: a kernel wait ran past its time limit";
    case SGEMM_ERR_NOMEM: return "SGEMM_ERR_NOMEM: host allocation failed";
    case SGEMM_ERR_BOUNDS: return "SGEMM_ERR_BOUNDS: a device-side bounds check of the checked build failed";
  }
  return "unknown sgemm status";
}

sgemm_status_t sgemm_device_status(int reset) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return SGEMM_ERR_CUDA;
  unsigned int* addr = nullptr;
  sgemm_status_t st = status_addr(device, &addr);
  if (st != SGEMM_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return SGEMM_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, addr, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return SGEMM_ERR_CUDA;
  if (reset && v != 0) {
    if (cudaMemset(addr, 0, sizeof(v)) != cudaSuccess) return SGEMM_ERR_CUDA;
  }
  if (v & kStatusBounds) return SGEMM_ERR_BOUNDS;
  return v ? SGEMM_ERR_TIMEOUT : SGEMM_OK;
}

sgemm_status_t sgemm_wait_limit_ns(int64_t M, int64_t N, int64_t K, int64_t batch, int num_sms, uint64_t* out) {
  if (!out || M < 0 || N < 0 || K < 0 || batch < 0 || num_sms < 1) return SGEMM_ERR_INVALID_ARG;
  *out = wait_limit_ns(work_floor_ns(M, N, K, batch, num_sms));
  return SGEMM_OK;
}

sgemm_status_t sgemm_table_choice(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t batch,
                                  int64_t stride_a, int64_t stride_b, int b_trans, int num_sms, char* name,
                                  size_t name_size, int* repack_a, int* repack_b) {
  if (!name || name_size == 0 || num_sms < 1 || batch < 0) return SGEMM_ERR_INVALID_ARG;
  sgemm_status_t st = check_dims(M, N, K, lda, ldb, N);
  if (st != SGEMM_OK) return st;
  bool rp_a = false, rp_b = false;
  const char* v = plan_table_choice(M, N, K, &lda, &ldb, num_sms, batch, stride_a, stride_b, -1, -1, b_trans ? 1 : 0,
                                    &rp_a, &rp_b);
  if (find_variant(v) < 0) v = registry().all[registry().first_generic]->name;
  if (strlen(v) + 1 > name_size) return SGEMM_ERR_INVALID_ARG;
  memcpy(name, v, strlen(v) + 1);
  if (repack_a) *repack_a = rp_a ? 1 : 0;
  if (repack_b) *repack_b = rp_b ? 1 : 0;
  return SGEMM_OK;
}

sgemm_status_t sgemm_streamk_schedule(int64_t tiles, int64_t k_slices, int num_sms, int ctas_per_sm, int64_t* grid,
                                      int* dp_waves, int64_t* sk_iters) {
  if (!grid || !dp_waves || !sk_iters || tiles < 0 || k_slices < 0 || num_sms < 1 || ctas_per_sm < 1)
    return SGEMM_ERR_INVALID_ARG;
  const StreamKSchedule s = api_streamk_schedule(tiles, k_slices, num_sms, ctas_per_sm, true);
  *grid = s.grid;
  *dp_waves = s.dp_waves;
  *sk_iters = s.sk_iters;
  return SGEMM_OK;
}

sgemm_status_t sgemm_set_wait_timeout_ns(uint64_t timeout_ns) {
  g_timeout_ns.store(timeout_ns ? timeout_ns : kDefaultTimeoutNs, std::memory_order_relaxed);
  return SGEMM_OK;
}

sgemm_status_t sgemm_selftest_wait_timeout(uint64_t timeout_ns, void* stream_) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return SGEMM_ERR_CUDA;
  unsigned int* addr = nullptr;
  sgemm_status_t st = status_addr(device, &addr);
  if (st != SGEMM_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (launch_wait_selftest(addr, timeout_ns, stream) != cudaSuccess) return SGEMM_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SGEMM_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, addr, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return SGEMM_ERR_CUDA;
  if (!(v & kStatusTimeoutSelftest)) return SGEMM_OK;
  if (cudaMemset(addr, 0, sizeof(v)) != cudaSuccess) return SGEMM_ERR_CUDA;
  return SGEMM_ERR_TIMEOUT;
}

}  // extern "C"

// ---- helpers shared with the static-scratch entry point (api_internal.h) ----
namespace sgemm {

sgemm_status_t api_check_dims(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc) {
  return check_dims(M, N, K, lda, ldb, ldc);
}

const Variant* api_find_variant(const char* name) {
  const int id = find_variant(name);
  return id < 0 ? nullptr : registry().all[id];
}

sgemm_status_t api_status_word(int device, unsigned int** out) { return status_addr(device, out); }

bool api_encoder_ready() { return encode_fn() != nullptr; }

sgemm_status_t api_encode_maps(const Variant* v, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                               const float* A, const float* B, LaunchArgs* a) {
  sgemm_plan_s shape;  // only the shape fields are read
  shape.M = M;
  shape.N = N;
  shape.K = K;
  shape.lda = lda;
  shape.ldb = ldb;
  shape.batch = 1;
  shape.stride_a = shape.stride_b = shape.stride_c = 0;
  return encode_maps(v, &shape, A, B, a);
}

uint64_t api_wait_timeout_ns(int64_t M, int64_t N, int64_t K, int sms) {
  return wait_limit_ns(work_floor_ns(M, N, K, 1, sms));
}

// Stream-K schedules (measured on GB300, CUDA events, L2 flushed):
//  * Tail: more tiles than resident CTAs and a partial last wave -- full
//    waves run data-parallel and the leftover tiles' k-slices are split over
//    every resident CTA (4096^3 on 128 x 256 tiles: 58.3 to 68.9 TFLOP/s).
//  * Fewer tiles than resident CTAs: every tile is split along K into s
//    pieces, one CTA each.  A piece's compute shrinks as KT / s, while the
//    tile's finisher pays one round trip to L2 per contributor, s - 1 in
//    all; the sweep's best s was about sqrt(3 KT), with an integer s and at
//    most one CTA per SM (512^3 on 128 x 64 tiles: 14.6 TFLOP/s with 4
//    pieces per tile on 128 CTAs, 11.9 spread over all 304 slots; 768^3 on
//    128 x 128: 31.5 with 4 per tile on 144 CTAs, 29.4 on 152;
//    256 x 256 x 2048: 8.4 with 16 per tile, 6.8 with 38).  When fewer than
//    three pieces per tile fit on the SMs, the tiles' slices are shared by
//    every resident CTA instead (1024^3 on 128 x 128: 43.8 on 152 CTAs,
//    40.7 with 2 per tile on 128).
StreamKSchedule api_streamk_schedule(int64_t tiles, int64_t KT, int sms, int ctas_per_sm, bool allowed) {
  const int64_t slots = static_cast<int64_t>(sms) * ctas_per_sm;
  StreamKSchedule s{tiles < slots ? tiles : slots, 0, 0};
  if (!allowed || tiles <= 0) return s;
  if (tiles > slots) {
    // The tail's k-slices go to every CTA only when there is at least one
    // slice per CTA: a finisher waits on every CTA between the first one that
    // holds a slice of its tile and itself, so no CTA may have an empty range.
    // (1152 x 1152 x 256 on 64 x 128 tiles: 10 tail tiles x 8 slices for 152
    // CTAs; the tail then runs as a plain partial wave.)
    const int64_t tail = tiles % slots;
    if (tail != 0 && KT >= 8 && tail * KT >= slots) s = {slots, static_cast<int>(tiles / slots), tail * KT};
    return s;
  }
  const int64_t cap = sms / tiles;  // pieces per tile with at most one CTA per SM
  if (cap >= 3) {
    int64_t pieces = static_cast<int64_t>(std::sqrt(3.0 * static_cast<double>(KT)) + 0.5);
    pieces = std::min(pieces, std::min(cap, KT));
    if (pieces >= 2) s = {tiles * pieces, 0, tiles * KT};
    return s;
  }
  if (tiles < slots && tiles * KT >= slots && KT >= 8) s = {slots, 0, tiles * KT};
  return s;
}

bool api_c_overlaps_operands(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                             const float* A, const float* B, const float* C) {
  sgemm_plan_s shape;  // only the shape fields spans_overlap reads
  shape.M = M;
  shape.N = N;
  shape.K = K;
  shape.ldc = ldc;
  shape.ex_lda = lda;
  shape.ex_ldb = ldb;
  shape.ex_swap = 0;
  shape.ex_ta = shape.ex_tb = 0;
  shape.batch = 1;
  shape.ex_stride_a = shape.ex_stride_b = shape.stride_c = 0;
  return spans_overlap(&shape, C, A, true) || spans_overlap(&shape, C, B, false);
}

}  // namespace sgemm
