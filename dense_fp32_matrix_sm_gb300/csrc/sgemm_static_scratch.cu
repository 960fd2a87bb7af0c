// sgemm_static_scratch.cu -- sgemm_run_static_scratch (include/sgemm.h):
// the 128 x 256 transposed-A kernel with its stream-K tail, run with no
// plan and no memory allocation.  The stream-K workspace (one partial tile
// per CTA) and its flags live in a file-scope __device__ array of fixed
// size whose address is looked up once per device.
//
// Nothing here changes the kernel: it is the same launcher the plan path
// uses, handed this array instead of a plan's cudaMalloc'd workspace.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "api_internal.h"
#include "kernels.h"
#include "sgemm.h"

using namespace sgemm;

namespace {

constexpr const char* kVariantName = "tmat_128x256x32_s3_b1";
constexpr int kTileM = 128;
constexpr int kTileN = 256;
constexpr int kMaxDevices = 64;
constexpr size_t kWorkspaceBytes =
    static_cast<size_t>(SGEMM_STATIC_SCRATCH_MAX_CTAS) * kTileM * kTileN * sizeof(float);
constexpr size_t kFlagBytes = (SGEMM_STATIC_SCRATCH_MAX_CTAS * sizeof(unsigned int) + 255) / 256 * 256;
static_assert(kWorkspaceBytes + kFlagBytes == SGEMM_STATIC_SCRATCH_BYTES,
              "the header's scratch size and this file's layout disagree");

}  // namespace

// The scratch: partial tiles first (float4 stores, 256-byte aligned), then
// the per-CTA flags.  Zero-filled when the module loads; set-up clears the
// flags again explicitly.
static __device__ __align__(256) unsigned char g_static_scratch[SGEMM_STATIC_SCRATCH_BYTES];

namespace {

struct DeviceState {
  std::atomic<bool> ready{false};
  float* ws = nullptr;
  unsigned int* flags = nullptr;
  unsigned int* status = nullptr;
  int sms = 0;          // SMs of the device
  int ctas_per_sm = 0;  // resident CTAs of the kernel per SM
  std::atomic<unsigned int> epoch{0};
};

DeviceState g_state[kMaxDevices];
std::mutex g_setup_mutex;
std::atomic<const Variant*> g_variant{nullptr};

// Once per device, with that device current.  A failed set-up leaves the
// device not ready, and the next call tries again.
sgemm_status_t setup(int device, cudaStream_t stream, DeviceState** out) {
  DeviceState& s = g_state[device];
  if (!s.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!s.ready.load(std::memory_order_relaxed)) {
      const Variant* v = api_find_variant(kVariantName);
      if (!v || v->bm != kTileM || v->bn != kTileN || !v->streamk) return SGEMM_ERR_UNSUPPORTED;
      if (!api_encoder_ready()) return SGEMM_ERR_CUDA;
      void* base = nullptr;
      if (cudaGetSymbolAddress(&base, g_static_scratch) != cudaSuccess) return SGEMM_ERR_CUDA;
      int sms = 0;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return SGEMM_ERR_CUDA;
      if (v->prepare() != cudaSuccess) return SGEMM_ERR_CUDA;
      int ctas = 0;
      if (v->occupancy(&ctas) != cudaSuccess || ctas < 1) return SGEMM_ERR_CUDA;
      unsigned int* status = nullptr;
      const sgemm_status_t st = api_status_word(device, &status);
      if (st != SGEMM_OK) return st;
      unsigned char* b = static_cast<unsigned char*>(base);
      unsigned int* flags = reinterpret_cast<unsigned int*>(b + kWorkspaceBytes);
      // flags compare equal to the call's epoch when a partial tile is
      // ready; they must start below every epoch used, i.e. at zero
      if (cudaMemsetAsync(flags, 0, kFlagBytes, stream) != cudaSuccess) return SGEMM_ERR_CUDA;
      s.ws = reinterpret_cast<float*>(b);
      s.flags = flags;
      s.status = status;
      s.sms = sms;
      s.ctas_per_sm = ctas;
      s.epoch.store(0, std::memory_order_relaxed);
      g_variant.store(v, std::memory_order_relaxed);
      s.ready.store(true, std::memory_order_release);
    }
  }
  *out = &s;
  return SGEMM_OK;
}

}  // namespace

extern "C" sgemm_status_t sgemm_run_static_scratch(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                                   int64_t ldc, float alpha, const float* A, const float* B,
                                                   float beta, float* C, void* stream_) {
  sgemm_status_t st = api_check_dims(M, N, K, lda, ldb, ldc);
  if (st != SGEMM_OK) return st;
  if (M == 0 || N == 0) return SGEMM_OK;
  if (!C) return SGEMM_ERR_INVALID_ARG;
  const bool product = K > 0 && alpha != 0.f;
  if (product && (!A || !B)) return SGEMM_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (!product)
    return launch_scale(C, ldc, static_cast<int>(M), static_cast<int>(N), beta, stream) == cudaSuccess
               ? SGEMM_OK
               : SGEMM_ERR_CUDA;
  // the kernel reads A and B with TMA: 16-byte rows and base addresses
  if (lda % 4 != 0 || ldb % 4 != 0 || (reinterpret_cast<uintptr_t>(A) & 15) != 0 ||
      (reinterpret_cast<uintptr_t>(B) & 15) != 0)
    return SGEMM_ERR_UNSUPPORTED;
  // C may not share its address span with A or B: the kernel reads A and B
  // by TMA while other CTAs write C (the same span test as sgemm_run)
  if (api_c_overlaps_operands(M, N, K, lda, ldb, ldc, A, B, C)) return SGEMM_ERR_UNSUPPORTED;

  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) return SGEMM_ERR_CUDA;
  if (device < 0 || device >= kMaxDevices) return SGEMM_ERR_UNSUPPORTED;
  DeviceState* s = nullptr;
  st = setup(device, stream, &s);
  if (st != SGEMM_OK) return st;
  const Variant* v = g_variant.load(std::memory_order_relaxed);

  LaunchArgs a;
  memset(&a, 0, sizeof(a));
  a.A = A;
  a.B = B;
  a.C = C;
  a.lda = lda;
  a.ldb = ldb;
  a.ldc = ldc;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.alpha = alpha;
  a.beta = beta;
  a.split_k = 1;
  a.status = s->status;
  a.timeout_ns = api_wait_timeout_ns(M, N, K, s->sms);

  // The same schedule as a plan of this variant (api_streamk_schedule):
  // full waves data-parallel and a partial last wave split along K; with
  // fewer tiles than CTA slots, every tile split into pieces along K.
  const int64_t tiles = ((M + kTileM - 1) / kTileM) * ((N + kTileN - 1) / kTileN);
  const int64_t KT = (K + v->bk - 1) / v->bk;
  // SGEMM_NO_STREAMK turns the split off here as it does for plans, so the
  // results stay bit-identical to a plan of the same variant
  const StreamKSchedule sk =
      api_streamk_schedule(tiles, KT, s->sms, s->ctas_per_sm, getenv("SGEMM_NO_STREAMK") == nullptr);
  int64_t grid = sk.grid;
  if (sk.sk_iters > 0) {
    if (grid > SGEMM_STATIC_SCRATCH_MAX_CTAS) return SGEMM_ERR_UNSUPPORTED;  // more partial tiles than the array holds
    a.dp_waves = sk.dp_waves;
    a.sk_iters = sk.sk_iters;
    a.ws = s->ws;
    a.ws_slots = SGEMM_STATIC_SCRATCH_MAX_CTAS;
    a.flags = s->flags;
    unsigned int e = s->epoch.fetch_add(1u, std::memory_order_relaxed) + 1u;
    if (e == 0u) {
      // the counter wrapped: a flag may still hold any earlier value, so
      // clear them all and start again from 1
      if (cudaMemsetAsync(s->flags, 0, kFlagBytes, stream) != cudaSuccess) return SGEMM_ERR_CUDA;
      s->epoch.store(1u, std::memory_order_relaxed);
      e = 1u;
    }
    a.epoch = e;
  }
  a.grid = static_cast<int>(grid);
  st = api_encode_maps(v, M, N, K, lda, ldb, A, B, &a);
  if (st != SGEMM_OK) return st;
  return v->launch(a, stream) == cudaSuccess ? SGEMM_OK : SGEMM_ERR_CUDA;
}
