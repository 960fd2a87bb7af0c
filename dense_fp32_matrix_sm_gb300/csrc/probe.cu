// probe.cu -- sgemm_probe_ffma (include/sgemm.h): the FP32 FMA pipe's
// achievable rate on this device, and the SM clock measured inside the
// kernel.  The FFMA-pipe roofline divides by SMs x 128 lanes x 2 x clock; an
// FMA-only kernel shows how much of that nominal rate an ideal instruction
// stream reaches (the pages report such a test at 96% of the nominal rate:
// "Writing a Fast Matmul in CUDA, Step by Step", the measurement set-up).
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"
#include "sgemm.h"

namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeCtasPerSm = 2;  // 16 warps per SM, as the FFMA GEMM kernels run
constexpr int kProbeIters = 8192;

// {clock64 at start, at end, globaltimer at start, at end} of CTA 0, thread 0
__device__ unsigned long long g_probe_clock[4];
__device__ float g_probe_sink;

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// The FFMA GEMM kernels' accumulation pattern without their loads, 128 FLOP
// per thread per step:
//  * PAIRED: acc[i][j] += a_pair[i] * b[j] as FFMA2 (a pair of two A rows
//    times one broadcast B value), 4 x 8 pair accumulators;
//  * else: acc[i][j] += a[i] * b[j] as FFMA, 8 x 8 accumulators (the
//    pages' register-blocked outer product).
// The operands are runtime values held in registers (no immediates).
// The result feeds a store guarded by a value the host never passes, so the
// arithmetic cannot be dropped.
template <bool PAIRED>
__global__ void __launch_bounds__(kProbeThreads) ffma_probe_kernel(int iters, float seed, unsigned int never) {
  const bool timer = blockIdx.x == 0 && threadIdx.x == 0;
  unsigned long long c0 = 0, t0 = 0;
  if (timer) {
    t0 = globaltimer();
    c0 = clock64();
  }
  const float x = seed + 1e-6f * static_cast<float>(threadIdx.x);
  float s = 0.f;
  if constexpr (PAIRED) {
    float2 acc[4][8], a[4];
    float b[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = make_float2(x + i, x - i);
#pragma unroll
    for (int j = 0; j < 8; ++j) b[j] = 1e-7f * (j + 1);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = make_float2(0.f, 0.f);
#pragma unroll 4
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = __ffma2_rn(a[i], make_float2(b[j], b[j]), acc[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) s += acc[i][j].x + acc[i][j].y;
  } else {
    float acc[8][8], a[8], b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = x + i;
#pragma unroll
    for (int j = 0; j < 8; ++j) b[j] = 1e-7f * (j + 1);
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
#pragma unroll 4
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) s += acc[i][j];
  }
  if (__float_as_uint(s) == never) g_probe_sink = s;
  if (timer) {
    const unsigned long long c1 = clock64();
    const unsigned long long t1 = globaltimer();
    g_probe_clock[0] = c0;
    g_probe_clock[1] = c1;
    g_probe_clock[2] = t0;
    g_probe_clock[3] = t1;
  }
}

}  // namespace

extern "C" sgemm_status_t sgemm_probe_ffma(int paired, double* tflops, double* sm_mhz) {
  if (!tflops || !sm_mhz || (paired != 0 && paired != 1)) return SGEMM_ERR_INVALID_ARG;
  int device = 0, sms = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return SGEMM_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return SGEMM_ERR_CUDA;
  const int grid = sms * kProbeCtasPerSm;
  cudaStream_t stream = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  sgemm_status_t st = SGEMM_ERR_CUDA;
  float ms = 0.f;
  unsigned long long clk[4] = {0, 0, 0, 0};
  auto launch = [&]() {
    if (paired)
      ffma_probe_kernel<true><<<grid, kProbeThreads, 0, stream>>>(kProbeIters, 1.0f, 0x7fc00001u);
    else
      ffma_probe_kernel<false><<<grid, kProbeThreads, 0, stream>>>(kProbeIters, 1.0f, 0x7fc00001u);
    return cudaGetLastError();
  };
  if (cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking) != cudaSuccess) return SGEMM_ERR_CUDA;
  if (cudaEventCreate(&e0) == cudaSuccess && cudaEventCreate(&e1) == cudaSuccess && launch() == cudaSuccess &&
      cudaEventRecord(e0, stream) == cudaSuccess && launch() == cudaSuccess &&
      cudaEventRecord(e1, stream) == cudaSuccess && cudaEventSynchronize(e1) == cudaSuccess &&
      cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess &&
      cudaMemcpyFromSymbol(clk, g_probe_clock, sizeof(clk)) == cudaSuccess && ms > 0.f && clk[3] > clk[2]) {
    const double flop = 128.0 * kProbeIters * static_cast<double>(grid) * kProbeThreads;
    *tflops = flop / (static_cast<double>(ms) * 1e-3) / 1e12;
    *sm_mhz = static_cast<double>(clk[1] - clk[0]) / static_cast<double>(clk[3] - clk[2]) * 1e3;
    st = SGEMM_OK;
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  cudaStreamDestroy(stream);
  return st;
}
