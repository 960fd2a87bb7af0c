// kernel_gemv.h -- host-side interface of the matrix-vector kernels
// (kernel_gemv.cu), beside the variant kinds of kernels.h.  Internal.
#pragma once

#include <stdint.h>

#include "kernels.h"

namespace sgemm {

// Variant::kind of the matrix-vector kernels (gemv_4x512: M <= 4;
// gemv_16x512: M <= 16): B streamed by plain loads, any alignment and
// leading dimension, B as stored or given transposed (LaunchArgs::b_trans);
// a.grid = the device's SM count, a.split_k = chunks the workspace a.ws
// holds per product.
constexpr int kKindGemv = 6;

const Variant* gemv_variants(int* count);

// Chunks of K a matrix-vector variant cuts each product of M rows into (B
// as stored or, b_trans = 1, transposed) on a device with `sms` SMs, sized
// to fill whole waves of the kernel instantiation that runs; -1 on a CUDA
// error.
int gemv_plan_chunks(const Variant* v, int64_t M, int64_t N, int64_t K, int64_t batch, int b_trans, int sms);

// Whether a matrix-vector variant takes M x N x K (over `batch` products).
bool gemv_takes(const Variant* v, int64_t M, int64_t N, int64_t K, int64_t batch);

}  // namespace sgemm
