// kernel_gemv.h -- host-side interface of the M <= 4 kernels
// (kernel_gemv.cu), beside the variant kinds of kernels.h.  Internal.
#pragma once

#include <stdint.h>

#include "kernels.h"

namespace sgemm {

// Variant::kind of the M <= 4 kernels: B streamed by plain loads, any
// alignment and leading dimension, B as stored or given transposed
// (LaunchArgs::b_trans); a.grid = resident CTA slots, a.split_k = chunks
// the workspace a.ws holds per product.
constexpr int kKindGemv = 6;

const Variant* gemv_variants(int* count);

// Chunks of K the M <= 4 kernels cut each product into (B as stored or,
// b_trans = 1, transposed), for a device with `slots` resident CTAs.
int gemv_chunks(int64_t N, int64_t K, int64_t batch, int b_trans, int64_t slots);

}  // namespace sgemm
