// api_internal.h -- helpers of the plan API (sgemm_api.cu) that the
// static-scratch entry point (sgemm_static_scratch.cu) shares, so both
// entry points check arguments, find variants, encode tensor maps and
// report timeouts the same way.  Not part of the C ABI.
#pragma once

#include <stdint.h>

#include "kernels.h"
#include "sgemm.h"

namespace sgemm {

// Dimension and leading-dimension checks of sgemm_plan.
sgemm_status_t api_check_dims(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc);
// The registered variant with this name, or nullptr.
const Variant* api_find_variant(const char* name);
// Device address of the per-device status word (looked up once per device).
sgemm_status_t api_status_word(int device, unsigned int** out);
// True once the driver's tensor-map encoder has been found.
bool api_encoder_ready();
// Encode a->tmA / a->tmB for variant v on these operands.
sgemm_status_t api_encode_maps(const Variant* v, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                               const float* A, const float* B, LaunchArgs* a);
// The current limit for in-kernel waits.
uint64_t api_wait_timeout_ns();

}  // namespace sgemm
