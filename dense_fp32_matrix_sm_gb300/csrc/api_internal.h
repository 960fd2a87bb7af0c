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
// The limit for the in-kernel waits of an M x N x K launch on `sms` SMs:
// the process-wide setting, or the launch's work-based floor if larger.
uint64_t api_wait_timeout_ns(int64_t M, int64_t N, int64_t K, int sms);
// The persistent grid of a transposed-A plan over `tiles` C tiles of KT
// k-slices, SMs x CTAs per SM resident: full waves data-parallel and, when
// stream-K is allowed, the last partial wave split along K (dp_waves full
// waves, then sk_iters k-slices shared by the grid).  A split always gives
// every CTA at least one k-slice (sk_iters >= grid): the kernel's finishers
// wait on every CTA between the first one holding a slice of their tile and
// themselves.  Pure host arithmetic.
struct StreamKSchedule {
  int64_t grid;
  int dp_waves;
  int64_t sk_iters;
};
StreamKSchedule api_streamk_schedule(int64_t tiles, int64_t KT, int sms, int ctas_per_sm, bool allowed);

// Whether C (M x N, ldc) shares its address span with A (M x K, lda) or
// B (K x N, ldb), all row-major and untransposed: the conservative span
// test sgemm_run applies before it launches.
bool api_c_overlaps_operands(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                             const float* A, const float* B, const float* C);

}  // namespace sgemm
