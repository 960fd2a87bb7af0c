// tma_variants_c.cu -- instantiations of the TMA-fed kernel (see
// tma_kernel.cuh).  Name: tma_<BM>x<BN>x<BK>_w<WM>x<WN>_s<STAGES>_<quad|scalar>_b<CTAs per SM>.
#include "tma_kernel.cuh"

namespace sgemm {
namespace {
using tma::kQuad;
using tma::kScalar;
const Variant kVariants[] = {
    tma::Variant_<128, 128, 32, 64, 32, 3, kScalar, 2, true>::describe("tma_128x128x32_w64x32_s3_scalar_b2"),
    tma::Variant_<128, 64, 32, 64, 32, 4, kQuad, 2, false>::describe("tma_128x64x32_w64x32_s4_quad_b2_ffma"),
    tma::Variant_<128, 128, 16, 64, 64, 4, kQuad, 2, true>::describe("tma_128x128x16_w64x64_s4_quad_b2"),
};
}  // namespace

const Variant* tma_variants_c(int* count) {
  *count = static_cast<int>(sizeof(kVariants) / sizeof(kVariants[0]));
  return kVariants;
}

}  // namespace sgemm
