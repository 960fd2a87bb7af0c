// cpa_variants.cu -- instantiations of the transposed-A kernel (see
// cpa_kernel.cuh).  Name: cpa_<BM>x<BN>x32_s<STAGES>_k<KW>_b<CTAs per SM>.
#include "cpa_kernel.cuh"

namespace sgemm {
namespace {
const Variant kVariants[] = {
    cpa::Variant_<128, 128, 3, 8, 2>::describe("cpa_128x128x32_s3_k8_b2"),
    cpa::Variant_<128, 128, 3, 4, 2>::describe("cpa_128x128x32_s3_k4_b2"),
    cpa::Variant_<128, 128, 3, 2, 2>::describe("cpa_128x128x32_s3_k2_b2"),
    cpa::Variant_<128, 128, 4, 2, 1>::describe("cpa_128x128x32_s4_k2_b1"),
    cpa::Variant_<128, 64, 3, 2, 3>::describe("cpa_128x64x32_s3_k2_b3"),
};
}  // namespace

const Variant* cpa_variants(int* count) {
  *count = static_cast<int>(sizeof(kVariants) / sizeof(kVariants[0]));
  return kVariants;
}

}  // namespace sgemm
