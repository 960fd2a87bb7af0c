// tmat_variants.cu -- instantiations of the TMA + in-shared-memory transposed-A
// kernel (see tmat_kernel.cuh).  Name: tmat_128x<BN>x32_s<STAGES>_b<CTAs per SM>.
#include "tmat_kernel.cuh"

namespace sgemm {
namespace {
const Variant kVariants[] = {
    tmat::Variant_<128, 4, 1>::describe("tmat_128x128x32_s4_b1"),
    tmat::Variant_<128, 3, 1>::describe("tmat_128x128x32_s3_b1"),
};
}  // namespace

const Variant* tmat_variants(int* count) {
  *count = static_cast<int>(sizeof(kVariants) / sizeof(kVariants[0]));
  return kVariants;
}

}  // namespace sgemm
