// tmat_variants.cu -- instantiations of the TMA + in-shared-memory transposed-A
// kernel (see tmat_kernel.cuh).  Name: tmat_<BM>x<BN>x32_s<STAGES>_b<CTAs per SM>.
#include "tmat_kernel.cuh"

namespace sgemm {
namespace {
const Variant kVariants[] = {
    // <BM, BN, stages, CTAs per SM, transpose step(s), split-phase slice sync>: measured best per shape
    tmat::Variant_<128, 128, 4, 1, 8, 24>::describe("tmat_128x128x32_s4_b1"),
    tmat::Variant_<128, 128, 5, 1, 8, 24>::describe("tmat_128x128x32_s5_b1"),
    tmat::Variant_<128, 128, 6, 1, 8, 24>::describe("tmat_128x128x32_s6_b1"),
    tmat::Variant_<128, 64, 3, 2, 16>::describe("tmat_128x64x32_s3_b2"),
    tmat::Variant_<256, 128, 3, 1, 24>::describe("tmat_256x128x32_s3_b1"),
    tmat::Variant_<128, 256, 3, 1, 24, -1, true>::describe("tmat_128x256x32_s3_b1"),
};
}  // namespace

const Variant* tmat_variants(int* count) {
  *count = static_cast<int>(sizeof(kVariants) / sizeof(kVariants[0]));
  return kVariants;
}

}  // namespace sgemm
