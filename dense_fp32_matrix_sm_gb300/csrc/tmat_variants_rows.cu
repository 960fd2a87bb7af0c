// tmat_variants_rows.cu -- 64-row instantiations of the TMA + in-shared-memory
// transposed-A kernel (see tmat_kernel.cuh), for products of 17 to 64 rows,
// where a 128-row tile would be half to three quarters padding.
// Name: tmat_<BM>x<BN>x32_s<STAGES>_b<CTAs per SM>.
#include "tmat_kernel.cuh"

namespace sgemm {
namespace {
const Variant kRowVariants[] = {
    // <BM, BN, stages, CTAs per SM, transpose step, second step (-1: none), split-phase slice sync>
    // 8 warps of 64 x 32, 168 registers: the table's choice up to 64 rows
    tmat::Variant_<64, 256, 3, 1, 24, -1, true>::describe("tmat_64x256x32_s3_b1"),
    // 4 warps, more and narrower tiles (113 KB: one CTA per SM in practice; autotuning only)
    tmat::Variant_<64, 128, 4, 2, 16>::describe("tmat_64x128x32_s4_b2"),
};
}  // namespace

const Variant* tmat_rows_variants(int* count) {
  *count = static_cast<int>(sizeof(kRowVariants) / sizeof(kRowVariants[0]));
  return kRowVariants;
}

}  // namespace sgemm
