// kernel_skinny.cu -- small-M (decode-shaped) SGEMM variants.
#include <cuda_runtime.h>

#include "kernels.h"

namespace sgemm {

const Variant* skinny_variants(int* count) {
  *count = 0;
  return nullptr;
}

}  // namespace sgemm
