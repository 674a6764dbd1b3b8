// Instantiations of the expert-range single kernel (bf16 weights).
#include "kernel_table.h"
#include "moe_flat.cuh"

namespace moe {

const void* kernel_flat(int maxm_t) {
  if (maxm_t == 1) return reinterpret_cast<const void*>(&moe_flat_kernel<FMT_BF16, 1>);
  if (maxm_t == 8) return reinterpret_cast<const void*>(&moe_flat_kernel<FMT_BF16, 8>);
  return nullptr;
}

}  // namespace moe
