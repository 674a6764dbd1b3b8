// Instantiations of the split-K single kernel (down matrices stored transposed;
// bf16 and FP8 weights).
#include "kernel_table.h"
#include "moe_sk.cuh"

namespace moe {

const void* kernel_sk(int fmt, int maxm_t) {
  if (fmt == FMT_BF16) {
    if (maxm_t == 1) return reinterpret_cast<const void*>(&moe_sk_kernel<FMT_BF16, 1>);
    if (maxm_t == 8) return reinterpret_cast<const void*>(&moe_sk_kernel<FMT_BF16, 8>);
  } else if (fmt == FMT_FP8) {
    if (maxm_t == 1) return reinterpret_cast<const void*>(&moe_sk_kernel<FMT_FP8, 1>);
    if (maxm_t == 8) return reinterpret_cast<const void*>(&moe_sk_kernel<FMT_FP8, 8>);
  }
  return nullptr;
}

}  // namespace moe
