// FP8 (e4m3 codes, one fp32 scale per 128 x 128 block) instantiations of the MoE decode layer kernels.
#include "kernel_table.h"
#include "moe_kernels.cuh"

namespace moe {

template <int MAXM>
static const void* pick(int phases) {
  switch (phases) {
    case PH_ALL: return reinterpret_cast<const void*>(&moe_layer_kernel<FMT_FP8, MAXM, PH_ALL>);
    case PH_R: return reinterpret_cast<const void*>(&moe_layer_kernel<FMT_FP8, MAXM, PH_R>);
    case PH_U: return reinterpret_cast<const void*>(&moe_layer_kernel<FMT_FP8, MAXM, PH_U>);
    case PH_D: return reinterpret_cast<const void*>(&moe_layer_kernel<FMT_FP8, MAXM, PH_D>);
    case PH_ILV:  // the interleaved kernel: one row, or any row count up to 8
      if constexpr (MAXM == 6) {
        return nullptr;
      } else {
        return reinterpret_cast<const void*>(&moe_ilv_kernel<FMT_FP8, MAXM>);
      }
    default: return nullptr;
  }
}

const void* kernel_fp8(int maxm_t, int phases) {
  if (maxm_t == 1) return pick<1>(phases);
  if (maxm_t == 6) return pick<6>(phases);
  if (maxm_t == 8) return pick<8>(phases);
  return nullptr;
}

}  // namespace moe
