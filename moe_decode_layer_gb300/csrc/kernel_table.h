// Host-side access to the kernel instantiations (one translation unit per
// weight format, so the two compile in parallel).
#pragma once

namespace moe {
// Kernel entry for (maxm_t in {1, 6, 8}, phases in Phase). NULL if not
// instantiated. maxm_t bounds the token rows of a launch; 6 (bf16 and FP8,
// phase-ordered and chained kernels) keeps the per-thread sums of up to six rows
// in registers where 8 spills, for runs of 2..6 rows.
const void* kernel_bf16(int maxm_t, int phases);
const void* kernel_nvfp4(int maxm_t, int phases);
const void* kernel_fp8(int maxm_t, int phases);
// The expert-range single kernel (bf16 weights) for maxm_t in {1, 8}.
const void* kernel_flat(int maxm_t);
// The split-K single kernel (down matrices transposed) for fmt in {FMT_BF16,
// FMT_FP8} and maxm_t in {1, 8}.
const void* kernel_sk(int fmt, int maxm_t);
}  // namespace moe
