// Internal interface between the C-ABI layer and the kernel translation units.
#pragma once

#include <cuda_runtime.h>

#include "ar.h"

namespace ar {

struct FusedParams;

// Kernel parameters of one validated fused call, each CTA handling `chunk` packs of a row
// and `csize` CTAs sharing a row (chunk = the row's packs and csize = 1: one CTA per row).
// Shared by every entry point that launches a fused kernel.
void fill_fused_params(FusedParams& p, const ar_fused_args& a, int chunk, int csize);

// Kernel entry for a plain reduce: dtype (kF32/kF16/kBF16), n in 1..8, unroll 1 or 4,
// vec = 16-byte path (else element-wise), has_tail = leftover packs/elements exist.
const void* reduce_kernel(int dtype, int n, int unroll, bool vec, bool has_tail);

// Kernel entry for the fused path: dtype kF16/kBF16, n in 1..8, ppt 1/2/4 packs per
// thread (vec only; the scalar tail form has ppt 1), quant = FP8 epilogue.
const void* fused_kernel_f16(int n, int ppt, bool quant, bool vec);
const void* fused_kernel_bf16(int n, int ppt, bool quant, bool vec);

// Staged (bulk-copy pipelined, persistent) fused kernel: n in 1..8, ppt 1, 2 or 4.
const void* staged_kernel_f16(int n, int ppt, bool quant);
const void* staged_kernel_bf16(int n, int ppt, bool quant);

// Cluster form of the staged kernel for rows longer than one CTA holds (a row split over
// the CTAs of a cluster; ppt 1 or 2 packs per thread).
const void* staged_cluster_kernel_f16(int n, int ppt, bool quant);
const void* staged_cluster_kernel_bf16(int n, int ppt, bool quant);

// Batched form of the staged kernel (2 packs per thread, one row per CTA).
const void* batch_kernel_f16(int n, bool quant);
const void* batch_kernel_bf16(int n, bool quant);

// Every fused kernel entry, for one-time attribute setup (non-portable cluster sizes).
int fused_kernel_list(const void** out, int cap);
int staged_kernel_list(const void** out, int cap);

}  // namespace ar
