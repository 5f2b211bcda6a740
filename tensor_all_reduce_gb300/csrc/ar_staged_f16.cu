// Instantiations of the staged fused kernel for the f16 element type (see ar_staged.cuh).
#include "ar_launch.h"
#include "ar_staged.cuh"

namespace ar {

template <int N, bool Q>
static const void* pick_staged_ppt_f16(int ppt) {
  switch (ppt) {
    case 1: return (const void*)&fused_staged_kernel<kF16, N, 1, Q>;
    case 2: return (const void*)&fused_staged_kernel<kF16, N, 2, Q>;
    case 4: return (const void*)&fused_staged_kernel<kF16, N, 4, Q>;
    default: return nullptr;
  }
}

const void* staged_kernel_f16(int n, int ppt, bool quant) {
  switch (n) {
#define AR_CASE(NN) \
  case NN: return quant ? pick_staged_ppt_f16<NN, true>(ppt) : pick_staged_ppt_f16<NN, false>(ppt);
    AR_CASE(1) AR_CASE(2) AR_CASE(3) AR_CASE(4) AR_CASE(5) AR_CASE(6) AR_CASE(7) AR_CASE(8)
#undef AR_CASE
    default: return nullptr;
  }
}

template <int N, bool Q>
static const void* pick_staged_cluster_ppt_f16(int ppt) {
  switch (ppt) {
    case 1: return (const void*)&fused_staged_cluster_kernel<kF16, N, 1, Q>;
    case 2: return (const void*)&fused_staged_cluster_kernel<kF16, N, 2, Q>;
    default: return nullptr;
  }
}

const void* staged_cluster_kernel_f16(int n, int ppt, bool quant) {
  switch (n) {
#define AR_CASE(NN) \
  case NN: return quant ? pick_staged_cluster_ppt_f16<NN, true>(ppt) : pick_staged_cluster_ppt_f16<NN, false>(ppt);
    AR_CASE(1) AR_CASE(2) AR_CASE(3) AR_CASE(4) AR_CASE(5) AR_CASE(6) AR_CASE(7) AR_CASE(8)
#undef AR_CASE
    default: return nullptr;
  }
}

const void* batch_kernel_f16(int n, bool quant) {
  switch (n) {
#define AR_CASE(NN) \
  case NN: return quant ? (const void*)&fused_batch_kernel<kF16, NN, 2, true> : (const void*)&fused_batch_kernel<kF16, NN, 2, false>;
    AR_CASE(1) AR_CASE(2) AR_CASE(3) AR_CASE(4) AR_CASE(5) AR_CASE(6) AR_CASE(7) AR_CASE(8)
#undef AR_CASE
    default: return nullptr;
  }
}

}  // namespace ar
