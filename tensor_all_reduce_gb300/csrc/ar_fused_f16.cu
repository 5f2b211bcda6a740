// Instantiations of the fused kernel for the f16 element type (see ar_fused.cuh).
#include "ar_fused.cuh"
#include "ar_launch.h"

namespace ar {

template <int N, bool Q>
static const void* pick_ppt_f16(int ppt, bool vec) {
  if (!vec) return (const void*)&fused_kernel<kF16, N, 1, Q, false>;
  switch (ppt) {
    case 1: return (const void*)&fused_kernel<kF16, N, 1, Q, true>;
    case 2: return (const void*)&fused_kernel<kF16, N, 2, Q, true>;
    case 4: return (const void*)&fused_kernel<kF16, N, 4, Q, true>;
    default: return nullptr;
  }
}

template <int N>
static const void* pick_q_f16(int ppt, bool quant, bool vec) {
  return quant ? pick_ppt_f16<N, true>(ppt, vec) : pick_ppt_f16<N, false>(ppt, vec);
}

const void* fused_kernel_f16(int n, int ppt, bool quant, bool vec) {
  switch (n) {
    case 1: return pick_q_f16<1>(ppt, quant, vec);
    case 2: return pick_q_f16<2>(ppt, quant, vec);
    case 3: return pick_q_f16<3>(ppt, quant, vec);
    case 4: return pick_q_f16<4>(ppt, quant, vec);
    case 5: return pick_q_f16<5>(ppt, quant, vec);
    case 6: return pick_q_f16<6>(ppt, quant, vec);
    case 7: return pick_q_f16<7>(ppt, quant, vec);
    case 8: return pick_q_f16<8>(ppt, quant, vec);
    default: return nullptr;
  }
}

}  // namespace ar
