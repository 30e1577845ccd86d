// cdist_d64.cu -- instantiations of the distance kernel for head dim 64.
#include "cdist_kernel.cuh"

namespace lapl {
namespace cdist_impl {

template <bool kBf16>
static const void* pick_s(int s) {
  switch (s) {
    case 1: return reinterpret_cast<const void*>(&cdist_exp_kernel<1, 4, 64, kBf16>);
    case 2: return reinterpret_cast<const void*>(&cdist_exp_kernel<2, 4, 64, kBf16>);
    case 3: return reinterpret_cast<const void*>(&cdist_exp_kernel<3, 4, 64, kBf16>);
    case 4: return reinterpret_cast<const void*>(&cdist_exp_kernel<4, 4, 64, kBf16>);
    case 5: return reinterpret_cast<const void*>(&cdist_exp_kernel<5, 4, 64, kBf16>);
    case 6: return reinterpret_cast<const void*>(&cdist_exp_kernel<6, 4, 64, kBf16>);
    case 7: return reinterpret_cast<const void*>(&cdist_exp_kernel<7, 4, 64, kBf16>);
    case 8: return reinterpret_cast<const void*>(&cdist_exp_kernel<8, 4, 64, kBf16>);
    default: return nullptr;
  }
}

const void* kernel_d64(int s, bool bf16) { return bf16 ? pick_s<true>(s) : pick_s<false>(s); }

}  // namespace cdist_impl
}  // namespace lapl
