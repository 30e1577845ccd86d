// cdist_gauss_d32.cu -- instantiations of the distance kernel for the Gaussian kernel (squared
// l2 distance), head dim 32.
#include "cdist_kernel.cuh"

namespace lapl {
namespace cdist_impl {

template <bool kBf16>
static const void* pick_s(int s) {
  switch (s) {
    case 1: return reinterpret_cast<const void*>(&cdist_exp_kernel<1, 4, 32, kBf16, true>);
    case 2: return reinterpret_cast<const void*>(&cdist_exp_kernel<2, 4, 32, kBf16, true>);
    case 3: return reinterpret_cast<const void*>(&cdist_exp_kernel<3, 4, 32, kBf16, true>);
    case 4: return reinterpret_cast<const void*>(&cdist_exp_kernel<4, 4, 32, kBf16, true>);
    case 5: return reinterpret_cast<const void*>(&cdist_exp_kernel<5, 4, 32, kBf16, true>);
    case 6: return reinterpret_cast<const void*>(&cdist_exp_kernel<6, 4, 32, kBf16, true>);
    case 7: return reinterpret_cast<const void*>(&cdist_exp_kernel<7, 4, 32, kBf16, true>);
    case 8: return reinterpret_cast<const void*>(&cdist_exp_kernel<8, 4, 32, kBf16, true>);
    default: return nullptr;
  }
}

const void* gauss_d32(int s, bool bf16) { return bf16 ? pick_s<true>(s) : pick_s<false>(s); }

}  // namespace cdist_impl
}  // namespace lapl
