// cdist_l1_bf16.cu -- instantiations of the fused L1 distance + exp kernel of cdist_l1.cuh for bf16 inputs, head dim 64,
// landmark grids s = 1 .. 8, one or two row groups per CTA.
#include "cdist_l1.cuh"

namespace lapl {
namespace cdist_l1 {

template <int DH, int G>
static const void* pick_s_bf16(int s) {
  switch (s) {
    case 1: return reinterpret_cast<const void*>(&cdist_l1_kernel<1, DH, G, true>);
    case 2: return reinterpret_cast<const void*>(&cdist_l1_kernel<2, DH, G, true>);
    case 3: return reinterpret_cast<const void*>(&cdist_l1_kernel<3, DH, G, true>);
    case 4: return reinterpret_cast<const void*>(&cdist_l1_kernel<4, DH, G, true>);
    case 5: return reinterpret_cast<const void*>(&cdist_l1_kernel<5, DH, G, true>);
    case 6: return reinterpret_cast<const void*>(&cdist_l1_kernel<6, DH, G, true>);
    case 7: return reinterpret_cast<const void*>(&cdist_l1_kernel<7, DH, G, true>);
    case 8: return reinterpret_cast<const void*>(&cdist_l1_kernel<8, DH, G, true>);
    default: return nullptr;
  }
}

const void* kernel_bf16(int s, int d, int g) {
  if (d != 64 || (g != 1 && g != 2)) return nullptr;
  return g == 1 ? pick_s_bf16<64, 1>(s) : pick_s_bf16<64, 2>(s);
}

}  // namespace cdist_l1
}  // namespace lapl
