// cdist_l1.cu -- instantiations of the fused L1 distance + exp kernel of cdist_l1.cuh for fp32
// inputs, head dims 32 and 64, landmark grids s = 1 .. 8, one or two row groups per CTA.
#include "cdist_l1.cuh"

namespace lapl {
namespace cdist_l1 {

template <int DH, int G>
static const void* pick_s(int s) {
  switch (s) {
    case 1: return reinterpret_cast<const void*>(&cdist_l1_kernel<1, DH, G>);
    case 2: return reinterpret_cast<const void*>(&cdist_l1_kernel<2, DH, G>);
    case 3: return reinterpret_cast<const void*>(&cdist_l1_kernel<3, DH, G>);
    case 4: return reinterpret_cast<const void*>(&cdist_l1_kernel<4, DH, G>);
    case 5: return reinterpret_cast<const void*>(&cdist_l1_kernel<5, DH, G>);
    case 6: return reinterpret_cast<const void*>(&cdist_l1_kernel<6, DH, G>);
    case 7: return reinterpret_cast<const void*>(&cdist_l1_kernel<7, DH, G>);
    case 8: return reinterpret_cast<const void*>(&cdist_l1_kernel<8, DH, G>);
    default: return nullptr;
  }
}

const void* kernel(int s, int d, int g) {
  if (g == 1) {
    if (d == 32) return pick_s<32, 1>(s);
    if (d == 64) return pick_s<64, 1>(s);
  } else if (g == 2) {
    if (d == 32) return pick_s<32, 2>(s);
    if (d == 64) return pick_s<64, 2>(s);
  }
  return nullptr;
}

}  // namespace cdist_l1
}  // namespace lapl
