// cdist_l1.cu -- instantiations of the fused L1 distance + exp kernel of cdist_l1.cuh for fp32
// inputs, head dims 32 and 64, landmark grids s = 1 .. 8.
#include "cdist_l1.cuh"

namespace lapl {
namespace cdist_l1 {

template <int DH>
static const void* pick_s(int s) {
  switch (s) {
    case 1: return reinterpret_cast<const void*>(&cdist_l1_kernel<1, DH>);
    case 2: return reinterpret_cast<const void*>(&cdist_l1_kernel<2, DH>);
    case 3: return reinterpret_cast<const void*>(&cdist_l1_kernel<3, DH>);
    case 4: return reinterpret_cast<const void*>(&cdist_l1_kernel<4, DH>);
    case 5: return reinterpret_cast<const void*>(&cdist_l1_kernel<5, DH>);
    case 6: return reinterpret_cast<const void*>(&cdist_l1_kernel<6, DH>);
    case 7: return reinterpret_cast<const void*>(&cdist_l1_kernel<7, DH>);
    case 8: return reinterpret_cast<const void*>(&cdist_l1_kernel<8, DH>);
    default: return nullptr;
  }
}

const void* kernel(int s, int d) {
  if (d == 32) return pick_s<32>(s);
  if (d == 64) return pick_s<64>(s);
  return nullptr;
}

}  // namespace cdist_l1
}  // namespace lapl
