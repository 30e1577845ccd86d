// cdist_l1.cu -- instantiations of the fused L1 distance + exp kernel of cdist_l1.cuh for fp32 inputs, head dims 32 and 64,
// landmark grids s = 1 .. 8, one or two row groups per CTA.
#include "cdist_l1.cuh"

namespace lapl {
namespace cdist_l1 {

template <int DH, int G>
static const void* pick_s_f32(int s) {
  switch (s) {
    case 1: return reinterpret_cast<const void*>(&cdist_l1_kernel<1, DH, G, false>);
    case 2: return reinterpret_cast<const void*>(&cdist_l1_kernel<2, DH, G, false>);
    case 3: return reinterpret_cast<const void*>(&cdist_l1_kernel<3, DH, G, false>);
    case 4: return reinterpret_cast<const void*>(&cdist_l1_kernel<4, DH, G, false>);
    case 5: return reinterpret_cast<const void*>(&cdist_l1_kernel<5, DH, G, false>);
    case 6: return reinterpret_cast<const void*>(&cdist_l1_kernel<6, DH, G, false>);
    case 7: return reinterpret_cast<const void*>(&cdist_l1_kernel<7, DH, G, false>);
    case 8: return reinterpret_cast<const void*>(&cdist_l1_kernel<8, DH, G, false>);
    default: return nullptr;
  }
}

const void* kernel_bf16(int s, int d, int g);   // cdist_l1_bf16.cu

const void* kernel(int s, int d, int g, bool bf16) {
  if (bf16) return kernel_bf16(s, d, g);
  if (g != 1 && g != 2) return nullptr;
  if (d == 32) return g == 1 ? pick_s_f32<32, 1>(s) : pick_s_f32<32, 2>(s);
  if (d == 64) return g == 1 ? pick_s_f32<64, 1>(s) : pick_s_f32<64, 2>(s);
  return nullptr;
}

}  // namespace cdist_l1
}  // namespace lapl
