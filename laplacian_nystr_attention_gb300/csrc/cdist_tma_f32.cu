// cdist_tma_f32.cu -- instantiations of the TMA-fed distance kernel for fp32 inputs, head dims
// 32 and 64 (one or two 128-byte boxes per token row).
#include "cdist_tma.cuh"

namespace lapl {
namespace cdist_tma {

template <int DH>
static const void* pick_s(int s) {
  switch (s) {
    case 1: return reinterpret_cast<const void*>(&cdist_tma_kernel<1, DH, false>);
    case 2: return reinterpret_cast<const void*>(&cdist_tma_kernel<2, DH, false>);
    case 3: return reinterpret_cast<const void*>(&cdist_tma_kernel<3, DH, false>);
    case 4: return reinterpret_cast<const void*>(&cdist_tma_kernel<4, DH, false>);
    case 5: return reinterpret_cast<const void*>(&cdist_tma_kernel<5, DH, false>);
    case 6: return reinterpret_cast<const void*>(&cdist_tma_kernel<6, DH, false>);
    case 7: return reinterpret_cast<const void*>(&cdist_tma_kernel<7, DH, false>);
    case 8: return reinterpret_cast<const void*>(&cdist_tma_kernel<8, DH, false>);
    default: return nullptr;
  }
}

const void* kernel_f32(int s, int d) {
  if (d == 32) return pick_s<32>(s);
  if (d == 64) return pick_s<64>(s);
  return nullptr;
}

}  // namespace cdist_tma
}  // namespace lapl
