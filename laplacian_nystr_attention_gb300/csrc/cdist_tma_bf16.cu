// cdist_tma_bf16.cu -- instantiations of the TMA-fed distance kernel for bf16 inputs, head dim
// 64 (one 128-byte box per token row).
#include "cdist_tma.cuh"

namespace lapl {
namespace cdist_tma {

const void* kernel_bf16(int s, int d) {
  if (d != 64) return nullptr;
  switch (s) {
    case 1: return reinterpret_cast<const void*>(&cdist_tma_kernel<1, 64, true>);
    case 2: return reinterpret_cast<const void*>(&cdist_tma_kernel<2, 64, true>);
    case 3: return reinterpret_cast<const void*>(&cdist_tma_kernel<3, 64, true>);
    case 4: return reinterpret_cast<const void*>(&cdist_tma_kernel<4, 64, true>);
    case 5: return reinterpret_cast<const void*>(&cdist_tma_kernel<5, 64, true>);
    case 6: return reinterpret_cast<const void*>(&cdist_tma_kernel<6, 64, true>);
    case 7: return reinterpret_cast<const void*>(&cdist_tma_kernel<7, 64, true>);
    case 8: return reinterpret_cast<const void*>(&cdist_tma_kernel<8, 64, true>);
    default: return nullptr;
  }
}

}  // namespace cdist_tma
}  // namespace lapl
