// cdist.cu -- host side of the fused L1 distance + exp kernel (cdist_kernel.cuh): shared
// memory size, occupancy, kernel choice and launch.
#include "cdist_kernel.cuh"

namespace lapl {
namespace cdist_impl {
const void* kernel_d32(int s, bool bf16);
const void* kernel_d64(int s, bool bf16);
const void* kernel_d0(int s, bool bf16);

constexpr int kRows = 4;   // tokens per thread; chunk = 128 tokens

// Kernel for (s, d, dtype): head dims 32 and 64 have compile-time instantiations (their channel
// loop is fully resolved at compile time); other dims use the runtime-d instantiation.
const void* pick(int s, int d, bool bf16) {
  if (d == 32) return kernel_d32(s, bf16);
  if (d == 64) return kernel_d64(s, bf16);
  return kernel_d0(s, bf16);
}

}  // namespace cdist_impl

using cdist_impl::pick;
using cdist_impl::CdistArgs;
using cdist_impl::kRows;

size_t cdist_smem_bytes(int s, int d, int tile, bool bf16) {
  const size_t m = (size_t)s * s;
  const size_t staged = 2 * (size_t)tile * d * (bf16 ? 2 : 4);
  return sizeof(float) * m * d + staged + (bf16 ? sizeof(float) * (size_t)tile * d : 0);
}

int cdist_tile_tokens() { return 32 * kRows; }

cudaError_t cdist_configure(int s, int d, bool bf16, size_t smem, int* ctas_per_sm) {
  const void* f = pick(s, d, bf16);
  if (!f) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, f, 32 * s, smem);
}

cudaError_t launch_cdist(const lapl_attn_plan& p, const void* q, const void* k, const void* v,
                         const float* landmarks, float* at, float* bt, float* stats,
                         float* dbg_dql, float* dbg_dlk, float* dbg_a, cudaStream_t st) {
  const Geometry& g = p.geo;
  CdistArgs a;
  a.q = q; a.k = k; a.v = v; a.landmarks = landmarks; a.at = at; a.bt = bt; a.stats = stats;
  a.dbg_dql = dbg_dql; a.dbg_dlk = dbg_dlk; a.dbg_a = dbg_a;
  a.part = g.cd_part;
  a.bh_count = g.bh;
  a.n = g.n; a.d = g.d; a.runs_q = g.cd_runs_q;
  a.c_exp = p.neg_log2e_over_lambda;
  const void* f = pick(g.s, g.d, p.cfg.in_dtype == LAPL_BF16);
  if (!f) return cudaErrorInvalidValue;
  void* args[] = {&a};
  return cudaLaunchKernel(f, dim3((unsigned)g.cd_part.ctas), dim3(32 * g.s), args, g.cd_smem, st);
}

}  // namespace lapl
