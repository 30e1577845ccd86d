// cdist.cu -- host side of the fused L1 distance + exp kernels: kernel choice, tensor maps,
// shared memory, occupancy and launch.
//
// Two kernels compute the same outputs (A^T and B^T):
//   cdist_tma_kernel (cdist_tma.cuh)   token chunks loaded by the Tensor Memory Accelerator into
//                                      a ring of 128B-swizzled stages, producer warp + consumer
//                                      warps on mbarriers; instantiated for fp32 with d in
//                                      {32, 64} and bf16 with d = 64;
//   cdist_exp_kernel (cdist_kernel.cuh) chunks loaded with cp.async by the whole CTA, every
//                                      shape, and the only one with Gaussian-kernel (squared
//                                      l2 distance) instantiations.
//   cdist_l1_kernel (cdist_l1.cuh)     TMA-fed like cdist_tma_kernel, with a helper warp and the
//                                      element work split between the FP32 and ALU pipes;
//                                      fp32 with d in {32, 64}, bf16 with d = 64, Laplacian
//                                      kernel.
//   gauss_tc_kernel (cdist_gauss_tc.cu) Gaussian kernel only: |x|^2 + |l|^2 - 2 x.l with x.l on
//                                      the tensor cores; fp32 or bf16, d in {32, 64}; the
//                                      automatic choice for the Gaussian kernel there.
// Automatic choice for the Laplacian kernel: cdist_l1_kernel wherever it is instantiated (fp32
// with d = 32 or 64, bf16 with d = 64); otherwise the TMA feed for fp32, d = 32, s <= 7; cp.async elsewhere (faster where the TMA
// kernel's extra producer warp costs registers, s = 8, or its consumer warps each widen the
// same bf16 chunk).  The environment variable LAPL_ATTN_CDIST_FEED=l1, =tma or =cp.async, read at
// plan creation, overrides the choice (l1 and tma only where instantiated and the tensor holds
// at least one chunk of rows).
#include <algorithm>
#include <stdlib.h>
#include <string.h>

#include "cdist_l1.cuh"
#include "cdist_tma.cuh"

namespace lapl {
namespace cdist_impl {
const void* kernel_d32(int s, bool bf16);
const void* kernel_d64(int s, bool bf16);
const void* kernel_d0(int s, bool bf16);
const void* gauss_d32(int s, bool bf16);
const void* gauss_d64(int s, bool bf16);
const void* gauss_d0(int s, bool bf16);

constexpr int kRows = 4;   // tokens per thread; chunk = 128 tokens

// Kernel for (s, d, dtype, distance): head dims 32 and 64 have compile-time instantiations
// (their channel loop is fully resolved at compile time); other dims use the runtime-d
// instantiation.
const void* pick(int s, int d, bool bf16, bool gauss) {
  if (gauss) {
    if (d == 32) return gauss_d32(s, bf16);
    if (d == 64) return gauss_d64(s, bf16);
    return gauss_d0(s, bf16);
  }
  if (d == 32) return kernel_d32(s, bf16);
  if (d == 64) return kernel_d64(s, bf16);
  return kernel_d0(s, bf16);
}

size_t smem_bytes(int s, int d, int tile, bool bf16) {
  const size_t m = (size_t)s * s;
  const size_t staged = 2 * (size_t)tile * d * (bf16 ? 2 : 4);
  return sizeof(float) * m * d + staged + (bf16 ? sizeof(float) * (size_t)tile * d : 0);
}
}  // namespace cdist_impl

namespace cdist_tma {
const void* kernel_f32(int s, int d);
const void* kernel_bf16(int s, int d);

const void* pick(int s, int d, bool bf16) { return bf16 ? kernel_bf16(s, d) : kernel_f32(s, d); }

// Dynamic shared memory: 1024 bytes of alignment slack, the stage ring, the landmark ring and
// the 2 * kStages mbarriers.
size_t smem_bytes(int s, int d, bool bf16) {
  const size_t m = (size_t)s * s;
  const size_t stage = (size_t)kTile * 128 * (bf16 ? 1 : d / 32);
  return 1024 + kStages * stage + (size_t)kLmSlots * m * d * sizeof(float) + 2 * kStages * 8;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, found once through the runtime (no link against libcuda).
EncodeTiledFn encoder() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    const cudaError_t e =
        cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// 2-D view [rows, d] of Q or K; a box is 128 rows of 128 bytes (32 fp32 or 64 bf16 channels),
// swizzled 128B; rows past the end read as zero.
bool encode(CUtensorMap* map, const void* base, long long rows, int d, bool bf16) {
  const EncodeTiledFn fn = encoder();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d * (bf16 ? 2 : 4)};
  const cuuint32_t box[2] = {bf16 ? 64u : 32u, (cuuint32_t)kTile};
  const cuuint32_t elem_strides[2] = {1, 1};
  const CUresult r =
      fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
         const_cast<void*>(base), dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
}  // namespace cdist_tma

bool tma_encode_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t inner,
                   uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  const cdist_tma::EncodeTiledFn fn = cdist_tma::encoder();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t elem_strides[2] = {1, 1};
  return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, elem_strides,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tma_encode_3d_sw128(CUtensorMap* map, const void* base, CUtensorMapDataType dtype,
                         uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2,
                         uint32_t b0, uint32_t b1) {
  const cdist_tma::EncodeTiledFn fn = cdist_tma::encoder();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
  const cuuint64_t strides[2] = {(cuuint64_t)s1, (cuuint64_t)s2};
  const cuuint32_t box[3] = {b0, b1, 1};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  return fn(map, dtype, 3, const_cast<void*>(base), dims, strides, box, elem_strides,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Error bits raised by device-side bounded waits; read and cleared by lapl_attn_device_errors.
__device__ unsigned g_device_errors;

cudaError_t device_error_word(unsigned** word) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_device_errors);
  *word = static_cast<unsigned*>(p);
  return e;
}

cudaError_t cdist_plan(lapl_attn_plan& p, int* ctas_per_sm) {
  Geometry& g = p.geo;
  const bool bf16 = p.cfg.in_dtype == LAPL_BF16;
  g.cd_rows = cdist_impl::kRows;
  g.cd_tile = 32 * g.cd_rows;
  const char* feed = getenv("LAPL_ATTN_CDIST_FEED");
  const bool want_l1 = feed && strcmp(feed, "l1") == 0;
  const bool want_tma = feed && strcmp(feed, "tma") == 0;
  const bool want_cpasync = feed && strcmp(feed, "cp.async") == 0;
  const bool gauss = p.cfg.kernel == LAPL_KERNEL_GAUSSIAN;
  const long long rows = (long long)g.bh * g.n;
  // Tensor-map coordinates are 32-bit; a box must not be taller than the tensor.
  const bool tma_ok = rows >= cdist_tma::kTile && rows < (1LL << 31) &&
                      cdist_tma::encoder() != nullptr;
  // The split-pipe kernel: fp32 with d = 32 or 64, or bf16 with d = 64; the Laplacian kernel.
  // Row groups per CTA: 1 (two CTAs of s consumer warps per SM) for s <= 7; 2 (one CTA of 2 s
  // consumer warps per SM) for s = 8, where one group's registers would not leave room for two
  // CTAs.  For s <= 7 two CTAs measured faster than one CTA of both groups (stage-1 shape 24.2
  // vs 24.7 us, 4x its heads 67.7 vs 71.9 us): their two copy pipelines fill each other's gaps.
  // LAPL_ATTN_CDIST_GROUPS=1 or 2 overrides.
  const char* grp = getenv("LAPL_ATTN_CDIST_GROUPS");
  g.cd_groups = grp && strcmp(grp, "1") == 0 ? 1 : grp && strcmp(grp, "2") == 0 ? 2
                                                                                 : (g.s == 8 ? 2 : 1);
  const void* fl1 = !gauss ? cdist_l1::kernel(g.s, g.d, g.cd_groups, bf16) : nullptr;
  g.cd_l1 = fl1 && tma_ok && (want_l1 || (!want_tma && !want_cpasync));
  // Gaussian kernel: the cross term x.l on the tensor cores where instantiated (d = 32 or 64;
  // the squared distance is |x|^2 + |l|^2 - 2 x.l); LAPL_ATTN_CDIST_FEED=cp.async forces the
  // CUDA-core kernel (direct sum of squared differences).
  const void* fg = gauss && !want_cpasync && g.m <= 64 ? gauss_tc_kernel_ptr(g.d, bf16) : nullptr;
  int smem_optin = 0;
  if (fg && (cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                    p.device) != cudaSuccess ||
             gauss_tc_smem_bytes(g.m, g.d, bf16) > (size_t)smem_optin)) {
    cudaGetLastError();
    fg = nullptr;
  }
  g.cd_gtc = fg != nullptr;
  const void* f = nullptr;
  if (g.cd_gtc) {
    f = fg;
    g.cd_l1 = false;
    g.cd_tma = false;
    g.cd_threads = gauss_tc_threads();
    g.cd_smem = gauss_tc_smem_bytes(g.m, g.d, bf16);
  } else if (g.cd_l1) {
    f = fl1;
    g.cd_tma = false;
    g.cd_threads = 32 * (g.cd_groups * g.s + 1);
    g.cd_smem = cdist_l1::smem_bytes(g.s, g.d, bf16, g.cd_groups);
  } else {
    const bool auto_tma = !bf16 && g.d == 32 && g.s <= 7;
    f = gauss ? nullptr : cdist_tma::pick(g.s, g.d, bf16);
    g.cd_tma = f && (want_tma || (auto_tma && !want_cpasync)) && tma_ok;
    if (g.cd_tma) {
      g.cd_threads = 32 * (g.s + 1);
      g.cd_smem = cdist_tma::smem_bytes(g.s, g.d, bf16);
    } else {
      f = cdist_impl::pick(g.s, g.d, bf16, gauss);
      g.cd_threads = 32 * g.s;
      g.cd_smem = cdist_impl::smem_bytes(g.s, g.d, g.cd_tile, bf16);
    }
  }
  if (!f) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)g.cd_smem);
  if (e != cudaSuccess) return e;
  if (g.cd_gtc) {
    // The tensor-core kernel asks for the largest shared-memory carveout; its CTAs per SM
    // follow from the SM's shared memory (with the per-CTA reservation), registers and
    // threads.  (The occupancy query reported one CTA per SM at d = 32, where two are
    // resident.)  Tensor memory is no limit: two CTAs take at most 2 x 128 of 512 columns.
    e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    int smem_sm = 0, reserved = 0, regs_sm = 0, threads_sm = 0;
    e = cudaFuncGetAttributes(&fa, f);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, p.device);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, p.device);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, p.device);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&threads_sm, cudaDevAttrMaxThreadsPerMultiProcessor, p.device);
    if (e != cudaSuccess) return e;
    const int by_smem = smem_sm / (int)(g.cd_smem + (size_t)reserved);
    const int regs_cta = ((fa.numRegs + 7) / 8 * 8) * g.cd_threads;
    const int by_regs = regs_cta > 0 ? regs_sm / regs_cta : 1;
    const int by_threads = threads_sm / g.cd_threads;
    *ctas_per_sm = std::max(1, std::min(std::min(by_smem, by_regs), std::min(by_threads, 2)));
    return cudaSuccess;
  }
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, f, g.cd_threads, g.cd_smem);
}

cudaError_t launch_cdist(const lapl_attn_plan& p, const void* q, const void* k, const void* v,
                         const float* landmarks, float* at, float* bt, float* dbg_dql,
                         float* dbg_dlk, float* dbg_a, cudaStream_t st) {
  const Geometry& g = p.geo;
  const bool bf16 = p.cfg.in_dtype == LAPL_BF16;
  if (g.cd_gtc)
    return launch_gauss_tc(p, q, k, landmarks, at, bt, dbg_dql, dbg_dlk, dbg_a, st);
  if (g.cd_tma || g.cd_l1) {
    const long long rows = (long long)g.bh * g.n;
    if (p.tmap_q_ptr != q) {
      if (!cdist_tma::encode(&p.tmap_q, q, rows, g.d, bf16)) return cudaErrorInvalidValue;
      p.tmap_q_ptr = q;
    }
    if (p.tmap_k_ptr != k) {
      if (!cdist_tma::encode(&p.tmap_k, k, rows, g.d, bf16)) return cudaErrorInvalidValue;
      p.tmap_k_ptr = k;
    }
    if (g.cd_l1) {
      cdist_l1::Args a;
      a.landmarks = landmarks; a.at = at; a.bt = bt; a.err = p.dev_err;
      a.dbg_dql = dbg_dql; a.dbg_dlk = dbg_dlk; a.dbg_a = dbg_a;
      a.part = g.cd_part;
      a.bh_count = g.bh;
      a.n = g.n;
      a.c_exp = p.neg_log2e_over_lambda;
      a.wait_ns = p.cd_wait_ns;
      a.skip_last_copy = p.cd_skip_last_copy == 1 ? 1 : 0;
      const void* f = cdist_l1::kernel(g.s, g.d, g.cd_groups, bf16);
      if (!f) return cudaErrorInvalidValue;
      void* args[] = {&a, &p.tmap_q, &p.tmap_k};
      return cudaLaunchKernel(f, dim3((unsigned)g.cd_part.ctas), dim3(g.cd_threads), args,
                              g.cd_smem, st);
    }
    cdist_tma::TmaArgs a;
    a.landmarks = landmarks; a.at = at; a.bt = bt; a.err = p.dev_err;
    a.dbg_dql = dbg_dql; a.dbg_dlk = dbg_dlk; a.dbg_a = dbg_a;
    a.part = g.cd_part;
    a.bh_count = g.bh;
    a.n = g.n;
    a.c_exp = p.neg_log2e_over_lambda;
    const void* f = cdist_tma::pick(g.s, g.d, bf16);
    if (!f) return cudaErrorInvalidValue;
    void* args[] = {&a, &p.tmap_q, &p.tmap_k};
    return cudaLaunchKernel(f, dim3((unsigned)g.cd_part.ctas), dim3(g.cd_threads), args, g.cd_smem,
                            st);
  }
  cdist_impl::CdistArgs a;
  a.q = q; a.k = k; a.v = v; a.landmarks = landmarks; a.at = at; a.bt = bt;
  a.dbg_dql = dbg_dql; a.dbg_dlk = dbg_dlk; a.dbg_a = dbg_a;
  a.part = g.cd_part;
  a.bh_count = g.bh;
  a.n = g.n; a.d = g.d;
  a.c_exp = p.neg_log2e_over_lambda;
  const void* f = cdist_impl::pick(g.s, g.d, bf16, p.cfg.kernel == LAPL_KERNEL_GAUSSIAN);
  if (!f) return cudaErrorInvalidValue;
  void* args[] = {&a};
  return cudaLaunchKernel(f, dim3((unsigned)g.cd_part.ctas), dim3(g.cd_threads), args, g.cd_smem, st);
}

}  // namespace lapl
