// pool.cu -- landmark pooling.
//
// Landmarks are average-pooled keys ("LaplacianFormer: Rethinking Linear Attention with
// Laplacian Kernel", English explainer page, 2.C.1): L[j] is the mean of K over the
// non-overlapping (grid_h/s) x (grid_w/s) window j = jr*s + jc of the token grid.
//
// One CTA per (landmark, head).  Threads are laid out as channel quads x token slices so that
// each warp reads whole 16-byte (fp32) or 8-byte (bf16) pieces of consecutive token rows; the
// slices are combined in a fixed order, so the result is deterministic.  HBM-bound: K is read
// exactly once.
#include "common.cuh"

namespace lapl {
namespace {

constexpr int kPoolThreads = 256;

template <bool kBf16>
__global__ void __launch_bounds__(kPoolThreads)
pool_landmarks_kernel(const void* __restrict__ kin, float* __restrict__ landmarks,
                      float* __restrict__ dbg, int grid_w, int n, int d, int s, int ph, int pw) {
  extern __shared__ float4 smem_pool[];
  const int m = s * s;
  const int j = (int)(blockIdx.x % m);   // landmark
  const long bh = blockIdx.x / m;        // (batch, head) slice
  const int d4 = d >> 2;               // channel quads
  const int slices = kPoolThreads / d4;
  const int quad = threadIdx.x % d4;
  const int slice = threadIdx.x / d4;
  const int jr = j / s, jc = j % s;
  const int win = ph * pw;

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (slice < slices) {
    // Four window positions per pass: their loads are issued before any is summed.
    for (int w0 = slice; w0 < win; w0 += 4 * slices) {
      float4 x[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int w = w0 + u * slices;
        x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (w < win) {
          const int r = jr * ph + w / pw;
          const int c = jc * pw + w % pw;
          const size_t tok = (size_t)bh * n + (size_t)r * grid_w + c;
          if constexpr (kBf16) {
            const uint2 raw = reinterpret_cast<const uint2*>(kin)[(tok * d >> 2) + quad];
            x[u] = make_float4(bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y));
          } else {
            x[u] = reinterpret_cast<const float4*>(kin)[(tok * d >> 2) + quad];
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc.x += x[u].x; acc.y += x[u].y; acc.z += x[u].z; acc.w += x[u].w;
      }
    }
    smem_pool[slice * d4 + quad] = acc;
  }
  __syncthreads();
  // Thread c < d combines the slices of channel c in slice order.
  for (int c = threadIdx.x; c < d; c += kPoolThreads) {
    const float* part = reinterpret_cast<const float*>(smem_pool);
    float sum = 0.f;
    for (int sl = 0; sl < slices; ++sl) sum += part[sl * d + c];
    const float val = sum / (float)win;
    const size_t o = ((size_t)bh * m + j) * d + c;
    landmarks[o] = val;
    if (dbg) dbg[o] = val;
  }
}

}  // namespace

cudaError_t launch_pool(const lapl_attn_plan& p, const void* k, float* landmarks,
                        float* dbg_landmarks, cudaStream_t st) {
  const Geometry& g = p.geo;
  const int s = g.s;
  const int ph = p.cfg.grid_h / s, pw = p.cfg.grid_w / s;
  const int d4 = g.d / 4;
  const int slices = kPoolThreads / d4;
  const size_t smem = (size_t)slices * d4 * sizeof(float4);
  const unsigned grid = (unsigned)(g.bh * g.m);
  if (p.cfg.in_dtype == LAPL_BF16)
    pool_landmarks_kernel<true><<<grid, kPoolThreads, smem, st>>>(
        k, landmarks, dbg_landmarks, p.cfg.grid_w, g.n, g.d, s, ph, pw);
  else
    pool_landmarks_kernel<false><<<grid, kPoolThreads, smem, st>>>(
        k, landmarks, dbg_landmarks, p.cfg.grid_w, g.n, g.d, s, ph, pw);
  return cudaGetLastError();
}

}  // namespace lapl
