// ns.cu -- landmark kernel matrix W and its Newton-Schulz inverse X.
//
// "LaplacianFormer: Rethinking Linear Attention with Laplacian Kernel", English explainer
// page, 2.C.2 (and German page, 2; Korean page, 2.3): W = k(L, L) + eps*I is inverted by the
// multiply-only Newton-Schulz iteration X <- X (2I - W X); eps*I keeps W strictly positive
// definite.  X0 = W^T / (|W|_1 |W|_inf) (largest absolute column sum times largest absolute
// row sum), exactly T steps.
//
// One CTA per (batch, head): the m x m matrices (m <= 64) live in shared memory, zero-padded
// to a multiple of 4 so that every thread owns a 4 x 4 register tile of each product; the
// padding rows and columns stay exactly zero through the iteration.  Each step is
// P = W X followed by X <- 2X - X P, in fp32.
#include "common.cuh"

namespace lapl {
namespace {

constexpr int kNsThreads = 256;

// C = A B (mp x mp, row-major, shared memory).  If kTwoXMinus, C = 2*Xs - A B instead.
template <bool kTwoXMinus>
__device__ __forceinline__ void small_matmul(const float* __restrict__ A,
                                             const float* __restrict__ Bm,
                                             const float* __restrict__ Xs, float* __restrict__ C,
                                             int mp) {
  const int nt = mp >> 2;
  for (int tile = threadIdx.x; tile < nt * nt; tile += kNsThreads) {
    const int ti = tile / nt, tj = tile % nt;
    float acc[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
    for (int k = 0; k < mp; ++k) {
      float a[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) a[r] = A[(4 * ti + r) * mp + k];
      const float4 b = *reinterpret_cast<const float4*>(&Bm[k * mp + 4 * tj]);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        acc[r][0] = fmaf(a[r], b.x, acc[r][0]);
        acc[r][1] = fmaf(a[r], b.y, acc[r][1]);
        acc[r][2] = fmaf(a[r], b.z, acc[r][2]);
        acc[r][3] = fmaf(a[r], b.w, acc[r][3]);
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float4 o;
      float* op = reinterpret_cast<float*>(&o);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int idx = (4 * ti + r) * mp + 4 * tj + c;
        op[c] = kTwoXMinus ? 2.f * Xs[idx] - acc[r][c] : acc[r][c];
      }
      *reinterpret_cast<float4*>(&C[(4 * ti + r) * mp + 4 * tj]) = o;
    }
  }
}

__global__ void __launch_bounds__(kNsThreads)
ns_inverse_kernel(const float* __restrict__ landmarks, float* __restrict__ xout,
                  float* __restrict__ dbg_dll, float* __restrict__ dbg_w,
                  float* __restrict__ dbg_x, int m, int d, int T, float eps, float c_exp) {
  extern __shared__ float4 smem_ns4[];
  float* smem = reinterpret_cast<float*>(smem_ns4);
  const int mp = (m + 3) & ~3;
  const long bh = blockIdx.x;
  float* sL = smem;              // [m][d]
  float* W = sL + m * d;         // [mp][mp]  (m*d is a multiple of 8: 16-byte aligned)
  float* X = W + mp * mp;
  float* P = X + mp * mp;
  float* Y = P + mp * mp;
  float* red = Y + mp * mp;      // column sums [64], row sums [64], scale

  const float4* Lg = reinterpret_cast<const float4*>(landmarks + (size_t)bh * m * d);
  for (int i = threadIdx.x; i < (m * d) >> 2; i += kNsThreads)
    reinterpret_cast<float4*>(sL)[i] = Lg[i];
  __syncthreads();

  // W = exp(-D_LL / lambda) + eps I, zero padding outside m x m.
  for (int idx = threadIdx.x; idx < mp * mp; idx += kNsThreads) {
    const int i = idx / mp, k = idx % mp;
    float w = 0.f;
    if (i < m && k < m) {
      float dist = 0.f;
      for (int c = 0; c < d; ++c) dist += fabsf(sL[i * d + c] - sL[k * d + c]);
      w = laplacian_from_distance(dist, c_exp);
      if (i == k) w += eps;
      const size_t o = ((size_t)bh * m + i) * m + k;
      if (dbg_dll) dbg_dll[o] = dist;
      if (dbg_w) dbg_w[o] = w;
    }
    W[idx] = w;
  }
  __syncthreads();

  // |W|_1 (largest absolute column sum) and |W|_inf (largest absolute row sum).
  if (threadIdx.x < m) {
    const int j = threadIdx.x;
    float cs = 0.f, rs = 0.f;
    for (int i = 0; i < m; ++i) {
      cs += fabsf(W[i * mp + j]);
      rs += fabsf(W[j * mp + i]);
    }
    red[j] = cs;
    red[64 + j] = rs;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float n1 = 0.f, ninf = 0.f;
    for (int j = 0; j < m; ++j) {
      n1 = fmaxf(n1, red[j]);
      ninf = fmaxf(ninf, red[64 + j]);
    }
    red[128] = n1 * ninf;
  }
  __syncthreads();
  const float scale = red[128];
  for (int idx = threadIdx.x; idx < mp * mp; idx += kNsThreads) {
    const int i = idx / mp, k = idx % mp;
    X[idx] = W[k * mp + i] / scale;     // X0 = W^T / (|W|_1 |W|_inf)
  }
  __syncthreads();

  for (int t = 0; t < T; ++t) {
    small_matmul<false>(W, X, nullptr, P, mp);   // P = W X
    __syncthreads();
    small_matmul<true>(X, P, X, Y, mp);          // Y = 2X - X P = X (2I - W X)
    __syncthreads();
    float* tmp = X; X = Y; Y = tmp;
  }

  for (int idx = threadIdx.x; idx < m * m; idx += kNsThreads) {
    const int i = idx / m, k = idx % m;
    const float x = X[i * mp + k];
    xout[(size_t)bh * m * m + idx] = x;
    if (dbg_x) dbg_x[(size_t)bh * m * m + idx] = x;
  }
}

}  // namespace

size_t ns_smem_bytes(int m, int d) {
  const int mp = (m + 3) & ~3;
  return sizeof(float) * ((size_t)m * d + 4 * (size_t)mp * mp + 132);
}

cudaError_t ns_configure(size_t smem) {
  return cudaFuncSetAttribute(ns_inverse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem);
}

cudaError_t launch_ns(const lapl_attn_plan& p, const float* landmarks, float* x, float* dbg_dll,
                      float* dbg_w, float* dbg_x, cudaStream_t st) {
  const Geometry& g = p.geo;
  ns_inverse_kernel<<<(unsigned)g.bh, kNsThreads, g.ns_smem, st>>>(
      landmarks, x, dbg_dll, dbg_w, dbg_x, g.m, g.d, p.cfg.ns_steps, p.cfg.eps,
      p.neg_log2e_over_lambda);
  return cudaGetLastError();
}

}  // namespace lapl
