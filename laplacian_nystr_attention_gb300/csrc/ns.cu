// ns.cu -- landmark kernel matrix W and its Newton-Schulz inverse X.
//
// "LaplacianFormer: Rethinking Linear Attention with Laplacian Kernel", English explainer
// page, 2.C.2 (and German page, 2; Korean page, 2.3): W = k(L, L) + eps*I is inverted by the
// multiply-only Newton-Schulz iteration X <- X (2I - W X); eps*I keeps W strictly positive
// definite.  X0 = W^T / (|W|_1 |W|_inf) (largest absolute column sum times largest absolute
// row sum), exactly T steps.
//
// One CTA per (batch, head); the m x m matrices (m <= 64) live in shared memory, zero-padded
// to MP = a multiple of 4 (the padding stays exactly zero through the iteration).
//
// Symmetry.  W is symmetric, X0 = W^T / c is symmetric, and X_{t+1} = X_t (2I - W X_t) is
// symmetric whenever X_t is a polynomial in W.  The update X <- 2X - X P is therefore evaluated
// on the upper-triangle 4 x 4 blocks only and mirrored, so every iterate is exactly symmetric.
// P = W X is computed in full: mirroring it as well drops its commutator part [W, X]/2, and in
// fp32 that error grows through the slow first phase of the iteration until it diverges
// (kappa(W) ~ 65 already does), whereas mirroring one of the two products stays within
// rounding of the plain iteration.  With A symmetric both factors are row reads,
// (A B)[i][j] = sum_k A[k][i] B[k][j]: one 128-bit load of A and one of B per 16 FMAs.
// The k range of each product is cut into slices over groups of warps (see sym_product), so
// that enough warps are in flight.
#include "common.cuh"

namespace lapl {
namespace {

constexpr int kNsThreads = 1024;

// Work split of one product over the CTA: the blocks of the product are laid out 32 per warp
// in row-major (bi, bj) order, so a warp's 128-bit reads of A hit at most a few distinct
// addresses (broadcast) and its reads of B are contiguous rows; the k range is cut into KS
// slices, one per group of warps, whose partial 4x4 tiles are summed through shared memory in
// slice order.
constexpr int slices_for(int mp, int blocks) {
  return (mp % 4 == 0 && ((blocks + 31) / 32) * 4 <= kNsThreads / 32) ? 4
       : (mp % 2 == 0 && ((blocks + 31) / 32) * 2 <= kNsThreads / 32) ? 2 : 1;
}

template <int S>
struct NsShape {
  static constexpr int M = S * S;
  static constexpr int MP = (M + 3) & ~3;
  static constexpr int NT = MP / 4;                  // 4x4 blocks per side
  static constexpr int NFULL = NT * NT;              // all blocks (P = W X)
  static constexpr int NB = NT * (NT + 1) / 2;       // upper-triangle blocks (X update)
  static constexpr int KS1 = slices_for(MP, NFULL);
  static constexpr int KS2 = slices_for(MP, NB);
  static constexpr int PART_FLOATS = (KS1 * NFULL > KS2 * NB ? KS1 * NFULL : KS2 * NB) * 16;
};

// Block index -> (bi, bj): row-major over all blocks, or over the upper triangle.
template <int NT, bool kUpper>
__device__ __forceinline__ void block_of(int item, int& bi, int& bj) {
  if constexpr (kUpper) {
    int b = 0, rem = item;
    while (rem >= NT - b) {
      rem -= NT - b;
      ++b;
    }
    bi = b;
    bj = b + rem;
  } else {
    bi = item / NT;
    bj = item % NT;
  }
}

// C = A B for symmetric A (MP x MP, row-major): (A B)[i][j] = sum_k A[k][i] B[k][j].
// kMirror: the blocks are the upper triangle and C = 2 Xs - A B is written to (i, j) and
// (j, i).  Otherwise every block is computed and C = A B.  Ends with a __syncthreads().
template <int MP, int NBLK, int KS, bool kMirror>
__device__ __forceinline__ void sym_product(const float* __restrict__ A,
                                            const float* __restrict__ B,
                                            const float* __restrict__ Xs, float* __restrict__ C,
                                            float* __restrict__ part) {
  constexpr int NT = MP / 4;
  constexpr int WPS = (NBLK + 31) / 32;          // warps per k slice
  constexpr int KL = MP / KS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ks = warp / WPS;
  const int item = (warp % WPS) * 32 + lane;
  if (ks < KS && item < NBLK) {
    int bi, bj;
    block_of<NT, kMirror>(item, bi, bj);
    float acc[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
    const float* a = A + (ks * KL) * MP + 4 * bi;
    const float* b = B + (ks * KL) * MP + 4 * bj;
#pragma unroll
    for (int kk = 0; kk < KL; ++kk) {
      const float4 av = *reinterpret_cast<const float4*>(a + kk * MP);
      const float4 bv = *reinterpret_cast<const float4*>(b + kk * MP);
      const float ar[4] = {av.x, av.y, av.z, av.w};
      const float br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(ar[r], br[c], acc[r][c]);
    }
    float4* dst = reinterpret_cast<float4*>(part) + ((size_t)ks * NBLK + item) * 4;
#pragma unroll
    for (int r = 0; r < 4; ++r) dst[r] = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
  }
  __syncthreads();
  // Sum the KS slices of every output element, in slice order.
  for (int e = threadIdx.x; e < NBLK * 16; e += kNsThreads) {
    const int item2 = e >> 4, rc = e & 15;
    float v = part[e];
#pragma unroll
    for (int q = 1; q < KS; ++q) v += part[(size_t)q * NBLK * 16 + e];
    int bi, bj;
    block_of<NT, kMirror>(item2, bi, bj);
    const int i = 4 * bi + (rc >> 2), j = 4 * bj + (rc & 3);
    if constexpr (kMirror) {
      if (bi < bj || (rc >> 2) <= (rc & 3)) {
        const float y = 2.f * Xs[i * MP + j] - v;
        C[i * MP + j] = y;
        C[j * MP + i] = y;
      }
    } else {
      C[i * MP + j] = v;
    }
  }
  __syncthreads();
}

template <int S>
__global__ void __launch_bounds__(kNsThreads)
ns_inverse_kernel(const float* __restrict__ landmarks, float* __restrict__ xout,
                  float* __restrict__ dbg_dll, float* __restrict__ dbg_w,
                  float* __restrict__ dbg_x, int d, int T, float eps, float c_exp) {
  using Sh = NsShape<S>;
  constexpr int M = Sh::M, MP = Sh::MP;
  extern __shared__ float4 smem_ns4[];
  float* smem = reinterpret_cast<float*>(smem_ns4);
  const long bh = blockIdx.x;
  float* W = smem;               // [MP][MP]
  float* X = W + MP * MP;
  float* P = X + MP * MP;
  float* Y = P + MP * MP;
  float* red = Y + MP * MP;      // column sums [64], row sums [64], scale
  float* part = red + 132;       // partial 4x4 tiles of the k slices
  float* sL = part + Sh::PART_FLOATS;   // [M][d]

  const float4* Lg = reinterpret_cast<const float4*>(landmarks + (size_t)bh * M * d);
  for (int i = threadIdx.x; i < (M * d) >> 2; i += kNsThreads)
    reinterpret_cast<float4*>(sL)[i] = Lg[i];
  __syncthreads();

  // W = exp(-D_LL / lambda) + eps I (exactly symmetric: |a-b| == |b-a| and the same order).
  for (int idx = threadIdx.x; idx < MP * MP; idx += kNsThreads) {
    const int i = idx / MP, k = idx % MP;
    float w = 0.f;
    if (i < M && k < M) {
      float dist = 0.f;
      for (int c = 0; c < d; ++c) dist += fabsf(sL[i * d + c] - sL[k * d + c]);
      // k(x, x) = 1 exactly: D_LL[i][i] = 0 and exp(0) = 1.
      w = (i == k) ? 1.f + eps : laplacian_from_distance(dist, c_exp);
      const size_t o = ((size_t)bh * M + i) * M + k;
      if (dbg_dll) dbg_dll[o] = dist;
      if (dbg_w) dbg_w[o] = w;
    }
    W[idx] = w;
  }
  __syncthreads();

  // |W|_1 (largest absolute column sum) and |W|_inf (largest absolute row sum).
  if (threadIdx.x < M) {
    const int j = threadIdx.x;
    float cs = 0.f, rs = 0.f;
    for (int i = 0; i < M; ++i) {
      cs += fabsf(W[i * MP + j]);
      rs += fabsf(W[j * MP + i]);
    }
    red[j] = cs;
    red[64 + j] = rs;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float n1 = 0.f, ninf = 0.f;
    for (int j = 0; j < M; ++j) {
      n1 = fmaxf(n1, red[j]);
      ninf = fmaxf(ninf, red[64 + j]);
    }
    red[128] = n1 * ninf;
  }
  __syncthreads();
  const float scale = red[128];
  for (int idx = threadIdx.x; idx < MP * MP; idx += kNsThreads) {
    const int i = idx / MP, k = idx % MP;
    X[idx] = W[k * MP + i] / scale;     // X0 = W^T / (|W|_1 |W|_inf)
  }

  __syncthreads();

  for (int t = 0; t < T; ++t) {
    sym_product<MP, Sh::NFULL, Sh::KS1, false>(W, X, nullptr, P, part);   // P = W X
    sym_product<MP, Sh::NB, Sh::KS2, true>(X, P, X, Y, part);             // Y = 2X - X P
    float* tmp = X; X = Y; Y = tmp;
  }

  for (int idx = threadIdx.x; idx < M * M; idx += kNsThreads) {
    const int i = idx / M, k = idx % M;
    const float x = X[i * MP + k];
    xout[(size_t)bh * M * M + idx] = x;
    if (dbg_x) dbg_x[(size_t)bh * M * M + idx] = x;
  }
}

template <int S>
const void* ns_ptr() { return reinterpret_cast<const void*>(&ns_inverse_kernel<S>); }

const void* pick_ns(int s) {
  switch (s) {
    case 1: return ns_ptr<1>();
    case 2: return ns_ptr<2>();
    case 3: return ns_ptr<3>();
    case 4: return ns_ptr<4>();
    case 5: return ns_ptr<5>();
    case 6: return ns_ptr<6>();
    case 7: return ns_ptr<7>();
    case 8: return ns_ptr<8>();
    default: return nullptr;
  }
}

}  // namespace

template <int S>
size_t ns_smem_of(int d) {
  using Sh = NsShape<S>;
  return sizeof(float) * (4 * (size_t)Sh::MP * Sh::MP + 132 + Sh::PART_FLOATS + (size_t)Sh::M * d);
}

size_t ns_smem_bytes(int m, int d) {
  switch (m) {
    case 1: return ns_smem_of<1>(d);
    case 4: return ns_smem_of<2>(d);
    case 9: return ns_smem_of<3>(d);
    case 16: return ns_smem_of<4>(d);
    case 25: return ns_smem_of<5>(d);
    case 36: return ns_smem_of<6>(d);
    case 49: return ns_smem_of<7>(d);
    case 64: return ns_smem_of<8>(d);
    default: return 0;
  }
}

cudaError_t ns_configure(int s, size_t smem) {
  const void* f = pick_ns(s);
  if (!f) return cudaErrorInvalidValue;
  return cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t launch_ns(const lapl_attn_plan& p, const float* landmarks, float* x, float* dbg_dll,
                      float* dbg_w, float* dbg_x, cudaStream_t st) {
  const Geometry& g = p.geo;
  const void* f = pick_ns(g.s);
  if (!f) return cudaErrorInvalidValue;
  int d = g.d, T = p.cfg.ns_steps;
  float eps = p.cfg.eps, c_exp = p.neg_log2e_over_lambda;
  void* args[] = {&landmarks, &x, &dbg_dll, &dbg_w, &dbg_x, &d, &T, &eps, &c_exp};
  return cudaLaunchKernel(f, dim3((unsigned)g.bh), dim3(kNsThreads), args, g.ns_smem, st);
}

}  // namespace lapl
