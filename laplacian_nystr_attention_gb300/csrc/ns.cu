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
// The k range of a block is split over KP adjacent lanes, combined with shuffles, so that
// enough warps are in flight.
#include "common.cuh"

namespace lapl {
namespace {

constexpr int kNsThreads = 1024;

// Lanes per block: largest power of two <= 8 that divides MP and keeps blocks*KP <= threads.
constexpr int lanes_per_block(int mp, int blocks) {
  return (mp % 8 == 0 && blocks * 8 <= kNsThreads) ? 8
       : (mp % 4 == 0 && blocks * 4 <= kNsThreads) ? 4
       : (mp % 2 == 0 && blocks * 2 <= kNsThreads) ? 2 : 1;
}

template <int S>
struct NsShape {
  static constexpr int M = S * S;
  static constexpr int MP = (M + 3) & ~3;
  static constexpr int NT = MP / 4;                  // 4x4 blocks per side
  static constexpr int NFULL = NT * NT;              // all blocks (P = W X)
  static constexpr int NB = NT * (NT + 1) / 2;       // upper-triangle blocks (X update)
  static constexpr int KP1 = lanes_per_block(MP, NFULL);
  static constexpr int KP2 = lanes_per_block(MP, NB);
};

// C = A B for symmetric A (MP x MP, row-major): (A B)[i][j] = sum_k A[k][i] B[k][j].
// kMirror: C = 2 Xs - A B on an upper-triangle block, written to (i, j) and (j, i).
// Otherwise: C = A B on any block.
template <int MP, int KP, bool kMirror>
__device__ __forceinline__ void sym_product(const float* __restrict__ A,
                                            const float* __restrict__ B,
                                            const float* __restrict__ Xs, float* __restrict__ C,
                                            int bi, int bj, int kp, bool active) {
  constexpr int KLEN = MP / KP;
  float acc[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
  if (active) {
    const float* a = A + (kp * KLEN) * MP + 4 * bi;
    const float* b = B + (kp * KLEN) * MP + 4 * bj;
#pragma unroll
    for (int kk = 0; kk < KLEN; ++kk) {
      const float4 av = *reinterpret_cast<const float4*>(a + kk * MP);
      const float4 bv = *reinterpret_cast<const float4*>(b + kk * MP);
      const float ar[4] = {av.x, av.y, av.z, av.w};
      const float br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(ar[r], br[c], acc[r][c]);
    }
  }
#pragma unroll
  for (int o = 1; o < KP; o <<= 1)
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r][c] += __shfl_xor_sync(0xffffffffu, acc[r][c], o);
  if (active && kp == 0) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      if constexpr (kMirror) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int i = 4 * bi + r, j = 4 * bj + c;
          if (bi < bj || r <= c) {
            const float v = 2.f * Xs[i * MP + j] - acc[r][c];
            C[i * MP + j] = v;
            C[j * MP + i] = v;
          }
        }
      } else {
        *reinterpret_cast<float4*>(&C[(4 * bi + r) * MP + 4 * bj]) =
            make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
      }
    }
  }
}

template <int S>
__global__ void __launch_bounds__(kNsThreads)
ns_inverse_kernel(const float* __restrict__ landmarks, float* __restrict__ xout,
                  float* __restrict__ dbg_dll, float* __restrict__ dbg_w,
                  float* __restrict__ dbg_x, int d, int T, float eps, float c_exp) {
  using Sh = NsShape<S>;
  constexpr int M = Sh::M, MP = Sh::MP, NT = Sh::NT;
  constexpr int KP1 = Sh::KP1, KP2 = Sh::KP2;
  extern __shared__ float4 smem_ns4[];
  float* smem = reinterpret_cast<float*>(smem_ns4);
  const long bh = blockIdx.x;
  float* W = smem;               // [MP][MP]
  float* X = W + MP * MP;
  float* P = X + MP * MP;
  float* Y = P + MP * MP;
  float* red = Y + MP * MP;      // column sums [64], row sums [64], scale
  float* sL = red + 132;         // [M][d]

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
      w = laplacian_from_distance(dist, c_exp);
      if (i == k) w += eps;
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

  // Blocks of this lane group: any block for P = W X, an upper-triangle block for the update.
  const int item1 = threadIdx.x / KP1, kp1 = threadIdx.x % KP1;
  const bool act1 = item1 < Sh::NFULL;
  const int bi1 = act1 ? item1 / NT : 0, bj1 = act1 ? item1 % NT : 0;
  const int item2 = threadIdx.x / KP2, kp2 = threadIdx.x % KP2;
  const bool act2 = item2 < Sh::NB;
  int bi2 = 0, bj2 = 0;
  if (act2) {
    int rem = item2;
    while (rem >= NT - bi2) {
      rem -= NT - bi2;
      ++bi2;
    }
    bj2 = bi2 + rem;
  }
  __syncthreads();

  for (int t = 0; t < T; ++t) {
    sym_product<MP, KP1, false>(W, X, nullptr, P, bi1, bj1, kp1, act1);  // P = W X
    __syncthreads();
    sym_product<MP, KP2, true>(X, P, X, Y, bi2, bj2, kp2, act2);         // Y = 2X - X P
    __syncthreads();
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

size_t ns_smem_bytes(int m, int d) {
  const int mp = (m + 3) & ~3;
  return sizeof(float) * (4 * (size_t)mp * mp + 132 + (size_t)m * d);
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
