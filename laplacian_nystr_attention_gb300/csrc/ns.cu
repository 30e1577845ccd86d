// ns.cu -- landmark kernel matrix W and its Newton-Schulz inverse X.
//
// "LaplacianFormer: Rethinking Linear Attention with Laplacian Kernel", English explainer
// page, 2.C.2 (and German page, 2; Korean page, 2.3): W = k(L, L) + eps*I is inverted by the
// multiply-only Newton-Schulz iteration X <- X (2I - W X); eps*I keeps W strictly positive
// definite.  X0 = W^T / (|W|_1 |W|_inf) (largest absolute column sum times largest absolute
// row sum), exactly T steps.
//
// One CTA per (batch, head); the m x m matrices (m <= 64) live in shared memory, zero-padded
// to 64 x 64 (the padding stays exactly zero through the iteration).
//
// Symmetry.  W is symmetric, X0 = W^T / c is symmetric, and X_{t+1} = X_t (2I - W X_t) is
// symmetric whenever X_t is a polynomial in W.  The update X <- 2X - X P is therefore evaluated
// on the upper-triangle tiles only and mirrored, so every iterate is exactly symmetric.
// P = W X is computed in full: mirroring it as well drops its commutator part [W, X]/2, and in
// fp32 that error grows through the slow first phase of the iteration until it diverges
// (kappa(W) ~ 65 already does), whereas mirroring one of the two products stays within
// rounding of the plain iteration.  With A symmetric both factors are row reads,
// (A B)[i][j] = sum_k A[k][i] B[k][j].
//
// Products.  Matrices are stored 64 x 64 (zero padding, row stride kMS).  A warp owns a 32 x 32
// output tile and a quarter of the k range; lane (rq, cq) = (lane / 8, lane % 8) owns rows
// 8rq..8rq+7 and columns 4cq..4cq+3 of it.  Per k a warp issues two 128-bit reads of A (all 8
// lanes of a quarter-warp read the same address) and one of B (a quarter reads 128 contiguous
// bytes): 8 shared-memory wavefronts per 32 FMAs per lane.  The k quarters meet through shared
// memory in a lane-major (conflict-free) layout.
#include "common.cuh"

namespace lapl {
namespace {

constexpr int kNsThreads = 512;

constexpr int kMS = 68;   // stored row stride: 64 columns (padded) + 4, 16-byte aligned, and
                          // column-direction stores spread over more banks than with 64

template <int S>
struct NsShape {
  static constexpr int M = S * S;
  static constexpr int MK = (M + 3) & ~3;            // k range actually summed
  static constexpr int NWT = (M + 31) / 32;          // 32x32 warp tiles per side (1 or 2)
  static constexpr int PART_FLOATS = 4 * 3 * 32 * 32;  // 4 tiles x 3 upper slices x 32 x 32
};

// C = A B for symmetric A (row stride kMS): (A B)[i][j] = sum_k A[k][i] B[k][j].
// kMirror: only warp tiles tr <= tc, C = 2 Xs - A B written to (i, j) and (j, i) (on a diagonal
// tile only the entries with i <= j, so C is exactly symmetric).  Otherwise every tile, C = A B.
// Warp w: tile w % NTILES, k quarter w / NTILES (the four slice-0 warps land on four different
// sub-partitions).  Ends with a __syncthreads().
template <int MK, int NWT, bool kMirror>
__device__ __forceinline__ void sym_product(const float* __restrict__ A,
                                            const float* __restrict__ B,
                                            const float* __restrict__ Xs, float* __restrict__ C,
                                            float* __restrict__ part) {
  constexpr int NTILES = kMirror ? NWT * (NWT + 1) / 2 : NWT * NWT;
  constexpr int KS = 4;
  constexpr int KQ = MK / KS;                        // MK is a multiple of 4
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = warp % NTILES, ks = warp / NTILES;
  const bool active = ks < KS;
  int tr = 0, tc = 0;
  if (kMirror) {
    tr = (tile == 2) ? 1 : 0;                        // tiles (0,0), (0,1), (1,1)
    tc = (tile >= 1) ? 1 : 0;
  } else {
    tr = tile / NWT;
    tc = tile % NWT;
  }
  const int rq = lane >> 3, cq = lane & 7;
  const int r0 = 32 * tr + 8 * rq, c0 = 32 * tc + 4 * cq;
  float acc[8][4];
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
  if (active) {
    const float* a = A + (ks * KQ) * kMS + r0;
    const float* b = B + (ks * KQ) * kMS + c0;
    // Operands of step kk+1 are loaded while the 32 FMAs of step kk issue.
    float4 a0 = *reinterpret_cast<const float4*>(a);
    float4 a1 = *reinterpret_cast<const float4*>(a + 4);
    float4 bv = *reinterpret_cast<const float4*>(b);
#pragma unroll
    for (int kk = 0; kk < KQ; ++kk) {
      const int kn = kk + 1 < KQ ? kk + 1 : kk;
      const float4 na0 = *reinterpret_cast<const float4*>(a + kn * kMS);
      const float4 na1 = *reinterpret_cast<const float4*>(a + kn * kMS + 4);
      const float4 nbv = *reinterpret_cast<const float4*>(b + kn * kMS);
      const float ar[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(ar[r], br[c], acc[r][c]);
      a0 = na0;
      a1 = na1;
      bv = nbv;
    }
    if (ks > 0) {
#pragma unroll
      for (int e = 0; e < 32; ++e)
        part[(((ks - 1) * NTILES + tile) * 32 + e) * 32 + lane] = acc[e >> 2][e & 3];
    }
  }
  __syncthreads();
  if (active && ks == 0) {
#pragma unroll
    for (int q = 1; q < KS; ++q)
#pragma unroll
      for (int e = 0; e < 32; ++e)
        acc[e >> 2][e & 3] += part[(((q - 1) * NTILES + tile) * 32 + e) * 32 + lane];
    if constexpr (kMirror) {
      float v[8][4];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float4 x4 = *reinterpret_cast<const float4*>(&Xs[(r0 + r) * kMS + c0]);
        v[r][0] = 2.f * x4.x - acc[r][0];
        v[r][1] = 2.f * x4.y - acc[r][1];
        v[r][2] = 2.f * x4.z - acc[r][2];
        v[r][3] = 2.f * x4.w - acc[r][3];
      }
      if (tr == tc) {
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int i = r0 + r, j = c0 + c;
            if (i <= j) {
              C[i * kMS + j] = v[r][c];
              C[j * kMS + i] = v[r][c];
            }
          }
      } else {
#pragma unroll
        for (int r = 0; r < 8; ++r)
          *reinterpret_cast<float4*>(&C[(r0 + r) * kMS + c0]) =
              make_float4(v[r][0], v[r][1], v[r][2], v[r][3]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          *reinterpret_cast<float4*>(&C[(c0 + c) * kMS + r0]) =
              make_float4(v[0][c], v[1][c], v[2][c], v[3][c]);
          *reinterpret_cast<float4*>(&C[(c0 + c) * kMS + r0 + 4]) =
              make_float4(v[4][c], v[5][c], v[6][c], v[7][c]);
        }
      }
    } else {
#pragma unroll
      for (int r = 0; r < 8; ++r)
        *reinterpret_cast<float4*>(&C[(r0 + r) * kMS + c0]) =
            make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
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
  constexpr int M = Sh::M, MP = kMS;
  extern __shared__ float4 smem_ns4[];
  float* smem = reinterpret_cast<float*>(smem_ns4);
  const long bh = blockIdx.x;
  float* W = smem;               // [64][MP]
  float* X = W + 64 * MP;
  float* P = X + 64 * MP;
  float* Y = P + 64 * MP;
  float* red = Y + 64 * MP;      // column sums [64], scale at [128]
  float* part = red + 132;       // partial 4x4 tiles of the k slices
  float* sL = part + Sh::PART_FLOATS;   // [d][64], channel-major

  // Landmarks, stored channel-major (sL[c * 64 + j]): in the distance loop below a warp reads
  // one broadcast value and 32 consecutive values per channel, free of bank conflicts.
  const float* Lg = landmarks + (size_t)bh * M * d;
  for (int i = threadIdx.x; i < M * d; i += kNsThreads) {
    const int j = i / d, c = i % d;
    sL[c * 64 + j] = Lg[i];
  }
  __syncthreads();

  // W = exp(-D_LL / lambda) + eps I, zero outside m x m.  Exactly symmetric: |a-b| == |b-a|
  // and both orders sum the channels in the same order.
  for (int idx = threadIdx.x; idx < 64 * 64; idx += kNsThreads) {
    const int i = idx >> 6, k = idx & 63;
    float w = 0.f;
    if (i < M && k < M) {
      float dist = 0.f;
      for (int c = 0; c < d; ++c) dist += fabsf(sL[c * 64 + i] - sL[c * 64 + k]);
      // k(x, x) = 1 exactly: D_LL[i][i] = 0 and exp(0) = 1.
      w = (i == k) ? 1.f + eps : laplacian_from_distance(dist, c_exp);
      const size_t o = ((size_t)bh * M + i) * M + k;
      if (dbg_dll) dbg_dll[o] = dist;
      if (dbg_w) dbg_w[o] = w;
    }
    W[i * MP + k] = w;
  }
  __syncthreads();

  // |W|_1 = largest absolute column sum.  W is exactly symmetric, so row j holds the same
  // values in the same order as column j and |W|_inf (largest absolute row sum) equals |W|_1
  // bit for bit.
  if (threadIdx.x < M) {
    const int j = threadIdx.x;
    float cs = 0.f;
    for (int i = 0; i < M; ++i) cs += fabsf(W[i * MP + j]);
    red[j] = cs;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float n1 = 0.f;
    for (int j = 0; j < M; ++j) n1 = fmaxf(n1, red[j]);
    red[128] = n1 * n1;            // |W|_1 |W|_inf
  }
  __syncthreads();
  const float scale = red[128];
  for (int idx = threadIdx.x; idx < 64 * 64; idx += kNsThreads) {
    const int i = idx >> 6, k = idx & 63;
    X[i * MP + k] = W[i * MP + k] / scale;     // X0 = W^T / (|W|_1 |W|_inf); W^T == W exactly
  }
  __syncthreads();

  for (int t = 0; t < T; ++t) {
    sym_product<Sh::MK, Sh::NWT, false>(W, X, nullptr, P, part);   // P = W X
    sym_product<Sh::MK, Sh::NWT, true>(X, P, X, Y, part);          // Y = 2X - X P
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
  return sizeof(float) * (4 * 64 * (size_t)kMS + 132 + Sh::PART_FLOATS + 64 * (size_t)d);
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
