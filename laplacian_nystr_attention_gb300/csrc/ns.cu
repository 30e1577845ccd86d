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
// symmetric whenever X_t is a polynomial in W.  Every iterate is kept exactly symmetric: the
// update V = 2X - X P is evaluated in full and X_{t+1} = (V + V^T) / 2, entry by entry (the
// two sums of a mirrored pair are the same fp32 addition).  Averaging drops the antisymmetric
// part of V's rounding error; keeping one triangle instead turns that part into a symmetric
// error of the same size, which the slow (unconverged) modes of an ill-conditioned W double at
// every step (a Gaussian-kernel W with kappa ~ 3e3 and 20 steps loses about 10x in O).
// P = W X is computed in full and not symmetrised: symmetrising it drops its commutator part
// [W, X]/2, and in fp32 that error grows through the slow first phase of the iteration until
// it diverges (kappa(W) ~ 65 already does).  With A symmetric both factors are row reads,
// (A B)[i][j] = sum_k A[k][i] B[k][j].
//
// Products.  Matrices are stored 64 x 64 (zero padding, row stride kMS).  A warp owns a 32 x 32
// output tile and a quarter of the k range; lane (rq, cq) = (lane / 8, lane % 8) owns rows
// 8rq..8rq+7 and columns 4cq..4cq+3 of it.  Per k a warp issues two 128-bit reads of A (all 8
// lanes of a quarter-warp read the same address) and one of B (a quarter reads 128 contiguous
// bytes): 8 shared-memory wavefronts per 32 FMAs per lane.  The k quarters meet through shared
// memory in a lane-major (conflict-free) layout.
//
// Pairs.  For m > 32 (2 x 2 warp tiles) a head can run on a cluster of two CTAs
// (ns_pair_kernel): both build W and X0, each computes half of every product's output rows and
// stores them into its own and its peer's shared memory (distributed shared memory), and one
// cluster barrier per product makes the halves visible.  Every CTA executes the same sequence
// of barriers and none leaves early, so every barrier completes.
#include <cooperative_groups.h>

#include "ns_common.cuh"

namespace lapl {
using namespace ns_detail;
namespace {

constexpr int kNsThreads = 512;

template <int S>
__global__ void __launch_bounds__(kNsThreads)
ns_inverse_kernel(const float* __restrict__ landmarks, float* __restrict__ xout,
                  float* __restrict__ dbg_dll, float* __restrict__ dbg_w,
                  float* __restrict__ dbg_x, float* __restrict__ xs, int d, int T, float eps,
                  float c_exp, int gauss) {
  using Sh = NsShape<S>;
  constexpr int M = Sh::M, MP = kMS;
  extern __shared__ float4 smem_ns4[];
  const NsSmem sm = ns_smem_layout<S>(reinterpret_cast<float*>(smem_ns4));
  const long bh = blockIdx.x;
  ns_prologue<S, kNsThreads>(sm, landmarks + (size_t)bh * M * d, d, eps, c_exp, gauss != 0, true,
                             dbg_dll, dbg_w, bh);
  float* W = sm.W;
  float* X = sm.X;
  float* P = sm.P;
  float* Y = sm.Y;
  float* part = sm.part;
  float* xsh = xs ? xs + (size_t)bh * (T + 1) * M * Sh::MK : nullptr;

  save_iterate<M, kNsThreads>(X, xsh);
  for (int t = 0; t < T; ++t) {
    sym_product<Sh::MK, Sh::NWT, kPlain>(W, X, nullptr, P, part);   // P = W X
    sym_product<Sh::MK, Sh::NWT, kAvgUpdate>(X, P, X, Y, part);          // Y = 2X - X P
    float* tmp = X; X = Y; Y = tmp;
    save_iterate<M, kNsThreads>(X, xsh ? xsh + (size_t)(t + 1) * M * Sh::MK : nullptr);
  }

  for (int idx = threadIdx.x; idx < M * M; idx += kNsThreads) {
    const int i = idx / M, k = idx % M;
    const float x = X[i * MP + k];
    xout[(size_t)bh * M * M + idx] = x;
    if (dbg_x) dbg_x[(size_t)bh * M * M + idx] = x;
  }
}

// One product on a CTA pair (m > 32, 2 x 2 warp tiles).  The product's 16 output strips (8 rows
// x 32 columns, four per 32 x 32 tile, tile-major) are cut in two: CTA rank `crank` computes
// strips 8 crank .. 8 crank + 7, i.e. rows 32 crank .. 32 crank + 31.  A warp job is two
// adjacent strips, 16 rows of one tile; lane (rq, cq) = (lane / 8, lane % 8) holds rows
// 4rq..4rq+3 and columns 4cq..4cq+3 of it, and warp w takes job w % 4 over k quarter w / 4.
// Results are stored into C (kUpdate: V = 2 Xs - A B; otherwise A B); pair_publish then copies
// this CTA's rows into the peer, and for kUpdate pair_symmetrise averages V with V^T.
template <int MK, bool kUpdate>
__device__ __forceinline__ void pair_product(const float* __restrict__ A,
                                             const float* __restrict__ B,
                                             const float* __restrict__ Xs, float* C,
                                             float* __restrict__ part, int crank) {
  constexpr int KS = 4;
  constexpr int KQ = MK / KS;
  constexpr int NJOBS = 4;                           // two-strip jobs per CTA
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int job = warp & 3, ks = warp >> 2;
  const bool active = job < NJOBS;
  const int pair = crank * NJOBS + job;
  const int tile = pair >> 1, half = pair & 1;
  const int tr = tile >> 1, tc = tile & 1;
  const int rq = lane >> 3, cq = lane & 7;
  const int r0 = 32 * tr + 16 * half + 4 * rq, c0 = 32 * tc + 4 * cq;
  float acc[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
  if (active) {
    const float* a = A + (ks * KQ) * kMS + r0;
    const float* b = B + (ks * KQ) * kMS + c0;
    float4 av = *reinterpret_cast<const float4*>(a);
    float4 bv = *reinterpret_cast<const float4*>(b);
#pragma unroll
    for (int kk = 0; kk < KQ; ++kk) {
      const int kn = kk + 1 < KQ ? kk + 1 : kk;
      const float4 nav = *reinterpret_cast<const float4*>(a + kn * kMS);
      const float4 nbv = *reinterpret_cast<const float4*>(b + kn * kMS);
      const float ar[4] = {av.x, av.y, av.z, av.w};
      const float br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(ar[r], br[c], acc[r][c]);
      av = nav;
      bv = nbv;
    }
    if (ks > 0) {
#pragma unroll
      for (int e = 0; e < 16; ++e)
        part[(((ks - 1) * 4 + job) * 16 + e) * 32 + lane] = acc[e >> 2][e & 3];
    }
  }
  __syncthreads();
  if (active && ks == 0) {
#pragma unroll
    for (int q = 1; q < KS; ++q)
#pragma unroll
      for (int e = 0; e < 16; ++e)
        acc[e >> 2][e & 3] += part[(((q - 1) * 4 + job) * 16 + e) * 32 + lane];
    if constexpr (kUpdate) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float4 x4 = *reinterpret_cast<const float4*>(&Xs[(r0 + r) * kMS + c0]);
        *reinterpret_cast<float4*>(&C[(r0 + r) * kMS + c0]) =
            make_float4(2.f * x4.x - acc[r][0], 2.f * x4.y - acc[r][1], 2.f * x4.z - acc[r][2],
                        2.f * x4.w - acc[r][3]);
      }
    } else {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        *reinterpret_cast<float4*>(&C[(r0 + r) * kMS + c0]) =
            make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
      }
    }
  }
  __syncthreads();
}

// Copy this CTA's rows of a pair product (rows 32 crank .. 32 crank + 31) from C into the
// peer's copy Cpeer: one 16-byte store per thread (512 threads x 4 floats = 2048 floats).
__device__ __forceinline__ void pair_publish(const float* __restrict__ C, float* Cpeer,
                                             int crank) {
  const int t = threadIdx.x;             // 0 .. 511
  const int row = 32 * crank + (t >> 4), col = 4 * (t & 15);
  *reinterpret_cast<float4*>(&Cpeer[row * kMS + col]) =
      *reinterpret_cast<const float4*>(&C[row * kMS + col]);
}

// C <- (C + C^T) / 2 over the m x m block, in place: each unordered pair (i < j) is read and
// written by one thread.  Both CTAs of a pair hold the same V and compute the same result.
// Ends with a __syncthreads().
template <int M>
__device__ __forceinline__ void pair_symmetrise(float* C) {
  for (int idx = threadIdx.x; idx < M * M; idx += kNsThreads) {
    const int i = idx / M, j = idx - i * M;
    if (i < j) {
      const float a = 0.5f * (C[i * kMS + j] + C[j * kMS + i]);
      C[i * kMS + j] = a;
      C[j * kMS + i] = a;
    }
  }
  __syncthreads();
}

// One head per cluster of two CTAs (m > 32).  Both CTAs build W and X0; each product is split
// between them (pair_product) and published by a cluster barrier.
template <int S>
__global__ void __launch_bounds__(kNsThreads)
ns_pair_kernel(const float* __restrict__ landmarks, float* __restrict__ xout,
               float* __restrict__ dbg_dll, float* __restrict__ dbg_w,
               float* __restrict__ dbg_x, float* __restrict__ xs, int d, int T, float eps,
               float c_exp, int gauss) {
  using Sh = NsShape<S>;
  static_assert(Sh::NWT == 2, "the pair split assumes 2 x 2 warp tiles");
  constexpr int M = Sh::M, MP = kMS;
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  extern __shared__ float4 smem_ns4[];
  const NsSmem sm = ns_smem_layout<S>(reinterpret_cast<float*>(smem_ns4));
  const long bh = blockIdx.x >> 1;
  ns_prologue<S, kNsThreads>(sm, landmarks + (size_t)bh * M * d, d, eps, c_exp, gauss != 0,
                             crank == 0, dbg_dll, dbg_w, bh);
  float* X = sm.X;
  float* Y = sm.Y;
  float* Yp = cluster.map_shared_rank(sm.Y, crank ^ 1);
  float* Xp = cluster.map_shared_rank(sm.X, crank ^ 1);
  float* Pp = cluster.map_shared_rank(sm.P, crank ^ 1);
  cluster.sync();                  // the peer is running before anything is stored into it
  float* xsh = (xs && crank == 0) ? xs + (size_t)bh * (T + 1) * M * Sh::MK : nullptr;
  save_iterate<M, kNsThreads>(X, xsh);

  for (int t = 0; t < T; ++t) {
    pair_product<Sh::MK, false>(sm.W, X, nullptr, sm.P, sm.part, crank);   // P = W X
    pair_publish(sm.P, Pp, crank);
    cluster.sync();
    pair_product<Sh::MK, true>(X, sm.P, X, Y, sm.part, crank);            // V = 2X - X P
    pair_publish(Y, Yp, crank);
    cluster.sync();
    pair_symmetrise<M>(Y);                                                // Y = (V + V^T) / 2
    float* tmp = X; X = Y; Y = tmp;
    tmp = Xp; Xp = Yp; Yp = tmp;
    save_iterate<M, kNsThreads>(X, xsh ? xsh + (size_t)(t + 1) * M * Sh::MK : nullptr);
  }

  // Both CTAs hold the final X; each writes half of it.
  const int total = M * M, half = (total + 1) / 2;
  const int lo = crank == 0 ? 0 : half, hi = crank == 0 ? half : total;
  for (int idx = lo + threadIdx.x; idx < hi; idx += kNsThreads) {
    const int i = idx / M, k = idx % M;
    const float x = X[i * MP + k];
    xout[(size_t)bh * M * M + idx] = x;
    if (dbg_x) dbg_x[(size_t)bh * M * M + idx] = x;
  }
}

template <int S>
const void* ns_ptr() { return reinterpret_cast<const void*>(&ns_inverse_kernel<S>); }

template <int S>
const void* ns_pair_ptr() { return reinterpret_cast<const void*>(&ns_pair_kernel<S>); }

// Kernel for landmark grid side s on clusters of `cluster` CTAs (1, or 2 for s >= 6).
const void* pick_ns(int s, int cluster) {
  if (cluster == 2) {
    switch (s) {
      case 6: return ns_pair_ptr<6>();
      case 7: return ns_pair_ptr<7>();
      case 8: return ns_pair_ptr<8>();
      default: return nullptr;
    }
  }
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
  return sizeof(float) * (4 * 64 * (size_t)kMS + kRedFloats + Sh::PART_FLOATS + 64 * (size_t)d);
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

bool ns_cluster_supported(int s, int cluster) { return pick_ns(s, cluster) != nullptr; }

cudaError_t ns_configure(int s, int cluster, size_t smem, int* clusters_per_gpu) {
  const void* f = pick_ns(s, cluster);
  if (!f) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess || !clusters_per_gpu) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(cluster);
  cfg.blockDim = dim3(kNsThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(clusters_per_gpu, f, &cfg);
}

cudaError_t launch_ns(const lapl_attn_plan& p, const float* landmarks, float* x, float* dbg_dll,
                      float* dbg_w, float* dbg_x, float* xs, cudaStream_t st) {
  const Geometry& g = p.geo;
  const void* f = pick_ns(g.s, g.ns_cluster);
  if (!f) return cudaErrorInvalidValue;
  int d = g.d, T = p.cfg.ns_steps;
  float eps = p.cfg.eps, c_exp = p.neg_log2e_over_lambda;
  int gauss = p.cfg.kernel == LAPL_KERNEL_GAUSSIAN;
  void* args[] = {&landmarks, &x, &dbg_dll, &dbg_w, &dbg_x, &xs, &d, &T, &eps, &c_exp, &gauss};
  if (g.ns_cluster == 1)
    return cudaLaunchKernel(f, dim3((unsigned)g.bh), dim3(kNsThreads), args, g.ns_smem, st);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = g.ns_cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(g.bh * g.ns_cluster));
  cfg.blockDim = dim3(kNsThreads);
  cfg.dynamicSmemBytes = g.ns_smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, f, args);
}

}  // namespace lapl
