// ns_common.cuh -- pieces shared by the Newton-Schulz kernels (ns.cu: CUDA-core products on one
// CTA or a CTA pair; ns_tc.cu: tensor-core products): the padded matrix shape, the
// shared-memory layout and the prologue that builds W = k(L, L) + eps I and X0.
#pragma once

#include "common.cuh"

namespace lapl {
namespace ns_detail {


constexpr int kMS = 68;   // stored row stride: 64 columns (padded) + 4, 16-byte aligned, and
                          // column-direction stores spread over more banks than with 64

constexpr int kRedFloats = 8 * 64 + 4;   // partial column sums of up to 8 row groups, maxima

template <int S>
struct NsShape {
  static constexpr int M = S * S;
  static constexpr int MK = (M + 3) & ~3;            // k range actually summed
  static constexpr int NWT = (M + 31) / 32;          // 32x32 warp tiles per side (1 or 2)
  static constexpr int PART_FLOATS = 4 * 3 * 32 * 32;  // 4 tiles x 3 upper slices x 32 x 32
};

// Shared-memory layout of both kernels.
struct NsSmem {
  float* W;
  float* X;
  float* P;
  float* Y;
  float* red;
  float* part;
  float* sL;
};

template <int S>
__device__ __forceinline__ NsSmem ns_smem_layout(float* smem) {
  NsSmem m;
  m.W = smem;                   // [64][kMS]
  m.X = m.W + 64 * kMS;
  m.P = m.X + 64 * kMS;
  m.Y = m.P + 64 * kMS;
  m.red = m.Y + 64 * kMS;       // partial column sums and maxima [kRedFloats]
  m.part = m.red + kRedFloats;  // partial tiles of the k slices
  m.sL = m.part + NsShape<S>::PART_FLOATS;   // [d][64], channel-major
  return m;
}

// W = k(L, L) + eps I and X0 = W^T / (|W|_1 |W|_inf) in shared memory (zero-padded to 64 x 64,
// row stride kMS), for a CTA of NT threads.  The debug copies of D_LL and W are written when
// write_debug is set.  red holds NT / 64 x 64 partial column sums plus two maxima
// (kRedFloats).  Ends synchronised.
//
// Thread t owns column k = t % 64 and the RPG = 64 / (NT / 64) rows starting at
// (t / 64) * RPG; per channel it reads its own landmark value and RPG / 4 broadcast 16-byte
// pieces, and keeps RPG independent sums.  Each distance adds |L_ic - L_kc| (or its square, for
// the Gaussian kernel) over c ascending, the same terms in the same order for (i, k) and (k, i),
// so W is exactly symmetric.
// acc[r] += D(L_{i0 + r}, L_k) over the d channels of the channel-major landmarks sL: the L1
// distance, or the squared l2 distance (gauss).  x - y and y - x are exact negatives of each
// other, so both distances are exactly symmetric in (i, k).
template <int RPG, bool kGauss>
__device__ __forceinline__ void landmark_distances(const float* __restrict__ sL, int d, int k,
                                                   int i0, float (&acc)[RPG]) {
#pragma unroll 4
  for (int c = 0; c < d; ++c) {
    const float lk = sL[c * 64 + k];
#pragma unroll
    for (int r4 = 0; r4 < RPG / 4; ++r4) {
      const float4 li = *reinterpret_cast<const float4*>(&sL[c * 64 + i0 + 4 * r4]);
      const float e0 = li.x - lk, e1 = li.y - lk, e2 = li.z - lk, e3 = li.w - lk;
      if constexpr (kGauss) {
        acc[4 * r4 + 0] = fmaf(e0, e0, acc[4 * r4 + 0]);
        acc[4 * r4 + 1] = fmaf(e1, e1, acc[4 * r4 + 1]);
        acc[4 * r4 + 2] = fmaf(e2, e2, acc[4 * r4 + 2]);
        acc[4 * r4 + 3] = fmaf(e3, e3, acc[4 * r4 + 3]);
      } else {
        acc[4 * r4 + 0] += fabsf(e0);
        acc[4 * r4 + 1] += fabsf(e1);
        acc[4 * r4 + 2] += fabsf(e2);
        acc[4 * r4 + 3] += fabsf(e3);
      }
    }
  }
}

template <int S, int NT>
__device__ __forceinline__ void ns_prologue(const NsSmem& sm, const float* __restrict__ Lg, int d,
                                            float eps, float c_exp, bool gauss, bool write_debug,
                                            float* __restrict__ dbg_dll,
                                            float* __restrict__ dbg_w, long bh) {
  constexpr int M = S * S, MP = kMS;
  constexpr int G = NT / 64, RPG = 64 / G;
  static_assert(NT % 64 == 0 && RPG % 4 == 0, "row groups of a multiple of 4 rows");
  float* W = sm.W;
  float* X = sm.X;
  float* red = sm.red;
  float* sL = sm.sL;
  // Landmarks, stored channel-major (sL[c * 64 + j], zero for j >= m).  Up to 8 loads per
  // thread are issued before any is stored.
  for (int i0 = threadIdx.x; i0 < 64 * d; i0 += 8 * NT) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * NT, c = i >> 6, j = i & 63;
      v[u] = (i < 64 * d && j < M) ? __ldg(&Lg[j * d + c]) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * NT;
      if (i < 64 * d) sL[i] = v[u];
    }
  }
  __syncthreads();

  const int k = threadIdx.x & 63, g = threadIdx.x >> 6, i0 = g * RPG;
  float acc[RPG];
#pragma unroll
  for (int r = 0; r < RPG; ++r) acc[r] = 0.f;
  if (i0 < M) {                                   // uniform over the 64 threads of a group
    if (gauss) landmark_distances<RPG, true>(sL, d, k, i0, acc);
    else landmark_distances<RPG, false>(sL, d, k, i0, acc);
  }
  // W = exp(-D_LL / lambda) + eps I, zero outside m x m; k(x, x) = 1 exactly (D_LL[i][i] = 0).
  float cs = 0.f;
#pragma unroll
  for (int r = 0; r < RPG; ++r) {
    const int i = i0 + r;
    float w = 0.f;
    if (i < M && k < M) {
      w = (i == k) ? 1.f + eps : laplacian_from_distance(acc[r], c_exp);
      if (write_debug) {
        const size_t o = ((size_t)bh * M + i) * M + k;
        if (dbg_dll) dbg_dll[o] = acc[r];
        if (dbg_w) dbg_w[o] = w;
      }
    }
    acc[r] = w;
    W[i * MP + k] = w;
    cs += fabsf(w);
  }
  red[g * 64 + k] = cs;
  __syncthreads();
  // |W|_1 = largest absolute column sum; W is exactly symmetric, so |W|_inf (largest absolute
  // row sum) equals it.
  if (threadIdx.x < 64) {
    float col = 0.f;
#pragma unroll
    for (int q = 0; q < G; ++q) col += red[q * 64 + threadIdx.x];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) col = fmaxf(col, __shfl_xor_sync(0xffffffffu, col, o));
    if ((threadIdx.x & 31) == 0) red[G * 64 + (threadIdx.x >> 5)] = col;
  }
  __syncthreads();
  const float n1 = fmaxf(red[G * 64], red[G * 64 + 1]);
  const float scale = n1 * n1;                    // |W|_1 |W|_inf
  // X0 = W^T / scale, as a product with 1 / scale: one division per thread (eight IEEE
  // divisions measured 2.4K cycles of the solve's critical path); X0 is the start of a
  // self-correcting iteration, and its last-bit rounding is the same in every solve kernel.
  const float inv_scale = 1.f / scale;
#pragma unroll
  for (int r = 0; r < RPG; ++r) X[(i0 + r) * MP + k] = acc[r] * inv_scale;
  __syncthreads();
}

// Barrier of the first `threads` threads of the CTA (whole warps), named barrier 1.
__device__ __forceinline__ void warps_barrier(int threads) {
  asm volatile("bar.sync 1, %0;\n" ::"r"(threads) : "memory");
}

// What sym_product does with the product P = A^T B.
enum ProductMode {
  kPlain = 0,      // C = P (and Ct = P^T when Ct is given)
  kAvgUpdate = 1,  // C = (V + V^T) / 2 with V = 2 Xs - P   (the Newton-Schulz update)
  kSymRecur = 2,   // C = V + V^T with V = Xs - P           (2 Xs - P - P^T for symmetric Xs)
  kSubtract = 3    // C -= P
};

// P = A^T B for 64 x 64 matrices with row stride kMS: P[i][j] = sum_k A[k][i] B[k][j], so
// for a symmetric A it is A B and both operands are read by rows; 512 threads.
// Warp w: tile w % NTILES, k quarter w / NTILES (the four slice-0 warps land on four different
// sub-partitions); the slice-0 warps (0 .. NTILES-1) reduce and store, and for the symmetrising
// modes meet at a named barrier between writing V and reading its transpose.  Ends with a
// __syncthreads().
template <int MK, int NWT, int kMode>
__device__ __forceinline__ void sym_product(const float* __restrict__ A,
                                            const float* __restrict__ B,
                                            const float* __restrict__ Xs, float* __restrict__ C,
                                            float* __restrict__ part, float* __restrict__ Ct = nullptr) {
  constexpr int NTILES = NWT * NWT;
  constexpr int KS = 4;
  constexpr int KQ = MK / KS;                        // MK is a multiple of 4
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = warp % NTILES, ks = warp / NTILES;
  const bool active = ks < KS;
  const int tr = tile / NWT, tc = tile % NWT;
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
    if constexpr (kMode == kAvgUpdate || kMode == kSymRecur) {
      constexpr float kx = kMode == kAvgUpdate ? 2.f : 1.f;     // V = kx Xs - P
      constexpr float kc = kMode == kAvgUpdate ? 0.5f : 1.f;    // C = kc (V + V^T)
      float v[8][4];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float4 x4 = *reinterpret_cast<const float4*>(&Xs[(r0 + r) * kMS + c0]);
        v[r][0] = kx * x4.x - acc[r][0];
        v[r][1] = kx * x4.y - acc[r][1];
        v[r][2] = kx * x4.z - acc[r][2];
        v[r][3] = kx * x4.w - acc[r][3];
        *reinterpret_cast<float4*>(&C[(r0 + r) * kMS + c0]) =
            make_float4(v[r][0], v[r][1], v[r][2], v[r][3]);
      }
      warps_barrier(32 * NTILES);                    // V complete
      float vt[8][4];                                // vt[r][c] = V[c0 + c][r0 + r]
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float4 t0 = *reinterpret_cast<const float4*>(&C[(c0 + c) * kMS + r0]);
        const float4 t1 = *reinterpret_cast<const float4*>(&C[(c0 + c) * kMS + r0 + 4]);
        vt[0][c] = t0.x; vt[1][c] = t0.y; vt[2][c] = t0.z; vt[3][c] = t0.w;
        vt[4][c] = t1.x; vt[5][c] = t1.y; vt[6][c] = t1.z; vt[7][c] = t1.w;
      }
      warps_barrier(32 * NTILES);                    // every transpose read before any write
#pragma unroll
      for (int r = 0; r < 8; ++r)
        *reinterpret_cast<float4*>(&C[(r0 + r) * kMS + c0]) =
            make_float4(kc * (v[r][0] + vt[r][0]), kc * (v[r][1] + vt[r][1]),
                        kc * (v[r][2] + vt[r][2]), kc * (v[r][3] + vt[r][3]));
    } else if constexpr (kMode == kSubtract) {
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        float4* cp = reinterpret_cast<float4*>(&C[(r0 + r) * kMS + c0]);
        const float4 o = *cp;
        *cp = make_float4(o.x - acc[r][0], o.y - acc[r][1], o.z - acc[r][2], o.w - acc[r][3]);
      }
    } else {
#pragma unroll
      for (int r = 0; r < 8; ++r)
        *reinterpret_cast<float4*>(&C[(r0 + r) * kMS + c0]) =
            make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
      if (Ct) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          *reinterpret_cast<float4*>(&Ct[(c0 + c) * kMS + r0]) =
              make_float4(acc[0][c], acc[1][c], acc[2][c], acc[3][c]);
          *reinterpret_cast<float4*>(&Ct[(c0 + c) * kMS + r0 + 4]) =
              make_float4(acc[4][c], acc[5][c], acc[6][c], acc[7][c]);
        }
      }
    }
  }
  __syncthreads();
}

// Copy the first M rows of X (row stride kMS) to dst as M rows of MK = 4 ceil(M / 4) floats
// (the columns past M are X's zero padding), one float4 per thread and step, with the CTA's
// NT threads: the iterates the backward pass runs through.  Nothing when dst is null.
template <int M, int NT>
__device__ __forceinline__ void save_iterate(const float* __restrict__ X, float* __restrict__ dst) {
  if (!dst) return;
  constexpr int Q = (M + 3) / 4;            // float4 per row
  for (int e = threadIdx.x; e < M * Q; e += NT) {
    const int r = e / Q, c4 = e - r * Q;
    *reinterpret_cast<float4*>(&dst[(r * Q + c4) * 4]) =
        *reinterpret_cast<const float4*>(&X[r * kMS + 4 * c4]);
  }
}

}  // namespace ns_detail
}  // namespace lapl
