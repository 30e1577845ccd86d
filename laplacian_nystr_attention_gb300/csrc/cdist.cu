// cdist.cu -- fused L1 distance + Laplacian kernel for the query and key blocks.
//
// "LaplacianFormer: Rethinking Linear Attention with Laplacian Kernel": the similarity is
// k(x, y) = exp(-||x - y||_1 / lambda) (English explainer page, 2.A), and the distance and the
// exponential are computed in one fused kernel (German page, 2, CUDA-Optimierung; Chinese page,
// 2.2).  The L1 distance is a sum of |a - b|, not a dot product, so it runs on the FP32 CUDA
// cores.
//
// Grid: blockIdx.y selects the side, blockIdx.x = (batch*head, split).
//   side 0 (queries):  A = k(Q, L) for a tile of tokens; the tile is stored landmark-major
//                      into A^T [BH, m, N] and its per-landmark (mean, M2) over the tile's
//                      tokens is reduced with warp shuffles into the per-tile statistics.
//   side 1 (keys):     B = k(L, K) for a tile of keys, immediately contracted with the tile of
//                      V into a per-CTA partial of B V [m, d] held in registers across the
//                      CTA's consecutive tiles (B is never written to memory).
//
// Block: s warps for m = s*s landmarks.  Warp w owns landmarks w*s .. w*s+s-1 (so every
// landmark read from shared memory is a warp-wide broadcast), lane l owns tokens
// l, l+32, .. l+32*(R-1) of the tile.  Per 4 channels a thread issues R + s 128-bit shared
// loads for 8*R*s FP32 instructions (subtract, then add the absolute value).  The token tile is
// kept in shared memory with its 16-byte chunks XOR-swizzled by the row, so the 8 lanes of a
// 128-bit load phase hit 8 different bank groups.
#include "common.cuh"

namespace lapl {
namespace {

struct CdistArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* landmarks;
  float* at;        // [BH, m, N]
  float* stats;     // [BH, tiles, 2, m]
  float* bvp;       // [BH, splits, m, d]
  float* dbg_dql;   // [BH, N, m]
  float* dbg_dlk;   // [BH, m, N]
  float* dbg_a;     // [BH, N, m]
  int n, d, tiles, tiles_per_split, splits;
  float c_exp;
};

__device__ __forceinline__ int swizzle_mask(int d) {
  const int d4 = d >> 2;
  const int low = d4 & (-d4);
  return (low < 8 ? low : 8) - 1;
}

// Stage rows [n0, n0+tile) of a [N, d] matrix into shared memory as fp32, zero beyond N.
// kSwizzle: 16-byte chunk c of row t is stored at chunk c ^ (t & mask).  Each thread keeps one
// chunk column and walks the rows, so no index needs a division inside the loop.
template <bool kBf16, bool kSwizzle>
__device__ __forceinline__ void stage_rows(const void* __restrict__ src, float* __restrict__ dst,
                                           size_t row0, int valid, int tile, int d, int mask,
                                           int nthreads) {
  if constexpr (kBf16) {
    const int d8 = d >> 3;
    const int rstep = nthreads / d8;
    const int c8 = threadIdx.x % d8;
    const int t0 = threadIdx.x / d8;
    if (t0 >= rstep) return;
    const uint4* s8 = reinterpret_cast<const uint4*>(src) + ((row0 * d) >> 3) + c8;
    const int c0 = 2 * c8, c1 = 2 * c8 + 1;
    for (int t = t0; t < tile; t += rstep) {
      uint4 raw = make_uint4(0u, 0u, 0u, 0u);
      if (t < valid) raw = s8[(size_t)t * d8];
      const float4 lo = make_float4(bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y));
      const float4 hi = make_float4(bf16_lo(raw.z), bf16_hi(raw.z), bf16_lo(raw.w), bf16_hi(raw.w));
      const int p0 = kSwizzle ? (c0 ^ (t & mask)) : c0;
      const int p1 = kSwizzle ? (c1 ^ (t & mask)) : c1;
      *reinterpret_cast<float4*>(&dst[t * d + 4 * p0]) = lo;
      *reinterpret_cast<float4*>(&dst[t * d + 4 * p1]) = hi;
    }
  } else {
    const int d4 = d >> 2;
    const int rstep = nthreads / d4;
    const int c4 = threadIdx.x % d4;
    const int t0 = threadIdx.x / d4;
    if (t0 >= rstep) return;
    const float4* s4 = reinterpret_cast<const float4*>(src) + ((row0 * d) >> 2) + c4;
    for (int t = t0; t < tile; t += rstep) {
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t < valid) x = s4[(size_t)t * d4];
      const int p = kSwizzle ? (c4 ^ (t & mask)) : c4;
      *reinterpret_cast<float4*>(&dst[t * d + 4 * p]) = x;
    }
  }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <int S, int R, int DC, bool kBf16>
__global__ void __launch_bounds__(32 * S)
cdist_exp_kernel(const CdistArgs a) {
  constexpr int kThreads = 32 * S;
  constexpr int kTile = 32 * R;
  constexpr int kTileP = kTile + 4;    // padded row of the kernel-value tile
  constexpr int M = S * S;
  extern __shared__ float4 smem_cd4[];
  float* smem = reinterpret_cast<float*>(smem_cd4);
  const int d = a.d, n = a.n;
  float* sL = smem;                    // [M][d]
  float* sX = sL + M * d;              // [kTile][d] swizzled token rows
  float* sOut = sX + kTile * d;        // [M][kTileP] kernel values, landmark-major
  float* sV = sOut + M * kTileP;       // [kTile][d] values (key side)

  const int side = blockIdx.y;
  const long bh = blockIdx.x / a.splits;
  const int split = blockIdx.x % a.splits;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mask = swizzle_mask(d);
  const int tile_begin = split * a.tiles_per_split;
  const int tile_end = min(a.tiles, tile_begin + a.tiles_per_split);
  const bool debug = a.dbg_dql || a.dbg_dlk || a.dbg_a;

  {
    const float4* Lg = reinterpret_cast<const float4*>(a.landmarks + (size_t)bh * M * d);
    for (int i = threadIdx.x; i < (M * d) >> 2; i += kThreads)
      reinterpret_cast<float4*>(sL)[i] = Lg[i];
  }

  // Key side, B V: thread (ks, lg, cq) accumulates landmarks lg*S .. lg*S+S-1 times channels
  // 4cq .. 4cq+3 over the token quads q == ks (mod KS) of every tile, in registers.
  const int cqn = d >> 2;
  const int set = S * cqn;
  const int KS = kThreads / set;       // token classes (>= 1 since d <= 128)
  const int bv_ks = threadIdx.x / set;
  const int bv_lg = (threadIdx.x % set) / cqn;
  const int bv_cq = threadIdx.x % cqn;
  const bool bv_on = bv_ks < KS;
  float bv[S][4];
#pragma unroll
  for (int jj = 0; jj < S; ++jj)
#pragma unroll
    for (int c = 0; c < 4; ++c) bv[jj][c] = 0.f;

  const void* src = side == 0 ? a.q : a.k;
  for (int tile = tile_begin; tile < tile_end; ++tile) {
    const int n0 = tile * kTile;
    const int valid = min(kTile, n - n0);
    const size_t row0 = (size_t)bh * n + n0;
    stage_rows<kBf16, true>(src, sX, row0, valid, kTile, d, mask, kThreads);
    if (side == 1) stage_rows<kBf16, false>(a.v, sV, row0, valid, kTile, d, 0, kThreads);
    __syncthreads();

    // ---- distances: acc[r][jj] = sum_c |x_{lane+32r, c} - L_{warp*S+jj, c}| ----
    float acc[R][S];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int jj = 0; jj < S; ++jj) acc[r][jj] = 0.f;
    const float* lrow = sL + warp * S * d;
    const int sw = lane & mask;
    for (int c4 = 0; c4 < (d >> 2); ++c4) {
      float4 x[R];
#pragma unroll
      for (int r = 0; r < R; ++r)
        x[r] = *reinterpret_cast<const float4*>(&sX[(lane + 32 * r) * d + 4 * (c4 ^ sw)]);
#pragma unroll
      for (int jj = 0; jj < S; ++jj) {
        const float4 l = *reinterpret_cast<const float4*>(&lrow[jj * d + 4 * c4]);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          float t = acc[r][jj];
          t += fabsf(x[r].x - l.x);
          t += fabsf(x[r].y - l.y);
          t += fabsf(x[r].z - l.z);
          t += fabsf(x[r].w - l.w);
          acc[r][jj] = t;
        }
      }
    }

    // ---- kernel values into the landmark-major tile ----
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int t = lane + 32 * r;
#pragma unroll
      for (int jj = 0; jj < S; ++jj) {
        const int j = warp * S + jj;
        const float val = t < valid ? laplacian_from_distance(acc[r][jj], a.c_exp) : 0.f;
        sOut[j * kTileP + t] = val;
        if (debug && t < valid) {
          const size_t tok = row0 + t;
          if (side == 0) {
            if (a.dbg_dql) a.dbg_dql[tok * M + j] = acc[r][jj];
            if (a.dbg_a) a.dbg_a[tok * M + j] = val;
          } else if (a.dbg_dlk) {
            a.dbg_dlk[((size_t)bh * M + j) * n + n0 + t] = acc[r][jj];
          }
        }
      }
    }
    __syncthreads();

    if (side == 0) {
      // A^T rows of this tile (coalesced along the tokens).
      for (int idx = threadIdx.x; idx < M * kTile; idx += kThreads) {
        const int j = idx / kTile, t = idx % kTile;
        if (t < valid) a.at[((size_t)bh * M + j) * n + n0 + t] = sOut[j * kTileP + t];
      }
      // Per-landmark mean and M2 over the tile's valid tokens: warp w reduces rows
      // w, w+S, ..., one row per pass, with shuffles (fixed order: deterministic).
      const float inv_valid = 1.f / (float)valid;
      for (int j = warp; j < M; j += S) {
        float sum = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int t = lane + 32 * r;
          if (t < valid) sum += sOut[j * kTileP + t];
        }
        const float mean = warp_sum(sum) * inv_valid;
        float ss = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int t = lane + 32 * r;
          if (t < valid) {
            const float dv = sOut[j * kTileP + t] - mean;
            ss = fmaf(dv, dv, ss);
          }
        }
        ss = warp_sum(ss);
        if (lane == 0) {
          float* st = a.stats + ((size_t)bh * a.tiles + tile) * 2 * M;
          st[j] = mean;
          st[M + j] = ss;
        }
      }
    } else if (bv_on) {
      // bv[jj][c] += sum_t B[lg*S+jj][t] * V[t][4cq+c]; padded tokens have B = 0 and V = 0.
      const float* brow = sOut + bv_lg * S * kTileP;
      for (int q = bv_ks; q < kTile / 4; q += KS) {
        const int t = 4 * q;
        float4 v4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          v4[u] = *reinterpret_cast<const float4*>(&sV[(t + u) * d + 4 * bv_cq]);
#pragma unroll
        for (int jj = 0; jj < S; ++jj) {
          const float4 b4 = *reinterpret_cast<const float4*>(&brow[jj * kTileP + t]);
          const float bu[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            bv[jj][0] = fmaf(bu[u], v4[u].x, bv[jj][0]);
            bv[jj][1] = fmaf(bu[u], v4[u].y, bv[jj][1]);
            bv[jj][2] = fmaf(bu[u], v4[u].z, bv[jj][2]);
            bv[jj][3] = fmaf(bu[u], v4[u].w, bv[jj][3]);
          }
        }
      }
    }
    __syncthreads();
  }

  if (side == 1) {
    // Combine the KS token classes (fixed order) through shared memory, then store the
    // CTA's partial B V.  sX and sOut are free now: KS * M * d <= 128 * M floats fit there.
    float* red = sX;
    if (bv_on) {
#pragma unroll
      for (int jj = 0; jj < S; ++jj)
        *reinterpret_cast<float4*>(&red[((size_t)bv_ks * M + bv_lg * S + jj) * d + 4 * bv_cq]) =
            make_float4(bv[jj][0], bv[jj][1], bv[jj][2], bv[jj][3]);
    }
    __syncthreads();
    float* dst = a.bvp + ((size_t)bh * a.splits + split) * M * d;
    for (int i = threadIdx.x; i < M * d; i += kThreads) {
      float sum = red[i];
      for (int q = 1; q < KS; ++q) sum += red[(size_t)q * M * d + i];
      dst[i] = sum;
    }
  }
}

constexpr int kRows = 4;   // tokens per thread; tile = 128 tokens

template <int S, bool kBf16>
const void* pick_dc(int dc) {
  switch (dc) {
    case 1: return reinterpret_cast<const void*>(&cdist_exp_kernel<S, kRows, 1, kBf16>);
    case 2: return reinterpret_cast<const void*>(&cdist_exp_kernel<S, kRows, 2, kBf16>);
    case 4: return reinterpret_cast<const void*>(&cdist_exp_kernel<S, kRows, 4, kBf16>);
    default: return nullptr;
  }
}

template <bool kBf16>
const void* pick_s(int s, int dc) {
  switch (s) {
    case 1: return pick_dc<1, kBf16>(dc);
    case 2: return pick_dc<2, kBf16>(dc);
    case 3: return pick_dc<3, kBf16>(dc);
    case 4: return pick_dc<4, kBf16>(dc);
    case 5: return pick_dc<5, kBf16>(dc);
    case 6: return pick_dc<6, kBf16>(dc);
    case 7: return pick_dc<7, kBf16>(dc);
    case 8: return pick_dc<8, kBf16>(dc);
    default: return nullptr;
  }
}

// Value columns per lane, rounded to an instantiated width.
int dc_of(int d) { return d <= 32 ? 1 : (d <= 64 ? 2 : 4); }

const void* pick(int s, int d, bool bf16) {
  return bf16 ? pick_s<true>(s, dc_of(d)) : pick_s<false>(s, dc_of(d));
}

}  // namespace

size_t cdist_smem_bytes(int s, int d, int tile) {
  const size_t m = (size_t)s * s;
  return sizeof(float) * (m * d + (size_t)tile * d + m * (tile + 4) + (size_t)tile * d);
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
                         const float* landmarks, float* at, float* stats, float* bvp,
                         float* dbg_dql, float* dbg_dlk, float* dbg_a, cudaStream_t st) {
  const Geometry& g = p.geo;
  CdistArgs a;
  a.q = q; a.k = k; a.v = v; a.landmarks = landmarks; a.at = at; a.stats = stats; a.bvp = bvp;
  a.dbg_dql = dbg_dql; a.dbg_dlk = dbg_dlk; a.dbg_a = dbg_a;
  a.n = g.n; a.d = g.d; a.tiles = g.cd_tiles; a.tiles_per_split = g.cd_tiles_per_split;
  a.splits = g.cd_splits; a.c_exp = p.neg_log2e_over_lambda;
  const void* f = pick(g.s, g.d, p.cfg.in_dtype == LAPL_BF16);
  if (!f) return cudaErrorInvalidValue;
  dim3 grid((unsigned)(g.bh * g.cd_splits), 2);
  void* args[] = {&a};
  return cudaLaunchKernel(f, grid, dim3(32 * g.s), args, g.cd_smem, st);
}

}  // namespace lapl
