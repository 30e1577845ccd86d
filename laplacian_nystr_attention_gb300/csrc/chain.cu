// chain.cu -- whitening statistics and the output chain O = A^ (X (B V)).
//
// "LaplacianFormer: Rethinking Linear Attention with Laplacian Kernel":
//  * whitening (Korean explainer page, 2.2; English page, 2.B): A^ = (A - mean) / sqrt(var +
//    delta) + bias with a diagonal estimator, i.e. one mean and one variance per landmark
//    column, taken over the N tokens of the (batch, head) slice (variance divides by N);
//  * low-rank product without the N x N matrix (Chinese page, 2.2), evaluated right to left.
//
// bv_kernel (the column-statistics CTAs, then one CTA per (batch, head, token split)):
//   partial B V of the split's tokens from B^T [BH, m, N] and V, register-tiled on the CUDA
//   cores (4 landmarks x 4 channels per thread, 8 shared loads per 64 FMAs).
// mix_kernel (per (batch, head, 8 value columns)), after B V and the Newton-Schulz solve:
//   reduces the per-split partials of B V in split order (while the solve may still run, when
//   it is this kernel's programmatic predecessor) and forms M = X (B V).
//   Fixed reduction orders: the result is bit-reproducible run to run.
// output_kernel (one CTA per (batch, head, token tile)):
//   loads the A^T tile and whitens it on the way into shared memory, then (after the M
//   kernel) writes O = A^ M with a 4 tokens x 4 channels register tile per thread.
#include "common.cuh"

namespace lapl {
namespace {

constexpr int kBvTile = 64;           // tokens per staged chunk
constexpr int kBvTileP = kBvTile + 4;  // padded row of the B^T chunk

__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, int src_bytes) {
  const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async4_zfill(void* dst, const void* src, int src_bytes) {
  const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(d), "l"(src), "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ float warp_allsum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Column statistics of A for the whitening: warp w of statistics CTA sidx takes landmark column
// j of head bh, the contiguous row A^T[bh][j][0..N), in one pass.  The values are shifted by c,
// the mean of the row's first (up to) 128 values, and each lane sums a - c and (a - c)^2 over
// every 32nd 16-byte piece (or element); the lanes are combined by a fixed xor tree.  Then
// mean = c + S1 / N and M2 = S2 - S1^2 / N (var = M2 / N).  c lies within a few standard
// deviations of the mean, so the subtraction keeps fp32 accuracy.
__device__ __forceinline__ void column_stats(const float* __restrict__ at, float* __restrict__ mu,
                                             float* __restrict__ rstd, float* __restrict__ dbg_mu,
                                             float* __restrict__ dbg_rstd, int m, int n,
                                             float delta, long sidx) {
  const int warps = (int)(blockDim.x >> 5), warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_head = (m + warps - 1) / warps;
  const long bh = sidx / per_head;
  const int j = (int)(sidx % per_head) * warps + warp;
  if (j >= m) return;
  const float* row = at + ((size_t)bh * m + j) * n;
  // Shift: mean of the first min(N, 128) values.
  const int nc = n < 128 ? n : 128;
  float c = 0.f;
  for (int i = lane; i < nc; i += 32) c += __ldcg(&row[i]);
  c = warp_allsum(c) / (float)nc;

  constexpr int kB = 4;                   // loads in flight per lane
  float s1 = 0.f, s2 = 0.f;
  if ((n & 3) == 0) {
    const float4* r4 = reinterpret_cast<const float4*>(row);
    const int n4 = n >> 2;
    for (int i0 = lane; i0 < n4; i0 += 32 * kB) {
      float4 v[kB];
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const int i = i0 + 32 * u;
        v[u] = i < n4 ? __ldcg(&r4[i]) : make_float4(c, c, c, c);   // c contributes 0
      }
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const float a = v[u].x - c, b = v[u].y - c, e = v[u].z - c, f = v[u].w - c;
        s1 += (a + b) + (e + f);
        s2 += (a * a + b * b) + (e * e + f * f);
      }
    }
  } else {
    for (int i0 = lane; i0 < n; i0 += 32 * kB) {
      float v[kB];
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const int i = i0 + 32 * u;
        v[u] = i < n ? __ldcg(&row[i]) : c;
      }
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const float a = v[u] - c;
        s1 += a;
        s2 = fmaf(a, a, s2);
      }
    }
  }
  s1 = warp_allsum(s1);
  s2 = warp_allsum(s2);
  if (lane == 0) {
    const float inv_n = 1.f / (float)n;
    const float mean = c + s1 * inv_n;
    const float m2 = fmaxf(s2 - s1 * s1 * inv_n, 0.f);
    const float rs = 1.f / sqrtf(m2 * inv_n + delta);
    mu[(size_t)bh * m + j] = mean;
    rstd[(size_t)bh * m + j] = rs;
    if (dbg_mu) dbg_mu[(size_t)bh * m + j] = mean;
    if (dbg_rstd) dbg_rstd[(size_t)bh * m + j] = rs;
  }
}

// Partial B V of the split's tokens.  Chunks of 64 tokens (B^T rows and V rows) are copied
// asynchronously into one of two shared buffers while the other is contracted.
template <bool kBf16>
__global__ void __launch_bounds__(512, 2)
bv_kernel(const float* __restrict__ bt, const void* __restrict__ vin, float* __restrict__ bvp,
          int m, int d, int n, int tiles_per_split, int splits, const float* __restrict__ at,
          float* __restrict__ mu, float* __restrict__ rstd, float* __restrict__ dbg_mu,
          float* __restrict__ dbg_rstd, long stat_ctas, float delta) {
  // A kernel launched as this grid's programmatic dependent (the conjugate-gradient solver)
  // may start its own preparation now; it waits for this grid before it reads any result.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  // The column-statistics CTAs come first: they are placed in the first wave, next to the
  // B V CTAs, instead of after them.
  if ((long)blockIdx.x < stat_ctas) {    // a column-statistics CTA (uniform per CTA)
    column_stats(at, mu, rstd, dbg_mu, dbg_rstd, m, n, delta, (long)blockIdx.x);
    return;
  }
  const long cta = (long)blockIdx.x - stat_ctas;
  extern __shared__ float4 smem_bv4[];
  float* smem = reinterpret_cast<float*>(smem_bv4);
  const int nthreads = blockDim.x;
  const int mp4 = (m + 3) & ~3;
  const int vrow = d * (kBf16 ? 2 : 4);                    // bytes per staged V row
  float* sB0 = smem;                                       // 2 x [mp4][kBvTileP]
  char* sV0 = reinterpret_cast<char*>(sB0 + 2 * mp4 * kBvTileP);   // 2 x [kBvTile][d]
  // bf16: each chunk of V is widened once into sVf (fp32 [kBvTile][d]) when it lands, instead
  // of at every use (each V value serves every landmark quad).
  float* sVf = reinterpret_cast<float*>(sV0 + 2 * kBvTile * d * (kBf16 ? 2 : 4));
  float* red = smem;   // [16][nthreads], reuses the staging buffers after the last chunk
  const long bh = cta / splits;
  const int sp = (int)(cta % splits);
  const int tiles = (n + kBvTile - 1) / kBvTile;
  const int t_begin = sp * tiles_per_split;
  const int t_end = min(tiles, t_begin + tiles_per_split);

  // Thread (ks, lg, cq): landmarks 4lg..4lg+3, channels 4cq..4cq+3, token quads == ks mod KS.
  const int cqn = d >> 2, lgn = mp4 >> 2;
  const int set = lgn * cqn;
  const int KS = max(1, nthreads / set);
  const int ks = threadIdx.x / set, lg = (threadIdx.x % set) / cqn, cq = threadIdx.x % cqn;
  const bool on = ks < KS;
  float acc[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;

  // Padding rows of the landmark dimension stay zero in both buffers.
  for (int i = threadIdx.x; i < (mp4 - m) * kBvTileP; i += nthreads) {
    sB0[m * kBvTileP + i] = 0.f;
    sB0[(mp4 + m) * kBvTileP + i] = 0.f;
  }

  const bool vec = (n & 3) == 0;
  auto issue = [&](int tile, int buf) {
    const int n0 = tile * kBvTile;
    const int valid = min(kBvTile, n - n0);
    float* sB = sB0 + buf * mp4 * kBvTileP;
    if (vec) {
      for (int i = threadIdx.x; i < m * (kBvTile / 4); i += nthreads) {
        const int j = i / (kBvTile / 4), q4 = i % (kBvTile / 4);
        const float* src = &bt[((size_t)bh * m + j) * n + n0 + (4 * q4 < valid ? 4 * q4 : 0)];
        cp_async16_zfill(&sB[j * kBvTileP + 4 * q4], src, 4 * q4 < valid ? 16 : 0);
      }
    } else {
      for (int i = threadIdx.x; i < m * kBvTile; i += nthreads) {
        const int j = i / kBvTile, t = i % kBvTile;
        const float* src = &bt[((size_t)bh * m + j) * n + n0 + (t < valid ? t : 0)];
        cp_async4_zfill(&sB[j * kBvTileP + t], src, t < valid ? 4 : 0);
      }
    }
    char* sV = sV0 + buf * kBvTile * vrow;
    const int pieces = vrow >> 4;
    const char* vbase = reinterpret_cast<const char*>(vin) + ((size_t)bh * n + n0) * vrow;
    for (int i = threadIdx.x; i < kBvTile * pieces; i += nthreads) {
      const int t = i / pieces, pc = i % pieces;
      cp_async16_zfill(sV + t * vrow + pc * 16, vbase + (size_t)(t < valid ? t : 0) * vrow + pc * 16,
                       t < valid ? 16 : 0);
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  };

  if (t_begin < t_end) issue(t_begin, 0);
  int buf = 0;
  for (int tile = t_begin; tile < t_end; ++tile) {
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    __syncthreads();
    if constexpr (kBf16) {
      const uint4* raw = reinterpret_cast<const uint4*>(sV0 + buf * kBvTile * vrow);
      for (int i = threadIdx.x; i < kBvTile * d / 8; i += nthreads) {
        const uint4 r = raw[i];
        float4* dst = reinterpret_cast<float4*>(sVf + 8 * i);
        dst[0] = make_float4(bf16_lo(r.x), bf16_hi(r.x), bf16_lo(r.y), bf16_hi(r.y));
        dst[1] = make_float4(bf16_lo(r.z), bf16_hi(r.z), bf16_lo(r.w), bf16_hi(r.w));
      }
      __syncthreads();
    }
    if (tile + 1 < t_end) issue(tile + 1, buf ^ 1);
    if (on) {
      const float* sB = sB0 + buf * mp4 * kBvTileP;
      const char* sV = kBf16 ? reinterpret_cast<const char*>(sVf) : sV0 + buf * kBvTile * vrow;
      const int vrow_f = d * 4;                            // bytes per fp32 row
      for (int q = ks; q < kBvTile / 4; q += KS) {
        const int t = 4 * q;
        float4 b4[4], v4[4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
          b4[r] = *reinterpret_cast<const float4*>(&sB[(4 * lg + r) * kBvTileP + t]);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          v4[u] = *reinterpret_cast<const float4*>(sV + (t + u) * vrow_f + 16 * cq);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float bu[4] = {b4[r].x, b4[r].y, b4[r].z, b4[r].w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            acc[r][0] = fmaf(bu[u], v4[u].x, acc[r][0]);
            acc[r][1] = fmaf(bu[u], v4[u].y, acc[r][1]);
            acc[r][2] = fmaf(bu[u], v4[u].z, acc[r][2]);
            acc[r][3] = fmaf(bu[u], v4[u].w, acc[r][3]);
          }
        }
      }
    }
    buf ^= 1;
  }
  // Combine the KS token classes in order: the class-0 thread of (lg, cq) adds the others'
  // register tiles to its own and stores the split's partial B V rows, 16 bytes at a time.
  __syncthreads();
  if (ks > 0 && on) {
#pragma unroll
    for (int e = 0; e < 16; ++e) red[e * nthreads + threadIdx.x] = acc[e >> 2][e & 3];
  }
  __syncthreads();
  if (ks == 0) {
    for (int q = 1; q < KS; ++q)
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[e >> 2][e & 3] += red[e * nthreads + q * set + threadIdx.x];
    float* dst = bvp + ((size_t)bh * splits + sp) * m * d + 4 * cq;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int j = 4 * lg + r;
      if (j < m)
        *reinterpret_cast<float4*>(&dst[(size_t)j * d]) =
            make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
    }
  }

}

constexpr int kFinishThreads = 256;
constexpr int kFinishCols = 8;     // value columns per finish CTA

__device__ __forceinline__ void cp_async4(float* dst, const float* src) {
  const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(d), "l"(src) : "memory");
}

// mix_kernel, grid (BH * column chunks) -- the one step that waits for the Newton-Schulz solve:
// CTA (bh, cc) sums the B V partials of columns [cc*8, cc*8+8) over the token splits (in split
// order) and forms those columns of M = X (B V).  The partials are complete when the kernel
// starts (B V precedes it on the stream, or through an event when the solve has SMs of its
// own); X is read after griddepcontrol.wait, which waits for the solve when this kernel is its
// programmatic dependent, so the partial sums overlap the end of the solve.  Rows of 8 columns
// are 32 bytes (d is a multiple of 8): every read is a 16-byte asynchronous copy but X's.
__global__ void __launch_bounds__(kFinishThreads)
mix_kernel(const float* __restrict__ xg, const float* __restrict__ bvp, float* __restrict__ mmat,
           float* __restrict__ bv_keep, float* __restrict__ dbg_bv, float* __restrict__ dbg_m,
           int m, int d, int bv_splits) {
  extern __shared__ float4 smem_fin4[];
  float* smem = reinterpret_cast<float*>(smem_fin4);
  const int chunks = d / kFinishCols;
  const long bh = blockIdx.x / chunks;
  const int cc = blockIdx.x % chunks;
  const int c0 = cc * kFinishCols;
  float* sP = smem;                                        // [bv_splits][m][8]
  float* sBV = sP + (size_t)bv_splits * m * kFinishCols;   // [m][8]
  float* sX = sBV + (size_t)m * kFinishCols;               // [m][m]
  // The output kernel may start now: it prepares its A tile and waits for this grid before
  // it reads M.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const float* pbase = bvp + (size_t)bh * bv_splits * m * d + c0;
  const int rows = bv_splits * m;                          // (split, landmark) rows
  for (int i = threadIdx.x; i < 2 * rows; i += kFinishThreads) {
    const int r = i >> 1, h = i & 1;
    cp_async16_zfill(&sP[r * kFinishCols + 4 * h], &pbase[(size_t)r * d + 4 * h], 16);
  }
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
  __syncthreads();
  for (int i = threadIdx.x; i < m * kFinishCols; i += kFinishThreads) {
    const int j = i >> 3, c = i & 7;
    float acc = 0.f;
    for (int sp = 0; sp < bv_splits; ++sp) acc += sP[(sp * m + j) * kFinishCols + c];
    sBV[i] = acc;
    if (bv_keep) bv_keep[((size_t)bh * m + j) * d + c0 + c] = acc;
    if (dbg_bv) dbg_bv[((size_t)bh * m + j) * d + c0 + c] = acc;
  }
  asm volatile("griddepcontrol.wait;\n" ::: "memory");     // X is complete and visible
  for (int i = threadIdx.x; i < m * m; i += kFinishThreads) cp_async4(&sX[i], &xg[(size_t)bh * m * m + i]);
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
  __syncthreads();
  for (int i = threadIdx.x; i < m * kFinishCols; i += kFinishThreads) {
    const int j = i >> 3, c = i & 7;
    float acc = 0.f;
    for (int k = 0; k < m; ++k) acc = fmaf(sX[j * m + k], sBV[k * kFinishCols + c], acc);
    const size_t o = ((size_t)bh * m + j) * d + c0 + c;
    mmat[o] = acc;
    if (dbg_m) dbg_m[o] = acc;
  }
}

constexpr int kOutThreads = 256;

// TPT: tokens per thread (4, or 8 for d >= 64 when the grid stays large: twice the tokens per
// CTA, so that each CTA's M load and A-tile prologue serve twice the work).
template <bool kOutBf16, int TPT>
__global__ void __launch_bounds__(kOutThreads)
output_kernel(const float* __restrict__ at, const float* __restrict__ mmat,
              const float* __restrict__ mu, const float* __restrict__ rstd,
              const float* __restrict__ bias, void* __restrict__ out, int m, int d, int n,
              int heads, int tile, int tiles, int whiten) {
  extern __shared__ float4 smem_out4[];
  float* smem = reinterpret_cast<float*>(smem_out4);
  const long bh = blockIdx.x / tiles;
  const int tix = blockIdx.x % tiles;
  const int h = (int)(bh % heads);
  const int n0 = tix * tile;
  float* sM = smem;                 // [m][d]
  float* sA = sM + m * d;           // [m][tile] whitened A, landmark-major
  float* sCoef = sA + m * tile;     // mean [m], scale [m], bias [m]

  // Everything up to the wait below reads results of earlier kernels only (A^T, mean, rstd),
  // so with a programmatic launch it overlaps the M = X (B V) kernel before it.
  for (int j = threadIdx.x; j < m; j += kOutThreads) {
    float mean = 0.f, scale = 1.f, b = 0.f;
    if (whiten) {
      mean = mu[(size_t)bh * m + j];
      scale = rstd[(size_t)bh * m + j];
      b = bias ? bias[(size_t)h * m + j] : 0.f;
    }
    sCoef[j] = mean;
    sCoef[m + j] = scale;
    sCoef[2 * m + j] = b;
  }
  __syncthreads();
  // A^T tile -> whitened, landmark-major shared tile.  With N % 4 == 0 every row piece is
  // 16-byte aligned: tile/4 threads per row read float4s, several rows per thread in flight.
  // Otherwise scalar loads, 16 issued per thread before any is consumed.
  if ((n & 3) == 0) {
    const int tq = tile >> 2;                 // float4 per row
    const int rpp = kOutThreads / tq;         // rows per pass
    const int r0 = threadIdx.x / tq, q4 = threadIdx.x % tq;
    const int tok = n0 + 4 * q4;
    if (r0 < rpp) {
      constexpr int kRows = 4;
      for (int jb = r0; jb < m; jb += kRows * rpp) {
        float4 a[kRows];
#pragma unroll
        for (int u = 0; u < kRows; ++u) {
          const int j = jb + u * rpp;
          a[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (j < m && tok < n)
            a[u] = *reinterpret_cast<const float4*>(&at[((size_t)bh * m + j) * n + tok]);
        }
#pragma unroll
        for (int u = 0; u < kRows; ++u) {
          const int j = jb + u * rpp;
          if (j < m) {
            const float mean = sCoef[j], sc = sCoef[m + j], b = sCoef[2 * m + j];
            *reinterpret_cast<float4*>(&sA[j * tile + 4 * q4]) =
                make_float4((a[u].x - mean) * sc + b, (a[u].y - mean) * sc + b,
                            (a[u].z - mean) * sc + b, (a[u].w - mean) * sc + b);
          }
        }
      }
    }
  } else {
    constexpr int kBatch = 16;
    const int total = m * tile;
    for (int base = 0; base < total; base += kBatch * kOutThreads) {
      float a[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = base + u * kOutThreads + threadIdx.x;
        a[u] = 0.f;
        if (i < total) {
          const int j = i / tile, tok = n0 + i % tile;
          if (tok < n) a[u] = at[((size_t)bh * m + j) * n + tok];
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = base + u * kOutThreads + threadIdx.x;
        if (i < total) {
          const int j = i / tile;
          sA[i] = (a[u] - sCoef[j]) * sCoef[m + j] + sCoef[2 * m + j];
        }
      }
    }
  }
  asm volatile("griddepcontrol.wait;\n" ::: "memory");      // M is complete and visible
  for (int i = threadIdx.x; i < m * d; i += kOutThreads) sM[i] = mmat[(size_t)bh * m * d + i];
  __syncthreads();

  const int cg = d >> 2;                     // channel quads
  const int q = threadIdx.x % cg;
  const int tg = threadIdx.x / cg;           // token group of TPT tokens
  if (TPT * tg >= tile) return;
  float acc[TPT][4];
#pragma unroll
  for (int r = 0; r < TPT; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
  for (int j = 0; j < m; ++j) {
    float av[TPT];
#pragma unroll
    for (int h = 0; h < TPT / 4; ++h) {
      const float4 a4 = *reinterpret_cast<const float4*>(&sA[j * tile + TPT * tg + 4 * h]);
      av[4 * h] = a4.x;
      av[4 * h + 1] = a4.y;
      av[4 * h + 2] = a4.z;
      av[4 * h + 3] = a4.w;
    }
    const float4 m4 = *reinterpret_cast<const float4*>(&sM[j * d + 4 * q]);
    const float mv[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
    for (int r = 0; r < TPT; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(av[r], mv[c], acc[r][c]);
  }
#pragma unroll
  for (int r = 0; r < TPT; ++r) {
    const int tok = n0 + TPT * tg + r;
    if (tok >= n) break;
    const size_t o = ((size_t)bh * n + tok) * d + 4 * q;
    if constexpr (kOutBf16) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc[r][0], acc[r][1]);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc[r][2], acc[r][3]);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + o) = pk;
    } else {
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + o) =
          make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
    }
  }
}

}  // namespace

size_t mix_smem_bytes(int m, int bv_splits) {
  return sizeof(float) * (((size_t)bv_splits + 1) * m * kFinishCols + (size_t)m * m);
}

cudaError_t mix_configure(size_t smem) {
  return cudaFuncSetAttribute(mix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

// Tokens per thread of the output kernel: 8 for d >= 64 when the 8192/d-token tiles still
// give at least two CTAs per SM, else 4.
int output_tile_tokens(int d, long bh, int n, int num_sms) {
  const int cg = d / 4;
  const int t8 = 8 * (kOutThreads / cg);
  const long ctas8 = bh * ((n + t8 - 1) / t8);
  return (d >= 64 && ctas8 >= 2L * num_sms ? 8 : 4) * (kOutThreads / cg);
}

size_t output_smem_bytes(int m, int d, int tile) {
  return sizeof(float) * ((size_t)m * d + (size_t)m * tile + 3 * (size_t)m);
}

cudaError_t output_configure(size_t smem) {
  const void* fs[] = {reinterpret_cast<const void*>(&output_kernel<false, 4>),
                      reinterpret_cast<const void*>(&output_kernel<false, 8>),
                      reinterpret_cast<const void*>(&output_kernel<true, 4>),
                      reinterpret_cast<const void*>(&output_kernel<true, 8>)};
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < 4 && e == cudaSuccess; ++i)
    e = cudaFuncSetAttribute(fs[i], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  return e;
}

size_t bv_smem_bytes(int m, int d, int threads, bool bf16) {
  const int mp4 = (m + 3) & ~3;
  const size_t staging = sizeof(float) * 2 * (size_t)mp4 * kBvTileP +
                         2 * (size_t)kBvTile * d * (bf16 ? 2 : 4) +
                         (bf16 ? sizeof(float) * (size_t)kBvTile * d : 0);
  const size_t red = sizeof(float) * 16 * (size_t)threads;
  return staging > red ? staging : red;
}

int bv_threads(int m, int d) {
  const int set = ((m + 3) / 4) * (d / 4);
  return set > 256 ? 512 : 256;
}

int bv_tile_tokens() { return kBvTile; }

int bv_occupancy(int threads, size_t smem) {
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, bv_kernel<false>, threads, smem) !=
      cudaSuccess)
    return 1;
  return occ > 0 ? occ : 1;
}

cudaError_t bv_configure(size_t smem) {
  cudaError_t e = cudaFuncSetAttribute(bv_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(bv_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t launch_bv(const lapl_attn_plan& p, const float* bt, const void* v, float* bvp,
                      const float* at, float* mu, float* rstd, float* dbg_mu, float* dbg_rstd,
                      cudaStream_t st) {
  const Geometry& g = p.geo;
  if (g.bv_tc) {
    // The column statistics (a launch of their own), then the tensor-core B V as its
    // programmatic dependent.
    if (g.stat_ctas > 0) {
      const cudaError_t e = launch_col_stats(p, at, mu, rstd, dbg_mu, dbg_rstd, st);
      if (e != cudaSuccess) return e;
    }
    return launch_bv_tc(p, bt, v, bvp, st, g.stat_ctas > 0);
  }
  const long bv_ctas = g.bh * g.bv_splits, stat_ctas = g.stat_ctas;
  const unsigned grid = (unsigned)(bv_ctas + stat_ctas);
  const float delta = p.cfg.delta;
  if (p.cfg.in_dtype == LAPL_BF16)
    bv_kernel<true><<<grid, g.bv_threads, g.bv_smem, st>>>(bt, v, bvp, g.m, g.d, g.n,
                                                           g.bv_tiles_per_split, g.bv_splits, at,
                                                           mu, rstd, dbg_mu, dbg_rstd, stat_ctas,
                                                           delta);
  else
    bv_kernel<false><<<grid, g.bv_threads, g.bv_smem, st>>>(bt, v, bvp, g.m, g.d, g.n,
                                                            g.bv_tiles_per_split, g.bv_splits, at,
                                                            mu, rstd, dbg_mu, dbg_rstd, stat_ctas,
                                                            delta);
  return cudaGetLastError();
}

cudaError_t launch_mix(const lapl_attn_plan& p, const float* x, const float* bvp, float* mmat,
                       float* bv_keep, float* dbg_bv, float* dbg_m, cudaStream_t st) {
  const Geometry& g = p.geo;
  const int chunks = g.d / kFinishCols;
  // With the solve on SMs of its own it precedes this kernel on the stream (B V comes through
  // an event): a programmatic dependent of the solve.  Otherwise B V precedes it, and its
  // partials must be complete at launch: a plain launch.
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)(g.bh * chunks));
  cfg.blockDim = dim3(kFinishThreads);
  cfg.dynamicSmemBytes = g.fin_smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = g.ns_exclusive ? 1 : 0;
  int m = g.m, d = g.d, splits = g.bv_splits;
  return cudaLaunchKernelEx(&cfg, mix_kernel, x, bvp, mmat, bv_keep, dbg_bv, dbg_m, m, d,
                            splits);
}

cudaError_t launch_output(const lapl_attn_plan& p, const float* at, const float* mmat,
                          const float* mu, const float* rstd, const float* bias, void* out,
                          cudaStream_t st) {
  const Geometry& g = p.geo;
  if (g.out_tc) return launch_output_tc(p, at, mmat, mu, rstd, bias, out, st);
  int tiles = (g.n + g.out_tile - 1) / g.out_tile;
  // Programmatic dependent launch: the kernel may begin while the preceding M kernel runs.
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)(g.bh * tiles));
  cfg.blockDim = dim3(kOutThreads);
  cfg.dynamicSmemBytes = g.out_smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int m = g.m, d = g.d, n = g.n, heads = p.cfg.heads, tile = g.out_tile, whiten = p.cfg.whiten;
  auto go = [&](auto kernel) {
    return cudaLaunchKernelEx(&cfg, kernel, at, mmat, mu, rstd, bias, out, m, d, n, heads, tile,
                              tiles, whiten);
  };
  const bool t8 = tile * (d / 4) == 8 * kOutThreads;
  if (p.cfg.out_dtype == LAPL_BF16)
    return t8 ? go(output_kernel<true, 8>) : go(output_kernel<true, 4>);
  return t8 ? go(output_kernel<false, 8>) : go(output_kernel<false, 4>);
}

}  // namespace lapl
