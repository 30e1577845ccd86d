// cdist_kernel.cuh -- the fused L1 distance + Laplacian kernel for the query and key blocks,
// fed by cp.async (cdist.cu chooses between it and the TMA-fed kernel of cdist_tma.cuh, which
// shares its helpers from this file).  Included by the translation units that instantiate it
// for given head dims.
#pragma once
//
// "LaplacianFormer: Rethinking Linear Attention with Laplacian Kernel": the similarity is
// k(x, y) = exp(-||x - y||_1 / lambda) (English explainer page, 2.A), and the distance and the
// exponential are computed in one fused kernel (German page, 2, CUDA-Optimierung; Chinese page,
// 2.2).  The L1 distance is a sum of |a - b|, not a dot product, so it runs on the FP32 CUDA
// cores.
//
// Persistent CTAs walk an equal share of the (side, head, token) positions (see Partition) in
// chunks of up to 32*R tokens of one head:
//   query chunk:  A = k(Q, L) is written from registers into A^T [BH, m, N] (each warp store
//                 covers 32 consecutive tokens); its column statistics are taken from A^T
//                 afterwards (statistics CTAs of bv_kernel, chain.cu).
//   key chunk:    B = k(L, K) is written the same way into B^T [BH, m, N]; the contraction with
//                 V runs in bv_kernel.
//
// Block: s warps for m = s*s landmarks.  Warp w owns landmarks w*s .. w*s+s-1 (so every
// landmark read from shared memory is a warp-wide broadcast), lane l owns tokens
// l, l+32, .. l+32*(R-1) of the chunk.  Per 4 channels a thread issues R + s 128-bit shared
// loads for 8*R*s FP32 instructions (subtract, then add the absolute value).  The token chunk
// is kept in shared memory with its 16-byte pieces XOR-swizzled by the row, so the 8 lanes of
// a 128-bit load phase hit 8 different bank groups.

#include "common.cuh"

namespace lapl {
namespace cdist_impl {

struct CdistArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* landmarks;
  float* at;        // [BH, m, N]  A^T
  float* bt;        // [BH, m, N]  B^T
  float* dbg_dql;   // [BH, N, m]
  float* dbg_dlk;   // [BH, m, N]
  float* dbg_a;     // [BH, N, m]
  Partition part;
  long long bh_count;
  int n, d;
  float c_exp;
};

__device__ __forceinline__ int swizzle_mask(int d) {
  const int d4 = d >> 2;
  const int low = d4 & (-d4);
  return (low < 8 ? low : 8) - 1;
}

// Asynchronous 16-byte copies global -> shared (zero-filled when src_bytes == 0).
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// Issue the copies of rows [row0, row0 + valid) of a [., d] matrix (fp32 or raw bf16) into a
// tile of `tile` rows; rows past `valid` are zero-filled.  fp32 tiles are stored with their
// 16-byte pieces XOR-swizzled by the row (piece c of row t at c ^ (t & mask)); raw bf16 tiles
// unswizzled (converted later).
template <bool kBf16>
__device__ __forceinline__ void issue_rows(const void* __restrict__ src, void* __restrict__ dst,
                                           size_t row0, int valid, int tile, int d, int mask,
                                           int nthreads) {
  const int row_bytes = d * (kBf16 ? 2 : 4);
  const int pieces = row_bytes >> 4;
  const int rstep = nthreads / pieces;
  const int pc = threadIdx.x % pieces;
  const int t0 = threadIdx.x / pieces;
  if (t0 >= rstep) return;
  const char* s0 = reinterpret_cast<const char*>(src) + row0 * row_bytes + pc * 16;
  char* d0 = reinterpret_cast<char*>(dst);
  for (int t = t0; t < tile; t += rstep) {
    const int p = kBf16 ? pc : (pc ^ (t & mask));
    cp_async16(d0 + t * row_bytes + p * 16, s0 + (size_t)(t < valid ? t : 0) * row_bytes,
               t < valid ? 16 : 0);
  }
}

// Raw bf16 tile -> fp32 swizzled tile.
__device__ __forceinline__ void convert_bf16_tile(const uint4* __restrict__ raw,
                                                  float* __restrict__ dst, int tile, int d,
                                                  int mask, int nthreads) {
  const int d8 = d >> 3;
  for (int i = threadIdx.x; i < tile * d8; i += nthreads) {
    const int t = i / d8, c8 = i % d8;
    const uint4 r = raw[i];
    const float4 lo = make_float4(bf16_lo(r.x), bf16_hi(r.x), bf16_lo(r.y), bf16_hi(r.y));
    const float4 hi = make_float4(bf16_lo(r.z), bf16_hi(r.z), bf16_lo(r.w), bf16_hi(r.w));
    *reinterpret_cast<float4*>(&dst[t * d + 4 * ((2 * c8) ^ (t & mask))]) = lo;
    *reinterpret_cast<float4*>(&dst[t * d + 4 * ((2 * c8 + 1) ^ (t & mask))]) = hi;
  }
}

// t += |x - l|: a subtract, then an add with the absolute value as an operand modifier (two
// FP32-pipe instructions per element).
__device__ __forceinline__ void abs_diff_acc(float& t, float x, float l) {
  asm("{\n\t.reg .f32 dd;\n\tsub.f32 dd, %1, %2;\n\tabs.f32 dd, dd;\n\tadd.f32 %0, %0, dd;\n\t}"
      : "+f"(t)
      : "f"(x), "f"(l));
}

// t += (x - l)^2: a subtract and a fused multiply-add (the Gaussian kernel's squared l2
// distance; also two FP32-pipe instructions per element).
__device__ __forceinline__ void sq_diff_acc(float& t, float x, float l) {
  const float dd = x - l;
  t = fmaf(dd, dd, t);
}

template <bool kGauss>
__device__ __forceinline__ void dist_acc(float& t, float x, float l) {
  if constexpr (kGauss) sq_diff_acc(t, x, l);
  else abs_diff_acc(t, x, l);
}

// acc[r][jj] = sum_c |x_{lane+32r, c} - L_{jj, c}| (squared terms for the Gaussian kernel) for
// the first RV row groups (the others 0).
template <int S, int R, int RV, bool kGauss>
__device__ __forceinline__ void l1_distances(const float* __restrict__ sX,
                                             const float* __restrict__ lrow, int d, int lane,
                                             int sw, float (&acc)[R][S]) {
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int jj = 0; jj < S; ++jj) acc[r][jj] = 0.f;
#pragma unroll 2
  for (int c4 = 0; c4 < (d >> 2); ++c4) {
    float4 x[RV];
#pragma unroll
    for (int r = 0; r < RV; ++r)
      x[r] = *reinterpret_cast<const float4*>(&sX[(lane + 32 * r) * d + 4 * (c4 ^ sw)]);
#pragma unroll
    for (int jj = 0; jj < S; ++jj) {
      const float4 l = *reinterpret_cast<const float4*>(&lrow[jj * d + 4 * c4]);
#pragma unroll
      for (int r = 0; r < RV; ++r) {
        float t = acc[r][jj];
        dist_acc<kGauss>(t, x[r].x, l.x);
        dist_acc<kGauss>(t, x[r].y, l.y);
        dist_acc<kGauss>(t, x[r].z, l.z);
        dist_acc<kGauss>(t, x[r].w, l.w);
        acc[r][jj] = t;
      }
    }
  }
}

template <int S, int R, int D, bool kBf16, bool kGauss = false>
__global__ void __launch_bounds__(32 * S)
cdist_exp_kernel(const CdistArgs a) {
  static_assert(S <= 8 && R == 4, "at most 8 landmarks per warp; 4 row groups");
  constexpr int kThreads = 32 * S;
  constexpr int kTile = 32 * R;
  constexpr int M = S * S;
  extern __shared__ float4 smem_cd4[];
  float* smem = reinterpret_cast<float*>(smem_cd4);
  const int d = D > 0 ? D : a.d;   // compile-time head dim when D > 0
  const int n = a.n;
  const int elt = kBf16 ? 2 : 4;
  float* sL = smem;                                       // [M][d]
  char* sbuf = reinterpret_cast<char*>(sL + M * d);       // 2 x [kTile][d] staged rows
  float* sXc = reinterpret_cast<float*>(sbuf + 2 * kTile * d * elt);   // bf16: converted tile

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mask = swizzle_mask(d);
  const bool debug = a.dbg_dql || a.dbg_dlk || a.dbg_a;
  const Partition& pt = a.part;
  const int cta = blockIdx.x;
  long long pos = part_start(pt, cta);
  const long long pend = part_start(pt, cta + 1);
  if (pos >= pend) return;

  // Chunk iterator: (side, head, first token); advanced without divisions.
  struct Chunk { int side; long long bh; int n0; int valid; };
  Chunk cur;
  {
    cur.side = pos < pt.uq ? 0 : 1;
    const long long local = pos - (cur.side ? pt.uq : 0);
    cur.bh = local / n;
    cur.n0 = (int)(local % n);
    cur.valid = (int)min((long long)min(kTile, n - cur.n0), pend - pos);
  }
  auto next_of = [&](const Chunk& c, long long p) {
    Chunk x = c;
    x.n0 += c.valid;
    if (x.n0 == n) {
      x.n0 = 0;
      x.bh += 1;
      if (x.side == 0 && x.bh == a.bh_count) {
        x.side = 1;
        x.bh = 0;
      }
    }
    x.valid = (int)min((long long)min(kTile, n - x.n0), pend - p);
    return x;
  };
  auto issue = [&](const Chunk& c, int buf) {
    issue_rows<kBf16>(c.side == 0 ? a.q : a.k, sbuf + buf * kTile * d * elt,
                      (size_t)c.bh * n + c.n0, c.valid, kTile, d, mask, kThreads);
    cp_async_commit();
  };

  long long cur_bh = -1;

  issue(cur, 0);
  int buf = 0;
  while (true) {
    cp_async_wait_all();
    __syncthreads();       // chunk `cur` is in sbuf[buf]; every warp is done with the last one
    const long long pnext = pos + cur.valid;
    const bool more = pnext < pend;
    Chunk nxt;
    if (more) {
      nxt = next_of(cur, pnext);
      issue(nxt, buf ^ 1);  // lands while this chunk is computed
    }
    const int side = cur.side, n0 = cur.n0, valid = cur.valid;
    const long long bh = cur.bh;
    if (bh != cur_bh) {
      const float4* Lg = reinterpret_cast<const float4*>(a.landmarks + (size_t)bh * M * d);
      for (int i = threadIdx.x; i < (M * d) >> 2; i += kThreads)
        reinterpret_cast<float4*>(sL)[i] = Lg[i];
      cur_bh = bh;
    }
    const float* sX;
    if constexpr (kBf16) {
      convert_bf16_tile(reinterpret_cast<const uint4*>(sbuf + buf * kTile * d * elt), sXc, kTile,
                        d, mask, kThreads);
      sX = sXc;
    } else {
      sX = reinterpret_cast<const float*>(sbuf + buf * kTile * d * elt);
    }
    __syncthreads();       // landmarks and (bf16) converted rows visible
    const size_t row0 = (size_t)bh * n + n0;

    // ---- distances over the row groups that hold valid tokens ----
    float acc[R][S];
    const float* lrow = sL + warp * S * d;
    const int sw = lane & mask;
    const int groups = (valid + 31) >> 5;
    if (groups == 4) l1_distances<S, R, 4, kGauss>(sX, lrow, d, lane, sw, acc);
    else if (groups == 3) l1_distances<S, R, 3, kGauss>(sX, lrow, d, lane, sw, acc);
    else if (groups == 2) l1_distances<S, R, 2, kGauss>(sX, lrow, d, lane, sw, acc);
    else l1_distances<S, R, 1, kGauss>(sX, lrow, d, lane, sw, acc);

    // ---- kernel values ----
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int t = lane + 32 * r;
#pragma unroll
      for (int jj = 0; jj < S; ++jj) {
        const float dist = acc[r][jj];
        acc[r][jj] = t < valid ? laplacian_from_distance(dist, a.c_exp) : 0.f;
        if (debug && t < valid) {
          const int j = warp * S + jj;
          const size_t tok = row0 + t;
          if (side == 0) {
            if (a.dbg_dql) a.dbg_dql[tok * M + j] = dist;
            if (a.dbg_a) a.dbg_a[tok * M + j] = acc[r][jj];
          } else if (a.dbg_dlk) {
            a.dbg_dlk[((size_t)bh * M + j) * n + n0 + t] = dist;
          }
        }
      }
    }

    // A^T / B^T straight from registers: per (r, jj) a warp stores 32 consecutive tokens.
#pragma unroll
    for (int jj = 0; jj < S; ++jj) {
      float* dst = (side == 0 ? a.at : a.bt) + ((size_t)bh * M + warp * S + jj) * n + n0;
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (lane + 32 * r < valid) dst[lane + 32 * r] = acc[r][jj];
    }
    if (!more) break;
    pos = pnext;
    cur = nxt;
    buf ^= 1;
  }
}


}  // namespace cdist_impl
}  // namespace lapl
