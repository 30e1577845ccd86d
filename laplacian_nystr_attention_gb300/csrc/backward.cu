// backward.cu -- gradients of a loss with dLoss/dO = G with respect to Q, K, V and the bias.
//
// The pages claim CUDA kernels for the forward and the backward pass ("LaplacianFormer:
// Rethinking Linear Attention with Laplacian Kernel", English explainer page, 2 "CUDA
// Acceleration"; German page, 2) and give no gradient: every kernel below applies the chain
// rule to one forward step, in reverse order.  The forward's workspace supplies what it saved
// (landmarks L, the iterates X_0 .. X_T, A^T, B^T, the column statistics, B V and M).
//
//   bwd_ahat_kernel   (head, token split)   dA^ = G M^T (stored), partials of dM = A^T G and
//                                           of the column sums s1 = sum dA^, s2 = sum dA^ Z
//   bwd_mid_kernel    (head, row quarter)   dM, dBV = X^T dM, S_T = sym(dM BV^T), the sums
//   bwd_ns_kernel     (head; side stream)   the Newton-Schulz steps backwards through the
//                                           forward's saved iterates to dW; the landmark-
//                                           block term of dL
//   bwd_query_kernel  (head, token tile)    g = dLoss/dD_QL = -(A / lambda) dA (stored) with
//                                           dA from the whitening backward; dQ
//   bwd_key_kernel    (head, token tile)    h = dLoss/dD_LK = -(B / lambda) (dBV V^T) (stored);
//                                           dK's distance term and dV = B^T dBV
//   bwd_lm_kernel     (head, split, side)   partials of dL from the query and key blocks
//   bwd_dl_kernel     (head)                dL = sum of the partials + the landmark term;
//                                           dbias = sum over the batch of s1
//   bwd_pool_kernel   (head, token tile)    dK += dL of the token's window / window size
//
// The distance derivative is sgn(x - y) with sgn(0) = 0 (Laplacian kernel) or 2 (x - y)
// (Gaussian kernel).  Reductions run in fixed orders: results are reproducible bit for bit.
#include <algorithm>

#include "ns_common.cuh"

namespace lapl {
using namespace ns_detail;
namespace {

constexpr int kBwdTile = 128;          // tokens per staged tile (bwd_ahat, bwd_lm)
constexpr int kBwdThreads = 256;
constexpr int kHeadThreads = 512;
constexpr int kMaxPairs = (kMaxM * kMaxD + kBwdThreads - 1) / kBwdThreads;   // 32

// The Gaussian kernel's distance slope d(x - y)^2 / dx.
__device__ __forceinline__ float gauss_slope(float x, float y) { return 2.f * (x - y); }

// The Laplacian kernel's sign on the multiply-add pipe.  With nc2 = -c 2^24,
//   step(x, nc2) = [x > c] + [x == c] / 2, exactly 0, 1/2 or 1,
// so that sgn(x - c) = 2 step - 1.  x - c is a multiple of 2^-149, so (x - c) 2^24, rounded
// once by the first multiply-add, is zero exactly when x == c and at least 2^-125 in magnitude
// otherwise (and keeps its sign); the second scales that to at least 1 in magnitude, adds 1/2
// and saturates to [0, 1].  Exact for all finite x and |c| < 2^104, denormals included (no flush
// to zero).  Three multiply-adds per element in all, against two compares, a subtract and a
// multiply-add for [x > c] - [x < c]; the weights' sum supplies the -1.
__device__ __forceinline__ float neg_scaled(float c) { return c * -0x1p24f; }
__device__ __forceinline__ float step(float x, float nc2) {
  return __saturatef(__fmaf_rn(__fmaf_rn(x, 0x1p24f, nc2), 0x1p125f, 0.5f));
}

// Element e of a [.., d] input row in fp32 or bf16.
__device__ __forceinline__ float load_in(const void* p, size_t e, bool bf16) {
  if (bf16) {
    const unsigned short u = reinterpret_cast<const unsigned short*>(p)[e];
    return __uint_as_float((unsigned)u << 16);
  }
  return reinterpret_cast<const float*>(p)[e];
}

// ---- dA^ = G M^T and the partial reductions over one token split -----------------------
// 512 threads, register tiles of 4 x 4 outputs over float4 operands in shared memory:
//   dA^[j][t]: warp w owns landmark quad w (w < m / 4), lane l tokens l, l + 32, l + 64,
//     l + 96 (rows a lane-stride apart: the eight lanes of a quarter-warp hit distinct banks;
//     the landmark rows are warp-wide broadcasts); the channels run in quads;
//   dM[j][c] += sum_t (Z[j][t] + beta_j) G[t][c]: thread (landmark quad, channel quad, token
//     class), token quads of its class, classes summed in order at the end.
constexpr int kAhatThreads = 512;

__global__ void __launch_bounds__(kAhatThreads)
bwd_ahat_kernel(const float* __restrict__ at, const float* __restrict__ mmat,
                const float* __restrict__ mu, const float* __restrict__ rstd,
                const float* __restrict__ bias, const float* __restrict__ gout,
                float* __restrict__ dahat, float* __restrict__ part_dm,
                float* __restrict__ part_s, int m, int d, int n, int heads, int tiles_per_split,
                int splits, int whiten) {
  extern __shared__ float4 smem_a4[];
  float* smem = reinterpret_cast<float*>(smem_a4);
  const int mp4 = (m + 3) & ~3;
  const int dq = d + 4, tq = kBwdTile + 4;     // padded row lengths (multiples of 4)
  float* sM = smem;                            // [mp4][d + 4]
  float* sG = sM + mp4 * dq;                   // [tile][d + 4]  token-major
  float* sZ = sG + kBwdTile * dq;              // [mp4][tile + 4] Z + beta (A^ without the bias
                                               //                 when whitening is off: A)
  float* sD = sZ + mp4 * tq;                   // [mp4][tile + 4] dA^
  float* sc = sD + mp4 * tq;                   // mu, r, beta [3][mp4]
  float* red = sG;                             // [16][threads] after the last tile
  const long bh = blockIdx.x / splits;
  const int sp = blockIdx.x % splits;
  const int h = (int)(bh % heads);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < mp4 * d; i += kAhatThreads) {
    const int j = i / d, c = i % d;
    sM[j * dq + c] = j < m ? mmat[((size_t)bh * m + j) * d + c] : 0.f;
  }
  for (int j = tid; j < mp4; j += kAhatThreads) {
    sc[j] = j < m ? mu[(size_t)bh * m + j] : 0.f;
    sc[mp4 + j] = j < m ? rstd[(size_t)bh * m + j] : 0.f;
    sc[2 * mp4 + j] = (j < m && whiten && bias) ? bias[(size_t)h * m + j] : 0.f;
  }
  // dM thread slots: (landmark quad lg, channel quad cq), KS token classes.
  const int cqn = d >> 2, set = (mp4 >> 2) * cqn;
  const int KS = max(1, kAhatThreads / set);
  const int ks = tid / set, lg = (tid % set) / cqn, cq = tid % cqn;
  const bool on = ks < KS;
  float acc[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
  float s1 = 0.f, s2 = 0.f;
  const int tiles = (n + kBwdTile - 1) / kBwdTile;
  const int t0 = sp * tiles_per_split, t1 = min(tiles, t0 + tiles_per_split);
  __syncthreads();
  for (int t = t0; t < t1; ++t) {
    const int n0 = t * kBwdTile;
    for (int i = tid; i < mp4 * kBwdTile; i += kAhatThreads) {
      const int j = i / kBwdTile, tt = i % kBwdTile, tok = n0 + tt;
      float z = 0.f;
      if (tok < n && j < m) {
        const float a = at[((size_t)bh * m + j) * n + tok];
        z = whiten ? (a - sc[j]) * sc[mp4 + j] : a;
      }
      sZ[j * tq + tt] = z;
    }
    for (int i = tid; i < kBwdTile * cqn; i += kAhatThreads) {
      const int tt = i / cqn, c4 = i % cqn, tok = n0 + tt;
      const float4 g = tok < n ? *reinterpret_cast<const float4*>(&gout[((size_t)bh * n + tok) * d + 4 * c4])
                               : make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(&sG[tt * dq + 4 * c4]) = g;
    }
    __syncthreads();
    // dA^ = G M^T
    for (int lq = warp; lq < (mp4 >> 2); lq += kAhatThreads / 32) {
      float o[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) o[a][b] = 0.f;
      for (int c4 = 0; c4 < cqn; ++c4) {
        float4 g[4], mv[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) g[b] = *reinterpret_cast<const float4*>(&sG[(lane + 32 * b) * dq + 4 * c4]);
#pragma unroll
        for (int a = 0; a < 4; ++a) mv[a] = *reinterpret_cast<const float4*>(&sM[(4 * lq + a) * dq + 4 * c4]);
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            o[a][b] = fmaf(g[b].x, mv[a].x, o[a][b]);
            o[a][b] = fmaf(g[b].y, mv[a].y, o[a][b]);
            o[a][b] = fmaf(g[b].z, mv[a].z, o[a][b]);
            o[a][b] = fmaf(g[b].w, mv[a].w, o[a][b]);
          }
      }
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int j = 4 * lq + a;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int tt = lane + 32 * b, tok = n0 + tt;
          sD[j * tq + tt] = o[a][b];
          if (j < m && tok < n) dahat[((size_t)bh * m + j) * n + tok] = o[a][b];
        }
      }
    }
    // dM partial: sum over the tile's token quads of this thread's class
    if (on) {
      for (int q = ks; q < kBwdTile / 4; q += KS) {
        const int tt = 4 * q;
        float4 z4[4], g4[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float beta = sc[2 * mp4 + 4 * lg + r];
          const float4 zz = *reinterpret_cast<const float4*>(&sZ[(4 * lg + r) * tq + tt]);
          z4[r] = make_float4(zz.x + beta, zz.y + beta, zz.z + beta, zz.w + beta);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) g4[u] = *reinterpret_cast<const float4*>(&sG[(tt + u) * dq + 4 * cq]);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float zu[4] = {z4[r].x, z4[r].y, z4[r].z, z4[r].w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            acc[r][0] = fmaf(zu[u], g4[u].x, acc[r][0]);
            acc[r][1] = fmaf(zu[u], g4[u].y, acc[r][1]);
            acc[r][2] = fmaf(zu[u], g4[u].z, acc[r][2]);
            acc[r][3] = fmaf(zu[u], g4[u].w, acc[r][3]);
          }
        }
      }
    }
    __syncthreads();
    if (tid < m) {
      for (int tt = 0; tt < kBwdTile; tt += 4) {
        const float4 dv = *reinterpret_cast<const float4*>(&sD[tid * tq + tt]);
        const float4 zv = *reinterpret_cast<const float4*>(&sZ[tid * tq + tt]);
        s1 += dv.x; s1 += dv.y; s1 += dv.z; s1 += dv.w;
        s2 = fmaf(dv.x, zv.x, s2); s2 = fmaf(dv.y, zv.y, s2);
        s2 = fmaf(dv.z, zv.z, s2); s2 = fmaf(dv.w, zv.w, s2);
      }
    }
    __syncthreads();
  }
  // Token classes combined in order (padding tokens contribute zeros: G is zero there).
#pragma unroll
  for (int e = 0; e < 16; ++e) red[e * kAhatThreads + tid] = on ? acc[e >> 2][e & 3] : 0.f;
  __syncthreads();
  float* pdm = part_dm + ((size_t)bh * splits + sp) * m * d;
  for (int i = tid; i < m * d; i += kAhatThreads) {
    const int j = i / d, c = i % d;
    const int lgi = j >> 2, r = j & 3, cqi = c >> 2, cc = c & 3;
    float sum = 0.f;
    for (int qq = 0; qq < KS; ++qq) sum += red[(r * 4 + cc) * kAhatThreads + qq * set + lgi * cqn + cqi];
    pdm[i] = sum;
  }
  if (tid < m) {
    float* ps = part_s + ((size_t)bh * splits + sp) * 2 * m;
    ps[tid] = s1;
    ps[m + tid] = s2;
  }
}

// ---- per head: dM, dBV = X^T dM, S_T = sym(dM BV^T), the whitening sums ------------------
// kMidParts CTAs per head.  Each sums the dM partials (every thread's elements loaded
// together, one split at a time, in split order) and forms its quarter of the rows of dBV and
// of S_T; part 0 also writes the whitening sums.
constexpr int kMidParts = 4;
constexpr int kMidElems = (kMaxM * kMaxD + kBwdThreads - 1) / kBwdThreads;   // 32

__global__ void __launch_bounds__(kBwdThreads)
bwd_mid_kernel(const float* __restrict__ xs, const float* __restrict__ bvg,
               const float* __restrict__ part_dm, const float* __restrict__ part_s,
               float* __restrict__ dbv, float* __restrict__ st, float* __restrict__ s12,
               float* __restrict__ dbias_bh, int m, int d, int T, int splits, int whiten) {
  extern __shared__ float4 smem_m4[];
  float* smem = reinterpret_cast<float*>(smem_m4);
  const int dp = d + 1;               // padded rows: threads of a warp read different rows
  float* sdM = smem;                  // [m][d + 1]
  float* sBV = sdM + m * dp;          // [m][d + 1]
  float* sX = sBV + m * dp;           // [m][m]  X_T
  const long bh = blockIdx.x / kMidParts;
  const int part = blockIdx.x % kMidParts;
  const int rows = (m + kMidParts - 1) / kMidParts;
  const int r0 = part * rows, r1 = min(m, r0 + rows);
  const int tid = threadIdx.x;
  const size_t mm = (size_t)m * m;
  const int md = m * d;
  {
    float a[kMidElems];
#pragma unroll
    for (int u = 0; u < kMidElems; ++u) a[u] = 0.f;
    const float* pa = part_dm + (size_t)bh * splits * md;
    for (int sp = 0; sp < splits; ++sp) {
      const float* src = pa + (size_t)sp * md;
#pragma unroll
      for (int u = 0; u < kMidElems; ++u) {
        const int e = tid + kBwdThreads * u;
        if (e < md) a[u] += src[e];
      }
    }
#pragma unroll
    for (int u = 0; u < kMidElems; ++u) {
      const int e = tid + kBwdThreads * u;
      if (e < md) {
        sdM[(e / d) * dp + e % d] = a[u];
        sBV[(e / d) * dp + e % d] = bvg[(size_t)bh * md + e];   // kept by the training forward
      }
    }
  }
  const int mk = (m + 3) & ~3;           // row length of the saved iterates
  for (int e = tid; e < m * m; e += kBwdThreads)
    sX[e] = xs[((size_t)bh * (T + 1) + T) * m * mk + (e / m) * mk + e % m];
  if (part == 0 && tid < m) {
    float a = 0.f, b = 0.f;
    for (int sp = 0; sp < splits; ++sp) {
      a += part_s[((size_t)bh * splits + sp) * 2 * m + tid];
      b += part_s[((size_t)bh * splits + sp) * 2 * m + m + tid];
    }
    s12[(size_t)bh * 2 * m + tid] = a;
    s12[(size_t)bh * 2 * m + m + tid] = b;
    dbias_bh[(size_t)bh * m + tid] = whiten ? a : 0.f;
  }
  __syncthreads();
  for (int e = r0 * d + tid; e < r1 * d; e += kBwdThreads) {
    const int j = e / d, c = e % d;
    float s = 0.f;
    for (int k = 0; k < m; ++k) s = fmaf(sX[k * m + j], sdM[k * dp + c], s);
    dbv[(size_t)bh * md + e] = s;
  }
  // (i, j) and (j, i) add the same two dot products: S_T is exactly symmetric.
  for (int e = r0 * m + tid; e < r1 * m; e += kBwdThreads) {
    const int i = e / m, j = e % m;
    float a = 0.f, b = 0.f;
    for (int c = 0; c < d; ++c) {
      a = fmaf(sdM[i * dp + c], sBV[j * dp + c], a);
      b = fmaf(sdM[j * dp + c], sBV[i * dp + c], b);
    }
    st[(size_t)bh * mm + e] = 0.5f * (a + b);
  }
}

// ---- per head: the Newton-Schulz steps backwards, the landmark-block term of dL ------------
// Only the symmetric part of dLoss/dW matters (W and D_LL are symmetric, and dL takes
// dW + dW^T), and X_t, W are exactly symmetric, so the reverse iteration carries
// S_t = sym(dLoss/dX_t):
//   S_t = 2 S - W X_t S - (W X_t S)^T;  dW -= X_t S_{t+1} X_t,
// three 64 x 64 products per step (U = X_t S and its transpose, W U, X_t U^T) on the tiled
// CUDA-core product of the Newton-Schulz kernels.  The iterates X_t are the ones the forward
// saved; X_{t-1} is copied in (cp.async) while step t's products run.  This kernel runs on
// the side stream, next to the token kernels that do not need its result.
template <int S>
__global__ void __launch_bounds__(kHeadThreads, 1)
bwd_ns_kernel(const float* __restrict__ landmarks, const float* __restrict__ xs,
              const float* __restrict__ st, float* __restrict__ dll, int d, int T, float eps,
              float c_exp, float lam, int gauss) {
  using Sh = NsShape<S>;
  constexpr int M = Sh::M, MK = Sh::MK, NWT = Sh::NWT;
  constexpr int MM = 64 * kMS;
  extern __shared__ float4 smem_h4[];
  float* smem = reinterpret_cast<float*>(smem_h4);
  float* Wb = smem;
  float* Xb[2] = {Wb + MM, Wb + 2 * MM};
  float* Sb = Wb + 3 * MM;
  float* Sn = Wb + 4 * MM;
  float* U = Wb + 5 * MM;
  float* Ut = Wb + 6 * MM;
  float* dW = Wb + 7 * MM;
  float* part = Wb + 8 * MM;               // [Sh::PART_FLOATS]
  float* red = part + Sh::PART_FLOATS;     // [kRedFloats]
  float* R = red + kRedFloats;             // landmarks (prologue)
  const long bh = blockIdx.x;
  const int tid = threadIdx.x;
  const size_t mm = (size_t)M * M;
  for (int e = tid; e < 7 * MM; e += kHeadThreads) Xb[0][e] = 0.f;   // zero padding
  __syncthreads();
  constexpr int Q = MK / 4;                // float4 per saved row
  const float* xsh = xs + (size_t)bh * (T + 1) * M * MK;
  auto fetch = [&](int t, float* dst) {
    for (int e = tid; e < M * Q; e += kHeadThreads) {
      const int r = e / Q, c4 = e - r * Q;
      const unsigned a = static_cast<unsigned>(__cvta_generic_to_shared(&dst[r * kMS + 4 * c4]));
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(a),
                   "l"(xsh + (size_t)t * M * MK + 4 * e)
                   : "memory");
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  };
  if (T > 0) fetch(T - 1, Xb[0]);

  NsSmem sm;
  sm.W = Wb;
  sm.X = U;                                // X0 of the prologue: not used
  sm.P = nullptr;
  sm.Y = nullptr;
  sm.red = red;
  sm.part = nullptr;
  sm.sL = R;
  ns_prologue<S, kHeadThreads>(sm, landmarks + (size_t)bh * M * d, d, eps, c_exp, gauss != 0,
                               false, nullptr, nullptr, bh);
  for (int e = tid; e < MM; e += kHeadThreads) U[e] = 0.f;
  for (int e = tid; e < M * M; e += kHeadThreads) Sb[(e / M) * kMS + e % M] = st[(size_t)bh * mm + e];

  int cur = 0;
  for (int t = T - 1; t >= 0; --t) {
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    __syncthreads();                                                  // X_t in Xb[cur]
    if (t > 0) fetch(t - 1, Xb[cur ^ 1]);
    const float* Xt = Xb[cur];
    sym_product<MK, NWT, kPlain>(Xt, Sb, nullptr, U, part, Ut);      // U = X_t S, Ut = U^T
    sym_product<MK, NWT, kSymRecur>(Wb, U, Sb, Sn, part);            // 2S - W U - (W U)^T
    sym_product<MK, NWT, kSubtract>(Xt, Ut, nullptr, dW, part);      // dW -= X_t S X_t
    float* tmp = Sb; Sb = Sn; Sn = tmp;
    cur ^= 1;
  }
  __syncthreads();

  // X0 = W^T / (|W|_1 |W|_inf): the symmetric part of dX0^T / scale, and the scale's
  // derivative through the first maximal column (row) sum.
  if (tid < 32) {
    const int lane = tid;
    float best_c = -1.f, best_r = -1.f;
    int jc = 0, ir = 0;
    for (int j = 0; j < M; ++j) {
      float cs = 0.f, rs = 0.f;
      for (int i = 0; i < M; ++i) {
        cs += fabsf(Wb[i * kMS + j]);
        rs += fabsf(Wb[j * kMS + i]);
      }
      if (cs > best_c) { best_c = cs; jc = j; }
      if (rs > best_r) { best_r = rs; ir = j; }
    }
    const float scale = best_c * best_r;
    float dsc = 0.f;
    for (int e = lane; e < M * M; e += 32) dsc -= Sb[(e / M) * kMS + e % M] * Wb[(e / M) * kMS + e % M];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dsc += __shfl_xor_sync(0xffffffffu, dsc, o);
    dsc /= scale * scale;
    if (lane == 0) {
      red[0] = scale;
      red[1] = dsc * best_r;       // d|W|_1
      red[2] = dsc * best_c;       // d|W|_inf
      red[3] = __int_as_float(jc);
      red[4] = __int_as_float(ir);
    }
  }
  __syncthreads();
  {
    const float scale = red[0], dn1 = red[1], dninf = red[2];
    const float inv_scale = 1.f / scale;          // one division, not one per element
    const int jc = __float_as_int(red[3]), ir = __float_as_int(red[4]);
    for (int e = tid; e < M * M; e += kHeadThreads) {
      const int i = e / M, j = e % M;
      float g = dW[i * kMS + j] + Sb[i * kMS + j] * inv_scale;
      const float w = Wb[i * kMS + j];
      const float sw = w > 0.f ? 1.f : (w < 0.f ? -1.f : 0.f);
      if (j == jc) g += dn1 * sw;
      if (i == ir) g += dninf * sw;
      // W = exp(-D_LL / lambda) + eps I: dLoss/dD_LL off the diagonal
      U[i * kMS + j] = (i == j) ? 0.f : -w / lam * g;
    }
  }
  __syncthreads();
  // dL_pc (landmark block) = sum_k (g[p][k] + g[k][p]) slope(L_pc, L_kc)
  const float* Lh = landmarks + (size_t)bh * M * d;
  for (int e = tid; e < M * d; e += kHeadThreads) {
    const int p = e / d, c = e % d;
    const float lp = Lh[p * d + c];
    float s = 0.f;
    for (int k = 0; k < M; ++k) {
      if (k == p) continue;
      const float g = U[p * kMS + k] + U[k * kMS + p];
      const float lk = Lh[k * d + c];
      s = fmaf(g, gauss ? 2.f * (lp - lk) : (lp > lk ? 1.f : (lp < lk ? -1.f : 0.f)), s);
    }
    dll[(size_t)bh * M * d + e] = s;
  }
}

// ---- query side: g = -(A / lambda) dA, dQ ------------------------------------------------
// One CTA (512 threads) per (head, 128-token tile): g for the tile (stored), then thread
// (token quad, channel quad) runs over the landmarks with g (float4 over its tokens) and L
// (float4 over its channels) for 16 dQ entries.
template <bool kGauss, int TU>
__global__ void __launch_bounds__(512)
bwd_query_kernel(const void* __restrict__ q, const float* __restrict__ at,
                 const float* __restrict__ dahat, const float* __restrict__ mu,
                 const float* __restrict__ rstd, const float* __restrict__ s12,
                 const float* __restrict__ landmarks, float* __restrict__ gq,
                 float* __restrict__ dq, int m, int d, int n, float lam, int whiten, int tiles,
                 int bf16) {
  extern __shared__ float4 smem_q4[];
  float* smem = reinterpret_cast<float*>(smem_q4);
  const int dq4 = d + 4, tq = kBwdTile + 4;
  float* sL = smem;                    // [m][d + 4]
  float* sg = sL + m * dq4;            // [m][tile + 4]
  const long bh = blockIdx.x / tiles;
  const int n0 = (blockIdx.x % tiles) * kBwdTile;
  const int tid = threadIdx.x;
  const int cqn = d >> 2;
  for (int i = tid; i < m * d; i += 512) sL[(i / d) * dq4 + i % d] = landmarks[(size_t)bh * m * d + i];
  const float inv_n = 1.f / (float)n, inv_lam = 1.f / lam;
  for (int i = tid; i < m * kBwdTile; i += 512) {
    const int j = i / kBwdTile, tt = i % kBwdTile, tok = n0 + tt;
    float g = 0.f;
    if (tok < n) {
      const size_t o = ((size_t)bh * m + j) * n + tok;
      const float a = at[o], dz = dahat[o];
      float da = dz;
      if (whiten) {
        const float r = rstd[(size_t)bh * m + j];
        const float z = (a - mu[(size_t)bh * m + j]) * r;
        const float s1 = s12[(size_t)bh * 2 * m + j], s2 = s12[(size_t)bh * 2 * m + m + j];
        da = r * (dz - s1 * inv_n - z * s2 * inv_n);
      }
      g = -a * inv_lam * da;
      gq[o] = g;
    }
    sg[j * tq + tt] = g;
  }
  __syncthreads();
  for (int slot = tid; slot < (kBwdTile / TU) * cqn; slot += 512) {
    const int c4 = slot % cqn, t0 = TU * (slot / cqn);
    // Laplacian: x holds -Q 2^24, acc sums g step(L, -Q 2^24) = g ([L > Q] + [L == Q] / 2) and
    // gs the weights: dQ = sum_j g sgn(Q - L) = gs - 2 acc.
    float x[TU][4], acc[TU][4], gs[TU];
#pragma unroll
    for (int u = 0; u < TU; ++u) {
      const int tok = n0 + t0 + u;
      gs[u] = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        x[u][c] = tok < n ? load_in(q, ((size_t)bh * n + tok) * d + 4 * c4 + c, bf16 != 0) : 0.f;
        if constexpr (!kGauss) x[u][c] = neg_scaled(x[u][c]);
        acc[u][c] = 0.f;
      }
    }
    for (int jj = 0; jj < m; ++jj) {
      float gg[TU];
      if constexpr (TU == 4) {
        const float4 g4 = *reinterpret_cast<const float4*>(&sg[jj * tq + t0]);
        gg[0] = g4.x; gg[1] = g4.y; gg[2] = g4.z; gg[3] = g4.w;
      } else {
        const float2 g2 = *reinterpret_cast<const float2*>(&sg[jj * tq + t0]);
        gg[0] = g2.x; gg[1] = g2.y;
      }
      const float4 l4 = *reinterpret_cast<const float4*>(&sL[jj * dq4 + 4 * c4]);
      const float ll[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
      for (int u = 0; u < TU; ++u) {
        if constexpr (kGauss) {
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[u][c] = fmaf(gg[u], gauss_slope(x[u][c], ll[c]), acc[u][c]);
        } else {
          gs[u] += gg[u];
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[u][c] = fmaf(gg[u], step(ll[c], x[u][c]), acc[u][c]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < TU; ++u) {
      const int tok = n0 + t0 + u;
      if constexpr (!kGauss) {
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[u][c] = fmaf(-2.f, acc[u][c], gs[u]);
      }
      if (tok < n)
        *reinterpret_cast<float4*>(dq + ((size_t)bh * n + tok) * d + 4 * c4) =
            make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
    }
  }
}

// ---- key side: h = -(B / lambda) (dBV V^T), dK's distance term, dV = B^T dBV --------------
// One CTA (512 threads) per (head, 128-token tile).  dB = dBV V^T on 4 x 4 register tiles as in
// bwd_ahat_kernel; then thread (token quad, channel quad) runs over the landmarks with h, B
// (float4 over its tokens) and L, dBV (float4 over its channels) for 16 dK and 16 dV entries.
template <bool kGauss, int TU>
__global__ void __launch_bounds__(512)
bwd_key_kernel(const void* __restrict__ k, const void* __restrict__ v,
               const float* __restrict__ bt, const float* __restrict__ dbv,
               const float* __restrict__ landmarks, float* __restrict__ hk,
               float* __restrict__ dk, float* __restrict__ dv, int m, int d, int n, float lam,
               int tiles, int bf16) {
  extern __shared__ float4 smem_k4[];
  float* smem = reinterpret_cast<float*>(smem_k4);
  const int mp4 = (m + 3) & ~3;
  const int dq = d + 4, tq = kBwdTile + 4;
  float* sL = smem;                    // [mp4][d + 4]
  float* sW = sL + mp4 * dq;           // [mp4][d + 4]  dBV
  float* sV = sW + mp4 * dq;           // [tile][d + 4]
  float* sh = sV + kBwdTile * dq;      // [mp4][tile + 4]
  float* sB = sh + mp4 * tq;           // [mp4][tile + 4]
  const long bh = blockIdx.x / tiles;
  const int n0 = (blockIdx.x % tiles) * kBwdTile;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cqn = d >> 2;
  for (int i = tid; i < mp4 * d; i += 512) {
    const int j = i / d, c = i % d;
    sL[j * dq + c] = j < m ? landmarks[((size_t)bh * m + j) * d + c] : 0.f;
    sW[j * dq + c] = j < m ? dbv[((size_t)bh * m + j) * d + c] : 0.f;
  }
  for (int i = tid; i < kBwdTile * d; i += 512) {
    const int tt = i / d, c = i % d, tok = n0 + tt;
    sV[tt * dq + c] = tok < n ? load_in(v, ((size_t)bh * n + tok) * d + c, bf16 != 0) : 0.f;
  }
  for (int i = tid; i < mp4 * kBwdTile; i += 512) {
    const int j = i / kBwdTile, tt = i % kBwdTile, tok = n0 + tt;
    sB[j * tq + tt] = (j < m && tok < n) ? bt[((size_t)bh * m + j) * n + tok] : 0.f;
  }
  __syncthreads();
  // h = -(B / lambda) (dBV V^T): warp w landmark quad w, lane l tokens l + 32 b
  const float inv_lam = 1.f / lam;
  for (int lq = warp; lq < (mp4 >> 2); lq += 16) {
    float o[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) o[a][b] = 0.f;
    for (int c4 = 0; c4 < cqn; ++c4) {
      float4 vv[4], wv[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) vv[b] = *reinterpret_cast<const float4*>(&sV[(lane + 32 * b) * dq + 4 * c4]);
#pragma unroll
      for (int a = 0; a < 4; ++a) wv[a] = *reinterpret_cast<const float4*>(&sW[(4 * lq + a) * dq + 4 * c4]);
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          o[a][b] = fmaf(wv[a].x, vv[b].x, o[a][b]);
          o[a][b] = fmaf(wv[a].y, vv[b].y, o[a][b]);
          o[a][b] = fmaf(wv[a].z, vv[b].z, o[a][b]);
          o[a][b] = fmaf(wv[a].w, vv[b].w, o[a][b]);
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int j = 4 * lq + a;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int tt = lane + 32 * b, tok = n0 + tt;
        const float h = -sB[j * tq + tt] * inv_lam * o[a][b];
        sh[j * tq + tt] = h;
        if (j < m && tok < n) hk[((size_t)bh * m + j) * n + tok] = h;
      }
    }
  }
  __syncthreads();
  for (int slot = tid; slot < (kBwdTile / TU) * cqn; slot += 512) {
    const int c4 = slot % cqn;
    const int t0 = TU * (slot / cqn);
    // Laplacian: x holds -K 2^24, gk sums h step(L, -K 2^24) = h ([L > K] + [L == K] / 2) and
    // hs the weights: dK's distance term -sum_j h sgn(L - K) = hs - 2 gk.
    float x[TU][4], gk[TU][4], gv[TU][4], hs[TU];
#pragma unroll
    for (int u = 0; u < TU; ++u) {
      const int tok = n0 + t0 + u;
      hs[u] = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        x[u][c] = tok < n ? load_in(k, ((size_t)bh * n + tok) * d + 4 * c4 + c, bf16 != 0) : 0.f;
        if constexpr (!kGauss) x[u][c] = neg_scaled(x[u][c]);
        gk[u][c] = 0.f;
        gv[u][c] = 0.f;
      }
    }
    for (int j = 0; j < m; ++j) {
      float hh[TU], bb[TU];
      if constexpr (TU == 4) {
        const float4 h4 = *reinterpret_cast<const float4*>(&sh[j * tq + t0]);
        const float4 b4 = *reinterpret_cast<const float4*>(&sB[j * tq + t0]);
        hh[0] = h4.x; hh[1] = h4.y; hh[2] = h4.z; hh[3] = h4.w;
        bb[0] = b4.x; bb[1] = b4.y; bb[2] = b4.z; bb[3] = b4.w;
      } else {
        const float2 h2 = *reinterpret_cast<const float2*>(&sh[j * tq + t0]);
        const float2 b2 = *reinterpret_cast<const float2*>(&sB[j * tq + t0]);
        hh[0] = h2.x; hh[1] = h2.y;
        bb[0] = b2.x; bb[1] = b2.y;
      }
      const float4 l4 = *reinterpret_cast<const float4*>(&sL[j * dq + 4 * c4]);
      const float4 w4 = *reinterpret_cast<const float4*>(&sW[j * dq + 4 * c4]);
      const float ll[4] = {l4.x, l4.y, l4.z, l4.w}, ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int u = 0; u < TU; ++u) {
        if constexpr (!kGauss) hs[u] += hh[u];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if constexpr (kGauss) gk[u][c] = fmaf(-hh[u], gauss_slope(ll[c], x[u][c]), gk[u][c]);
          else gk[u][c] = fmaf(hh[u], step(ll[c], x[u][c]), gk[u][c]);
          gv[u][c] = fmaf(bb[u], ww[c], gv[u][c]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < TU; ++u) {
      const int tok = n0 + t0 + u;
      if constexpr (!kGauss) {
#pragma unroll
        for (int c = 0; c < 4; ++c) gk[u][c] = fmaf(-2.f, gk[u][c], hs[u]);
      }
      if (tok < n) {
        const size_t row = ((size_t)bh * n + tok) * d + 4 * c4;
        *reinterpret_cast<float4*>(dk + row) = make_float4(gk[u][0], gk[u][1], gk[u][2], gk[u][3]);
        *reinterpret_cast<float4*>(dv + row) = make_float4(gv[u][0], gv[u][1], gv[u][2], gv[u][3]);
      }
    }
  }
}

// ---- partials of dL over one token split: side 0 from the query block, 1 from the key block --
// Both sides add -w sgn(X - L) (side 0: X = Q, w = g; side 1: X = K, w = h, from
// +h sgn(L - K)).  Thread: quads (landmark j, channels 4 c4 .. 4 c4 + 3); per staged token one
// float4 of the token row and one weight, shared by the four channels.  Laplacian kernel: l holds
// -L 2^24, acc sums w step(X, -L 2^24) and ws the weights, and the partial is ws - 2 acc.
constexpr int kMaxQuads = kMaxPairs / 4;    // 8 quads per thread at m = 64, d = 128

// Quads per thread of the dL-partials kernel: 2, 4 or 8 (m d / 4 quads over 256 threads).
int lm_quads_per_thread(int m, int d) {
  const int need = (m * (d / 4) + kBwdThreads - 1) / kBwdThreads;
  return need <= 2 ? 2 : (need <= 4 ? 4 : kMaxQuads);
}

template <bool kGauss, int QPT>
__device__ __forceinline__ void lm_tile(const float* __restrict__ sX, const float* __restrict__ sw,
                                        int dp, int tp, int d4, int quads, const float4 (&lv)[QPT],
                                        float4 (&acc)[QPT], float (&ws)[QPT]) {
#pragma unroll
  for (int u = 0; u < QPT; ++u) {
    const int qd = threadIdx.x + kBwdThreads * u;
    if (qd < quads) {
      const int j = qd / d4, c4 = qd % d4;
      const float4 l = lv[u];
      float4 a = acc[u];
      float s = ws[u];
      const float* xp = sX + 4 * c4;
      const float* wp = sw + j * tp;
      for (int tt = 0; tt < kBwdTile; tt += 4) {
        const float4 w4 = *reinterpret_cast<const float4*>(wp + tt);
        const float w[4] = {w4.x, w4.y, w4.z, w4.w};
        if constexpr (!kGauss) s += (w4.x + w4.y) + (w4.z + w4.w);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float4 x = *reinterpret_cast<const float4*>(xp + (tt + r) * dp);
          if constexpr (kGauss) {
            a.x = fmaf(-w[r], gauss_slope(x.x, l.x), a.x);
            a.y = fmaf(-w[r], gauss_slope(x.y, l.y), a.y);
            a.z = fmaf(-w[r], gauss_slope(x.z, l.z), a.z);
            a.w = fmaf(-w[r], gauss_slope(x.w, l.w), a.w);
          } else {
            a.x = fmaf(w[r], step(x.x, l.x), a.x);
            a.y = fmaf(w[r], step(x.y, l.y), a.y);
            a.z = fmaf(w[r], step(x.z, l.z), a.z);
            a.w = fmaf(w[r], step(x.w, l.w), a.w);
          }
        }
      }
      acc[u] = a;
      ws[u] = s;
    }
  }
}

template <bool kGauss, int QPT>
__global__ void __launch_bounds__(kBwdThreads)
bwd_lm_kernel(const void* __restrict__ q, const void* __restrict__ k,
              const float* __restrict__ gq, const float* __restrict__ hk,
              const float* __restrict__ landmarks, float* __restrict__ part_dl, int m, int d,
              int n, int tiles_per_split, int splits, int bf16) {
  extern __shared__ float4 smem_l4[];
  float* smem = reinterpret_cast<float*>(smem_l4);
  const int dp = d + 4, tp = kBwdTile + 4;
  float* sX = smem;                      // [tile][d + 4]
  float* sw = sX + kBwdTile * dp;        // [m][tile + 4]
  const int side = blockIdx.x & 1;
  const long rest = blockIdx.x >> 1;
  const long bh = rest / splits;
  const int sp = (int)(rest % splits);
  const void* x = side == 0 ? q : k;
  const float* wgt = side == 0 ? gq : hk;
  const float* Lh = landmarks + (size_t)bh * m * d;
  const int d4 = d >> 2, quads = m * d4;
  float4 acc[QPT], lv[QPT];
  float ws[QPT];
#pragma unroll
  for (int u = 0; u < QPT; ++u) {
    const int qd = threadIdx.x + kBwdThreads * u;
    acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    ws[u] = 0.f;
    lv[u] = qd < quads ? *reinterpret_cast<const float4*>(&Lh[4 * qd]) : acc[u];
    if constexpr (!kGauss)
      lv[u] = make_float4(neg_scaled(lv[u].x), neg_scaled(lv[u].y), neg_scaled(lv[u].z),
                          neg_scaled(lv[u].w));
  }
  const int tiles = (n + kBwdTile - 1) / kBwdTile;
  const int t0 = sp * tiles_per_split, t1 = min(tiles, t0 + tiles_per_split);
  for (int t = t0; t < t1; ++t) {
    const int n0 = t * kBwdTile;
    for (int i = threadIdx.x; i < kBwdTile * d4; i += kBwdThreads) {
      const int tt = i / d4, c4 = i % d4, tok = n0 + tt;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (tok < n) {
        const size_t e = ((size_t)bh * n + tok) * d + 4 * c4;
        if (bf16) {
          v = make_float4(load_in(x, e, true), load_in(x, e + 1, true), load_in(x, e + 2, true),
                          load_in(x, e + 3, true));
        } else {
          v = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(x) + e);
        }
      }
      *reinterpret_cast<float4*>(&sX[tt * dp + 4 * c4]) = v;
    }
    for (int i = threadIdx.x; i < m * kBwdTile; i += kBwdThreads) {
      const int j = i / kBwdTile, tt = i % kBwdTile, tok = n0 + tt;
      sw[j * tp + tt] = tok < n ? wgt[((size_t)bh * m + j) * n + tok] : 0.f;
    }
    __syncthreads();
    lm_tile<kGauss, QPT>(sX, sw, dp, tp, d4, quads, lv, acc, ws);
    __syncthreads();
  }
  float* out = part_dl + (((size_t)bh * 2 + side) * splits + sp) * m * d;
#pragma unroll
  for (int u = 0; u < QPT; ++u) {
    const int qd = threadIdx.x + kBwdThreads * u;
    float4 a = acc[u];
    if constexpr (!kGauss)
      a = make_float4(fmaf(-2.f, a.x, ws[u]), fmaf(-2.f, a.y, ws[u]), fmaf(-2.f, a.z, ws[u]),
                      fmaf(-2.f, a.w, ws[u]));
    if (qd < quads) *reinterpret_cast<float4*>(&out[4 * qd]) = a;
  }
}

// ---- dL per head (one element per thread, every partial load in flight); dbias ----------
__global__ void __launch_bounds__(kBwdThreads)
bwd_dl_kernel(const float* __restrict__ part_dl, const float* __restrict__ dll,
              const float* __restrict__ dbias_bh, float* __restrict__ dl,
              float* __restrict__ dbias, int m, int d, int splits, int batch, int heads,
              int chunks) {
  const long bh = blockIdx.x / chunks;
  const int e = (blockIdx.x % chunks) * kBwdThreads + threadIdx.x;
  const size_t md = (size_t)m * d;
  if (e < m * d) {
    float s = 0.f;
    for (int side = 0; side < 2; ++side) {
      const float* src = part_dl + ((size_t)bh * 2 + side) * splits * md + e;
#pragma unroll 16
      for (int sp = 0; sp < splits; ++sp) s += src[(size_t)sp * md];
    }
    dl[(size_t)bh * md + e] = s + dll[(size_t)bh * md + e];
  }
  if (dbias && bh < heads && blockIdx.x % chunks == 0) {   // batch 0: head h = bh sums the batch
    for (int j = threadIdx.x; j < m; j += kBwdThreads) {
      float s = 0.f;
      for (int b = 0; b < batch; ++b) s += dbias_bh[((size_t)b * heads + bh) * m + j];
      dbias[(size_t)bh * m + j] = s;
    }
  }
}

// ---- pooling backward: dK_n += dL_{window(n)} / (ph pw) ----------------------------------
// Thread: one 4-channel piece c4 of every tpp-th token of the tile; the token's window is
// found once per token, and dK moves in 16-byte pieces.
__global__ void __launch_bounds__(kBwdThreads)
bwd_pool_kernel(const float* __restrict__ dl, float* __restrict__ dk, int m, int d, int n,
                int grid_w, int s, int ph, int pw, int tiles) {
  const long bh = blockIdx.x / tiles;
  const int n0 = (blockIdx.x % tiles) * kBwdTile;
  const float inv = 1.f / (float)(ph * pw);
  const int d4 = d >> 2, tpp = kBwdThreads / d4;
  const int c4 = threadIdx.x % d4, t0 = threadIdx.x / d4;
  if (t0 >= tpp) return;
  const float* dlh = dl + (size_t)bh * m * d + 4 * c4;
#pragma unroll 4
  for (int tt = t0; tt < kBwdTile; tt += tpp) {
    const int tok = n0 + tt;
    if (tok >= n) break;
    const int r = tok / grid_w, col = tok - r * grid_w;
    const int j = (r / ph) * s + col / pw;
    const float4 g = *reinterpret_cast<const float4*>(dlh + (size_t)j * d);
    float4* p = reinterpret_cast<float4*>(dk + ((size_t)bh * n + tok) * d + 4 * c4);
    float4 v = *p;
    v.x += g.x * inv;
    v.y += g.y * inv;
    v.z += g.z * inv;
    v.w += g.w * inv;
    *p = v;
  }
}

template <int S>
const void* ns_bwd_ptr() { return reinterpret_cast<const void*>(&bwd_ns_kernel<S>); }

const void* pick_ns_bwd(int s) {
  switch (s) {
    case 1: return ns_bwd_ptr<1>();
    case 2: return ns_bwd_ptr<2>();
    case 3: return ns_bwd_ptr<3>();
    case 4: return ns_bwd_ptr<4>();
    case 5: return ns_bwd_ptr<5>();
    case 6: return ns_bwd_ptr<6>();
    case 7: return ns_bwd_ptr<7>();
    case 8: return ns_bwd_ptr<8>();
    default: return nullptr;
  }
}


size_t ahat_smem(int m, int d) {
  const size_t mp4 = (m + 3) & ~3;
  const size_t stage = mp4 * (d + 4) + (size_t)kBwdTile * (d + 4) + 2 * mp4 * (kBwdTile + 4) +
                       3 * mp4;
  const size_t red = 16 * (size_t)kAhatThreads + mp4 * (d + 4);   // red aliases sG onwards
  return sizeof(float) * (stage > red ? stage : red);
}
size_t ns_bwd_smem(int d) {
  return sizeof(float) * (8 * 64 * (size_t)kMS + 4 * 3 * 32 * 32 + kRedFloats + 64 * (size_t)d);
}
size_t mid_smem(int m, int d) { return sizeof(float) * (2 * (size_t)m * (d + 1) + (size_t)m * m); }
size_t query_smem(int m, int d) {
  return sizeof(float) * ((size_t)m * (d + 4) + (size_t)m * (kBwdTile + 4));
}
size_t key_smem(int m, int d) {
  const size_t mp4 = (m + 3) & ~3;
  return sizeof(float) * (2 * mp4 * (d + 4) + (size_t)kBwdTile * (d + 4) +
                          2 * mp4 * (kBwdTile + 4));
}
size_t lm_smem(int m, int d) {
  return sizeof(float) * ((size_t)kBwdTile * (d + 4) + (size_t)m * (kBwdTile + 4));
}
const void* lm_kernel(bool gauss, int qpt) {
  if (gauss) {
    if (qpt == 2) return reinterpret_cast<const void*>(&bwd_lm_kernel<true, 2>);
    if (qpt == 4) return reinterpret_cast<const void*>(&bwd_lm_kernel<true, 4>);
    return reinterpret_cast<const void*>(&bwd_lm_kernel<true, kMaxQuads>);
  }
  if (qpt == 2) return reinterpret_cast<const void*>(&bwd_lm_kernel<false, 2>);
  if (qpt == 4) return reinterpret_cast<const void*>(&bwd_lm_kernel<false, 4>);
  return reinterpret_cast<const void*>(&bwd_lm_kernel<false, kMaxQuads>);
}

}  // namespace

// Token splits of a kernel over `units` independent units of `tiles` chunks each: its time is
// about the waves of resident CTAs times the chunks of one CTA (plus half a chunk for its
// prologue and the store of its partial); take the split count that minimises that, the
// fewest CTAs among equals.
static void choose_splits(long long slots, long long units, int tiles, int max_splits,
                          int* splits_out, int* tps_out) {
  double best = 0.0;
  for (int want = 1; want <= std::min(tiles, max_splits); ++want) {
    const int tps = (tiles + want - 1) / want, splits = (tiles + tps - 1) / tps;
    const long long waves = (units * splits + slots - 1) / slots;
    const double cost = (double)waves * (tps + 0.5);
    if (want == 1 || cost < best) {
      best = cost;
      *tps_out = tps;
      *splits_out = splits;
    }
  }
}

BwdLayout bwd_layout(const lapl_attn_plan& p) {
  const Geometry& g = p.geo;
  const size_t bh = (size_t)g.bh, m = g.m, d = g.d, n = g.n, sp = g.ahat_splits;
  BwdLayout L;
  size_t off = 0;
  auto take = [&](size_t floats) {
    const size_t at = off;
    off = align_up(off + floats * sizeof(float), kAlign);
    return at;
  };
  L.dahat = take(bh * m * n);
  L.part_dm = take(bh * sp * m * d);
  L.part_s = take(bh * sp * 2 * m);
  L.s12 = take(bh * 2 * m);
  L.dbv = take(bh * m * d);
  L.dll = take(bh * m * d);
  L.dbias_bh = take(bh * m);
  L.gq = take(bh * m * n);
  L.hk = take(bh * m * n);
  L.part_dl = take(bh * 2 * (size_t)g.lm_splits * m * d);
  L.dl = take(bh * m * d);
  L.st = take(bh * m * m);
  L.total = off;
  return L;
}

cudaError_t bwd_configure(lapl_attn_plan& p) {
  Geometry& g = p.geo;
  cudaError_t e = cudaFuncSetAttribute(bwd_ahat_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)ahat_smem(g.m, g.d));
  const void* hf = pick_ns_bwd(g.s);
  if (!hf) return cudaErrorInvalidValue;
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(hf, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ns_bwd_smem(g.d));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_mid_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)mid_smem(g.m, g.d));
  const int qs = (int)query_smem(g.m, g.d), ks = (int)key_smem(g.m, g.d),
            ls = (int)lm_smem(g.m, g.d);
  const void* tok_kernels[] = {
      reinterpret_cast<const void*>(&bwd_query_kernel<false, 2>),
      reinterpret_cast<const void*>(&bwd_query_kernel<false, 4>),
      reinterpret_cast<const void*>(&bwd_query_kernel<true, 2>),
      reinterpret_cast<const void*>(&bwd_query_kernel<true, 4>),
      reinterpret_cast<const void*>(&bwd_key_kernel<false, 2>),
      reinterpret_cast<const void*>(&bwd_key_kernel<false, 4>),
      reinterpret_cast<const void*>(&bwd_key_kernel<true, 2>),
      reinterpret_cast<const void*>(&bwd_key_kernel<true, 4>)};
  for (int i = 0; i < 8 && e == cudaSuccess; ++i)
    e = cudaFuncSetAttribute(tok_kernels[i], cudaFuncAttributeMaxDynamicSharedMemorySize, i < 4 ? qs : ks);
  const bool gauss = p.cfg.kernel == LAPL_KERNEL_GAUSSIAN;
  const void* lmk = lm_kernel(gauss, lm_quads_per_thread(g.m, g.d));
  if (e == cudaSuccess) e = cudaFuncSetAttribute(lmk, cudaFuncAttributeMaxDynamicSharedMemorySize, ls);
  int occ = 0, aocc = 0;
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, lmk, kBwdThreads, ls);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&aocc, bwd_ahat_kernel, kAhatThreads,
                                                      ahat_smem(g.m, g.d));
  if (e != cudaSuccess) return e;
  const int tiles = std::max(1, (g.n + kBwdTile - 1) / kBwdTile);
  const long long heads = std::max<long long>(g.bh, 1);
  choose_splits((long long)p.num_sms * std::max(occ, 1), 2 * heads, tiles, 256, &g.lm_splits,
                &g.lm_tiles_per_split);
  choose_splits((long long)p.num_sms * std::max(aocc, 1), heads, tiles, 64, &g.ahat_splits,
                &g.ahat_tiles_per_split);
  return cudaSuccess;
}

cudaError_t launch_backward(const lapl_attn_plan& p, const void* q, const void* k, const void* v,
                            const float* bias, const float* gout, float* dq, float* dk,
                            float* dv, float* dbias, const char* fws, char* bws,
                            cudaStream_t st) {
  const Geometry& g = p.geo;
  const WorkspaceLayout& F = p.ws;
  const BwdLayout B = bwd_layout(p);
  const int m = g.m, d = g.d, n = g.n, splits = g.ahat_splits, tps = g.ahat_tiles_per_split;
  const int lsp = g.lm_splits, ltps = g.lm_tiles_per_split;
  const int heads = p.cfg.heads, whiten = p.cfg.whiten, bf16 = p.cfg.in_dtype == LAPL_BF16;
  const bool gauss = p.cfg.kernel == LAPL_KERNEL_GAUSSIAN;
  const float lam = p.cfg.lambda;
  const float* L = reinterpret_cast<const float*>(fws + F.landmarks);
  const float* Xs = reinterpret_cast<const float*>(fws + F.xs);
  const float* At = reinterpret_cast<const float*>(fws + F.at);
  const float* Bt = reinterpret_cast<const float*>(fws + F.bt);
  const float* BV = reinterpret_cast<const float*>(fws + F.bv);
  const float* M = reinterpret_cast<const float*>(fws + F.mmat);
  const float* mu = reinterpret_cast<const float*>(fws + F.mu);
  const float* rstd = reinterpret_cast<const float*>(fws + F.rstd);
  auto W = [&](size_t off) { return reinterpret_cast<float*>(bws + off); };
  float *dahat = W(B.dahat), *part_dm = W(B.part_dm), *part_s = W(B.part_s), *s12 = W(B.s12),
        *dbv = W(B.dbv), *dll = W(B.dll), *dbias_bh = W(B.dbias_bh), *gq = W(B.gq),
        *hk = W(B.hk), *part_dl = W(B.part_dl), *dl = W(B.dl), *sT = W(B.st);
  const unsigned bh = (unsigned)g.bh;
  const int ptiles = (n + kBwdTile - 1) / kBwdTile;

  bwd_ahat_kernel<<<bh * splits, kAhatThreads, ahat_smem(m, d), st>>>(
      At, M, mu, rstd, bias, gout, dahat, part_dm, part_s, m, d, n, heads, tps, splits, whiten);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bwd_mid_kernel<<<bh * kMidParts, kBwdThreads, mid_smem(m, d), st>>>(
      Xs, BV, part_dm, part_s, dbv, sT, s12, dbias_bh, m, d, p.cfg.ns_steps, splits, whiten);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // The Newton-Schulz backward (only the landmark-block term of dL needs it) on the side
  // stream, next to the token kernels.
  cudaStream_t side = p.side_stream;
  e = cudaEventRecord(p.ev_pool, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(side, p.ev_pool, 0);
  if (e != cudaSuccess) return e;
  {
    const void* f = pick_ns_bwd(g.s);
    int T = p.cfg.ns_steps, gs = gauss, dd = d;
    float eps = p.cfg.eps, c_exp = p.neg_log2e_over_lambda, lm = lam;
    void* args[] = {&L, &Xs, &sT, &dll, &dd, &T, &eps, &c_exp, &lm, &gs};
    e = cudaLaunchKernel(f, dim3(bh), dim3(kHeadThreads), args, ns_bwd_smem(d), side);
    if (e == cudaSuccess) e = cudaEventRecord(p.ev_join, side);
    if (e != cudaSuccess) return e;
  }
  // Tokens per thread in the token kernels: 4, or 2 when 32 token quads x d / 4 channel quads
  // would leave threads idle.
  const bool tu4 = (kBwdTile / 4) * (d / 4) >= 512;
  auto launch_tok = [&](auto qk, auto kk) {
    qk<<<bh * ptiles, 512, query_smem(m, d), st>>>(q, At, dahat, mu, rstd, s12, L, gq, dq, m, d,
                                                   n, lam, whiten, ptiles, bf16);
    kk<<<bh * ptiles, 512, key_smem(m, d), st>>>(k, v, Bt, dbv, L, hk, dk, dv, m, d, n, lam,
                                                 ptiles, bf16);
  };
  if (gauss) {
    if (tu4) launch_tok(bwd_query_kernel<true, 4>, bwd_key_kernel<true, 4>);
    else launch_tok(bwd_query_kernel<true, 2>, bwd_key_kernel<true, 2>);
  } else {
    if (tu4) launch_tok(bwd_query_kernel<false, 4>, bwd_key_kernel<false, 4>);
    else launch_tok(bwd_query_kernel<false, 2>, bwd_key_kernel<false, 2>);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    const void* f = lm_kernel(gauss, lm_quads_per_thread(m, d));
    int mm = m, dd = d, nn = n, ltps_ = ltps, lsp_ = lsp, bf = bf16;
    void* args[] = {&q, &k, &gq, &hk, &L, &part_dl, &mm, &dd, &nn, &ltps_, &lsp_, &bf};
    e = cudaLaunchKernel(f, dim3(bh * lsp * 2), dim3(kBwdThreads), args, lm_smem(m, d), st);
  }
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, p.ev_join, 0);
  if (e != cudaSuccess) return e;
  const unsigned dl_chunks = (unsigned)((m * d + kBwdThreads - 1) / kBwdThreads);
  bwd_dl_kernel<<<bh * dl_chunks, kBwdThreads, 0, st>>>(part_dl, dll, dbias_bh, dl, dbias, m, d,
                                                         lsp, p.cfg.batch, heads, dl_chunks);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int s = g.s;
  bwd_pool_kernel<<<bh * ptiles, kBwdThreads, 0, st>>>(dl, dk, m, d, n, p.cfg.grid_w, s,
                                                        p.cfg.grid_h / s, p.cfg.grid_w / s, ptiles);
  return cudaGetLastError();
}

}  // namespace lapl
