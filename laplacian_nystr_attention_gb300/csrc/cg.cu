// cg.cu -- conjugate-gradient solve of W M = B V, the solver the Newton-Schulz iteration is
// compared with.
//
// "LaplacianFormer: Rethinking Linear Attention with Laplacian Kernel", German explainer page,
// 4 (ablation) and English page, 4 ("Solver Robustness"): the pages weigh the multiply-only
// Newton-Schulz inverse against a conjugate-gradient (CG) solver, which they find less
// accurate and less stable when W is ill-conditioned.  With this solver X is never formed:
// each column b of B V is solved by T iterations of classical CG on W y = b from y = 0
// (q = W p; alpha = r.r / p.q; y += alpha p; r -= alpha q; beta = r.r_new / r.r_old;
// p = r + beta p), and a column stops only where no step is defined (r.r == 0 or p.q <= 0).
//
// One CTA (8 warps) per (batch, head).
//   * W = k(L, L) + eps I is built from the landmarks with the Newton-Schulz prologue.  The
//     kernel is launched as a programmatic dependent of the B V kernel, so this overlaps the
//     B V kernel's tail; griddepcontrol.wait then waits for that grid.
//   * The B V partials of the head (contiguous) are copied into shared memory with cp.async,
//     every copy of a chunk in flight at once, while each lane loads its rows of W into
//     registers; they are summed in split order (the order of the M kernel of the
//     Newton-Schulz path, so B V is the same bit for bit).
//   * Warp w owns columns j = w + 8 c (c < NC), in passes of 8 NC columns; lane l holds rows
//     l and l + 32 of W, y, r, p and q.  q = W p multiplies the register-resident rows of W
//     by p, which the warp exchanges through its own shared-memory slots (one float4
//     broadcast per 4 k).  The 2 NC dot products of an iteration are xor-butterfly sums over
//     the warp, all columns interleaved (every lane gets the same bits).  No CTA barrier is
//     taken inside the iteration.
#include "ns_common.cuh"

namespace lapl {
using namespace ns_detail;
namespace {

constexpr int kCgThreads = 256;
constexpr int kCgWarps = kCgThreads / 32;
constexpr int kMaxNc = 8;                 // columns per warp and pass
// Floats of the staging buffer for the B V partials (96 KB; at least one split of m x d).
constexpr int kStageFloats = 24576;

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(src) : "memory");
}

// v[c] <- sum over the warp's lanes of v[c], for every c (the same bits in every lane).
template <int NC>
__device__ __forceinline__ void warp_sums(float (&v)[NC]) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int c = 0; c < NC; ++c) v[c] += __shfl_xor_sync(0xffffffffu, v[c], o);
}

template <int S, int NC>
__global__ void __launch_bounds__(kCgThreads, 1)
cg_kernel(const float* __restrict__ landmarks, const float* __restrict__ bvp,
          float* __restrict__ mmat, float* __restrict__ dbg_dll, float* __restrict__ dbg_w,
          float* __restrict__ dbg_bv, float* __restrict__ dbg_m, int d, int T, float eps,
          float c_exp, int gauss, int splits, int region) {
  using Sh = NsShape<S>;
  constexpr int M = Sh::M, MK = Sh::MK, NH = Sh::NWT;    // NH rows per lane: lane + 32 h
  extern __shared__ float4 smem_cg4[];
  float* smem = reinterpret_cast<float*>(smem_cg4);
  NsSmem sm;
  sm.W = smem;                          // [64][kMS]
  sm.X = sm.W + 64 * kMS;               // X0 of the prologue (not used here)
  sm.P = nullptr;
  sm.Y = nullptr;
  sm.red = sm.X + 64 * kMS;             // [kRedFloats]
  sm.part = nullptr;
  sm.sL = sm.red + kRedFloats;          // landmarks, then the staged partials, then the
                                        // search directions: `region` floats
  float* sB = sm.sL + region;           // B V, [M][d]
  const long bh = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // W from the landmarks (written by the pooling kernel, which finished before the B V kernel
  // started), while the B V kernel may still run.
  ns_prologue<S, kCgThreads>(sm, landmarks + (size_t)bh * M * d, d, eps, c_exp, gauss != 0,
                             true, dbg_dll, dbg_w, bh);
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  // B V and the column statistics are complete: the output kernel may start its A tiles.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

  const int md = M * d;                          // a multiple of 8
  const int chunk = kStageFloats / md;           // >= 1 (md <= 64 * 128)
  float* stage = sm.X;                           // X, red and the region: free now
  const float* src = bvp + (size_t)bh * splits * md;
  auto issue = [&](int sp0) {
    const int nsp = splits - sp0 < chunk ? splits - sp0 : chunk;
    const float* c0 = src + (size_t)sp0 * md;
    for (int i = 4 * threadIdx.x; i < nsp * md; i += 4 * kCgThreads) cp_async16(&stage[i], &c0[i]);
    asm volatile("cp.async.commit_group;\n" ::: "memory");
    return nsp;
  };
  int nsp = issue(0);

  // Rows lane and lane + 32 of W into registers while the first copies are in flight.
  float w[NH][MK];
#pragma unroll
  for (int h = 0; h < NH; ++h)
#pragma unroll
    for (int k0 = 0; k0 < MK; k0 += 4) {
      const float4 v = *reinterpret_cast<const float4*>(&sm.W[(lane + 32 * h) * kMS + k0]);
      w[h][k0] = v.x;
      w[h][k0 + 1] = v.y;
      w[h][k0 + 2] = v.z;
      w[h][k0 + 3] = v.w;
    }

  // B V = sum of the split partials, in split order.
  for (int sp0 = 0; sp0 < splits; sp0 += chunk) {
    if (sp0 > 0) nsp = issue(sp0);
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    __syncthreads();
    // Four consecutive entries per thread (md is a multiple of 8), four splits loaded ahead.
    const float4* st4 = reinterpret_cast<const float4*>(stage);
    float4* sB4 = reinterpret_cast<float4*>(sB);
    const int md4 = md >> 2;
    for (int e = threadIdx.x; e < md4; e += kCgThreads) {
      float4 a = sp0 == 0 ? make_float4(0.f, 0.f, 0.f, 0.f) : sB4[e];
      int q = 0;
      for (; q + 4 <= nsp; q += 4) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = st4[(q + u) * md4 + e];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          a.x += v[u].x;
          a.y += v[u].y;
          a.z += v[u].z;
          a.w += v[u].w;
        }
      }
      for (; q < nsp; ++q) {
        const float4 v = st4[q * md4 + e];
        a.x += v.x;
        a.y += v.y;
        a.z += v.z;
        a.w += v.w;
      }
      sB4[e] = a;
    }
    __syncthreads();
  }

  float* dir = sm.sL + warp * NC * 64;   // this warp's p columns, [NC][64]
  for (int j0 = 0; j0 < d; j0 += kCgWarps * NC) {
    float y[NC][NH], r[NC][NH], p[NC][NH], rr[NC];
    bool live[NC];
    // r = p = b, y = 0.
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int j = j0 + warp + kCgWarps * c;
      rr[c] = 0.f;
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        const int i = lane + 32 * h;
        float b = 0.f;
        if (j < d && i < M) {
          b = sB[i * d + j];
          if (dbg_bv) dbg_bv[((size_t)bh * M + i) * d + j] = b;
        }
        y[c][h] = 0.f;
        r[c][h] = b;
        p[c][h] = b;
        rr[c] = fmaf(b, b, rr[c]);
        dir[c * 64 + i] = b;
      }
    }
    warp_sums<NC>(rr);
#pragma unroll
    for (int c = 0; c < NC; ++c) live[c] = (j0 + warp + kCgWarps * c) < d && rr[c] != 0.f;
    __syncwarp();

    for (int t = 0; t < T; ++t) {
      // q = W p: k ascending.
      float q[NC][NH];
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int h = 0; h < NH; ++h) q[c][h] = 0.f;
#pragma unroll
      for (int k0 = 0; k0 < MK; k0 += 4) {
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const float4 pk = *reinterpret_cast<const float4*>(&dir[c * 64 + k0]);
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            q[c][h] = fmaf(w[h][k0], pk.x, q[c][h]);
            q[c][h] = fmaf(w[h][k0 + 1], pk.y, q[c][h]);
            q[c][h] = fmaf(w[h][k0 + 2], pk.z, q[c][h]);
            q[c][h] = fmaf(w[h][k0 + 3], pk.w, q[c][h]);
          }
        }
      }
      __syncwarp();                   // every lane has read dir before it is overwritten
      float pq[NC], rn[NC];
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        pq[c] = 0.f;
#pragma unroll
        for (int h = 0; h < NH; ++h) pq[c] = fmaf(p[c][h], q[c][h], pq[c]);
      }
      warp_sums<NC>(pq);
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        live[c] = live[c] && pq[c] > 0.f;
        // alpha and beta by the fast division (within 2 ulp): the dot products they divide
        // carry about n u of rounding already, and an IEEE division costs hundreds of cycles
        // on this chain.
        const float alpha = live[c] ? __fdividef(rr[c], pq[c]) : 0.f;
        rn[c] = 0.f;
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          if (live[c]) {
            y[c][h] = fmaf(alpha, p[c][h], y[c][h]);
            r[c][h] = fmaf(-alpha, q[c][h], r[c][h]);
          }
          rn[c] = fmaf(r[c][h], r[c][h], rn[c]);
        }
      }
      warp_sums<NC>(rn);
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        if (live[c]) {
          const float beta = __fdividef(rn[c], rr[c]);
          rr[c] = rn[c];
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            p[c][h] = fmaf(beta, p[c][h], r[c][h]);
            dir[c * 64 + lane + 32 * h] = p[c][h];
          }
          live[c] = rn[c] != 0.f;
        }
      }
      __syncwarp();                   // the new directions are visible to the whole warp
    }

#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int j = j0 + warp + kCgWarps * c;
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        const int i = lane + 32 * h;
        if (j < d && i < M) {
          const size_t o = ((size_t)bh * M + i) * d + j;
          mmat[o] = y[c][h];
          if (dbg_m) dbg_m[o] = y[c][h];
        }
      }
    }
    __syncwarp();                     // dir is rewritten by the next pass
  }
}

// Columns per warp and pass: the power of two >= ceil(d / 8), at most 8 (d = 128 takes two
// passes).
int cols_per_warp(int d) {
  const int need = (d + kCgWarps - 1) / kCgWarps;
  int nc = 1;
  while (nc < need && nc < kMaxNc) nc *= 2;
  return nc;
}

template <int S>
const void* pick_nc(int nc) {
  switch (nc) {
    case 1: return reinterpret_cast<const void*>(&cg_kernel<S, 1>);
    case 2: return reinterpret_cast<const void*>(&cg_kernel<S, 2>);
    case 4: return reinterpret_cast<const void*>(&cg_kernel<S, 4>);
    case 8: return reinterpret_cast<const void*>(&cg_kernel<S, 8>);
    default: return nullptr;
  }
}

const void* pick_cg(int s, int d) {
  const int nc = cols_per_warp(d);
  switch (s) {
    case 1: return pick_nc<1>(nc);
    case 2: return pick_nc<2>(nc);
    case 3: return pick_nc<3>(nc);
    case 4: return pick_nc<4>(nc);
    case 5: return pick_nc<5>(nc);
    case 6: return pick_nc<6>(nc);
    case 7: return pick_nc<7>(nc);
    case 8: return pick_nc<8>(nc);
    default: return nullptr;
  }
}

}  // namespace

// Floats after W of the region shared by X0, the landmarks, the staged partials and the
// directions (X and red are part of it).
int cg_region_floats(int d) {
  int r = kStageFloats - (64 * kMS + kRedFloats);      // staging starts at X
  if (64 * d > r) r = 64 * d;
  if (kCgWarps * kMaxNc * 64 > r) r = kCgWarps * kMaxNc * 64;
  return r;
}

size_t cg_smem_bytes(int m, int d) {
  return sizeof(float) * (2 * 64 * (size_t)kMS + kRedFloats + (size_t)cg_region_floats(d) +
                          (size_t)m * d);
}

cudaError_t cg_configure(int s, int d, size_t smem) {
  const void* f = pick_cg(s, d);
  if (!f) return cudaErrorInvalidValue;
  return cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t launch_cg(const lapl_attn_plan& p, const float* landmarks, const float* bvp,
                      float* mmat, float* dbg_dll, float* dbg_w, float* dbg_bv, float* dbg_m,
                      cudaStream_t st) {
  const Geometry& g = p.geo;
  const void* f = pick_cg(g.s, g.d);
  if (!f) return cudaErrorInvalidValue;
  int d = g.d, T = p.cfg.ns_steps, splits = g.bv_splits, region = cg_region_floats(g.d);
  float eps = p.cfg.eps, c_exp = p.neg_log2e_over_lambda;
  int gauss = p.cfg.kernel == LAPL_KERNEL_GAUSSIAN;
  void* args[] = {&landmarks, &bvp, &mmat,  &dbg_dll, &dbg_w,  &dbg_bv, &dbg_m,
                  &d,         &T,   &eps,   &c_exp,   &gauss,  &splits, &region};
  // Programmatic dependent launch: the CTAs may start (and build W) while the B V kernel runs.
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)g.bh);
  cfg.blockDim = dim3(kCgThreads);
  cfg.dynamicSmemBytes = g.cg_smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, f, args);
}

}  // namespace lapl
