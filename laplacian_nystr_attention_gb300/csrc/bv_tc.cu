// bv_tc.cu -- B V on the tensor cores (tcgen05, TF32 operands split into an exact high/low pair,
// fp32 accumulation in tensor memory).
//
// "LaplacianFormer: Rethinking Linear Attention with Laplacian Kernel": the output is
// O = A^ (X (B V)), evaluated right to left so that the N x N matrix is never formed (Chinese
// explainer page, 2.2); B V is the first product, a contraction over the N tokens.
//
// One CTA per (batch, head, token split), 10 warps, chunks of 32 tokens:
//   warp 8     one thread copies each chunk with the Tensor Memory Accelerator into a ring of
//              kRaw raw stages: B^T[bh] rows 0..m-1 x 32 tokens (landmark-major, as stored) and
//              V[bh] 32 tokens x d (token-major, as stored); tokens past N read as zero.
//   warps 0-7  converters (two per scheduler: one warp alone left the conversion waiting on its
//              own shared-memory latencies): from a raw stage they build the two operands of one accumulation in
//              a ring of kOps operand stages (K-major, no swizzle, core matrices of 8 rows x 16
//              bytes; the strides between core matrices are padded by 16 bytes so that the
//              converters' 16-byte stores of a quarter-warp fall in 8 different bank groups):
//                A = [B_hi; B_lo]   128 rows: landmark j's TF32 high part in row j, its low
//                                   part in row 64 + j (rows m..63 and 64+m..127 stay zero);
//                Bop = [V_hi; V_lo] rows c and d + c hold value column c (fp32 V), or V's rows
//                                   alone (bf16 V is exact in TF32); 4 tokens x 4 columns are
//                                   transposed in registers.
//              After the last chunk warps 0-3 read the accumulator back.
//   warp 9     owns the tensor memory; one thread issues tcgen05.mma (M = 128, N = 2d or d,
//              K = 8) for each 8 tokens and commits each operand stage back to the converters.
// The column statistics of A run as a separate launch just before this one (col_stats_kernel,
// one CTA per landmark column); this grid is its programmatic dependent, so the two overlap.
// The accumulator D then holds
//   D[j][c] = B_hi V_hi,  D[j][d + c] = B_hi V_lo,  D[64 + j][c] = B_lo V_hi   (j < 64, c < d)
// and the split's partial (B V)[j][c] = D[j][c] + D[j][d + c] + D[64 + j][c] (the product of the
// two low parts, 2^-20 relative, is left out), written to the same partial buffer the M kernel
// reduces in split order.  Every barrier wait is bounded (one second); on a timeout the CTA sets
// the chain bit of the device error word, waits (bounded) for its copies and its tensor-core
// work, and frees its tensor memory.
#include <algorithm>

#include "common.cuh"

namespace lapl {
namespace {

constexpr int kTok = 32;                    // tokens (K) per chunk
constexpr int kRawMax = 12;                 // raw (copied) stages: as many as fit, <= 12
constexpr int kOps = 3;                     // operand stages
constexpr int kConvThreads = 256;           // warps 0-7: two per scheduler
constexpr int kTmaWarp = 8, kMmaWarp = 9;
constexpr int kBvTcThreads = 32 * 10;
constexpr unsigned kRawBt = 64 * kTok * 4;               // B^T part of a raw stage (m <= 64)
constexpr unsigned kSboA = 128, kLboA = 16 * 128 + 16;   // A: 128 rows
constexpr unsigned kOpABytes = (kTok / 4) * kLboA;       // 8 K-groups
constexpr unsigned kSboB = 144;                          // B: padded row-group stride

__host__ __device__ constexpr unsigned align128(unsigned x) { return (x + 127u) & ~127u; }
__host__ __device__ inline unsigned raw_v_bytes(int d, bool bf16) {
  return (unsigned)(kTok * d * (bf16 ? 2 : 4));
}
__host__ __device__ inline unsigned raw_stage_bytes(int d, bool bf16) {
  return align128(kRawBt + raw_v_bytes(d, bf16));
}
__host__ __device__ inline unsigned lbo_b(int nb) { return (unsigned)(nb / 8) * kSboB; }
__host__ __device__ inline unsigned op_stage_bytes(int nb) {
  return align128(kOpABytes + (kTok / 4) * lbo_b(nb));
}

__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ float tf32_rna(float x) {
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}
// K-major, no swizzle, descriptor version 1.
__device__ __forceinline__ uint64_t op_desc(unsigned addr, unsigned lbo, unsigned sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}
// D fp32, A and B TF32, both K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc(unsigned n) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}
__device__ __forceinline__ void mbar_init(unsigned bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_test(unsigned bar, unsigned parity) {
  unsigned done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait: gives up after `bound` ns of %globaltimer.
__device__ __forceinline__ bool mbar_wait(unsigned bar, unsigned parity,
                                          unsigned long long bound) {
  if (mbar_test(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_test(bar, parity))
    if (global_ns() - t0 > bound) return false;
  return true;
}
__device__ __forceinline__ void tma_load_2d(unsigned dst, const CUtensorMap* map, int x, int y,
                                            unsigned bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<unsigned long long>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(unsigned addr, float (&v)[16]) {
  unsigned r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(addr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// Column statistics of A for the whitening, a launch of its own before the tensor-core B V
// (whose programmatic dependent it is).  CTA t takes landmark column t of the (head, landmark)
// list, the row A^T[t][0..N); its 8 warps stream 8 contiguous segments of the row, up to 16
// independent 16-byte loads per lane in flight.  Every segment is shifted by the row's first
// value c, so the partial sums S1 = Sum (a - c) and S2 = Sum (a - c)^2 simply add (warp sums,
// then the 8 warps in a fixed order); mean = c + S1 / N and var = (S2 - S1^2 / N) / N.  c is a
// value of the row, so the subtraction keeps fp32 accuracy.
constexpr int kStatThreads = 256;

__device__ __forceinline__ float warp_allsum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(kStatThreads)
col_stats_kernel(const float* __restrict__ at, float* __restrict__ mu, float* __restrict__ rstd,
                 float* __restrict__ dbg_mu, float* __restrict__ dbg_rstd, int n, float delta) {
  // The B V kernel after this one may start now (it does not read these results).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float part[2][kStatThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long t = blockIdx.x;
  const float* row = at + (size_t)t * n;
  const float c = __ldcg(row);
  float s1 = 0.f, s2 = 0.f;
  constexpr int kW = kStatThreads / 32;
  if ((n & 3) == 0) {
    constexpr int kB = 16;
    const float4* r4 = reinterpret_cast<const float4*>(row);
    const int n4 = n >> 2;
    const int per = (n4 + kW - 1) / kW;                 // float4 per warp segment
    const int beg = warp * per, end = min(n4, beg + per);
    for (int i0 = beg + lane; i0 < end; i0 += 32 * kB) {
      float4 v[kB];
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const int i = i0 + 32 * u;
        v[u] = i < end ? __ldcg(&r4[i]) : make_float4(c, c, c, c);
      }
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const float a = v[u].x - c, b = v[u].y - c, e = v[u].z - c, f = v[u].w - c;
        s1 += (a + b) + (e + f);
        s2 += (a * a + b * b) + (e * e + f * f);
      }
    }
  } else {
    for (int i = threadIdx.x; i < n; i += kStatThreads) {
      const float a = __ldcg(&row[i]) - c;
      s1 += a;
      s2 = fmaf(a, a, s2);
    }
  }
  s1 = warp_allsum(s1);
  s2 = warp_allsum(s2);
  if (lane == 0) {
    part[0][warp] = s1;
    part[1][warp] = s2;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float a1 = 0.f, a2 = 0.f;
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      a1 += part[0][w];
      a2 += part[1][w];
    }
    const float inv_n = 1.f / (float)n;
    const float mean = c + a1 * inv_n;
    const float m2 = fmaxf(a2 - a1 * a1 * inv_n, 0.f);
    const float rs = 1.f / sqrtf(m2 * inv_n + delta);
    mu[t] = mean;
    rstd[t] = rs;
    if (dbg_mu) dbg_mu[t] = mean;
    if (dbg_rstd) dbg_rstd[t] = rs;
  }
}

struct BvTcArgs {
  float* bvp;           // [BH, splits, m, d]
  unsigned* err;
  int m, d, n;
  int tiles_per_split, splits;
  int nraw;             // raw stages (<= kRawMax)
  unsigned long long wait_ns;   // bound of every barrier wait
  int skip_last;        // fault injection: the copy warp never copies a CTA's last tile
};

template <bool kBf16>
__global__ void __launch_bounds__(kBvTcThreads, 1)
bv_tc_kernel(const BvTcArgs a, const __grid_constant__ CUtensorMap map_bt,
             const __grid_constant__ CUtensorMap map_v) {
  // A kernel launched as this grid's programmatic dependent (the conjugate-gradient solver)
  // may start its own preparation now; it waits for this grid before it reads any result.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ __align__(128) unsigned char smem_bv[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = a.m, d = a.d, n = a.n;
  const int nb = kBf16 ? d : 2 * d;                     // B operand rows = MMA N
  const unsigned raw_bytes = raw_stage_bytes(d, kBf16);
  const unsigned op_bytes = op_stage_bytes(nb);
  const unsigned lboB = lbo_b(nb);
  const int kRaw = a.nraw;
  unsigned char* raw = smem_bv;                                        // kRaw raw stages
  unsigned char* ops = raw + kRaw * raw_bytes;                         // kOps operand stages
  unsigned long long* bars = reinterpret_cast<unsigned long long*>(ops + kOps * op_bytes);
  const unsigned rfull0 = smem_u32(bars), rempty0 = rfull0 + 8 * kRawMax,
                 ofull0 = rempty0 + 8 * kRawMax, oempty0 = ofull0 + 8 * kOps,
                 done_bar = oempty0 + 8 * kOps;
  unsigned* slot = reinterpret_cast<unsigned*>(bars + 2 * kRawMax + 2 * kOps + 1);

  const long bh = blockIdx.x / a.splits;
  const int sp = blockIdx.x % a.splits;
  const int tiles_total = (n + kTok - 1) / kTok;
  const int t_begin = sp * a.tiles_per_split;
  const int t_end = min(tiles_total, t_begin + a.tiles_per_split);
  const int ntiles = max(0, t_end - t_begin);
  const unsigned tmem_cols = nb <= 32 ? 32u : nb <= 64 ? 64u : nb <= 128 ? 128u : 256u;

  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(slot)),
                 "r"(tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRaw; ++s) {
      mbar_init(rfull0 + 8 * s, 1);
      mbar_init(rempty0 + 8 * s, kConvThreads / 32);
    }
    for (int s = 0; s < kOps; ++s) {
      mbar_init(ofull0 + 8 * s, kConvThreads / 32);
      mbar_init(oempty0 + 8 * s, 1);
    }
    mbar_init(done_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // Zero the operand stages once: the padding rows of A (landmarks m..63) are never written
  // again.
  for (unsigned i = threadIdx.x; i < kOps * op_bytes / 16; i += kBvTcThreads)
    reinterpret_cast<float4*>(ops)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const unsigned tmem = *slot;
  bool ok = true;

  if (warp == kTmaWarp) {
    // ---------------- copies ----------------
    if (lane == 0) {
      const unsigned bytes = (unsigned)m * kTok * 4 + raw_v_bytes(d, kBf16);
      int issued = 0;
      for (int i = 0; i < ntiles; ++i) {
        const int s = i % kRaw;
        if (i >= kRaw && !mbar_wait(rempty0 + 8 * s, ((i / kRaw) - 1) & 1, a.wait_ns)) {
          ok = false;
          break;
        }
        if (a.skip_last && i == ntiles - 1) break;   // fault injection: never copied
        const int n0 = (t_begin + i) * kTok;
        const unsigned dst = smem_u32(raw + s * raw_bytes);
        mbar_expect_tx(rfull0 + 8 * s, bytes);
        tma_load_2d(dst, &map_bt, n0, (int)(bh * m), rfull0 + 8 * s);
        tma_load_2d(dst + kRawBt, &map_v, 0, (int)(bh * n + n0), rfull0 + 8 * s);
        issued = i + 1;
      }
      // Every issued copy lands before the CTA may finish.
      for (int i = max(0, issued - kRaw); i < issued; ++i)
        mbar_wait(rfull0 + 8 * (i % kRaw), (i / kRaw) & 1, a.wait_ns);
    }
  } else if (warp < kConvThreads / 32) {
    // ---------------- converters ----------------
    const int tid = threadIdx.x;
    const int cq = d >> 2;
    for (int i = 0; i < ntiles; ++i) {
      const int rs = i % kRaw, os = i % kOps;
      bool w = mbar_wait(rfull0 + 8 * rs, (i / kRaw) & 1, a.wait_ns);
      if (w && i >= kOps) w = mbar_wait(oempty0 + 8 * os, ((i / kOps) - 1) & 1, a.wait_ns);
      // The whole warp takes the same branch (a lane-by-lane exit would strand the others at
      // the warp barrier below).
      if (!__all_sync(0xffffffffu, w)) {
        ok = false;
        break;
      }
      const float* rbt = reinterpret_cast<const float*>(raw + rs * raw_bytes);
      const unsigned char* rv = raw + rs * raw_bytes + kRawBt;
      unsigned char* opa = ops + os * op_bytes;
      unsigned char* opb = opa + kOpABytes;
      // A: (landmark j, token quad q); a quarter-warp covers one landmark row.  All of a
      // thread's loads are issued before any is converted.
      constexpr int kAItems = 64 * (kTok / 4) / kConvThreads;
      float4 av[kAItems];
#pragma unroll
      for (int k = 0; k < kAItems; ++k) {
        const int e = tid + k * kConvThreads, j = e >> 3, q = e & 7;
        av[k] = j < m ? *reinterpret_cast<const float4*>(&rbt[j * kTok + 4 * q])
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < kAItems; ++k) {
        const int e = tid + k * kConvThreads, j = e >> 3, q = e & 7;
        if (j < m) {
          const float4 v = av[k];
          const float4 hi =
              make_float4(tf32_rna(v.x), tf32_rna(v.y), tf32_rna(v.z), tf32_rna(v.w));
          const float4 lo = make_float4(v.x - hi.x, v.y - hi.y, v.z - hi.z, v.w - hi.w);
          unsigned char* p = opa + q * kLboA + (j & 7) * 16;
          *reinterpret_cast<float4*>(p + (j >> 3) * kSboA) = hi;
          *reinterpret_cast<float4*>(p + ((64 + j) >> 3) * kSboA) = lo;
        }
      }
      // B: (token quad q, column quad c4); a quarter-warp covers consecutive column quads.
      for (int e = tid; e < (kTok / 4) * cq; e += kConvThreads) {
        const int q = e / cq, c4 = e % cq;
        float x[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int t = 4 * q + u;
          if constexpr (kBf16) {
            const uint2 r = *reinterpret_cast<const uint2*>(rv + (t * d + 4 * c4) * 2);
            x[u][0] = bf16_lo(r.x); x[u][1] = bf16_hi(r.x);
            x[u][2] = bf16_lo(r.y); x[u][3] = bf16_hi(r.y);
          } else {
            const float4 r = *reinterpret_cast<const float4*>(rv + (t * d + 4 * c4) * 4);
            x[u][0] = r.x; x[u][1] = r.y; x[u][2] = r.z; x[u][3] = r.w;
          }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float4 col = make_float4(x[0][c], x[1][c], x[2][c], x[3][c]);
          const int row = 4 * c4 + c;
          unsigned char* p = opb + q * lboB;
          if constexpr (kBf16) {
            *reinterpret_cast<float4*>(p + (row >> 3) * kSboB + (row & 7) * 16) = col;
          } else {
            const float4 hi = make_float4(tf32_rna(col.x), tf32_rna(col.y), tf32_rna(col.z),
                                          tf32_rna(col.w));
            const int lrow = d + row;
            *reinterpret_cast<float4*>(p + (row >> 3) * kSboB + (row & 7) * 16) = hi;
            *reinterpret_cast<float4*>(p + (lrow >> 3) * kSboB + (lrow & 7) * 16) =
                make_float4(col.x - hi.x, col.y - hi.y, col.z - hi.z, col.w - hi.w);
          }
        }
      }
      // Generic-proxy stores -> visible to the tensor core (async proxy).
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(ofull0 + 8 * os);
        mbar_arrive(rempty0 + 8 * rs);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issue ----------------
    if (lane == 0) {
      const uint32_t id = idesc((unsigned)nb);
      for (int i = 0; i < ntiles; ++i) {
        const int os = i % kOps;
        if (!mbar_wait(ofull0 + 8 * os, (i / kOps) & 1, a.wait_ns)) {
          ok = false;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const unsigned sa = smem_u32(ops + os * op_bytes), sb = sa + kOpABytes;
#pragma unroll
        for (int kk = 0; kk < kTok / 8; ++kk) {
          const uint64_t ad = op_desc(sa + kk * 2 * kLboA, kLboA, kSboA);
          const uint64_t bd = op_desc(sb + kk * 2 * lboB, lboB, kSboB);
          const unsigned acc = (i > 0 || kk > 0) ? 1u : 0u;
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
              "l"(ad), "l"(bd), "r"(id), "r"(acc)
              : "memory");
        }
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                oempty0 + 8 * os)
            : "memory");
      }
      // Everything issued so far completes before `done`.
      asm volatile(
          "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
              done_bar)
          : "memory");
    }
  }

  // ---------------- accumulator -> partial B V ----------------
  // Agree on failures first: a timed-out copy, converter or issuer leaves `done` unreached.
  ok = __syncthreads_and(ok ? 1 : 0) != 0;
  bool done = ok && (ntiles == 0 || mbar_wait(done_bar, 0, a.wait_ns));
  done = __syncthreads_and(done ? 1 : 0) != 0;
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  // [64][d + 4]: rows padded by 16 bytes so that the lanes' row-wise accesses spread over the
  // banks (unpadded, every lane of a warp hit the same bank); every copy has been consumed.
  float* xchg = reinterpret_cast<float*>(raw);
  const int xs = d + 4;
  float* dst = a.bvp + ((size_t)bh * a.splits + sp) * m * d;
  if (done && warp < 4) {
    const int r = 32 * warp + lane;                // accumulator row = tensor-memory lane
    const unsigned row_addr = tmem + ((unsigned)(32 * warp) << 16);
    // Rows 64..127 (low parts of B) hand their B_lo V_hi columns to rows 0..63.
    if (warp >= 2 && ntiles > 0) {
      for (int c0 = 0; c0 < d; c0 += 16) {
        float v[16];
        tmem_ld16(row_addr + c0, v);
#pragma unroll
        for (int c = 0; c < 16; c += 4)
          *reinterpret_cast<float4*>(&xchg[(r - 64) * xs + c0 + c]) =
              make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
      }
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (warp < 2 && ntiles == 0) {
      if (r < m)
        for (int c = 0; c < d; c += 4)      // no tokens in this split: a zero partial
          *reinterpret_cast<float4*>(&dst[(size_t)r * d + c]) = make_float4(0.f, 0.f, 0.f, 0.f);
    } else if (warp < 2) {
      // tcgen05.ld is warp-collective: every lane loads, only rows r < m are stored.
      for (int c0 = 0; c0 < d; c0 += 16) {
        float v[16];
        tmem_ld16(row_addr + c0, v);
        if constexpr (!kBf16) {
          float w[16];
          tmem_ld16(row_addr + d + c0, w);
#pragma unroll
          for (int c = 0; c < 16; ++c) v[c] += w[c];
        }
        if (r < m) {
#pragma unroll
          for (int c = 0; c < 16; c += 4)
            *reinterpret_cast<float4*>(&dst[(size_t)r * d + c0 + c]) = make_float4(
                v[c] + xchg[r * xs + c0 + c], v[c + 1] + xchg[r * xs + c0 + c + 1],
                v[c + 2] + xchg[r * xs + c0 + c + 2], v[c + 3] + xchg[r * xs + c0 + c + 3]);
        }
      }
    }
  } else if (!done && threadIdx.x == 0) {
    atomicOr(a.err, kErrBitChain);
    // Wait (bounded) for whatever the tensor core may still be doing before the memory goes.
    mbar_wait(done_bar, 0, a.wait_ns);
  }
  // Launched as a programmatic dependent of the column-statistics kernel, which it does not
  // read: this grid completes only after that one has, so whatever waits for B V also finds
  // the statistics complete.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(tmem_cols)
                 : "memory");
  }
}

}  // namespace

cudaError_t launch_col_stats(const lapl_attn_plan& p, const float* at, float* mu, float* rstd,
                             float* dbg_mu, float* dbg_rstd, cudaStream_t st) {
  const Geometry& g = p.geo;
  const unsigned grid = (unsigned)(g.bh * g.m);     // one CTA per (head, landmark) column
  col_stats_kernel<<<grid, kStatThreads, 0, st>>>(at, mu, rstd, dbg_mu, dbg_rstd, g.n,
                                                   p.cfg.delta);
  return cudaGetLastError();
}

int bv_tc_threads() { return kBvTcThreads; }
int bv_tc_tile_tokens() { return kTok; }

// Raw stages that fit next to the operand stages in `smem_limit` bytes (0 if fewer than 4).
int bv_tc_raw_stages(int d, bool bf16, size_t smem_limit) {
  const int nb = bf16 ? d : 2 * d;
  const size_t fixed = (size_t)kOps * op_stage_bytes(nb) + (2 * kRawMax + 2 * kOps + 1) * 8 + 16;
  if (smem_limit <= fixed) return 0;
  const int n = (int)std::min<size_t>(kRawMax, (smem_limit - fixed) / raw_stage_bytes(d, bf16));
  return n >= 4 ? n : 0;
}

size_t bv_tc_smem_bytes(int d, bool bf16, int nraw) {
  const int nb = bf16 ? d : 2 * d;
  const size_t body = (size_t)nraw * raw_stage_bytes(d, bf16) + (size_t)kOps * op_stage_bytes(nb);
  return body + (2 * kRawMax + 2 * kOps + 1) * 8 + 16;
}

cudaError_t bv_tc_configure(size_t smem) {
  cudaError_t e = cudaFuncSetAttribute(bv_tc_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(bv_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem);
}

int bv_tc_occupancy(size_t smem, bool bf16) {
  int occ = 0;
  const cudaError_t e = bf16 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                   &occ, bv_tc_kernel<true>, kBvTcThreads, smem)
                             : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                   &occ, bv_tc_kernel<false>, kBvTcThreads, smem);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  return occ > 0 ? occ : 1;
}

cudaError_t launch_bv_tc(const lapl_attn_plan& p, const float* bt, const void* v, float* bvp,
                         cudaStream_t st, bool pdl) {
  const Geometry& g = p.geo;
  const bool bf16 = p.cfg.in_dtype == LAPL_BF16;
  // B^T viewed as [BH m, N] fp32, boxes of 32 tokens x m rows; V as [BH N, d], boxes of d x 32.
  if (p.tmap_bt_ptr != bt) {
    if (!tma_encode_2d(&p.tmap_bt, bt, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (uint64_t)g.n,
                       (uint64_t)g.bh * g.m, (uint64_t)g.n * 4, kTok, (uint32_t)g.m))
      return cudaErrorInvalidValue;
    p.tmap_bt_ptr = bt;
  }
  if (p.tmap_v_ptr != v) {
    if (!tma_encode_2d(&p.tmap_v, v,
                       bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                       (uint64_t)g.d, (uint64_t)g.bh * g.n, (uint64_t)g.d * (bf16 ? 2 : 4),
                       (uint32_t)g.d, kTok))
      return cudaErrorInvalidValue;
    p.tmap_v_ptr = v;
  }
  BvTcArgs a;
  a.bvp = bvp; a.err = p.dev_err;
  a.m = g.m; a.d = g.d; a.n = g.n;
  a.tiles_per_split = g.bv_tiles_per_split; a.splits = g.bv_splits;
  a.nraw = g.bv_raw_stages;
  a.wait_ns = p.cd_wait_ns;
  a.skip_last = p.cd_skip_last_copy == 3 ? 1 : 0;
  const void* f = bf16 ? reinterpret_cast<const void*>(&bv_tc_kernel<true>)
                       : reinterpret_cast<const void*>(&bv_tc_kernel<false>);
  void* args[] = {&a, &p.tmap_bt, &p.tmap_v};
  // A programmatic dependent of the statistics launch before it when that one precedes it on
  // the stream (see the kernel's end); a plain launch when the statistics run beside it.
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)(g.bh * g.bv_splits));
  cfg.blockDim = dim3(kBvTcThreads);
  cfg.dynamicSmemBytes = g.bv_smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, f, args);
}

}  // namespace lapl
