// ns_tc.cu -- Newton-Schulz inverse of W with the products on the tensor cores (tcgen05, TF32
// operands split into an exact high/low pair, fp32 accumulation in tensor memory).
//
// "LaplacianFormer: Rethinking Linear Attention with Laplacian Kernel", English explainer page,
// 2.C.2 (German page, 2; Korean page, 2.3): X <- X (2I - W X) from X0 = W^T / (|W|_1 |W|_inf),
// exactly T steps; W = k(L, L) + eps I.  Same iterate as the CUDA-core kernels of ns.cu, with
// the products evaluated differently.
//
// One CTA (16 warps) per (batch, head).  The m x m matrices are zero-padded to 64 x 64.  A
// product C = A B is one accumulation of ceil(m / 8) tcgen05.mma instructions, M = N = 128,
// K = 8 each, into 128 columns of tensor memory:
//     D = [A_hi; A_lo] [Bt_hi; Bt_lo]^T
// with Bt = B^T stored K-major, a_hi = tf32(a) rounded to nearest and a_lo = tf32(a - a_hi).
// The four 64 x 64 blocks of D are the four cross products, so
//     C = D[0:64, 0:64] + D[0:64, 64:128] + D[64:128, 0:64] + D[64:128, 64:128]
// reproduces the fp32 operands to about 2^-22 relative.
//
// Both products take A = X.  The first forms P^T = X W, which equals (W X)^T because X and W
// are exactly symmetric; its rows are the K-major rows of the second product's Bt, so
// Q = X P needs no transpose.  The epilogues write whole operand rows (contiguous 16-byte
// pieces).  As in the CUDA-core kernel, X_{t+1} = (V + V^T) / 2 with V = 2X - Q, exactly
// symmetric (the first product relies on X^T == X), and averaging drops the antisymmetric part
// of V's rounding error instead of doubling it into the slow modes.
//
// Operands live in shared memory in the tensor cores' K-major layout without swizzle: core
// matrices of 8 rows x 16 bytes (8 x 4 TF32), cores adjacent in K kLbo bytes apart, adjacent in
// rows 128 bytes apart.  Completion of each product is signalled on an mbarrier; every wait is
// bounded (one second of %globaltimer), and on a timeout the CTA sets the device error word,
// waits once more (also bounded) for the tensor core, frees its tensor memory and returns.
#include "ns_common.cuh"

namespace lapl {
using namespace ns_detail;
namespace {

constexpr int kTcThreads = 512;
constexpr unsigned kLbo = 16 * 128;            // bytes between K-adjacent core matrices
constexpr unsigned kSbo = 128;                 // bytes between row-adjacent core matrices
constexpr unsigned kOpBytes = 128 * 64 * 4;    // one 128 x 64 TF32 operand
constexpr unsigned kTmemCols = 128;
constexpr unsigned long long kWaitNs = 1000000000ull;
constexpr unsigned kErrTimeout = kErrBitSolve;

// Offsets (bytes) in dynamic shared memory.
constexpr unsigned kOffWW = 0;                         // [W_hi; W_lo]      (Bt of P^T = X W)
constexpr unsigned kOffXX = kOffWW + kOpBytes;         // [X_hi; X_lo]      (A of both)
constexpr unsigned kOffPP = kOffXX + kOpBytes;         // [Pt_hi; Pt_lo]    (Bt of Q = X P)
constexpr unsigned kOffXf = kOffPP + kOpBytes;         // X fp32 [64][kMS]
constexpr unsigned kOffSc = kOffXf + 64 * kMS * 4;     // W fp32 in the prologue, then the
                                                       // exchange of the low-row partials
constexpr unsigned kOffRed = kOffSc + 64 * kMS * 4;    // column sums [kRedFloats]
constexpr unsigned kOffBar = kOffRed + kRedFloats * 4; // mbarrier (8-byte aligned)
constexpr unsigned kOffSlot = kOffBar + 8;             // tensor-memory address
constexpr unsigned kOffL = kOffSlot + 8;               // landmarks, channel-major [d][64]

__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

// Byte offset of element (r, k) of a 128-row K-major operand.
__device__ __forceinline__ unsigned op_off(int r, int k) {
  return (unsigned)((k >> 2) * kLbo + (r >> 3) * kSbo + (r & 7) * 16 + (k & 3) * 4);
}

// Round to the nearest TF32 value (10 explicit mantissa bits), ties away from zero: add half
// of the dropped 13 bits' range to the sign-magnitude pattern and clear them (a carry moves
// into the exponent exactly when rounding up crosses a binade).  Finite inputs only.
__device__ __forceinline__ float tf32_rna(float x) {
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}

// Store 4 consecutive k of operand row r (r < 64) as high part (row r) and low part (r + 64).
__device__ __forceinline__ void store_split(unsigned char* op, int r, int k0, float4 v) {
  const float4 hi = make_float4(tf32_rna(v.x), tf32_rna(v.y), tf32_rna(v.z), tf32_rna(v.w));
  const float4 lo = make_float4(tf32_rna(v.x - hi.x), tf32_rna(v.y - hi.y), tf32_rna(v.z - hi.z),
                                tf32_rna(v.w - hi.w));
  *reinterpret_cast<float4*>(op + op_off(r, k0)) = hi;
  *reinterpret_cast<float4*>(op + op_off(r + 64, k0)) = lo;
}

// Shared-memory matrix descriptor: K-major, no swizzle, descriptor version 1.
__device__ __forceinline__ uint64_t op_desc(unsigned addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)((kLbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((kSbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// Instruction descriptor: D fp32, A and B TF32, both K-major, N = 128, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (2u << 7) | (2u << 10) | ((128u >> 3) << 17) |
                            ((128u >> 4) << 24);

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void proxy_fence() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// D (tensor memory) = A Bt^T over ksteps x 8 columns of K, then arrive on bar when done.
__device__ __forceinline__ void issue_product(unsigned tmem, unsigned a_base, unsigned b_base,
                                              int ksteps, unsigned bar) {
  for (int kk = 0; kk < ksteps; ++kk) {
    const uint64_t ad = op_desc(a_base + kk * 2 * kLbo);
    const uint64_t bd = op_desc(b_base + kk * 2 * kLbo);
    const unsigned acc = kk > 0 ? 1u : 0u;
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem),
        "l"(ad), "l"(bd), "r"(kIdesc), "r"(acc)
        : "memory");
  }
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                   bar)
               : "memory");
}

__device__ __forceinline__ bool mbar_try(unsigned bar, unsigned parity) {
  unsigned done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
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

// Bounded wait of every thread for the given phase; the CTA agrees on the outcome.
__device__ __forceinline__ bool wait_product(unsigned bar, unsigned parity) {
  bool ok = mbar_try(bar, parity);
  if (!ok) {
    const unsigned long long t0 = global_ns();
    while (!(ok = mbar_try(bar, parity)))
      if (global_ns() - t0 > kWaitNs) break;
  }
  return __syncthreads_and(ok ? 1 : 0) != 0;
}

// 16 consecutive fp32 columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_ld16(unsigned addr, float (&v)[16]) {
  unsigned r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(addr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// Two 16-column loads, one wait: both round trips to tensor memory overlap.
__device__ __forceinline__ void tmem_ld16x2(unsigned addr_a, unsigned addr_b, float (&a)[16],
                                            float (&b)[16]) {
  unsigned r[16], q[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(addr_a));
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];\n"
      : "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3]), "=r"(q[4]), "=r"(q[5]), "=r"(q[6]),
        "=r"(q[7]), "=r"(q[8]), "=r"(q[9]), "=r"(q[10]), "=r"(q[11]), "=r"(q[12]), "=r"(q[13]),
        "=r"(q[14]), "=r"(q[15])
      : "r"(addr_b));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    a[j] = __uint_as_float(r[j]);
    b[j] = __uint_as_float(q[j]);
  }
}

// C = sum of the four blocks of D, 8 columns of one row per thread.  Warp w reads tensor-memory
// lanes 32(w % 4).. (D rows dr) and columns 16h.. and 64 + 16h.. (h = w / 4); D rows dr and
// dr + 64 hold the A_hi and A_lo parts of C row i = dr % 64.  The A_hi thread keeps columns
// 16h..16h+7 and the A_lo thread 16h+8..16h+15; each hands the other half of its sums to the
// other through sc.  On return c holds C[i][col0 .. col0+7].
__device__ __forceinline__ void combine_product(unsigned tmem, float* sc, float (&c)[8], int& i,
                                                int& col0) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sp = warp & 3, h = warp >> 2;
  const int dr = 32 * sp + lane;
  i = dr & 63;
  const bool low = dr >= 64;
  const unsigned lane_base = (unsigned)(32 * sp) << 16;
  float a[16], v[16];
  tmem_ld16x2(tmem + lane_base + 16 * h, tmem + lane_base + 64 + 16 * h, a, v);
#pragma unroll
  for (int j = 0; j < 16; ++j) a[j] += v[j];
  // kept half: a[8..15] for the low thread, a[0..7] for the high one (selects, so that a stays
  // in registers)
  float kept[8], given[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    kept[j] = low ? a[8 + j] : a[j];
    given[j] = low ? a[j] : a[8 + j];
  }
  col0 = 16 * h + (low ? 8 : 0);
  const int give0 = 16 * h + (low ? 0 : 8);
#pragma unroll
  for (int j = 0; j < 8; j += 4)
    *reinterpret_cast<float4*>(&sc[i * kMS + give0 + j]) =
        make_float4(given[j], given[j + 1], given[j + 2], given[j + 3]);
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 8; j += 4) {
    const float4 o = *reinterpret_cast<const float4*>(&sc[i * kMS + col0 + j]);
    c[j] = kept[j] + o.x;
    c[j + 1] = kept[j + 1] + o.y;
    c[j + 2] = kept[j + 2] + o.z;
    c[j + 3] = kept[j + 3] + o.w;
  }
}

template <int S>
__global__ void __launch_bounds__(kTcThreads, 1)
ns_tc_kernel(const float* __restrict__ landmarks, float* __restrict__ xout,
             float* __restrict__ dbg_dll, float* __restrict__ dbg_w, float* __restrict__ dbg_x,
             float* __restrict__ xs, int d, int T, float eps, float c_exp, int gauss,
             unsigned* __restrict__ err) {
  using Sh = NsShape<S>;
  constexpr int M = Sh::M;
  constexpr int KSTEPS = (Sh::MK + 7) / 8;
  extern __shared__ __align__(1024) unsigned char smem_tc[];
  unsigned char* WW = smem_tc + kOffWW;
  unsigned char* XX = smem_tc + kOffXX;
  unsigned char* PP = smem_tc + kOffPP;
  float* Xf = reinterpret_cast<float*>(smem_tc + kOffXf);
  float* sc = reinterpret_cast<float*>(smem_tc + kOffSc);
  unsigned long long* bar = reinterpret_cast<unsigned long long*>(smem_tc + kOffBar);
  unsigned* slot = reinterpret_cast<unsigned*>(smem_tc + kOffSlot);
  const int warp = threadIdx.x >> 5;
  const long bh = blockIdx.x;
  // The M kernel after this one reduces the B V partials before it waits for this grid.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     smem_u32(slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  if (threadIdx.x == 32) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }

  // Launched as a programmatic dependent of the pooling kernel: L is complete past this wait.
  asm volatile("griddepcontrol.wait;\n" ::: "memory");

  // W (into sc) and X0 (into Xf), fp32, row stride kMS.
  NsSmem sm;
  sm.W = sc;
  sm.X = Xf;
  sm.P = nullptr;
  sm.Y = nullptr;
  sm.red = reinterpret_cast<float*>(smem_tc + kOffRed);
  sm.part = nullptr;
  sm.sL = reinterpret_cast<float*>(smem_tc + kOffL);
  ns_prologue<S, kTcThreads>(sm, landmarks + (size_t)bh * M * d, d, eps, c_exp, gauss != 0, true,
                             dbg_dll, dbg_w, bh);

  // Operands W and X0 as TF32 high/low pairs.  A warp takes 32 consecutive rows of one
  // 4-column piece: its 16-byte stores are contiguous in the operand layout.
  for (int g = threadIdx.x; g < 64 * 16; g += kTcThreads) {
    const int r = g & 63, k0 = (g >> 6) * 4;
    store_split(WW, r, k0, *reinterpret_cast<const float4*>(&sc[r * kMS + k0]));
    store_split(XX, r, k0, *reinterpret_cast<const float4*>(&Xf[r * kMS + k0]));
  }
  proxy_fence();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const unsigned tmem = *slot;
  const unsigned bar_a = smem_u32(bar);
  const unsigned xx_a = smem_u32(XX), ww_a = smem_u32(WW), pp_a = smem_u32(PP);

  unsigned phase = 0;
  bool ok = true;
  float* xsh = xs ? xs + (size_t)bh * (T + 1) * M * Sh::MK : nullptr;
  for (int t = 0; t < T && ok; ++t) {
    // ---- P^T = X W ----
    if (threadIdx.x == 0) issue_product(tmem, xx_a, ww_a, KSTEPS, bar_a);
    // X_t is kept for the backward pass while the tensor cores work (they read XX, not Xf).
    save_iterate<M, kTcThreads>(Xf, xsh ? xsh + (size_t)t * M * Sh::MK : nullptr);
    ok = wait_product(bar_a, phase);
    phase ^= 1;
    if (!ok) break;
    tc_fence_after();
    {
      float c[8];
      int i, col0;
      combine_product(tmem, sc, c, i, col0);
#pragma unroll
      for (int j = 0; j < 8; j += 4)
        store_split(PP, i, col0 + j, make_float4(c[j], c[j + 1], c[j + 2], c[j + 3]));
    }
    proxy_fence();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- Q = X P;  V = 2X - Q;  X <- (V + V^T) / 2, exactly symmetric ----
    if (threadIdx.x == 0) issue_product(tmem, xx_a, pp_a, KSTEPS, bar_a);
    ok = wait_product(bar_a, phase);
    phase ^= 1;
    if (!ok) break;
    tc_fence_after();
    float y[8];
    int i, col0;
    combine_product(tmem, sc, y, i, col0);
    // V into sc, at the entries this thread alone read in combine_product.
#pragma unroll
    for (int j = 0; j < 8; j += 4) {
      const float4 xo = *reinterpret_cast<const float4*>(&Xf[i * kMS + col0 + j]);
      y[j] = 2.f * xo.x - y[j];
      y[j + 1] = 2.f * xo.y - y[j + 1];
      y[j + 2] = 2.f * xo.z - y[j + 2];
      y[j + 3] = 2.f * xo.w - y[j + 3];
      *reinterpret_cast<float4*>(&sc[i * kMS + col0 + j]) =
          make_float4(y[j], y[j + 1], y[j + 2], y[j + 3]);
    }
    __syncthreads();
    // (i, col) and (col, i) add the same two values: the result is exactly symmetric.
#pragma unroll
    for (int j = 0; j < 8; ++j) y[j] = 0.5f * (y[j] + sc[(col0 + j) * kMS + i]);
#pragma unroll
    for (int j = 0; j < 8; j += 4)
      *reinterpret_cast<float4*>(&Xf[i * kMS + col0 + j]) =
          make_float4(y[j], y[j + 1], y[j + 2], y[j + 3]);
#pragma unroll
    for (int j = 0; j < 8; j += 4)
      store_split(XX, i, col0 + j, make_float4(y[j], y[j + 1], y[j + 2], y[j + 3]));
    proxy_fence();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  if (ok) save_iterate<M, kTcThreads>(Xf, xsh ? xsh + (size_t)T * M * Sh::MK : nullptr);

  if (!ok) {
    if (threadIdx.x == 0) atomicOr(err, kErrTimeout);
    wait_product(bar_a, phase ^ 1);      // let an unfinished product drain (bounded)
  } else {
    for (int idx = threadIdx.x; idx < M * M; idx += kTcThreads) {
      const int i = idx / M, k = idx % M;
      const float x = Xf[i * kMS + k];
      xout[(size_t)bh * M * M + idx] = x;
      if (dbg_x) dbg_x[(size_t)bh * M * M + idx] = x;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

template <int S>
const void* tc_ptr() { return reinterpret_cast<const void*>(&ns_tc_kernel<S>); }

const void* pick_tc(int s) {
  switch (s) {
    case 1: return tc_ptr<1>();
    case 2: return tc_ptr<2>();
    case 3: return tc_ptr<3>();
    case 4: return tc_ptr<4>();
    case 5: return tc_ptr<5>();
    case 6: return tc_ptr<6>();
    case 7: return tc_ptr<7>();
    case 8: return tc_ptr<8>();
    default: return nullptr;
  }
}

}  // namespace

size_t ns_tc_smem_bytes(int d) { return kOffL + sizeof(float) * 64 * (size_t)d; }

cudaError_t ns_tc_configure(int s, size_t smem) {
  const void* f = pick_tc(s);
  if (!f) return cudaErrorInvalidValue;
  return cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t launch_ns_tc(const lapl_attn_plan& p, const float* landmarks, float* x,
                         float* dbg_dll, float* dbg_w, float* dbg_x, float* xs, cudaStream_t st) {
  const Geometry& g = p.geo;
  const void* f = pick_tc(g.s);
  if (!f) return cudaErrorInvalidValue;
  int d = g.d, T = p.cfg.ns_steps;
  float eps = p.cfg.eps, c_exp = p.neg_log2e_over_lambda;
  unsigned* err = p.dev_err;
  int gauss = p.cfg.kernel == LAPL_KERNEL_GAUSSIAN;
  void* args[] = {&landmarks, &x, &dbg_dll, &dbg_w, &dbg_x, &xs, &d, &T, &eps, &c_exp, &gauss, &err};
  // When the solve follows the pooling kernel on the same stream (the solve has SMs of its
  // own), it is a programmatic dependent of it: its launch and set-up overlap the pooling.
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)g.bh);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = g.ns_smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = g.ns_exclusive ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, f, args);
}

}  // namespace lapl
