// cdist_gauss_tc.cu -- fused squared-l2 distance + exp for the Gaussian kernel, the cross term
// on the tensor cores (tcgen05, TF32 operands split into an exact high/low pair, fp32
// accumulation in tensor memory).
//
// The Gaussian kernel k(x, y) = exp(-|x - y|_2^2 / lambda) is the similarity of earlier linear
// attention that "LaplacianFormer: Rethinking Linear Attention with Laplacian Kernel" sets
// against its Laplacian kernel (English explainer page, 1 "Theoretical Mismatch"); A = k(Q, L)
// and B = k(L, K) are formed as for the Laplacian kernel (English page, 2.C), stored
// landmark-major.  Unlike |x - y|_1, the squared l2 distance expands into a dot product:
//   |x - l|^2 = |x|^2 + |l|^2 - 2 x.l,
// and x.l for a chunk of 128 tokens against every landmark of the head is the product
// [128 x d] [d x m], a dense contraction.  Per chunk the accumulator D (128 token rows =
// tensor-memory lanes, 2 np columns, np = m rounded up to 16) receives
//   D[:, 0:2np]  = X_hi [L_hi | L_lo]      (one MMA chain, N = 2 np)
//   D[:, 0:np]  += X_lo L_hi               (fp32 inputs only; bf16 inputs are exact in TF32)
// so x.l = D[t][j] + D[t][np + j] to about 2^-21 relative.  The epilogue forms
// max(|x|^2 + |l|^2 - 2 x.l, 0) and the exponential.  On small-integer inputs with dyadic
// landmarks every term is exact in fp32, so the distances equal the direct sum bit for bit.
//
// Persistent CTAs walk balanced ranges of (side, head, token) positions in chunks of up to 128
// tokens of one head (the Partition of the other distance kernels).  Warps:
//   0-3  converters: 16-byte loads of the chunk's rows (the next chunk's loads are in flight
//        while this one is converted), |x|^2 by a shuffle sum over the lanes that hold a row,
//        X_hi / X_lo stored in the K-major operand layout (core matrices of 8 rows x 16 bytes;
//        the K-direction stride padded by 16 bytes so a quarter-warp's stores, one row's
//        consecutive 16-byte pieces, fall in 8 bank groups); for a new head they also build
//        [L_hi; L_lo] and |l|^2 (two buffers, by head parity);
//   4-7  epilogue: read the accumulator (one token row per thread), form the distances and
//        kernel values, store them (a warp store is 32 consecutive tokens of one landmark row);
//        the values of 16 landmarks are formed without a branch before any is stored;
//   8    owns the tensor memory; one thread issues the MMAs.
// Two operand stages and two accumulators: the conversion of chunk i + 1 and the stores of
// chunk i - 1 overlap the MMAs of chunk i.  Every barrier wait is bounded (wait_ns); on a
// timeout the CTA sets the distance bit of the device error word, waits (bounded) for its
// tensor-core work and frees the tensor memory.
#include "common.cuh"

namespace lapl {
namespace {

constexpr int kTile = 128;
constexpr int kEpiWarp0 = 4, kMmaWarp = 8;
constexpr int kThreads = 32 * 9;
constexpr unsigned kSbo = 128;                  // stride between 8-row core groups
constexpr unsigned kLboA = 16 * kSbo + 16;      // X operand: 128 rows, padded

__host__ __device__ inline int np16(int m) { return m <= 16 ? 16 : (m + 15) & ~15; }
__host__ __device__ inline unsigned lbo_l(int np) { return (unsigned)(2 * np / 8) * kSbo + 16; }
__host__ __device__ inline unsigned align128(unsigned x) { return (x + 127u) & ~127u; }

__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ float tf32_rna(float x) {
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}
__device__ __forceinline__ uint64_t op_desc(unsigned addr, unsigned lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((kSbo >> 4) & 0x3FFFu) << 32;
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
// Waiting warps back off (a short sleep between polls): the converter, epilogue and MMA warps
// share the SM's four schedulers, and a hot polling loop takes issue slots from the warp that
// does the work.
__device__ __forceinline__ bool mbar_wait(unsigned bar, unsigned parity,
                                          unsigned long long bound) {
  if (mbar_test(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_test(bar, parity)) {
    __nanosleep(32);
    if (global_ns() - t0 > bound) return false;
  }
  return true;
}
__device__ __forceinline__ void commit(unsigned bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ void mma(unsigned tmem, uint64_t ad, uint64_t bd, uint32_t id,
                                    unsigned acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
      "l"(ad), "l"(bd), "r"(id), "r"(acc)
      : "memory");
}
// Two 16-column loads of this warp's 32 lanes, one wait.
__device__ __forceinline__ void tmem_ld16x2(unsigned addr_v, unsigned addr_w, float (&v)[16],
                                            float (&w)[16]) {
  unsigned r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%32];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,"
      "%28,%29,%30,%31}, [%33];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(addr_v), "r"(addr_w)
      : "memory");
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    v[j] = __uint_as_float(r[j]);
    w[j] = __uint_as_float(r[16 + j]);
  }
}
__device__ __forceinline__ float4 bf16x4_to_f32(unsigned lo, unsigned hi) {
  return make_float4(__uint_as_float(lo << 16), __uint_as_float(lo & 0xFFFF0000u),
                     __uint_as_float(hi << 16), __uint_as_float(hi & 0xFFFF0000u));
}

struct GaussTcArgs {
  const void* q;             // [BH, N, d] fp32 or bf16
  const void* k;
  const float* landmarks;    // [BH, m, d]
  float* at;                 // [BH, m, N]
  float* bt;                 // [BH, m, N]
  float* dbg_dql;            // optional [BH, N, m]
  float* dbg_dlk;            // optional [BH, m, N]
  float* dbg_a;              // optional [BH, N, m]
  unsigned* err;
  long long tiles;           // 2 * BH * tiles_per_head: (side, head, 128-token tile) units
  int tiles_per_head;
  long long bh_count;
  int n, m, np;
  int tma_store;             // 1: kernel values leave through TMA tensor stores (N % 4 == 0)
  float c_exp;
  unsigned long long wait_ns;
  int skip_last;             // fault injection: the converters never publish a CTA's last chunk
};

// Tile sequence of a CTA: the CTA takes units [tiles * c / ctas, tiles * (c + 1) / ctas) of the
// list (side, head, tile), query side first; a tile is 128 tokens of one head from a multiple of
// 128 (fewer at the end of a head).
struct TileIter {
  long long u, uend;
  int side;
  long long bh;
  int t, n0, valid;

  __device__ void init(long long tiles, int ctas, int cta, int tph, long long bh_count, int n) {
    u = tiles * cta / ctas;
    uend = tiles * (cta + 1) / ctas;
    if (u >= uend) return;
    const long long per_side = bh_count * tph;
    side = u >= per_side ? 1 : 0;
    const long long r = u - side * per_side;
    bh = r / tph;
    t = (int)(r % tph);
    n0 = t * kTile;
    valid = min(kTile, n - n0);
  }
  __device__ bool done() const { return u >= uend; }
  __device__ bool last() const { return u + 1 >= uend; }
  __device__ void next(int tph, long long bh_count, int n) {
    if (++u >= uend) return;
    if (++t == tph) {
      t = 0;
      if (++bh == bh_count) {
        bh = 0;
        side = 1;
      }
    }
    n0 = t * kTile;
    valid = min(kTile, n - n0);
  }
};

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];\n\t"
      "cp.async.bulk.commit_group;" ::"l"(reinterpret_cast<unsigned long long>(map)),
      "r"(x), "r"(y), "r"(smem_u32(src))
      : "memory");
}
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

template <bool kBf16, int DH>
struct GCfg {
  static constexpr int kPieces = kBf16 ? DH / 8 : DH / 4;     // 16-byte pieces per input row
  static constexpr int kItems = kPieces;                      // pieces per converter thread
  static constexpr int kRowsPerPass = 128 / kPieces;
  static constexpr unsigned kAPart = (DH / 4) * kLboA;        // one of X_hi, X_lo
  static constexpr unsigned kAStage = (kBf16 ? 1 : 2) * kAPart;
};

template <bool kBf16, int DH>
__global__ void __launch_bounds__(kThreads, DH == 32 ? 2 : 1)
    gauss_tc_kernel(const GaussTcArgs a, const __grid_constant__ CUtensorMap map_at,
                    const __grid_constant__ CUtensorMap map_bt) {
  using C = GCfg<kBf16, DH>;
  extern __shared__ __align__(128) unsigned char smem_g[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = a.m, n = a.n, np = a.np;
  const unsigned lboL = lbo_l(np);
  const unsigned lbytes = align128((DH / 4) * lboL);
  unsigned char* astage = smem_g;                                    // [2][X_hi (, X_lo)]
  unsigned char* lbuf = astage + 2 * C::kAStage;                     // [L_hi; L_lo]
  float* ostage = reinterpret_cast<float*>(lbuf + lbytes);           // [4 warps][m][32]
  float* nxs = ostage + align128(4u * m * 32 * 4) / 4;               // [2][128] |x|^2
  float* nls = nxs + 2 * kTile;                                      // [64]     |l|^2
  unsigned long long* bars = reinterpret_cast<unsigned long long*>(nls + 64);
  const unsigned ofull0 = smem_u32(bars), afull0 = ofull0 + 16, aempty0 = afull0 + 16,
                 done_bar = aempty0 + 16;
  unsigned* slot = reinterpret_cast<unsigned*>(bars + 7);
  // Accumulator s at column s * acc_stride (2 np rounded up to 32, 64 or 128).
  const unsigned acc_stride = np <= 16 ? 32u : np <= 32 ? 64u : 128u;
  const unsigned tmem_cols = 2 * acc_stride;
  const unsigned long long bound = a.wait_ns;

  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(slot)),
                 "r"(tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(ofull0 + 8 * s, 4);      // converter warps
      mbar_init(afull0 + 8 * s, 1);      // tensor-core commit
      mbar_init(aempty0 + 8 * s, 4);     // epilogue warps
    }
    mbar_init(done_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const unsigned tmem = *slot;
  bool ok = true;
  TileIter it;
  it.init(a.tiles, gridDim.x, blockIdx.x, a.tiles_per_head, a.bh_count, n);
  const int tph = a.tiles_per_head;

  if (warp < 4) {
    // ---------------- converters ----------------
    // Piece q = item * 128 + t of the chunk: row q / kPieces, 16-byte piece q % kPieces; the
    // lanes holding one row are kPieces consecutive lanes (kPieces divides 32).
    const int t = threadIdx.x;
    const int prow = t / C::kPieces, pc = t % C::kPieces;
    const char* qb = static_cast<const char*>(a.q);
    const char* kb = static_cast<const char*>(a.k);
    constexpr size_t kRowBytes = (size_t)DH * (kBf16 ? 2 : 4);
    uint4 nxt[C::kItems];
    auto load_chunk = [&](const TileIter& c, uint4 (&v)[C::kItems]) {
      const char* base = (c.side == 0 ? qb : kb) + ((size_t)c.bh * n + c.n0) * kRowBytes;
#pragma unroll
      for (int i = 0; i < C::kItems; ++i) {
        const int row = i * C::kRowsPerPass + prow;
        v[i] = make_uint4(0u, 0u, 0u, 0u);
        if (row < c.valid)
          v[i] = __ldcs(reinterpret_cast<const uint4*>(base + (size_t)row * kRowBytes) + pc);
      }
    };
    TileIter ld = it;
    if (!ld.done()) load_chunk(ld, nxt);
    long long prev_bh = -1;
    for (int i = 0; !it.done(); ++i) {
      const int s = i & 1;
      uint4 cur[C::kItems];
#pragma unroll
      for (int j = 0; j < C::kItems; ++j) cur[j] = nxt[j];
      ld.next(tph, a.bh_count, n);
      if (!ld.done()) load_chunk(ld, nxt);
      if (a.skip_last && it.last()) break;       // fault injection: never published
      // Stage s and |x|^2 slot s were last read by chunk i - 2, the landmark operand (for a new
      // head) by chunk i - 1: the epilogue of that chunk (after its MMAs) released them.
      const bool new_head = it.bh != prev_bh;
      const int wc = new_head ? i - 1 : i - 2;
      if (wc >= 0 && !__all_sync(0xffffffffu,
                                 mbar_wait(aempty0 + 8 * (wc & 1), (wc >> 1) & 1, bound))) {
        ok = false;
        break;
      }
      unsigned char* xhi = astage + s * C::kAStage;
      unsigned char* xlo = xhi + C::kAPart;
#pragma unroll
      for (int j = 0; j < C::kItems; ++j) {
        const int row = j * C::kRowsPerPass + prow;
        const unsigned ro = (row >> 3) * kSbo + (row & 7) * 16;
        float part;
        if constexpr (kBf16) {
          const float4 x0 = bf16x4_to_f32(cur[j].x, cur[j].y);
          const float4 x1 = bf16x4_to_f32(cur[j].z, cur[j].w);
          part = x0.x * x0.x;
          part = fmaf(x0.y, x0.y, part);
          part = fmaf(x0.z, x0.z, part);
          part = fmaf(x0.w, x0.w, part);
          part = fmaf(x1.x, x1.x, part);
          part = fmaf(x1.y, x1.y, part);
          part = fmaf(x1.z, x1.z, part);
          part = fmaf(x1.w, x1.w, part);
          // bf16 values are exact in TF32: no low part.
          *reinterpret_cast<float4*>(xhi + (2 * pc) * kLboA + ro) = x0;
          *reinterpret_cast<float4*>(xhi + (2 * pc + 1) * kLboA + ro) = x1;
        } else {
          const float4 x = make_float4(__uint_as_float(cur[j].x), __uint_as_float(cur[j].y),
                                       __uint_as_float(cur[j].z), __uint_as_float(cur[j].w));
          part = x.x * x.x;
          part = fmaf(x.y, x.y, part);
          part = fmaf(x.z, x.z, part);
          part = fmaf(x.w, x.w, part);
          const float4 hi = make_float4(tf32_rna(x.x), tf32_rna(x.y), tf32_rna(x.z), tf32_rna(x.w));
          *reinterpret_cast<float4*>(xhi + pc * kLboA + ro) = hi;
          *reinterpret_cast<float4*>(xlo + pc * kLboA + ro) =
              make_float4(x.x - hi.x, x.y - hi.y, x.z - hi.z, x.w - hi.w);
        }
#pragma unroll
        for (int o = 1; o < C::kPieces; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (pc == 0) nxs[s * kTile + row] = part;
      }
      if (new_head) {
        // [L_hi; L_lo] and |l|^2 of the new head: rows j < np hold L_hi (zero past m), rows
        // np + j hold L_lo.
        prev_bh = it.bh;
        unsigned char* lb = lbuf;
        float* nl = nls;
        const float* lg = a.landmarks + (size_t)it.bh * m * DH;
        // np * kQ is a multiple of 128 (np of 16, kQ >= 8): every pass is warp-uniform, as
        // the shuffles need.  The MMA waits for all four converter warps, so no barrier
        // between them is needed before the landmark operand is used.
        constexpr int kQ = DH / 4;                  // quads per landmark row
        for (int e = t; e < np * kQ; e += 128) {
          const int j = e / kQ, c = e % kQ;
          const float4 l = j < m ? *reinterpret_cast<const float4*>(lg + (size_t)j * DH + 4 * c)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
          float part = l.x * l.x;
          part = fmaf(l.y, l.y, part);
          part = fmaf(l.z, l.z, part);
          part = fmaf(l.w, l.w, part);
#pragma unroll
          for (int o = 1; o < kQ; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
          if (c == 0 && j < 64) nl[j] = part;
          const float4 hi = make_float4(tf32_rna(l.x), tf32_rna(l.y), tf32_rna(l.z), tf32_rna(l.w));
          const int lr = np + j;
          *reinterpret_cast<float4*>(lb + c * lboL + (j >> 3) * kSbo + (j & 7) * 16) = hi;
          *reinterpret_cast<float4*>(lb + c * lboL + (lr >> 3) * kSbo + (lr & 7) * 16) =
              make_float4(l.x - hi.x, l.y - hi.y, l.z - hi.z, l.w - hi.w);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(ofull0 + 8 * s);
      it.next(tph, a.bh_count, n);
    }
  } else if (warp < kMmaWarp) {
    // ---------------- epilogue ----------------
    const int ew = warp - kEpiWarp0;                   // tensor-memory lanes 32 ew ..
    const int r = 32 * ew + lane;                      // token row of the chunk
    const bool debug = a.dbg_dql || a.dbg_dlk || a.dbg_a;
    const bool tma_store = a.tma_store != 0;
    // This warp's 32 tokens of the chunk, landmark-major, for the tensor store: [m][32].
    float* stg = ostage + ew * m * 32;
    for (int i = 0; !it.done(); ++i) {
      const int b = i & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(afull0 + 8 * b, (i >> 1) & 1, bound))) {
        ok = false;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if (tma_store && i > 0) {
        if (lane == 0) bulk_wait_read();           // the last tensor store has read the slice
        __syncwarp();
      }
      const float xr = nxs[b * kTile + r];
      const float* nl = nls;
      const bool live = r < it.valid;
      float* dst = (it.side == 0 ? a.at : a.bt) + (size_t)it.bh * m * n + it.n0 + r;
      const unsigned row_addr = tmem + ((unsigned)(32 * ew) << 16) + b * acc_stride;
      // Per 16 landmarks: both accumulator halves in one wait, the 16 values without a branch
      // (independent chains the scheduler can interleave), then the stores; a branch around
      // each value's arithmetic would serialise the latency of every chain.
      auto values16 = [&](int c0, float (&v)[16], const float (&w)[16]) {
        const float4* nl4 = reinterpret_cast<const float4*>(nl + c0);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float4 l = nl4[q4];
          v[4 * q4 + 0] = fmaxf(fmaf(-2.f, v[4 * q4 + 0] + w[4 * q4 + 0], xr + l.x), 0.f);
          v[4 * q4 + 1] = fmaxf(fmaf(-2.f, v[4 * q4 + 1] + w[4 * q4 + 1], xr + l.y), 0.f);
          v[4 * q4 + 2] = fmaxf(fmaf(-2.f, v[4 * q4 + 2] + w[4 * q4 + 2], xr + l.z), 0.f);
          v[4 * q4 + 3] = fmaxf(fmaf(-2.f, v[4 * q4 + 3] + w[4 * q4 + 3], xr + l.w), 0.f);
        }
        float kv[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) kv[jj] = laplacian_from_distance(v[jj], a.c_exp);
        if (tma_store) {
          // Tokens past the head's end land in the slice and are clipped by the tensor store.
          float* s0 = stg + c0 * 32 + lane;
          if (c0 + 16 <= m) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) s0[jj * 32] = kv[jj];
          } else {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj)
              if (c0 + jj < m) s0[jj * 32] = kv[jj];
          }
        }
        if (live) {
          float* d0 = dst + (size_t)c0 * n;
          if (tma_store) {
          } else if (c0 + 16 <= m) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) d0[(size_t)jj * n] = kv[jj];
          } else {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj)
              if (c0 + jj < m) d0[(size_t)jj * n] = kv[jj];
          }
          if (debug) {
            const size_t tok = (size_t)it.bh * n + it.n0 + r;
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int j = c0 + jj;
              if (j >= m) continue;
              if (it.side == 0) {
                if (a.dbg_dql) a.dbg_dql[tok * m + j] = v[jj];
                if (a.dbg_a) a.dbg_a[tok * m + j] = kv[jj];
              } else if (a.dbg_dlk) {
                a.dbg_dlk[((size_t)it.bh * m + j) * n + it.n0 + r] = v[jj];
              }
            }
          }
        }
      };
      for (int c0 = 0; c0 < np; c0 += 16) {
        float v[16], w[16];
        tmem_ld16x2(row_addr + c0, row_addr + np + c0, v, w);
        values16(c0, v, w);
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      if (tma_store) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(aempty0 + 8 * b);
        // This warp's [m x 32] box at token n0 + 32 ew of landmark row bh m; x is a multiple
        // of 32 (128 bytes); a box past the head's end is clipped, one wholly past it skipped.
        const int x = it.n0 + 32 * ew;
        if (tma_store && x < n)
          tma_store_2d(it.side == 0 ? &map_at : &map_bt, stg, x, (int)(it.bh * m));
      }
      it.next(tph, a.bh_count, n);
    }
    if (lane == 0 && tma_store) bulk_wait_all();   // stores done before the CTA's memory goes
  } else {
    // ---------------- MMA issue ----------------
    if (lane == 0) {
      const uint32_t id2 = idesc((unsigned)(2 * np)), id1 = idesc((unsigned)np);
      for (int i = 0; !it.done(); ++i) {
        const int s = i & 1;
        if (!mbar_wait(ofull0 + 8 * s, (i >> 1) & 1, bound) ||
            (i >= 2 && !mbar_wait(aempty0 + 8 * s, ((i >> 1) - 1) & 1, bound))) {
          ok = false;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const unsigned xhi = smem_u32(astage + s * C::kAStage), xlo = xhi + C::kAPart;
        const unsigned lb = smem_u32(lbuf);
        const unsigned acc = tmem + s * acc_stride;
#pragma unroll
        for (int kk = 0; kk < DH / 8; ++kk)
          mma(acc, op_desc(xhi + kk * 2 * kLboA, kLboA), op_desc(lb + kk * 2 * lboL, lboL), id2,
              kk > 0 ? 1u : 0u);
        if constexpr (!kBf16) {
#pragma unroll
          for (int kk = 0; kk < DH / 8; ++kk)
            mma(acc, op_desc(xlo + kk * 2 * kLboA, kLboA), op_desc(lb + kk * 2 * lboL, lboL), id1,
                1u);
        }
        commit(afull0 + 8 * s);
        it.next(tph, a.bh_count, n);
      }
      commit(done_bar);
    }
  }

  ok = __syncthreads_and(ok ? 1 : 0) != 0;
  if (threadIdx.x == 0) {
    if (!ok) atomicOr(a.err, kErrBitCdist);
    mbar_wait(done_bar, 0, bound);      // issued tensor-core work drains (bounded)
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(tmem_cols)
                 : "memory");
  }
}

template <bool kBf16, int DH>
size_t smem_of(int m) {
  using C = GCfg<kBf16, DH>;
  const int np = np16(m);
  return 2 * (size_t)C::kAStage + (size_t)align128((DH / 4) * lbo_l(np)) +
         align128(4u * m * 32 * 4) + (2 * kTile + 64) * sizeof(float) + 7 * 8 + 8;
}

const void* kernel_of(bool bf16, int d) {
  if (d == 32) return bf16 ? (const void*)gauss_tc_kernel<true, 32> : (const void*)gauss_tc_kernel<false, 32>;
  if (d == 64) return bf16 ? (const void*)gauss_tc_kernel<true, 64> : (const void*)gauss_tc_kernel<false, 64>;
  return nullptr;
}

}  // namespace

size_t gauss_tc_smem_bytes(int m, int d, bool bf16) {
  if (d == 32) return bf16 ? smem_of<true, 32>(m) : smem_of<false, 32>(m);
  if (d == 64) return bf16 ? smem_of<true, 64>(m) : smem_of<false, 64>(m);
  return 0;
}

int gauss_tc_threads() { return kThreads; }

const void* gauss_tc_kernel_ptr(int d, bool bf16) { return kernel_of(bf16, d); }

cudaError_t launch_gauss_tc(const lapl_attn_plan& p, const void* q, const void* k,
                            const float* landmarks, float* at, float* bt, float* dbg_dql,
                            float* dbg_dlk, float* dbg_a, cudaStream_t st) {
  const Geometry& g = p.geo;
  const bool bf16 = p.cfg.in_dtype == LAPL_BF16;
  const void* f = kernel_of(bf16, g.d);
  if (!f) return cudaErrorInvalidValue;
  GaussTcArgs a;
  a.q = q; a.k = k; a.landmarks = landmarks; a.at = at; a.bt = bt;
  a.dbg_dql = dbg_dql; a.dbg_dlk = dbg_dlk; a.dbg_a = dbg_a;
  a.err = p.dev_err;
  a.tiles_per_head = (g.n + kTile - 1) / kTile;
  a.tiles = 2LL * g.bh * a.tiles_per_head;
  a.bh_count = g.bh;
  a.n = g.n; a.m = g.m; a.np = np16(g.m);
  a.c_exp = p.neg_log2e_over_lambda;
  a.wait_ns = p.cd_wait_ns;
  a.skip_last = p.cd_skip_last_copy == 1 ? 1 : 0;
  // Tensor stores of [m x 32] boxes of A^T and B^T, viewed as [BH m rows, N columns]; rows of
  // N fp32 must be a multiple of 16 bytes.  Otherwise plain stores.
  a.tma_store = g.n % 4 == 0 && (long long)g.bh * g.m < (1LL << 31);
  if (a.tma_store) {
    const uint64_t rows = (uint64_t)g.bh * g.m;
    if (p.tmap_at_st_ptr != at) {
      if (!tma_encode_2d(&p.tmap_at_st, at, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (uint64_t)g.n, rows,
                         (uint64_t)g.n * 4, 32, (uint32_t)g.m))
        return cudaErrorInvalidValue;
      p.tmap_at_st_ptr = at;
    }
    if (p.tmap_bt_st_ptr != bt) {
      if (!tma_encode_2d(&p.tmap_bt_st, bt, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (uint64_t)g.n, rows,
                         (uint64_t)g.n * 4, 32, (uint32_t)g.m))
        return cudaErrorInvalidValue;
      p.tmap_bt_st_ptr = bt;
    }
  }
  void* args[] = {&a, &p.tmap_at_st, &p.tmap_bt_st};
  return cudaLaunchKernel(f, dim3((unsigned)g.cd_part.ctas), dim3(kThreads), args, g.cd_smem, st);
}

}  // namespace lapl
