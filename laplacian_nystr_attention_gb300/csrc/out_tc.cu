// out_tc.cu -- O = A^ M on the tensor cores (tcgen05, TF32 operands split into an exact high/low
// pair, fp32 accumulation in tensor memory), whitening applied on the way into the operand.
//
// "LaplacianFormer: Rethinking Linear Attention with Laplacian Kernel": the output is
// O = A^ (X (B V)) with A^ = (A - mean) / sqrt(var + delta) + bias column by column (Korean
// explainer page, 2.2; English page, 2.B), evaluated right to left so that the N x N matrix is
// never formed (Chinese page, 2.2); this is the last product, O = A^ M with M = X (B V).
//
// Persistent: one CTA per SM, each walking a contiguous range of 128-token tiles (head-major
// order).  Per tile the accumulator D (128 token rows = tensor-memory lanes) receives
//   D[:, 0:2d]  = A^_hi [M_hi | M_lo]      (one MMA chain with N = 2d)
//   D[:, 0:d]  += A^_lo  M_hi              (a second chain with N = d into the same columns)
// so O[t][c] = D[t][c] + D[t][d + c]: the three cross products that reproduce fp32 operands to
// about 2^-21, summed within one tensor-memory lane (no exchange between warps).
// Warps:
//   0-7  converters (two per scheduler): take the A^T tile (landmark-major [m][N], copied into
//        shared memory by TMA while the previous tile is converted), whiten it, transpose
//        4 x 4 in registers and store A^_hi / A^_lo in the K-major operand
//        layout (core matrices of 8 rows x 16 bytes, row-group stride padded to 144 bytes so
//        that a quarter-warp's stores fall in 8 bank groups); per head they also build
//        [M_hi; M_lo] (2d rows, K = landmarks) from M after the programmatic wait;
//   8-11 epilogue: read the accumulator (one row per thread), add the two halves, store O: for
//        fp32 O with d = 32 or 64 and bf16 O with d = 64 each warp stages its 32 rows in shared
//        memory (128-byte swizzle: 16-byte piece c of row t at c ^ (t % 8), conflict-free) and
//        writes them with TMA tensor stores of a [B H, N, d] view that clip at the head's end
//        (per-thread row stores of 16 bytes touch 32 rows per warp instruction and measured
//        about a quarter of the kernel's time at the high-resolution shape); otherwise each
//        thread stores its row;
//   12   owns the tensor memory; one thread issues the MMAs.
// Two operand stages and two accumulators (2 x 2d tensor-memory columns): the conversion of
// tile i + 1 and the stores of tile i - 1 overlap the MMAs of tile i.  One M buffer: a new
// head's M is written once the previous tile's MMAs are complete.
// The first tile's loads and whitening run before the programmatic wait, overlapping the M
// kernel.  Every barrier wait is bounded (one second); on a timeout the CTA sets the chain bit
// of the device error word, waits (bounded) for its tensor-core work and frees the tensor
// memory.
#include "common.cuh"

namespace lapl {
namespace {

constexpr int kTileT = 128;
constexpr int kStagesO = 2;
constexpr int kConvWarps = 8;
constexpr int kConvThreadsO = 32 * kConvWarps;
constexpr int kEpiWarp0 = 8, kMmaWarpO = 12;
constexpr int kOutTcThreads = 32 * 13;
constexpr unsigned kSboO = 144;                 // A^: padded stride between 8-row core groups
constexpr unsigned kLboA = 16 * kSboO;          // A^ operand: 128 rows
constexpr unsigned kSboB = 128;                 // [M_hi; M_lo]: unpadded (written once per head)
constexpr int kItems = 16 / kConvWarps;         // landmark quads per converter thread (m <= 64)
// Whitening coefficients (mean, scale, bias) of each converter warp's 4 kItems landmarks.
constexpr unsigned kCoefFloatsPerWarp = 3 * 4 * kItems;
constexpr unsigned kCoefBytes = kConvWarps * kCoefFloatsPerWarp * 4;
constexpr unsigned kBarBytes = 11 * 8;          // 11 mbarriers, then the tensor-memory slot

__host__ __device__ inline int mk8(int m) { return (m + 7) & ~7; }
__host__ __device__ inline unsigned a_part_bytes(int mk) { return (unsigned)(mk / 4) * kLboA; }
__host__ __device__ inline unsigned lbo_b(int rows) { return (unsigned)(rows / 8) * kSboB; }
__host__ __device__ inline unsigned b_bytes(int d, int mk) {
  return (unsigned)(mk / 4) * lbo_b(2 * d);
}
__host__ __device__ inline unsigned align128(unsigned x) { return (x + 127u) & ~127u; }
// The copied A^T tile: m landmark rows x 128 tokens, fp32.
__host__ __device__ inline unsigned raw_bytes(int m) { return align128((unsigned)m * kTileT * 4); }

__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ float tf32_rna(float x) {
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}
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
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y,
                                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];\n\t"
      "cp.async.bulk.commit_group;" ::"l"(reinterpret_cast<unsigned long long>(map)),
      "r"(x), "r"(y), "r"(z), "r"(smem_u32(src))
      : "memory");
}
// A^T tile (128 tokens x m landmark rows) into shared memory; tokens past N read as zero.
__device__ __forceinline__ void tma_load_2d(unsigned dst, const CUtensorMap* map, int x, int y,
                                            unsigned bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<unsigned long long>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// The same tile into L2 only; coordinates past the tensor read nothing.
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<unsigned long long>(map)),
               "r"(x), "r"(y)
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

struct OutTcArgs {
  const float* at;      // [BH, m, N]
  const float* mmat;    // [BH, m, d]
  const float* mu;      // [BH, m]
  const float* rstd;    // [BH, m]
  const float* bias;    // [H, m] or null
  void* out;            // [BH, N, d] fp32 or bf16
  unsigned* err;
  int m, d, n, heads;
  int tiles_per_head;
  long tiles;
  int whiten;
  int ahead;            // A^T tiles prefetched into L2 beyond the one being copied (0: off)
  unsigned long long wait_ns;   // bound of every barrier wait
  int skip_last;        // fault injection: thread 0 never copies a CTA's last A^T tile
};

// Shared memory after the operand stages, the M buffer and the A^T tile, from a 1024-byte
// boundary: the epilogue warps' store stages, one box (32 rows x 128 bytes) each.
constexpr unsigned kOstageBytes = 4u * 32u * 128u;

template <bool kOutBf16, bool kTmaStore>
__global__ void __launch_bounds__(kOutTcThreads, 1)
    out_tc_kernel(const OutTcArgs a, const __grid_constant__ CUtensorMap map_o,
                  const __grid_constant__ CUtensorMap map_at) {
  extern __shared__ __align__(128) unsigned char smem_o[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = a.m, d = a.d, n = a.n;
  const int mk = mk8(m);
  const unsigned apart = a_part_bytes(mk);
  const unsigned bbytes = b_bytes(d, mk);
  const unsigned lboB = lbo_b(2 * d);
  unsigned char* astage = smem_o;                                       // [stage][hi, lo]
  unsigned char* bbuf = astage + kStagesO * 2 * apart;                  // [2d x mk]
  unsigned char* raw = bbuf + align128(bbytes);                         // A^T tile [m][128]
  unsigned kCoefOff = kStagesO * 2 * apart + align128(bbytes) + raw_bytes(m);
  unsigned char* ostage = nullptr;
  if constexpr (kTmaStore) {
    // 1024-byte aligned (the swizzle pattern's period), by pointer arithmetic on the array.
    const unsigned at = smem_u32(smem_o + kCoefOff);
    ostage = smem_o + kCoefOff + ((1024u - (at & 1023u)) & 1023u);
    kCoefOff = (unsigned)(ostage - smem_o) + kOstageBytes;
  }
  unsigned long long* bars = reinterpret_cast<unsigned long long*>(smem_o + kCoefOff + kCoefBytes);
  const unsigned ofull0 = smem_u32(bars), oempty0 = ofull0 + 16, afull0 = oempty0 + 16,
                 aempty0 = afull0 + 16, done_bar = aempty0 + 16, rfull = done_bar + 8,
                 rempty = rfull + 8;
  unsigned* slot = reinterpret_cast<unsigned*>(bars + 11);
  const unsigned tmem_cols = 4 * d <= 64 ? 64u : 4 * d <= 128 ? 128u : 4 * d <= 256 ? 256u : 512u;

  const long t_begin = (long)blockIdx.x * a.tiles / gridDim.x;
  const long t_end = (long)(blockIdx.x + 1) * a.tiles / gridDim.x;
  const int ntiles = (int)(t_end - t_begin);

  if (warp == kMmaWarpO) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(slot)),
                 "r"(tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(ofull0 + 8 * s, kConvWarps);
      mbar_init(oempty0 + 8 * s, 1);     // tensor-core commit
      mbar_init(afull0 + 8 * s, 1);      // tensor-core commit
      mbar_init(aempty0 + 8 * s, 4);     // epilogue warps
    }
    mbar_init(done_bar, 1);
    mbar_init(rfull, 1);                 // the copying thread's expect_tx arrival
    mbar_init(rempty, kConvWarps);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const unsigned tmem = *slot;
  bool ok = true;
  int copied = 0;                      // A^T copies issued (thread 0)

  if (warp < kConvWarps) {
    // ---------------- converters ----------------
    // Thread (warp w, lane q) handles token quad q of landmark quads w, w + 8.
    // Thread 0 copies each A^T tile with the Tensor Memory Accelerator into the one raw stage
    // (16-byte register loads of the landmark-major rows, 32 KB per SM in flight, measured
    // about 1600 cycles per tile just to issue); the converters move the tile to registers,
    // free the stage (the copy of tile i + 1 starts) and convert tile i meanwhile.
    const int tid = threadIdx.x;
    // This warp's whitening coefficients: mean, scale, bias of its 4 kItems landmarks.
    float* coef = reinterpret_cast<float*>(smem_o + kCoefOff) + warp * kCoefFloatsPerWarp;
    long prev_bh = -1;
    bool waited = false;
    const unsigned tile_bytes = (unsigned)m * kTileT * 4;
    auto copy_tile = [&](int j) {
      const long tile = t_begin + j;
      mbar_expect_tx(rfull, tile_bytes);
      tma_load_2d(smem_u32(raw), &map_at, (int)(tile % a.tiles_per_head) * kTileT,
                  (int)(tile / a.tiles_per_head) * m, rfull);
    };
    // Thread 0 also keeps the Tensor Memory Accelerator prefetching A^T into L2 `ahead` tiles
    // beyond the copy: tile j is prefetched while tile j - 1 - ahead is converted.
    auto prefetch = [&](int j) {
      if (tid == 0 && j < ntiles) {
        const long tile = t_begin + j;
        tma_prefetch_l2_2d(&map_at, (int)(tile % a.tiles_per_head) * kTileT,
                           (int)(tile / a.tiles_per_head) * m);
      }
    };
    // Fault injection: a CTA's last tile is never copied, so the waits on it run out.
    const bool skip_last = a.skip_last != 0;
    if (tid == 0 && ntiles > 0 && !(skip_last && ntiles == 1)) {
      copy_tile(0);
      copied = 1;
    }
    for (int j = 2; j <= a.ahead; ++j) prefetch(j);
    for (int i = 0; i < ntiles; ++i) {
      if (a.ahead > 0) prefetch(i + 1 + a.ahead);
      const long tile = t_begin + i;
      const long bh = tile / a.tiles_per_head;
      const int s = i & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(rfull, i & 1, a.wait_ns))) {
        ok = false;
        break;
      }
      float4 cur[kItems][4];
      const float* rt = reinterpret_cast<const float*>(raw) + 4 * lane;
#pragma unroll
      for (int it = 0; it < kItems; ++it) {
        const int p = warp + kConvWarps * it;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = 4 * p + u;
          cur[it][u] = j < m ? *reinterpret_cast<const float4*>(rt + j * kTileT)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(rempty);
      if (warp == 0 && i + 1 < ntiles) {
        // The next copy overwrites the stage once every converter warp holds this tile.
        const bool freed = lane != 0 || mbar_wait(rempty, i & 1, a.wait_ns);
        if (!__all_sync(0xffffffffu, freed)) {
          ok = false;
          break;
        }
        if (lane == 0 && !(skip_last && i + 1 == ntiles - 1)) {
          copied = i + 2;
          copy_tile(i + 1);
        }
      }
      const bool new_head = bh != prev_bh;
      if (new_head) {
        // Whitening coefficients of this head for this warp's landmarks (kItems quads); the
        // warp alone reads them, so a warp barrier orders the refresh.
        __syncwarp();
        if (lane < 4 * kItems) {
          const int j = 4 * (warp + kConvWarps * (lane >> 2)) + (lane & 3);
          float mean = 0.f, sc = 1.f, b = 0.f;
          if (a.whiten && j < m) {
            const int h = (int)(bh % a.heads);
            mean = a.mu[(size_t)bh * m + j];
            sc = a.rstd[(size_t)bh * m + j];
            b = a.bias ? a.bias[(size_t)h * m + j] : 0.f;
          }
          coef[lane] = mean;
          coef[4 * kItems + lane] = sc;
          coef[8 * kItems + lane] = b;
        }
        __syncwarp();
      }
      if (i >= kStagesO &&
          !__all_sync(0xffffffffu, mbar_wait(oempty0 + 8 * s, ((i >> 1) - 1) & 1, a.wait_ns))) {
        ok = false;
        break;
      }
      unsigned char* ahi = astage + s * 2 * apart;
      unsigned char* alo = ahi + apart;
#pragma unroll
      for (int it = 0; it < kItems; ++it) {
        const int p = warp + kConvWarps * it;
        if (p < mk / 4) {
          float4 v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = 4 * p + u;
            const float mean = coef[4 * it + u], sc = coef[4 * kItems + 4 * it + u],
                        b = coef[8 * kItems + 4 * it + u];
            v[u] = j < m ? make_float4((cur[it][u].x - mean) * sc + b, (cur[it][u].y - mean) * sc + b,
                                       (cur[it][u].z - mean) * sc + b, (cur[it][u].w - mean) * sc + b)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int row = 4 * lane + t;
            const float4 col = t == 0 ? make_float4(v[0].x, v[1].x, v[2].x, v[3].x)
                             : t == 1 ? make_float4(v[0].y, v[1].y, v[2].y, v[3].y)
                             : t == 2 ? make_float4(v[0].z, v[1].z, v[2].z, v[3].z)
                                      : make_float4(v[0].w, v[1].w, v[2].w, v[3].w);
            const float4 hi = make_float4(tf32_rna(col.x), tf32_rna(col.y), tf32_rna(col.z),
                                          tf32_rna(col.w));
            const unsigned o = p * kLboA + (row >> 3) * kSboO + (row & 7) * 16;
            *reinterpret_cast<float4*>(ahi + o) = hi;
            *reinterpret_cast<float4*>(alo + o) =
                make_float4(col.x - hi.x, col.y - hi.y, col.z - hi.z, col.w - hi.w);
          }
        }
      }
      if (new_head) {
        // M of this head: needs the M kernel (programmatic predecessor) complete, and the
        // previous tile's MMAs (the last readers of the one M buffer) done.
        if (!waited) {
          asm volatile("griddepcontrol.wait;" ::: "memory");
          waited = true;
        }
        if (i >= 1 && !__all_sync(0xffffffffu,
                                  mbar_wait(oempty0 + 8 * ((i - 1) & 1), ((i - 1) >> 1) & 1, a.wait_ns))) {
          ok = false;
          break;
        }
        unsigned char* bb = bbuf;
        const float* mg = a.mmat + (size_t)bh * m * d;
        // [M_hi; M_lo]: row c (c < d) = column c of M_hi, row d + c = column c of M_lo;
        // items (landmark quad p, value-column quad c4).
        const int cq = d >> 2;
        for (int e = tid; e < (mk / 4) * cq; e += kConvThreadsO) {
          const int c4 = e % cq, p = e / cq;
          float4 r[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = 4 * p + u;
            r[u] = j < m ? *reinterpret_cast<const float4*>(&mg[(size_t)j * d + 4 * c4])
                         : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float4 col = c == 0 ? make_float4(r[0].x, r[1].x, r[2].x, r[3].x)
                             : c == 1 ? make_float4(r[0].y, r[1].y, r[2].y, r[3].y)
                             : c == 2 ? make_float4(r[0].z, r[1].z, r[2].z, r[3].z)
                                      : make_float4(r[0].w, r[1].w, r[2].w, r[3].w);
            const float4 hi = make_float4(tf32_rna(col.x), tf32_rna(col.y), tf32_rna(col.z),
                                          tf32_rna(col.w));
            const int row = 4 * c4 + c, lrow = d + row;
            *reinterpret_cast<float4*>(bb + p * lboB + (row >> 3) * kSboB + (row & 7) * 16) = hi;
            *reinterpret_cast<float4*>(bb + p * lboB + (lrow >> 3) * kSboB + (lrow & 7) * 16) =
                make_float4(col.x - hi.x, col.y - hi.y, col.z - hi.z, col.w - hi.w);
          }
        }
        prev_bh = bh;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(ofull0 + 8 * s);
    }
  } else if (warp < kMmaWarpO) {
    // ---------------- epilogue ----------------
    const int ew = warp - kEpiWarp0;                   // tensor-memory lanes 32 ew ..
    const int r = 32 * ew + lane;                      // token row of the tile
    // This warp's store stage: one box of 32 rows x 128 bytes, 16-byte piece c of row `lane`
    // at (c ^ (lane % 8)) * 16; a row of O is one or two boxes, staged and stored in turn.
    unsigned char* stg = kTmaStore ? ostage + ew * (kOstageBytes / 4) : nullptr;
    constexpr int kElt = kOutBf16 ? 2 : 4;
    for (int i = 0; i < ntiles; ++i) {
      const long tile = t_begin + i;
      const long bh = tile / a.tiles_per_head;
      const int n0 = (int)(tile % a.tiles_per_head) * kTileT;
      const int b = i & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(afull0 + 8 * b, (i >> 1) & 1, a.wait_ns))) {
        ok = false;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const unsigned row_addr = tmem + ((unsigned)(32 * ew) << 16) + (unsigned)(b * 2 * d);
      const int tok = n0 + r;
      // Rows n0 + 32 ew .. of head bh; rows past the head's end are clipped by the store, a
      // box wholly past it is not issued.
      const bool rows_in = n0 + 32 * ew < n;
      for (int c0 = 0; c0 < d; c0 += 16) {
        float v[16], w[16];
        tmem_ld16(row_addr + c0, v);
        tmem_ld16(row_addr + d + c0, w);
        if constexpr (kTmaStore) {
          if ((c0 * kElt) % 128 == 0) {
            // A new box: the stage's previous store has finished reading it.
            if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            __syncwarp();
          }
          if constexpr (kOutBf16) {
            uint4 pk[2];
            unsigned* pw = reinterpret_cast<unsigned*>(pk);
#pragma unroll
            for (int c = 0; c < 16; c += 2) {
              __nv_bfloat162 t2 = __floats2bfloat162_rn(v[c] + w[c], v[c + 1] + w[c + 1]);
              pw[c / 2] = *reinterpret_cast<unsigned*>(&t2);
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int gc = c0 / 8 + u;                      // 16-byte piece of the row
              *reinterpret_cast<uint4*>(stg + lane * 128 + (((gc & 7) ^ (lane & 7)) << 4)) =
                  pk[u];
            }
          } else {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int gc = c0 / 4 + u;
              *reinterpret_cast<float4*>(stg + lane * 128 + (((gc & 7) ^ (lane & 7)) << 4)) =
                  make_float4(v[4 * u] + w[4 * u], v[4 * u + 1] + w[4 * u + 1],
                              v[4 * u + 2] + w[4 * u + 2], v[4 * u + 3] + w[4 * u + 3]);
            }
          }
          if (((c0 + 16) * kElt) % 128 == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0 && rows_in)
              tma_store_3d(&map_o, stg, c0 + 16 - 128 / kElt, n0 + 32 * ew, (int)bh);
          }
        } else if (tok < n) {
          const size_t o = ((size_t)bh * n + tok) * d + c0;
          if constexpr (kOutBf16) {
            uint4 pk[2];
            unsigned* pw = reinterpret_cast<unsigned*>(pk);
#pragma unroll
            for (int c = 0; c < 16; c += 2) {
              __nv_bfloat162 t2 = __floats2bfloat162_rn(v[c] + w[c], v[c + 1] + w[c + 1]);
              pw[c / 2] = *reinterpret_cast<unsigned*>(&t2);
            }
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + o);
            dst[0] = pk[0];
            dst[1] = pk[1];
          } else {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + o);
#pragma unroll
            for (int c = 0; c < 16; c += 4)
              dst[c / 4] = make_float4(v[c] + w[c], v[c + 1] + w[c + 1], v[c + 2] + w[c + 2],
                                       v[c + 3] + w[c + 3]);
          }
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(aempty0 + 8 * b);
    }
    if (kTmaStore && lane == 0)
      asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");   // stores done before exit
  } else {
    // ---------------- MMA issue ----------------
    if (lane == 0) {
      const uint32_t id2 = idesc((unsigned)(2 * d)), id1 = idesc((unsigned)d);
      for (int i = 0; i < ntiles; ++i) {
        const int s = i & 1, b = i & 1;
        if (!mbar_wait(ofull0 + 8 * s, (i >> 1) & 1, a.wait_ns) ||
            (i >= 2 && !mbar_wait(aempty0 + 8 * b, ((i >> 1) - 1) & 1, a.wait_ns))) {
          ok = false;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const unsigned ahi = smem_u32(astage + s * 2 * apart), alo = ahi + apart;
        const unsigned bb = smem_u32(bbuf);
        const unsigned acc_addr = tmem + (unsigned)(b * 2 * d);
        for (int kk = 0; kk < mk / 8; ++kk) {
          const uint64_t bd = op_desc(bb + kk * 2 * lboB, lboB, kSboB);
          mma(acc_addr, op_desc(ahi + kk * 2 * kLboA, kLboA, kSboO), bd, id2, kk > 0 ? 1u : 0u);
          mma(acc_addr, op_desc(alo + kk * 2 * kLboA, kLboA, kSboO), bd, id1, 1u);
        }
        commit(oempty0 + 8 * s);
        commit(afull0 + 8 * b);
      }
      commit(done_bar);
    }
  }

  // Every issued copy lands before the CTA may finish (at once unless a wait gave up).
  if (threadIdx.x == 0 && copied > 0) mbar_wait(rfull, (copied - 1) & 1, a.wait_ns);
  ok = __syncthreads_and(ok ? 1 : 0) != 0;
  if (!ok && threadIdx.x == 0) {
    atomicOr(a.err, kErrBitChain);
    mbar_wait(done_bar, 0, a.wait_ns);   // let issued tensor-core work drain (bounded)
  }
  if (ok && threadIdx.x == 0) mbar_wait(done_bar, 0, a.wait_ns);
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == kMmaWarpO) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(tmem_cols)
                 : "memory");
  }
}

}  // namespace

size_t out_tc_smem_bytes(int m, int d, bool tma_store, bool out_bf16) {
  const int mk = mk8(m);
  (void)out_bf16;
  return (size_t)kStagesO * 2 * a_part_bytes(mk) + (size_t)align128(b_bytes(d, mk)) +
         raw_bytes(m) + (tma_store ? 1024 + (size_t)kOstageBytes : 0) + kCoefBytes + kBarBytes + 16;
}

bool out_tc_tma_store(int d, bool out_bf16) { return out_bf16 ? d == 64 : (d == 32 || d == 64); }

int out_tc_threads() { return kOutTcThreads; }

cudaError_t out_tc_configure(size_t smem) {
  const void* fs[4] = {(const void*)out_tc_kernel<false, false>, (const void*)out_tc_kernel<true, false>,
                       (const void*)out_tc_kernel<false, true>, (const void*)out_tc_kernel<true, true>};
  for (const void* f : fs) {
    const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)smem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_output_tc(const lapl_attn_plan& p, const float* at, const float* mmat,
                             const float* mu, const float* rstd, const float* bias, void* out,
                             cudaStream_t st) {
  const Geometry& g = p.geo;
  const bool bf16 = p.cfg.out_dtype == LAPL_BF16;
  OutTcArgs a;
  a.at = at; a.mmat = mmat; a.mu = mu; a.rstd = rstd; a.bias = bias; a.out = out;
  a.err = p.dev_err;
  a.m = g.m; a.d = g.d; a.n = g.n; a.heads = p.cfg.heads;
  a.tiles_per_head = (g.n + kTileT - 1) / kTileT;
  a.tiles = g.bh * a.tiles_per_head;
  a.whiten = p.cfg.whiten;
  a.ahead = g.out_ahead;
  a.wait_ns = p.cd_wait_ns;
  a.skip_last = p.cd_skip_last_copy == 2 ? 1 : 0;
  if (p.tmap_at_pf_ptr != at) {
    // A^T as [B H m, N] fp32, boxes of one tile: 128 tokens x m landmark rows (the copies and
    // the L2 prefetches).
    if (!tma_encode_2d(&p.tmap_at_pf, at, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (uint64_t)g.n,
                       (uint64_t)g.bh * g.m, (uint64_t)g.n * 4, kTileT, (uint32_t)g.m))
      return cudaErrorInvalidValue;
    p.tmap_at_pf_ptr = at;
  }
  if (g.out_tma && p.tmap_o_ptr != out) {
    // O as [B H, N, d]: boxes of 128 bytes x 32 rows of one head, 128-byte swizzle.
    const int elt = bf16 ? 2 : 4;
    if (!tma_encode_3d_sw128(&p.tmap_o, out,
                             bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                             (uint64_t)g.d, (uint64_t)g.n, (uint64_t)g.bh, (uint64_t)g.d * elt,
                             (uint64_t)g.n * g.d * elt, (uint32_t)(128 / elt), 32))
      return cudaErrorInvalidValue;
    p.tmap_o_ptr = out;
  }
  const long grid = std::min<long>(a.tiles, p.num_sms);
  // Programmatic dependent launch: the first tile's loads and whitening overlap the kernel
  // before (the M kernel, or the CG solver).
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kOutTcThreads);
  cfg.dynamicSmemBytes = g.out_smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const CUtensorMap& map = p.tmap_o;
  const CUtensorMap& map_at = p.tmap_at_pf;
  if (g.out_tma)
    return bf16 ? cudaLaunchKernelEx(&cfg, out_tc_kernel<true, true>, a, map, map_at)
                : cudaLaunchKernelEx(&cfg, out_tc_kernel<false, true>, a, map, map_at);
  return bf16 ? cudaLaunchKernelEx(&cfg, out_tc_kernel<true, false>, a, map, map_at)
              : cudaLaunchKernelEx(&cfg, out_tc_kernel<false, false>, a, map, map_at);
}

}  // namespace lapl
