// cdist_l1.cuh -- fused L1 distance + exp for the query and key blocks, TMA-fed, with the
// element work split between the FP32 pipe and the integer/ALU pipe.
//
// For a balanced range of (side, head, token) positions this computes A = k(Q, L) or
// B = k(L, K) with k(x, y) = exp(-|x - y|_1 / lambda) ("LaplacianFormer: Rethinking Linear
// Attention with Laplacian Kernel", English explainer page, 2.A; distance and exponential in
// one kernel: German page, 2; Chinese page, 2.2), stored landmark-major like the other
// distance kernels.
//
// Element arithmetic.  Each (token, landmark, channel) term |q - l| needs two FP32-pipe
// instructions written directly (a subtract, then an add with an absolute-value operand).  The
// identity |q - l| = q + l - 2 min(q, l) moves half of that work to the ALU pipe:
//   sum_c |q_c - l_c| = Sq + Sl - 2 sum_c min(q_c, l_c),   Sq = sum_c q_c,  Sl = sum_c l_c,
// where the minimum is one ALU instruction and the running sum one packed FP32 add for two
// channels (add.f32x2).  A warp takes the first s/2 of its s landmarks the direct way
// (sub.f32x2, then two abs-adds) and the others through the identity, so both pipes are busy.
// On integer-valued inputs every partial sum is exact in fp32, so both forms give the same
// distance bit for bit; on float inputs the identity's rounding is that of sums of magnitude
// at most sum_c (|q_c| + |l_c|).
//
// CTA: G row groups of s consumer warps (warp w owns landmarks (w mod s)*s .. +s-1; in group
// w / s, lane l owns tokens l, l+32, ... of its 4/G 32-row groups of a 128-token chunk) and one
// helper warp.  Inputs are fp32 (d = 32 or 64) or bf16 (d = 64; each 4-channel piece of a row
// is widened to fp32 once in registers for all of the warp's landmarks).  Lane 0 of the helper
// issues the cp.async.bulk.tensor loads of the chunks (128 rows of 128 bytes per box, SWIZZLE_128B:
// 16-byte piece c of row t lands at c ^ (t % 8)) into a ring of kStages stages, plus a bulk
// copy of a head's landmarks when the head changes; the whole helper warp then computes, per
// chunk, the token sums Sq (and for a new head the landmark sums Sl).  Barriers per stage: full
// (copies landed; the consumers start the chunk's loop), ready (sums written, 32 helper
// arrivals; the consumers wait on it before their epilogue), empty (every consumer warp done
// with the stage and its sums).
//
// Every wait is bounded (wait_ns of %globaltimer).  On timeout the waiting warp sets
// kErrCdistTimeout in the device error word and leaves; the producer lane, on every exit path,
// first waits (with the same bound) until every bulk copy it issued has landed, so no copy is
// left writing into the shared memory of a finished CTA.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace lapl {
namespace cdist_l1 {

constexpr int kTile = 128;       // tokens per chunk
constexpr unsigned kErrCdistTimeout = kErrBitCdist;

struct Args {
  const float* landmarks;    // [BH, m, d]
  float* at;                 // [BH, m, N]
  float* bt;                 // [BH, m, N]
  unsigned* err;             // device error word
  float* dbg_dql;
  float* dbg_dlk;
  float* dbg_a;
  Partition part;
  long long bh_count;
  int n;
  float c_exp;
  unsigned long long wait_ns;   // bound of one barrier wait
  int skip_last_copy;           // fault injection for tests: never issue the last chunk's copy
};

// Stages of the copy ring (and landmark slots, as many): 4 of one 128-byte box per row, 2 of
// two; 3 for bf16 rows of 64 channels with one row group, so that two CTAs (stages plus slots of
// 64 x 49 fp32 landmarks) fit in one SM's shared memory.  (Four stages of two boxes with one CTA
// per SM measured no faster.)
__host__ __device__ constexpr int l1_stages(int boxes, bool bf16, int d, int g) {
  return boxes == 1 ? (bf16 && d == 64 && g == 1 ? 3 : 4) : 2;
}
template <int DH, bool kBf16, int G>
struct Cfg {
  static constexpr int kElemBytes = kBf16 ? 2 : 4;
  static constexpr int kBoxElems = 128 / kElemBytes;                 // elements per 128-byte box
  static constexpr int kBoxes = DH / kBoxElems;                      // 128-byte boxes per row
  static constexpr int kStages = l1_stages(kBoxes, kBf16, DH, G);
  static constexpr unsigned kStageBytes = kTile * 128 * kBoxes;
};

__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(unsigned long long* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned long long* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_test(unsigned long long* bar, unsigned parity) {
  unsigned done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait until the phase with the given parity has completed; false after `bound` ns.
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, unsigned parity,
                                          unsigned long long bound) {
  if (mbar_test(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_test(bar, parity))
    if (global_ns() - t0 > bound) return false;
  return true;
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<unsigned long long>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, unsigned bytes,
                                          unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// t += |x0 - l0| + |x1 - l1| (in that order): one packed subtract, two abs-adds.
__device__ __forceinline__ void sub_abs2(float& t, float x0, float x1, float l0, float l1) {
  asm("{\n\t.reg .b64 a, b, d;\n\t.reg .f32 d0, d1;\n\t"
      "mov.b64 a, {%1, %2};\n\tmov.b64 b, {%3, %4};\n\t"
      "sub.f32x2 d, a, b;\n\tmov.b64 {d0, d1}, d;\n\t"
      "abs.f32 d0, d0;\n\tabs.f32 d1, d1;\n\tadd.f32 %0, %0, d0;\n\tadd.f32 %0, %0, d1;\n\t}"
      : "+f"(t)
      : "f"(x0), "f"(x1), "f"(l0), "f"(l1));
}
// (t0, t1) += (min(x0, l0), min(x1, l1)): two ALU minimums, one packed add.
__device__ __forceinline__ void min_acc2(float& t0, float& t1, float x0, float x1, float l0,
                                         float l1) {
  asm("{\n\t.reg .b64 a, m;\n\t.reg .f32 m0, m1;\n\t"
      "min.f32 m0, %2, %4;\n\tmin.f32 m1, %3, %5;\n\t"
      "mov.b64 m, {m0, m1};\n\tmov.b64 a, {%0, %1};\n\t"
      "add.f32x2 a, a, m;\n\tmov.b64 {%0, %1}, a;\n\t}"
      : "+f"(t0), "+f"(t1)
      : "f"(x0), "f"(x1), "f"(l0), "f"(l1));
}

// Channel quad c4 of token row t in a swizzled stage, as fp32 (bf16 rows widen exactly: a bf16
// value is the upper half of the fp32 with the same value).
template <bool kBf16>
__device__ __forceinline__ float4 stage_quad(const char* stage, int t, int c4) {
  if constexpr (kBf16) {
    const int p = c4 >> 1;                        // 16-byte piece of 8 channels
    const uint2 w = *reinterpret_cast<const uint2*>(stage + (p >> 3) * (kTile * 128) + t * 128 +
                                                    (((p & 7) ^ (t & 7)) << 4) + (c4 & 1) * 8);
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                       __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
  } else {
    return *reinterpret_cast<const float4*>(stage + (c4 >> 3) * (kTile * 128) + t * 128 +
                                            (((c4 & 7) ^ (t & 7)) << 4));
  }
}

// Distances of one chunk for the first RV of this warp's RPL row groups (token rows
// row0 + lane + 32 r): sub-path accumulators accS (landmarks 0 .. NS-1 of the warp) and min-path
// pair accumulators accM (landmarks NS .. S-1).
template <int S, int NS, int DH, int RV, int RPL, bool kBf16>
__device__ __forceinline__ void chunk_sums(const char* __restrict__ stage,
                                           const float* __restrict__ lrow, int lane, int row0,
                                           float (&accS)[RPL][NS > 0 ? NS : 1],
                                           float (&accM)[RPL][S - NS][2]) {
#pragma unroll
  for (int r = 0; r < RPL; ++r) {
#pragma unroll
    for (int j = 0; j < NS; ++j) accS[r][j] = 0.f;
#pragma unroll
    for (int j = 0; j < S - NS; ++j) accM[r][j][0] = accM[r][j][1] = 0.f;
  }
  // Lane row base and swizzle: row t = row0 + lane + 32 r keeps t % 8 = lane % 8 for every r
  // (row0 is a multiple of 32).
  const char* rowp = stage + (row0 + lane) * 128;
  const int sw = lane & 7;
#pragma unroll 2
  for (int c4 = 0; c4 < DH / 4; ++c4) {
    float4 x[RV];
    if constexpr (kBf16) {
      // 4 bf16 channels (8 bytes) per row, widened to fp32 once for all of the warp's landmarks.
      const int p = c4 >> 1;
      const char* pc = rowp + (p >> 3) * (kTile * 128) + (((p & 7) ^ sw) << 4) + (c4 & 1) * 8;
#pragma unroll
      for (int r = 0; r < RV; ++r) {
        const uint2 w = *reinterpret_cast<const uint2*>(pc + r * 32 * 128);
        x[r] = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                           __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
      }
    } else {
      const char* pc = rowp + (c4 >> 3) * (kTile * 128) + (((c4 & 7) ^ sw) << 4);
#pragma unroll
      for (int r = 0; r < RV; ++r) x[r] = *reinterpret_cast<const float4*>(pc + r * 32 * 128);
    }
#pragma unroll
    for (int jj = 0; jj < S; ++jj) {
      const float4 l = *reinterpret_cast<const float4*>(&lrow[jj * DH + 4 * c4]);
#pragma unroll
      for (int r = 0; r < RV; ++r) {
        if (jj < NS) {
          sub_abs2(accS[r][jj < NS ? jj : 0], x[r].x, x[r].y, l.x, l.y);
          sub_abs2(accS[r][jj < NS ? jj : 0], x[r].z, x[r].w, l.z, l.w);
        } else {
          float* p = accM[r][jj >= NS ? jj - NS : 0];
          min_acc2(p[0], p[1], x[r].x, x[r].y, l.x, l.y);
          min_acc2(p[0], p[1], x[r].z, x[r].w, l.z, l.w);
        }
      }
    }
  }
}

// G row groups: G * S consumer warps; warp w owns landmarks (w mod S) * S .. + S - 1 and the
// token rows of group w / S (4 / G row groups of 32 tokens each).  G = 1: two CTAs per SM;
// G = 2: one CTA per SM with the same 2 S consumer warps, all on the same chunk sequence (two
// CTAs on one SM do not progress at the same rate: the warp scheduler favours the older CTA,
// which finishes its equal share well before the other).
template <int S, int DH, int G, bool kBf16>
__global__ void __launch_bounds__(32 * (G * S + 1), G == 1 ? 2 : 1)
cdist_l1_kernel(const Args a, const __grid_constant__ CUtensorMap map_q,
                const __grid_constant__ CUtensorMap map_k) {
  using C = Cfg<DH, kBf16, G>;
  constexpr int CW = G * S;                     // consumer warps; the helper warp is CW
  constexpr int RPL = 4 / G;                    // 32-row groups per consumer warp
  constexpr int kStages = C::kStages;
  constexpr int kLmSlots = kStages;
  constexpr int M = S * S;
  constexpr int NS = S / 2;                     // landmarks per warp on the direct path
  constexpr unsigned kLmBytes = M * DH * 4;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte alignment of the stages (128-byte swizzle atom), by pointer arithmetic on the
  // shared array itself so that every access stays a shared-memory access (a round trip through
  // an integer would turn them into generic loads).
  unsigned char* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* stages = base;                                              // kStages stages
  float* lms = reinterpret_cast<float*>(stages + kStages * C::kStageBytes);  // [slot][M][DH]
  float* sq = lms + kLmSlots * M * DH;                                       // [stage][kTile]
  float* sl = sq + kStages * kTile;                                          // [slot][64]
  unsigned long long* full = reinterpret_cast<unsigned long long*>(sl + kLmSlots * 64);
  unsigned long long* ready = full + kStages;
  unsigned long long* empty = ready + kStages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = a.n;
  const unsigned long long bound = a.wait_ns;

  if (threadIdx.x == 32 * CW) {
    // The producer's first copies need the tensor maps: fetch the descriptors now.
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<unsigned long long>(&map_q))
                 : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<unsigned long long>(&map_k))
                 : "memory");
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&ready[s], 32);
      mbar_init(&empty[s], CW);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  ChunkIter it;
  it.init(a.part, blockIdx.x, n);
  __syncthreads();
  if (it.done()) return;

  if (warp == CW) {
    // ---------------- helper warp: copies (lane 0), token and landmark sums ----------------
    ChunkIter is = it;             // next chunk to issue (lane 0)
    int issued = 0, skipped = -1;
    long long issued_bh = -1;
    int issue_slot = -1;
    bool ok = true;
    long long cur_bh = -1;
    int lm_slot = -1;
    for (int i = 0; !it.done(); ++i) {
      if (lane == 0) {
        // Issue every chunk up to i (waiting for its stage if needed), then any further chunk,
        // up to i + kStages - 1, whose stage is already free.
        while (ok && !is.done() && issued < i + kStages) {
          const int s = issued % kStages;
          if (issued >= kStages) {
            const unsigned par = ((issued / kStages) - 1) & 1;
            if (issued <= i) {
              if (!mbar_wait(&empty[s], par, bound)) {
                atomicOr(a.err, kErrCdistTimeout);
                ok = false;
                break;
              }
            } else if (!mbar_test(&empty[s], par)) {
              break;
            }
          }
          const bool new_head = is.bh != issued_bh;
          if (new_head) issue_slot = (issue_slot + 1) % kLmSlots;
          if (a.skip_last_copy && is.last()) {
            skipped = issued;        // fault injection: this chunk's stage never fills
          } else {
            mbar_expect_tx(&full[s], C::kStageBytes + (new_head ? kLmBytes : 0u));
            const CUtensorMap* map = is.side == 0 ? &map_q : &map_k;
            const int row = (int)(is.bh * n + is.n0);
#pragma unroll
            for (int b = 0; b < C::kBoxes; ++b)
              tma_load_2d(stages + s * C::kStageBytes + b * (kTile * 128), map,
                          b * C::kBoxElems, row, &full[s]);
            if (new_head)
              bulk_load(lms + issue_slot * M * DH, a.landmarks + (size_t)is.bh * M * DH,
                        kLmBytes, &full[s]);
          }
          issued_bh = is.bh;
          ++issued;
          is.next(n, a.bh_count);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const int s = i % kStages;
      const bool new_head = it.bh != cur_bh;
      if (new_head) {
        lm_slot = (lm_slot + 1) % kLmSlots;
        cur_bh = it.bh;
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (i / kStages) & 1, bound))) {
        if (lane == 0) atomicOr(a.err, kErrCdistTimeout);
        break;
      }
      const char* stage = reinterpret_cast<const char*>(stages + s * C::kStageBytes);
      if (new_head) {
        const float* L = lms + lm_slot * M * DH;
        // Lane j sums landmark j starting at channel j mod DH (conflict-free banks).
        for (int j = lane; j < M; j += 32) {
          float t = 0.f;
#pragma unroll 8
          for (int c = 0; c < DH; ++c) t += L[j * DH + ((c + lane) & (DH - 1))];
          sl[lm_slot * 64 + j] = t;
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int t = lane + 32 * r;
        float acc = 0.f;
#pragma unroll
        for (int c4 = 0; c4 < DH / 4; ++c4) {
          const float4 x = stage_quad<kBf16>(stage, t, c4);
          acc += x.x;
          acc += x.y;
          acc += x.z;
          acc += x.w;
        }
        sq[s * kTile + t] = acc;
      }
      mbar_arrive(&ready[s]);
      it.next(n, a.bh_count);
    }
    // Every issued copy lands before the CTA may exit.
    if (lane == 0) {
      for (int j = issued - 1; j >= 0 && j >= issued - kStages; --j) {
        if (j == skipped) continue;
        if (!mbar_wait(&full[j % kStages], (j / kStages) & 1, bound))
          atomicOr(a.err, kErrCdistTimeout);
      }
    }
    return;
  }

  // ---------------- consumers ----------------
  const int lg = warp % S;                       // landmark group
  const int row0 = (warp / S) * RPL * 32;        // first token row of this warp's row groups
  long long cur_bh = -1;
  int lm_slot = -1;
  const bool debug = a.dbg_dql || a.dbg_dlk || a.dbg_a;
  for (int i = 0; !it.done(); ++i) {
    const int s = i % kStages;
    const int side = it.side, n0 = it.n0, valid = it.valid;
    const long long bh = it.bh;
    if (bh != cur_bh) {
      lm_slot = (lm_slot + 1) % kLmSlots;
      cur_bh = bh;
    }
    // The distances need only the copied rows and landmarks; the helper's sums are first used
    // in the epilogue, so its work on this chunk overlaps the loop.
    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (i / kStages) & 1, bound))) {
      if (lane == 0) atomicOr(a.err, kErrCdistTimeout);
      return;
    }
    const char* stage = reinterpret_cast<const char*>(stages + s * C::kStageBytes);
    const float* lrow = lms + lm_slot * M * DH + lg * S * DH;

    float accS[RPL][NS > 0 ? NS : 1];
    float accM[RPL][S - NS][2];
    // 32-row groups of the chunk that hold tokens, counted within this warp's groups.
    const int rv = min(max(((valid + 31) >> 5) - row0 / 32, 0), RPL);
    if (rv == RPL) chunk_sums<S, NS, DH, RPL, RPL, kBf16>(stage, lrow, lane, row0, accS, accM);
    else if (RPL > 3 && rv == 3) chunk_sums<S, NS, DH, 3, RPL, kBf16>(stage, lrow, lane, row0, accS, accM);
    else if (RPL > 2 && rv == 2) chunk_sums<S, NS, DH, 2, RPL, kBf16>(stage, lrow, lane, row0, accS, accM);
    else if (rv >= 1) chunk_sums<S, NS, DH, 1, RPL, kBf16>(stage, lrow, lane, row0, accS, accM);
    if (!__all_sync(0xffffffffu, mbar_wait(&ready[s], (i / kStages) & 1, bound))) {
      if (lane == 0) atomicOr(a.err, kErrCdistTimeout);
      return;
    }
    float sqr[RPL], slj[S - NS];
#pragma unroll
    for (int r = 0; r < RPL; ++r) sqr[r] = sq[s * kTile + row0 + lane + 32 * r];
#pragma unroll
    for (int j = 0; j < S - NS; ++j) slj[j] = sl[lm_slot * 64 + lg * S + NS + j];
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);     // this warp is done with the stage

    // Kernel values, stored straight from registers: per (landmark, row group) one warp store of
    // 32 consecutive tokens.  Every value is formed first, without a branch, then stored; the
    // debug copies have a loop of their own.
    float* dst0 = (side == 0 ? a.at : a.bt) + ((size_t)bh * M + lg * S) * n + n0;
    float dist[S][RPL];
#pragma unroll
    for (int jj = 0; jj < S; ++jj) {
#pragma unroll
      for (int r = 0; r < RPL; ++r) {
        if (jj < NS) {
          dist[jj][r] = accS[r][jj < NS ? jj : 0];
        } else {
          const float* p = accM[r][jj >= NS ? jj - NS : 0];
          dist[jj][r] = fmaf(-2.f, p[0] + p[1], sqr[r] + slj[jj >= NS ? jj - NS : 0]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < RPL; ++r) {
      const int t = row0 + lane + 32 * r;
      if (t < valid) {
#pragma unroll
        for (int jj = 0; jj < S; ++jj)
          dst0[(size_t)jj * n + t] = laplacian_from_distance(dist[jj][r], a.c_exp);
      }
    }
    if (debug) {
#pragma unroll
      for (int r = 0; r < RPL; ++r) {
        const int t = row0 + lane + 32 * r;
        if (t >= valid) continue;
        const size_t tok = (size_t)bh * n + n0 + t;
#pragma unroll
        for (int jj = 0; jj < S; ++jj) {
          const int j = lg * S + jj;
          if (side == 0) {
            if (a.dbg_dql) a.dbg_dql[tok * M + j] = dist[jj][r];
            if (a.dbg_a) a.dbg_a[tok * M + j] = laplacian_from_distance(dist[jj][r], a.c_exp);
          } else if (a.dbg_dlk) {
            a.dbg_dlk[((size_t)bh * M + j) * n + n0 + t] = dist[jj][r];
          }
        }
      }
    }
    it.next(n, a.bh_count);
  }
}

// Dynamic shared memory: 1024 bytes of alignment slack, stages, landmark slots, token sums,
// landmark sums and 3 barriers per stage.
inline size_t smem_bytes(int s, int d, bool bf16, int g) {
  const size_t m = (size_t)s * s;
  const int boxes = d * (bf16 ? 2 : 4) / 128;
  const int stages = l1_stages(boxes, bf16, d, g);
  const size_t stage = (size_t)kTile * 128 * boxes;
  return 1024 + stages * stage + (size_t)stages * m * d * sizeof(float) +
         (size_t)stages * kTile * sizeof(float) + (size_t)stages * 64 * sizeof(float) +
         3 * stages * 8;
}

// Instantiations: fp32 with d = 32 or 64 (cdist_l1.cu), bf16 with d = 64 (cdist_l1_bf16.cu);
// g row groups (1 or 2).
const void* kernel(int s, int d, int g, bool bf16);

}  // namespace cdist_l1
}  // namespace lapl
