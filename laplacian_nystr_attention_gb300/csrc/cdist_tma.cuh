// cdist_tma.cuh -- fused L1 distance + exp kernel fed by the Tensor Memory Accelerator.
//
// Same computation and outputs as cdist_exp_kernel (cdist_kernel.cuh): for a balanced range of
// (side, head, token) positions, A = k(Q, L) or B = k(L, K) with k(x, y) = exp(-|x - y|_1 /
// lambda) ("LaplacianFormer: Rethinking Linear Attention with Laplacian Kernel", English
// explainer page, 2.A), stored landmark-major.
//
// Pipeline (warp-specialised, no CTA-wide barrier per chunk):
//   * producer warp (warp s): one lane issues cp.async.bulk.tensor loads of 128-token chunks of
//     Q or K (SWIZZLE_128B: 16-byte piece c of a 128-byte row t lands at c ^ (t % 8)) into a
//     ring of kStages buffers, and a 1-D bulk copy of the head's landmarks into a ring of
//     kStages slots whenever the head changes; both complete on the stage's "full" mbarrier;
//   * consumer warps (warps 0..s-1, one landmark group each): wait on "full", compute, store,
//     and release the stage on its "empty" mbarrier (one arrival per warp).
// Landmark slots: before loading chunk i the producer waits until every consumer warp has
// released chunk i - kStages, so consumers can only be reading the landmarks of chunks
// i-kStages+1 .. i-1, which occupy at most kStages-1 slots; a new head takes the next slot of
// the ring, never one of those.
//
// Every mbarrier wait is bounded (one second of %globaltimer); on timeout the waiting thread
// sets kErrTimeout in the library's device error word and its warp leaves the kernel.  Copies
// already issued are still awaited (with the same bound) by the consumers that wait on them.
#pragma once

#include <cuda.h>

#include "cdist_kernel.cuh"

namespace lapl {
namespace cdist_tma {

using cdist_impl::abs_diff_acc;

constexpr int kStages = 2;
constexpr int kLmSlots = kStages;
constexpr int kTile = 128;                          // tokens per chunk (rows of a TMA box)
constexpr unsigned kErrTimeout = kErrBitCdist;
constexpr unsigned long long kWaitNs = 1000000000ull;   // bound of one mbarrier wait

struct TmaArgs {
  const float* landmarks;    // [BH, m, d]
  float* at;                 // [BH, m, N]
  float* bt;                 // [BH, m, N]
  unsigned* err;             // device error word (kErrTimeout)
  float* dbg_dql;
  float* dbg_dlk;
  float* dbg_a;
  Partition part;
  long long bh_count;
  int n;
  float c_exp;
};

__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(unsigned long long* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_tx(unsigned long long* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned addr, unsigned parity) {
  unsigned done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(done)
      : "r"(addr), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the completion of the phase with the given parity; false after kWaitNs.
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, unsigned parity) {
  const unsigned addr = smem_u32(bar);
  if (mbar_try_wait(addr, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(addr, parity))
    if (global_ns() - t0 > kWaitNs) return false;
  return true;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<unsigned long long>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, unsigned bytes,
                                          unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Distances of one chunk from the swizzled stage: acc[r][jj] = sum_c |x_t,c - L_(warp*S+jj),c|
// for tokens t = lane + 32 r (r < RV; the other rows are zero).
template <int S, int DH, bool kBf16, int RV>
__device__ __forceinline__ void chunk_distances(const char* __restrict__ stage,
                                                const float* __restrict__ lrow, int lane,
                                                float (&acc)[4][S]) {
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int jj = 0; jj < S; ++jj) acc[r][jj] = 0.f;
  const int sw = lane & 7;
  constexpr int kUnroll = S >= 8 ? 1 : 2;   // S = 8 at two CTAs per SM has no registers to spare
  if constexpr (!kBf16) {
    // fp32: 128-byte rows of 32 channels; DH = 64 uses two such sub-tiles.
#pragma unroll kUnroll
    for (int c4 = 0; c4 < DH / 4; ++c4) {
      const char* sub = stage + (c4 >> 3) * (kTile * 128);
      float4 x[RV];
#pragma unroll
      for (int r = 0; r < RV; ++r)
        x[r] = *reinterpret_cast<const float4*>(sub + (lane + 32 * r) * 128 + (((c4 & 7) ^ sw) << 4));
#pragma unroll
      for (int jj = 0; jj < S; ++jj) {
        const float4 l = *reinterpret_cast<const float4*>(&lrow[jj * DH + 4 * c4]);
#pragma unroll
        for (int r = 0; r < RV; ++r) {
          float t = acc[r][jj];
          abs_diff_acc(t, x[r].x, l.x);
          abs_diff_acc(t, x[r].y, l.y);
          abs_diff_acc(t, x[r].z, l.z);
          abs_diff_acc(t, x[r].w, l.w);
          acc[r][jj] = t;
        }
      }
    }
  } else {
    // bf16: 128-byte rows of 64 channels, 16-byte pieces of 8 channels, widened to fp32 four
    // channels at a time.
    static_assert(DH == 64, "bf16 stages hold 64 channels per row");
#pragma unroll 1
    for (int c8 = 0; c8 < 8; ++c8) {
      uint4 raw[RV];
#pragma unroll
      for (int r = 0; r < RV; ++r)
        raw[r] = *reinterpret_cast<const uint4*>(stage + (lane + 32 * r) * 128 + ((c8 ^ sw) << 4));
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float4 x[RV];
#pragma unroll
        for (int r = 0; r < RV; ++r) {
          const uint32_t u0 = half ? raw[r].z : raw[r].x;
          const uint32_t u1 = half ? raw[r].w : raw[r].y;
          x[r] = make_float4(bf16_lo(u0), bf16_hi(u0), bf16_lo(u1), bf16_hi(u1));
        }
#pragma unroll
        for (int jj = 0; jj < S; ++jj) {
          const float4 l = *reinterpret_cast<const float4*>(&lrow[jj * DH + 8 * c8 + 4 * half]);
#pragma unroll
          for (int r = 0; r < RV; ++r) {
            float t = acc[r][jj];
            abs_diff_acc(t, x[r].x, l.x);
            abs_diff_acc(t, x[r].y, l.y);
            abs_diff_acc(t, x[r].z, l.z);
            abs_diff_acc(t, x[r].w, l.w);
            acc[r][jj] = t;
          }
        }
      }
    }
  }
}

template <int S, int DH, bool kBf16>
__global__ void __launch_bounds__(32 * (S + 1), 2)
cdist_tma_kernel(const TmaArgs a, const __grid_constant__ CUtensorMap map_q,
                 const __grid_constant__ CUtensorMap map_k) {
  constexpr int M = S * S;
  constexpr int kBoxes = kBf16 ? 1 : DH / 32;              // 128-byte-wide boxes per chunk
  constexpr unsigned kStageBytes = kTile * 128 * kBoxes;
  constexpr unsigned kLmBytes = M * DH * 4;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // Stages need 1024-byte alignment (128-byte swizzle atom).
  // 1024-byte alignment of the stages (128-byte swizzle atom), by pointer arithmetic on the
  // shared array itself so that every access stays a shared-memory access (a round trip through
  // an integer would turn them into generic loads).
  unsigned char* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* stages = base;                                          // kStages x kStageBytes
  float* lms = reinterpret_cast<float*>(stages + kStages * kStageBytes);  // kLmSlots x [M][DH]
  unsigned long long* full = reinterpret_cast<unsigned long long*>(lms + kLmSlots * M * DH);
  unsigned long long* empty = full + kStages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = a.n;
  const int cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], S);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();

  ChunkIter it;
  it.init(a.part, cta, n);
  if (it.done()) return;

  if (warp == S) {
    // ---------------- producer ----------------
    if (lane == 0) {
      long long prev_bh = -1;
      int lm_slot = -1;
      for (int i = 0; !it.done(); ++i) {
        const int s = i % kStages;
        if (i >= kStages && !mbar_wait(&empty[s], ((i / kStages) - 1) & 1)) {
          atomicOr(a.err, kErrTimeout);
          return;
        }
        const bool new_head = it.bh != prev_bh;
        if (new_head) lm_slot = (lm_slot + 1) % kLmSlots;
        mbar_arrive_tx(&full[s], kStageBytes + (new_head ? kLmBytes : 0u));
        const CUtensorMap* map = it.side == 0 ? &map_q : &map_k;
        const int row = (int)(it.bh * n + it.n0);
#pragma unroll
        for (int b = 0; b < kBoxes; ++b)
          tma_load_2d(stages + s * kStageBytes + b * (kTile * 128), map, b * (kBf16 ? 64 : 32), row,
                      &full[s]);
        if (new_head)
          bulk_load(lms + lm_slot * M * DH, a.landmarks + (size_t)it.bh * M * DH, kLmBytes, &full[s]);
        prev_bh = it.bh;
        it.next(n, a.bh_count);
      }
    }
    return;
  }

  // ---------------- consumers ----------------
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
    // Every lane waits (acquiring the copied bytes); the warp leaves together on a timeout.
    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (i / kStages) & 1))) {
      if (lane == 0) atomicOr(a.err, kErrTimeout);
      return;
    }
    const char* stage = reinterpret_cast<const char*>(stages + s * kStageBytes);
    const float* lrow = lms + lm_slot * M * DH + warp * S * DH;

    float acc[4][S];
    const int groups = (valid + 31) >> 5;
    if (groups == 4) chunk_distances<S, DH, kBf16, 4>(stage, lrow, lane, acc);
    else if (groups == 3) chunk_distances<S, DH, kBf16, 3>(stage, lrow, lane, acc);
    else if (groups == 2) chunk_distances<S, DH, kBf16, 2>(stage, lrow, lane, acc);
    else chunk_distances<S, DH, kBf16, 1>(stage, lrow, lane, acc);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);     // this warp is done with the stage

    const size_t row0 = (size_t)bh * n + n0;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
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
#pragma unroll
    for (int jj = 0; jj < S; ++jj) {
      float* dst = (side == 0 ? a.at : a.bt) + ((size_t)bh * M + warp * S + jj) * n + n0;
#pragma unroll
      for (int r = 0; r < 4; ++r)
        if (lane + 32 * r < valid) dst[lane + 32 * r] = acc[r][jj];
    }
    it.next(n, a.bh_count);
  }
}

}  // namespace cdist_tma
}  // namespace lapl
