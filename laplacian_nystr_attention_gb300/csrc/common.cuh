// common.cuh -- internal declarations shared by the CUDA translation units of liblapl_attn.
//
// Nothing here is part of the public ABI (include/lapl_attn.h is).  The plan holds host
// state only; every device buffer belongs to the caller.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

#include "lapl_attn.h"

namespace lapl {

// Bits of the device error word (set by a kernel whose bounded barrier wait gave up).
constexpr unsigned kErrBitCdist = 1u;   // distance kernel (TMA pipeline)
constexpr unsigned kErrBitSolve = 2u;   // Newton-Schulz solve on the tensor cores
constexpr unsigned kErrBitChain = 4u;   // tensor-core B V or output product

constexpr int kMaxS = 8;            // landmark grid side: m = s*s <= 64
constexpr int kMaxM = kMaxS * kMaxS;
constexpr int kMaxD = 128;
constexpr size_t kAlign = 256;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Balanced split of the distance kernel's work.  Positions 0 .. 2*BH*N-1 list every (side,
// head, token): query tokens first (position bh*N + n), then key tokens (BH*N + bh*N + n).  The
// `ctas` CTAs take consecutive ranges of q or q+1 positions (q = total / ctas; the first
// total % ctas CTAs take one more), so every CTA gets the same work up to one token.
struct Partition {
  long long uq;      // query positions, BH * N (key positions follow)
  long long total;   // 2 * uq
  long long q;       // total / ctas
  int rem;           // total % ctas
  int ctas;
};

// First position of CTA c (c == ctas gives the end of the list).
__host__ __device__ inline long long part_start(const Partition& pt, int c) {
  return (long long)c * pt.q + (c < pt.rem ? c : pt.rem);
}

// The CTA whose range holds position x (for q > 0).
__host__ __device__ inline int part_owner(const Partition& pt, long long x) {
  const long long big = (long long)pt.rem * (pt.q + 1);
  if (x < big) return (int)(x / (pt.q + 1));
  return pt.rem + (int)((x - big) / pt.q);
}

// Tokens per chunk of the persistent distance kernels that walk a Partition.
constexpr int kChunkTokens = 128;

// Chunk sequence of a CTA: (side, head, first token, token count), advanced without divisions.
struct ChunkIter {
  long long pos, pend;
  int side;
  long long bh;
  int n0, valid;

  __device__ void init(const Partition& pt, int cta, int n) {
    pos = part_start(pt, cta);
    pend = part_start(pt, cta + 1);
    if (pos >= pend) return;
    side = pos < pt.uq ? 0 : 1;
    const long long local = pos - (side ? pt.uq : 0);
    bh = local / n;
    n0 = (int)(local % n);
    valid = (int)min((long long)min(kChunkTokens, n - n0), pend - pos);
  }
  __device__ bool done() const { return pos >= pend; }
  __device__ bool last() const { return pos + valid >= pend; }
  __device__ void next(int n, long long bh_count) {
    pos += valid;
    if (pos >= pend) return;
    n0 += valid;
    if (n0 == n) {
      n0 = 0;
      bh += 1;
      if (side == 0 && bh == bh_count) {
        side = 1;
        bh = 0;
      }
    }
    valid = (int)min((long long)min(kChunkTokens, n - n0), pend - pos);
  }
};

// Offsets (bytes) of the workspace regions for one configuration.  All fp32.  The regions
// only the training forward writes (xs, bv) come last, so a plain forward needs only the
// first fwd_total bytes.
struct WorkspaceLayout {
  size_t landmarks;    // [BH, m, d]         pooled keys L
  size_t x;            // [BH, m, m]         Newton-Schulz result X
  size_t at;           // [BH, m, N]         A = k(Q, L), landmark-major (A transposed)
  size_t bt;           // [BH, m, N]         B = k(L, K)
  size_t bvp;          // [BH, bv_splits, m, d]  per-split partial sums of B V
  size_t mmat;         // [BH, m, d]         M = X (B V)
  size_t mu;           // [BH, m]            column means of A
  size_t rstd;         // [BH, m]            1 / sqrt(column variance + delta)
  size_t fwd_total;    // bytes a plain forward reads or writes (everything above)
  size_t xs;           // [BH, T + 1, m, mk] every Newton-Schulz iterate X_0 .. X_T, rows
                       //                    padded to mk = 4 ceil(m / 4) (kept for the
                       //                    backward pass; Newton-Schulz plans only)
  size_t bv;           // [BH, m, d]         B V (kept for the backward pass)
  size_t total;
};

// Offsets (bytes) of the backward pass's own workspace regions.  All fp32.
struct BwdLayout {
  size_t dahat;      // [BH, m, N]          dLoss/dA^ (landmark-major)
  size_t part_dm;    // [BH, splits, m, d]  partial dM = A^T G
  size_t part_s;     // [BH, splits, 2, m]  partial column sums of dA^ and dA^ Z
  size_t s12;        // [BH, 2, m]          the sums
  size_t dbv;        // [BH, m, d]          dLoss/d(B V)
  size_t dll;        // [BH, m, d]          the landmark block's term of dL
  size_t dbias_bh;   // [BH, m]             per-slice bias gradient
  size_t gq;         // [BH, m, N]          dLoss/dD_QL
  size_t hk;         // [BH, m, N]          dLoss/dD_LK
  size_t part_dl;    // [BH, 2, splits, m, d]  partial dL (query side, key side)
  size_t dl;         // [BH, m, d]          dLoss/dL
  size_t st;         // [BH, m, m]          sym(dLoss/dX_T)
  size_t total;
};

// Launch geometry decided once per plan.
struct Geometry {
  int s, m, d, n;          // landmark grid side, landmarks, head dim, tokens per head
  long bh;                 // batch * heads
  int cd_rows;             // tokens per thread in the distance kernel
  int cd_tile;             // tokens per distance chunk = 32 * cd_rows
  bool cd_tma;             // distance kernel fed by TMA (cdist_tma.cuh), else by cp.async
  bool cd_l1;              // the TMA-fed kernel with the split FP32/ALU element arithmetic
                           // (cdist_l1.cuh); excludes cd_tma
  int cd_groups;           // split-pipe kernel: row groups per CTA (1: two CTAs per SM, 2: one)
  bool cd_gtc;             // Gaussian kernel with the cross term on the tensor cores
                           // (cdist_gauss_tc.cu); excludes cd_tma and cd_l1
  int cd_threads;          // threads of a distance-kernel CTA
  Partition cd_part;       // balanced split over cd_part.ctas persistent CTAs
  int bv_splits;           // B V: CTAs per head
  int stat_ctas;           // column-statistics CTAs appended to the B V grid (0: no whitening)
  int bv_tiles_per_split;  // B V: 64-token chunks per CTA
  int bv_threads;
  size_t bv_smem;
  bool bv_tc;              // B V on the tensor cores (bv_tc.cu), after a launch of the
                           // statistics CTAs alone (stat_ctas of stat_threads threads)
  int stat_threads;
  bool stats_beside;       // the statistics launch runs on a stream of its own beside the
                           // tensor-core B V (the distance chain on the launching stream)
  int bv_raw_stages;       // tensor-core B V: raw copy stages (as many as fit, <= 12)
  bool out_tc;             // O = A^ M on the tensor cores (out_tc.cu)
  bool out_tma;            // ... with its rows written by TMA tensor stores
  int out_ahead;           // ... and A^T tiles prefetched into L2 this far ahead (0: off)
  size_t fin_smem;
  size_t cd_smem;          // dynamic shared memory of the distance kernel
  int out_tile;            // tokens per output-kernel CTA
  int out_threads;
  size_t out_smem;
  size_t ns_smem;
  int ns_cluster;          // Newton-Schulz CTAs per head (a cluster of 1 or 2)
  bool ns_tc;              // Newton-Schulz products on the tensor cores (ns_tc.cu)
  bool ns_exclusive;       // Newton-Schulz CTAs own their SMs (few heads)
  bool cg;                 // conjugate-gradient solver (cg.cu) instead of Newton-Schulz
  size_t cg_smem;
  size_t pool_threads;
  int ahat_splits;         // backward dA^ / dM partials: CTAs per head
  int ahat_tiles_per_split;  // backward dA^ / dM partials: 128-token chunks per CTA
  int lm_splits;           // backward dL partials: CTAs per (head, side)
  int lm_tiles_per_split;  // backward dL partials: 128-token chunks per CTA
};

// Timing marks of one forward (events recorded when timing is on).
enum Mark {
  kMarkStart, kMarkPoolDone, kMarkNsStart, kMarkNsDone, kMarkCdistStart, kMarkCdistDone,
  kMarkBvDone, kMarkMixDone, kMarkOutputDone, kMarks
};

}  // namespace lapl

struct lapl_attn_plan {
  lapl_attn_config cfg;
  lapl::Geometry geo;
  lapl::WorkspaceLayout ws;
  int device;
  int num_sms;
  float neg_log2e_over_lambda;  // exp(-D/lambda) == exp2(D * this)
  cudaStream_t side_stream;     // runs the shorter of the two chains of a forward
  cudaEvent_t ev_pool, ev_join;   // pooling done; side-stream chain done
  cudaStream_t stat_stream;     // the column statistics beside the tensor-core B V
  cudaEvent_t ev_cdist, ev_stats;   // distances done; statistics done
  bool timing;                  // record stage events in forward
  bool timed_once;              // a forward ran with timing on
  cudaEvent_t ev_stage[lapl::kMarks];   // indexed by lapl::Mark
  unsigned* dev_err;            // the library's device error word on this device
  // Tensor maps of Q and K for the TMA-fed distance kernel, re-encoded when the pointers change.
  mutable CUtensorMap tmap_q, tmap_k;
  mutable const void* tmap_q_ptr;
  mutable const void* tmap_k_ptr;
  // Tensor maps of B^T and V for the tensor-core B V kernel, re-encoded when the pointers change.
  mutable CUtensorMap tmap_bt, tmap_v;
  mutable const void* tmap_bt_ptr;
  mutable const void* tmap_v_ptr;
  // Tensor maps of A^T and B^T for the tensor stores of the Gaussian tensor-core distance
  // kernel, re-encoded when the pointers change.
  mutable CUtensorMap tmap_at_st, tmap_bt_st;
  // Tensor map of O for the tensor stores of the tensor-core output kernel.
  mutable CUtensorMap tmap_o;
  mutable const void* tmap_o_ptr;
  // Tensor map of A^T for the tensor-core output kernel's tile copies and L2 prefetches.
  mutable CUtensorMap tmap_at_pf;
  mutable const void* tmap_at_pf_ptr;
  mutable const void* tmap_at_st_ptr;
  mutable const void* tmap_bt_st_ptr;
  // Fault injection for tests (lapl_attn_set_fault_injection): bound of the barrier waits of
  // the distance kernels and the tensor-core chain kernels, and which kernel skips each CTA's
  // last copy (0 none, 1 the distance kernel, 2 the tensor-core output kernel, 3 the
  // tensor-core B V kernel).
  unsigned long long cd_wait_ns;
  int cd_skip_last_copy;
  // lapl_attn_forward_host: two half-batch plans (first ceil(B/2), then floor(B/2) batches; null
  // when it runs one forward), the stream the second half runs on, and its fork and join events.
  lapl_attn_plan* half[2];
  cudaStream_t pipe_stream;
  cudaEvent_t ev_pipe_start, ev_pipe_join;
  char last_error[256];
};

namespace lapl {

// Kernel launchers, one per translation unit.  Each returns the launch's cudaError_t.
cudaError_t launch_pool(const lapl_attn_plan& p, const void* k, float* landmarks,
                        float* dbg_landmarks, cudaStream_t st);
cudaError_t launch_ns(const lapl_attn_plan& p, const float* landmarks, float* x, float* dbg_dll,
                      float* dbg_w, float* dbg_x, float* xs, cudaStream_t st);
cudaError_t launch_cdist(const lapl_attn_plan& p, const void* q, const void* k, const void* v,
                         const float* landmarks, float* at, float* bt, float* dbg_dql,
                         float* dbg_dlk, float* dbg_a, cudaStream_t st);
cudaError_t launch_bv(const lapl_attn_plan& p, const float* bt, const void* v, float* bvp,
                      const float* at, float* mu, float* rstd, float* dbg_mu, float* dbg_rstd,
                      cudaStream_t st);
cudaError_t launch_mix(const lapl_attn_plan& p, const float* x, const float* bvp, float* mmat,
                       float* bv_keep, float* dbg_bv, float* dbg_m, cudaStream_t st);
cudaError_t launch_output(const lapl_attn_plan& p, const float* at, const float* mmat,
                          const float* mu, const float* rstd, const float* bias, void* out,
                          cudaStream_t st);

// 2-D tensor map, no swizzle, rows past the extent read as zero: `inner` elements per row
// (contiguous), `outer` rows `row_bytes` apart, boxes of box_inner x box_outer.  False if the
// driver's encoder is unavailable or rejects the map.
bool tma_encode_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t inner,
                   uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);

// 3-D tensor map with 128-byte swizzle, for tensor stores: dims d0 (contiguous) x d1 x d2,
// strides s1 and s2 bytes, boxes of b0 x b1 x 1.
bool tma_encode_3d_sw128(CUtensorMap* map, const void* base, CUtensorMapDataType dtype,
                         uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2,
                         uint32_t b0, uint32_t b1);
// Distance kernel choice for a plan: sets geo.cd_tma, cd_tile, cd_rows, cd_threads and cd_smem,
// opts in to the shared memory and returns the resident CTAs per SM.
cudaError_t cdist_plan(lapl_attn_plan& p, int* ctas_per_sm);
// Address of the library's device error word: one bit per kernel whose bounded wait gave up
// (kErrBitCdist, kErrBitSolve).
cudaError_t device_error_word(unsigned** word);
// Shared-memory sizes, needed at plan time to size grids and opt in to > 48 KB.
size_t ns_smem_bytes(int m, int d);
bool ns_cluster_supported(int s, int cluster);
// Sets the shared-memory attribute; with clusters_per_gpu, also how many clusters of the
// kernel can be resident at once.
cudaError_t ns_configure(int s, int cluster, size_t smem, int* clusters_per_gpu);
size_t ns_tc_smem_bytes(int d);
cudaError_t ns_tc_configure(int s, size_t smem);
cudaError_t launch_ns_tc(const lapl_attn_plan& p, const float* landmarks, float* x,
                         float* dbg_dll, float* dbg_w, float* dbg_x, float* xs, cudaStream_t st);
size_t output_smem_bytes(int m, int d, int tile);
cudaError_t output_configure(size_t smem);
size_t bv_smem_bytes(int m, int d, int threads, bool bf16);
int bv_threads(int m, int d);
int bv_tile_tokens();
cudaError_t bv_configure(size_t smem);
int bv_occupancy(int threads, size_t smem);   // resident B V CTAs per SM
// B V on the tensor cores (bv_tc.cu).
int bv_tc_threads();
int bv_tc_tile_tokens();
int bv_tc_raw_stages(int d, bool bf16, size_t smem_limit);
size_t bv_tc_smem_bytes(int d, bool bf16, int nraw);
cudaError_t bv_tc_configure(size_t smem);
int bv_tc_occupancy(size_t smem, bool bf16);
// pdl: launched as the programmatic dependent of the statistics launch just before it.
cudaError_t launch_bv_tc(const lapl_attn_plan& p, const float* bt, const void* v, float* bvp,
                         cudaStream_t st, bool pdl);
// O = A^ M on the tensor cores (out_tc.cu); tma_store: O rows written by TMA tensor stores
// (fp32 O with d = 32 or 64, bf16 O with d = 64: out_tc_tma_store).
size_t out_tc_smem_bytes(int m, int d, bool tma_store, bool out_bf16);
bool out_tc_tma_store(int d, bool out_bf16);
int out_tc_threads();
cudaError_t out_tc_configure(size_t smem);
cudaError_t launch_output_tc(const lapl_attn_plan& p, const float* at, const float* mmat,
                             const float* mu, const float* rstd, const float* bias, void* out,
                             cudaStream_t st);
// Gaussian-kernel distances with the cross term on the tensor cores (cdist_gauss_tc.cu):
// fp32 or bf16 inputs with d in {32, 64}, m <= 64.  smem 0 (and kernel_ptr null) where there is
// no instantiation.
size_t gauss_tc_smem_bytes(int m, int d, bool bf16);
int gauss_tc_threads();
const void* gauss_tc_kernel_ptr(int d, bool bf16);
cudaError_t launch_gauss_tc(const lapl_attn_plan& p, const void* q, const void* k,
                            const float* landmarks, float* at, float* bt, float* dbg_dql,
                            float* dbg_dlk, float* dbg_a, cudaStream_t st);
// Column statistics of A as a launch of their own (with the tensor-core B V).
cudaError_t launch_col_stats(const lapl_attn_plan& p, const float* at, float* mu, float* rstd,
                             float* dbg_mu, float* dbg_rstd, cudaStream_t st);
size_t mix_smem_bytes(int m, int bv_splits);
cudaError_t mix_configure(size_t smem);
// Backward pass (backward.cu).
BwdLayout bwd_layout(const lapl_attn_plan& p);
cudaError_t bwd_configure(lapl_attn_plan& p);
cudaError_t launch_backward(const lapl_attn_plan& p, const void* q, const void* k, const void* v,
                            const float* bias, const float* gout, float* dq, float* dk,
                            float* dv, float* dbias, const char* fws, char* bws,
                            cudaStream_t st);
// Conjugate-gradient solver: M = T CG iterations on W M = B V (replaces Newton-Schulz + mix).
size_t cg_smem_bytes(int m, int d);
cudaError_t cg_configure(int s, int d, size_t smem);
cudaError_t launch_cg(const lapl_attn_plan& p, const float* landmarks, const float* bvp,
                      float* mmat, float* dbg_dll, float* dbg_w, float* dbg_bv, float* dbg_m,
                      cudaStream_t st);

// ---- device helpers ---------------------------------------------------------------------
__device__ __forceinline__ float laplacian_from_distance(float dist, float neg_log2e_over_lambda) {
  // exp(-dist/lambda) = 2^(dist * (-log2(e)/lambda)), with the hardware base-2 exponential
  // (relative error of a few ulp; results below 2^-126 flush to zero).
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(dist * neg_log2e_over_lambda));
  return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t two) { return __uint_as_float(two << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t two) { return __uint_as_float(two & 0xffff0000u); }

}  // namespace lapl
