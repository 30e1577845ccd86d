// api.cu -- the C ABI (include/lapl_attn.h): validation, plan, workspace layout, and the
// stream-ordered launch sequence of one forward pass.
//
// When the solve is the longer chain and needs few SMs (B*H <= SMs/4; the solve's CTAs then
// get SMs of their own):
//   launching stream                               side stream
//   K1 pool      L = avg-pool(K)
//   fork (L) -------------------------------------> K2 cdist  A^T + run statistics, B^T
//   K3 solve     W, X (Newton-Schulz)               K2b bv    B V partials per token split
//   join <----------------------------------------- done (long before the solve)
//   K4 mix       B V = sum of partials, M = X (B V)
//   K5 output    column statistics, O = whiten(A) M
// The solve follows pooling on the same stream, so its CTAs are placed the moment pooling
// ends; the distance kernel takes the SMs that are left.
//
// Otherwise the distance kernel is the longest chain: K1 pool, K2 cdist and K2b bv run on the
// launching stream and the solve on the side stream, joined before K4.
//
// K5 is a programmatic dependent launch of K4: it merges the column statistics and loads and
// whitens its A tile while M is computed.
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <new>

#include "common.cuh"

namespace lapl {

int output_tile_tokens(int d, long bh, int n, int num_sms);

namespace {

int isqrt_exact(int m) {
  for (int s = 1; s * s <= m; ++s)
    if (s * s == m) return s;
  return -1;
}

lapl_status validate(const lapl_attn_config* c) {
  if (!c) return LAPL_ERR_INVALID_ARG;
  if (c->batch < 0 || c->heads < 1 || c->grid_h < 1 || c->grid_w < 1) return LAPL_ERR_INVALID_ARG;
  if (c->head_dim < 1 || c->num_landmarks < 1) return LAPL_ERR_INVALID_ARG;
  if (!(c->lambda > 0.f) || !isfinite(c->lambda)) return LAPL_ERR_INVALID_ARG;
  if (!(c->eps >= 0.f) || !isfinite(c->eps)) return LAPL_ERR_INVALID_ARG;
  if (c->whiten != 0 && c->whiten != 1) return LAPL_ERR_INVALID_ARG;
  if (c->whiten && (!(c->delta > 0.f) || !isfinite(c->delta))) return LAPL_ERR_INVALID_ARG;
  if (c->ns_steps < 0 || c->ns_steps > 1000) return LAPL_ERR_INVALID_ARG;
  if ((c->in_dtype != LAPL_F32 && c->in_dtype != LAPL_BF16) ||
      (c->out_dtype != LAPL_F32 && c->out_dtype != LAPL_BF16))
    return LAPL_ERR_INVALID_ARG;
  if (c->kernel != LAPL_KERNEL_LAPLACIAN && c->kernel != LAPL_KERNEL_GAUSSIAN)
    return LAPL_ERR_INVALID_ARG;
  if (c->solver != LAPL_SOLVER_NEWTON_SCHULZ && c->solver != LAPL_SOLVER_CG)
    return LAPL_ERR_INVALID_ARG;
  const int s = isqrt_exact(c->num_landmarks);
  if (s < 0 || s > kMaxS) return LAPL_ERR_UNSUPPORTED;
  if (c->grid_h % s != 0 || c->grid_w % s != 0) return LAPL_ERR_UNSUPPORTED;
  if (c->head_dim % 8 != 0 || c->head_dim > kMaxD) return LAPL_ERR_UNSUPPORTED;
  const long long n = (long long)c->grid_h * c->grid_w;
  if (n > (1LL << 24)) return LAPL_ERR_UNSUPPORTED;
  if ((long long)c->batch * c->heads > (1LL << 24)) return LAPL_ERR_UNSUPPORTED;
  if ((long long)c->batch * c->heads * n > (1LL << 40)) return LAPL_ERR_UNSUPPORTED;
  return LAPL_OK;
}

void set_error(lapl_attn_plan* p, cudaError_t e, const char* where) {
  snprintf(p->last_error, sizeof(p->last_error), "%s: %s (%s)", where, cudaGetErrorName(e),
           cudaGetErrorString(e));
}

bool aligned16(const void* ptr) { return ((uintptr_t)ptr & 15u) == 0; }

size_t elem_bytes(int dtype) { return dtype == LAPL_BF16 ? 2 : 4; }

// Split of the distance kernel over `ctas` persistent CTAs (see Partition).
void setup_cdist_partition(Geometry& g, int ctas) {
  Partition& pt = g.cd_part;
  pt.uq = (long long)g.bh * g.n;
  pt.total = 2 * pt.uq;
  if (ctas > pt.total) ctas = (int)std::max<long long>(pt.total, 1);
  pt.ctas = ctas;
  pt.q = pt.total / ctas;
  pt.rem = (int)(pt.total % ctas);
}
}  // namespace
}  // namespace lapl

namespace lapl {
namespace {
// A plan for cfg.  force_tps > 0: B V takes force_tps tiles per split (the split count follows),
// in place of the plan's own choice; the host entry point's half-batch plans use this so that
// every slice is reduced in the same order as by the full plan.
lapl_status create_plan(const lapl_attn_config* cfg, lapl_attn_plan** out, int force_tps);
}  // namespace
}  // namespace lapl

using namespace lapl;

extern "C" {

int lapl_attn_version(void) { return 100; }

const char* lapl_attn_status_string(lapl_status s) {
  switch (s) {
    case LAPL_OK: return "LAPL_OK";
    case LAPL_ERR_INVALID_ARG: return "LAPL_ERR_INVALID_ARG";
    case LAPL_ERR_UNSUPPORTED: return "LAPL_ERR_UNSUPPORTED";
    case LAPL_ERR_WORKSPACE: return "LAPL_ERR_WORKSPACE";
    case LAPL_ERR_ALIGNMENT: return "LAPL_ERR_ALIGNMENT";
    case LAPL_ERR_CUDA: return "LAPL_ERR_CUDA";
    case LAPL_ERR_DEVICE_TIMEOUT: return "LAPL_ERR_DEVICE_TIMEOUT";
    case LAPL_ERR_NOT_IMPLEMENTED: return "LAPL_ERR_NOT_IMPLEMENTED";
  }
  return "LAPL_ERR_UNKNOWN";
}

const char* lapl_attn_last_error(lapl_attn_handle h) { return h ? h->last_error : ""; }

lapl_status lapl_attn_create(const lapl_attn_config* cfg, lapl_attn_handle* out) {
  if (!out) return LAPL_ERR_INVALID_ARG;
  *out = nullptr;
  lapl_attn_plan* p = nullptr;
  lapl_status st = create_plan(cfg, &p, 0);
  if (st != LAPL_OK) return st;
  // lapl_attn_forward_host runs two half-batch forwards on two streams, so that the copies of
  // one half overlap the other's kernels and the first half's output leaves while the second
  // computes.  LAPL_ATTN_HOST_SPLIT=0, read here, keeps one forward.
  const char* split_env = getenv("LAPL_ATTN_HOST_SPLIT");
  const bool split = cfg->batch >= 2 && !(split_env && strcmp(split_env, "0") == 0);
  if (split) {
    for (int i = 0; i < 2 && st == LAPL_OK; ++i) {
      lapl_attn_config hc = *cfg;
      hc.batch = i == 0 ? (cfg->batch + 1) / 2 : cfg->batch / 2;
      st = create_plan(&hc, &p->half[i], p->geo.bv_tiles_per_split);
    }
    // The halves must compute every slice with the full plan's kernels (a half too small for a
    // TMA box of rows, for instance, would take another distance kernel): else one forward.
    for (int i = 0; i < 2 && st == LAPL_OK; ++i) {
      const Geometry &a = p->geo, &b = p->half[i]->geo;
      if (a.cd_l1 != b.cd_l1 || a.cd_tma != b.cd_tma || a.cd_gtc != b.cd_gtc ||
          a.cd_groups != b.cd_groups || a.bv_tc != b.bv_tc || a.out_tc != b.out_tc ||
          a.ns_tc != b.ns_tc || a.ns_cluster != b.ns_cluster || a.bv_splits != b.bv_splits) {
        for (int j = 0; j < 2; ++j) {
          lapl_attn_destroy(p->half[j]);
          p->half[j] = nullptr;
        }
        *out = p;
        return LAPL_OK;
      }
    }
    cudaError_t e = cudaSuccess;
    if (st == LAPL_OK) e = cudaStreamCreateWithFlags(&p->pipe_stream, cudaStreamNonBlocking);
    if (st == LAPL_OK && e == cudaSuccess)
      e = cudaEventCreateWithFlags(&p->ev_pipe_start, cudaEventDisableTiming);
    if (st == LAPL_OK && e == cudaSuccess)
      e = cudaEventCreateWithFlags(&p->ev_pipe_join, cudaEventDisableTiming);
    if (st == LAPL_OK && e != cudaSuccess) st = LAPL_ERR_CUDA;
    if (st != LAPL_OK) {
      lapl_attn_destroy(p);
      return st;
    }
  }
  *out = p;
  return LAPL_OK;
}

}  // extern "C"

namespace lapl {
namespace {
lapl_status create_plan(const lapl_attn_config* cfg, lapl_attn_plan** out, int force_tps) {
  if (!out) return LAPL_ERR_INVALID_ARG;
  *out = nullptr;
  lapl_status st = validate(cfg);
  if (st != LAPL_OK) return st;

  lapl_attn_plan* p = new (std::nothrow) lapl_attn_plan();
  if (!p) return LAPL_ERR_INVALID_ARG;
  p->cfg = *cfg;
  p->last_error[0] = '\0';
  p->cd_wait_ns = 1000000000ull;   // one second
  p->cd_skip_last_copy = 0;
  p->neg_log2e_over_lambda = (float)(-1.4426950408889634 / (double)cfg->lambda);

  Geometry& g = p->geo;
  g.s = isqrt_exact(cfg->num_landmarks);
  g.m = cfg->num_landmarks;
  g.d = cfg->head_dim;
  g.n = cfg->grid_h * cfg->grid_w;
  g.bh = (long)cfg->batch * cfg->heads;

  cudaError_t e = cudaGetDevice(&p->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
  if (e != cudaSuccess) {
    set_error(p, e, "create/device");
    delete p;
    return LAPL_ERR_CUDA;
  }

  // Distance kernel: persistent CTAs, one wave of resident CTAs, balanced ranges.
  int per_sm = 1;
  e = device_error_word(&p->dev_err);
  if (e == cudaSuccess) e = cdist_plan(*p, &per_sm);
  g.cg = cfg->solver == LAPL_SOLVER_CG;
  if (e == cudaSuccess && g.cg) {
    // Conjugate gradient: one kernel after B V, on the launching stream; no Newton-Schulz.
    g.ns_cluster = 1;
    g.ns_tc = false;
    g.ns_exclusive = false;
    g.cg_smem = cg_smem_bytes(g.m, g.d);
    e = cg_configure(g.s, g.d, g.cg_smem);
  } else if (e == cudaSuccess) {
    // Newton-Schulz is the longest dependency chain of the forward.  Kernels: "tc" (one CTA per
    // head, products on the tensor cores; the default for m >= 25), "ffma" (one CTA per head,
    // CUDA-core products; the default for m <= 16) and "pair" (a cluster of two CTAs per head
    // that split every CUDA-core product; m > 32).  LAPL_ATTN_NS_KERNEL, read here, picks one.
    const char* nk = getenv("LAPL_ATTN_NS_KERNEL");
    g.ns_cluster = 1;
    g.ns_tc = g.s >= 5;
    if (nk && strcmp(nk, "ffma") == 0) g.ns_tc = false;
    if (nk && strcmp(nk, "pair") == 0 && ns_cluster_supported(g.s, 2)) {
      g.ns_cluster = 2;
      g.ns_tc = false;
    }
    if (nk && strcmp(nk, "tc") == 0) g.ns_tc = true;
    // The solve goes first, on SMs of its own (its CTAs ask for almost a whole SM's shared
    // memory, so no other kernel's CTA shares their SM), when it uses few SMs and is the
    // longer of the two chains after pooling.  Chain estimates, from GB300 measurements: the
    // solve about 15 us + 2.2 us per step (4 us on the CUDA cores); the distance and B V
    // kernels about 6e6 (token, landmark, channel) elements per us.
    const double ns_us = 15.0 + (g.ns_tc ? 2.2 : 4.0) * cfg->ns_steps;
    const double cd_us = 2.0 * (double)g.bh * g.n * g.m * g.d / 6e6;
    g.ns_exclusive = g.bh * g.ns_cluster <= p->num_sms / 4 && ns_us >= cd_us;
    int smem_max = 0;
    e = cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, p->device);
    g.ns_smem = g.ns_tc ? ns_tc_smem_bytes(g.d) : ns_smem_bytes(g.m, g.d);
    if (e == cudaSuccess && g.ns_exclusive && (size_t)smem_max > g.ns_smem) g.ns_smem = smem_max;
    if (e == cudaSuccess && g.ns_tc) {
      e = ns_tc_configure(g.s, g.ns_smem);
    } else if (e == cudaSuccess && g.ns_cluster == 2) {
      int clusters = 0;
      e = ns_configure(g.s, 2, g.ns_smem, &clusters);
      if (e != cudaSuccess || clusters < 1) {   // no room for a pair: one CTA per head
        cudaGetLastError();
        g.ns_cluster = 1;
        g.ns_exclusive = g.bh <= p->num_sms / 4;
        e = cudaSuccess;
      }
    }
    if (e == cudaSuccess && !g.ns_tc && g.ns_cluster == 1)
      e = ns_configure(g.s, 1, g.ns_smem, nullptr);
  }
  if (e == cudaSuccess) {
    // O = A^ M on the tensor cores where the shapes allow it (d a multiple of 16 and two
    // accumulators of 2d columns in at most 256 tensor-memory columns; N a multiple of 4 for
    // the A^T rows' tensor map; the operand stages within the shared memory) and where it
    // measured faster: at d = 64 for every sequence length (stage-2/3 shape, N = 784 and 128
    // heads: output 26.6 -> 19.5 us; N = 1024 and 4096 sweeps equal or faster), for smaller d
    // from N = 4096 (stage-1 shape, d = 32 and 2.6 tiles per persistent CTA: 14.3 against
    // 12.5 us for the CUDA-core kernel).  LAPL_ATTN_OUT=cuda or =tc forces either.
    const char* ok_env = getenv("LAPL_ATTN_OUT");
    const bool want_tc = ok_env && strcmp(ok_env, "tc") == 0;
    const bool want_cuda = (ok_env && strcmp(ok_env, "cuda") == 0) ||
                           (!want_tc && g.d < 64 && g.n < 4096);
    int smem_optin = 0;
    if (cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                               p->device) != cudaSuccess)
      smem_optin = 0;
    const bool out_bf16 = cfg->out_dtype == LAPL_BF16;
    g.out_tma = out_tc_tma_store(g.d, out_bf16) && g.bh < (1LL << 31) && g.n < (1LL << 31);
    g.out_tc = !want_cuda && g.d % 16 == 0 && 4 * g.d <= 256 && g.n % 4 == 0 &&
               g.bh * g.m < (1LL << 31) && g.n < (1LL << 31) &&
               out_tc_smem_bytes(g.m, g.d, g.out_tma, out_bf16) <= (size_t)smem_optin;
    if (!g.out_tc) g.out_tma = false;
    if (g.out_tc) {
      // A^T tiles prefetched into L2 beyond the tile being copied: LAPL_ATTN_OUT_AHEAD
      // overrides the distance, 0 turns it off.
      g.out_ahead = 3;
      if (const char* ah = getenv("LAPL_ATTN_OUT_AHEAD"))
        g.out_ahead = std::max(0, std::min(8, atoi(ah)));
      g.out_tile = 128;
      g.out_threads = out_tc_threads();
      g.out_smem = out_tc_smem_bytes(g.m, g.d, g.out_tma, out_bf16);
      e = out_tc_configure(g.out_smem);
    } else {
      g.out_tile = output_tile_tokens(g.d, g.bh, g.n, p->num_sms);
      g.out_threads = 256;
      g.out_smem = output_smem_bytes(g.m, g.d, g.out_tile);
      e = output_configure(g.out_smem);
    }
  }
  if (e != cudaSuccess) {
    set_error(p, e, "create/configure");
    delete p;
    return LAPL_ERR_CUDA;
  }
  if (e == cudaSuccess && !g.cg) e = bwd_configure(*p);
  if (e == cudaSuccess) {
    // B V on the tensor cores where the shapes allow it: the MMA's N (d for bf16 V, 2d for
    // fp32 V) at most 256, and d a multiple of 16 (the accumulator is read 16 columns at a
    // time); LAPL_ATTN_BV=cuda forces the CUDA-core kernel.
    const bool bf16 = cfg->in_dtype == LAPL_BF16;
    const int nb = bf16 ? g.d : 2 * g.d;
    const char* bvk = getenv("LAPL_ATTN_BV");
    // The B^T tensor map needs rows of 16-byte multiples (N % 4 == 0); its boxes are m <= 64
    // rows and the M kernel's reduction order is unchanged.
    // Automatic choice, as measured: d = 64 at every sequence length (stage-2/3 shape, N =
    // 784 and 128 heads: B V stage 69.8 -> 63.5 us; N = 4096 sweeps 20.5 -> 16.4 us; N = 1024
    // equal), smaller d from N = 4096 (stage-1 shape, d = 32 fp32: the CUDA-core kernel 16.4
    // against 19.7 us).  LAPL_ATTN_BV=tc or =cuda forces either.
    const bool want_tc = bvk && strcmp(bvk, "tc") == 0;
    const bool want_cuda = bvk && strcmp(bvk, "cuda") == 0;
    g.bv_tc = g.d % 16 == 0 && nb <= 256 && g.n % 4 == 0 && g.bh * g.n < (1LL << 31) &&
              g.bh * g.m < (1LL << 31) && !want_cuda &&
              (want_tc || g.d >= 64 || g.n >= 4096);
    int smem_optin = 0;
    if (g.bv_tc) {
      if (cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                 p->device) != cudaSuccess)
        smem_optin = 0;
      // As many raw copy stages as fit (bytes in flight per SM); fp32 V with d = 128 leaves
      // room for too few: the CUDA-core kernel then.
      g.bv_raw_stages = bv_tc_raw_stages(g.d, bf16, (size_t)smem_optin);
      if (g.bv_raw_stages == 0) g.bv_tc = false;
    }
    if (g.bv_tc) {
      g.bv_threads = bv_tc_threads();
      g.bv_smem = bv_tc_smem_bytes(g.d, bf16, g.bv_raw_stages);
      e = bv_tc_configure(g.bv_smem);
    } else {
      g.bv_threads = bv_threads(g.m, g.d);
      g.bv_smem = bv_smem_bytes(g.m, g.d, g.bv_threads, bf16);
      e = bv_configure(g.bv_smem);
    }
  }
  if (e != cudaSuccess) {
    set_error(p, e, "create/configure");
    delete p;
    return LAPL_ERR_CUDA;
  }
  if (per_sm < 1) per_sm = 1;
  {
    // Column statistics of A: one warp per landmark column, placed before the B V CTAs in
    // their grid.
    // With the tensor-core B V they are a launch of their own, 256 threads each.
    g.stat_threads = g.bv_tc ? 256 : g.bv_threads;
    const int warps = g.stat_threads / 32;
    g.stat_ctas = cfg->whiten ? (int)(g.bh * ((g.m + warps - 1) / warps)) : 0;
    const long long stat_in_grid = g.bv_tc ? 0 : g.stat_ctas;
    // B V: whole 64-token chunks per CTA, on the SMs the solve leaves free (it keeps its own
    // when ns_exclusive).  The kernel's time is about the waves of resident CTAs (statistics
    // CTAs counted as B V CTAs) times the chunks of one CTA plus one for its prologue and
    // partial store: pick the split count that minimises it, the fewest CTAs among equals.  At
    // most kMaxBvSplits CTAs per head: the M kernel stages every split's partial of its 8
    // columns in shared memory (64 splits at m = 64: 146 KB).
    constexpr int kMaxBvSplits = 64;
    const long long bh1 = g.bh > 0 ? g.bh : 1;
    const int tile_tokens = g.bv_tc ? bv_tc_tile_tokens() : bv_tile_tokens();
    const int tiles = std::max(1, (g.n + tile_tokens - 1) / tile_tokens);
    long long sms = p->num_sms;
    if (g.ns_exclusive) sms -= g.bh * g.ns_cluster;
    const int occ = g.bv_tc ? bv_tc_occupancy(g.bv_smem, cfg->in_dtype == LAPL_BF16)
                            : bv_occupancy(g.bv_threads, g.bv_smem);
    const long long slots = std::max<long long>(sms, 1) * occ;
    long long best = -1;
    // The tensor-core kernel streams its tiles through a pipeline whose start-up and epilogue
    // cost several tiles: one wave of as few CTAs as fill the SMs.
    const int startup = g.bv_tc ? 8 : 1;
    for (int want = 1; want <= std::min(tiles, kMaxBvSplits); ++want) {
      const int tps = (tiles + want - 1) / want, splits = (tiles + tps - 1) / tps;
      const long long waves = (bh1 * splits + stat_in_grid + slots - 1) / slots;
      const long long cost = waves * (tps + startup);
      if (best < 0 || cost < best) {
        best = cost;
        g.bv_tiles_per_split = tps;
        g.bv_splits = splits;
      }
    }
    if (force_tps > 0) {
      g.bv_tiles_per_split = force_tps;
      g.bv_splits = (tiles + force_tps - 1) / force_tps;
    }
  }
  {
    // No more CTAs than chunks of work.
    const long long chunks = 2LL * (g.bh > 0 ? g.bh : 1) * ((g.n + g.cd_tile - 1) / g.cd_tile);
    // When the Newton-Schulz solve needs few SMs (one CTA per head, at most a quarter of the
    // SMs), it gets those SMs to itself: the distance kernel's persistent grid covers the
    // others (see ns_exclusive).
    long long slots = (long long)p->num_sms * per_sm;
    if (g.ns_exclusive) slots -= g.bh * g.ns_cluster * per_sm;
    const long long ctas = std::min<long long>(slots, chunks);
    setup_cdist_partition(g, (int)std::max<long long>(ctas, 1));
    g.fin_smem = mix_smem_bytes(g.m, g.bv_splits);
    e = mix_configure(g.fin_smem);
    if (e != cudaSuccess) {
      set_error(p, e, "create/configure-finish");
      delete p;
      return LAPL_ERR_CUDA;
    }
  }

  // Workspace regions.
  WorkspaceLayout& w = p->ws;
  const size_t bh = (size_t)g.bh, m = g.m, d = g.d, n = g.n;
  size_t off = 0;
  auto take = [&](size_t floats) {
    const size_t at = off;
    off = align_up(off + floats * sizeof(float), kAlign);
    return at;
  };
  w.landmarks = take(bh * m * d);
  w.x = take(bh * m * m);
  w.at = take(bh * m * n);
  w.bt = take(bh * m * n);
  w.bvp = take(bh * g.bv_splits * m * d);
  w.mmat = take(bh * m * d);
  w.mu = take(bh * m);
  w.rstd = take(bh * m);
  w.fwd_total = off;
  // Written only by lapl_attn_forward_train, read only by the backward pass.
  w.xs = take(g.cg ? 0 : bh * ((size_t)cfg->ns_steps + 1) * m * ((m + 3) & ~(size_t)3));
  w.bv = take(g.cg ? 0 : bh * m * d);
  w.total = off;

  // The column statistics (an HBM-bound read of A^T that only the output kernel needs) run on
  // a stream of their own beside the tensor-core B V, whose converters leave HBM bandwidth to
  // spare, when the distance chain is on the launching stream and B V takes more than one
  // wave of CTAs; otherwise they precede B V on its stream.  Measured both ways: the
  // high-resolution shape (B V in two waves) 527.7 -> 513.5 us per forward; one-wave shapes
  // lose 1-6 us (the N = 65536 sweeps, the stage-2/3 shape), the statistics CTAs taking issue
  // slots from B V's converters for its whole duration.  LAPL_ATTN_STATS_BESIDE=1 / =0 forces
  // either.
  {
    const char* sb = getenv("LAPL_ATTN_STATS_BESIDE");
    const bool can = g.bv_tc && g.stat_ctas > 0 && !g.ns_exclusive && !g.cg;
    const bool auto_on = g.bh * g.bv_splits > (long long)p->num_sms;
    g.stats_beside = can && (sb ? strcmp(sb, "1") == 0 : auto_on);
  }

  // The side stream runs the shorter of the two chains (see the launch sequence).
  e = cudaStreamCreateWithFlags(&p->side_stream, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_join, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_pool, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->stat_stream, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_cdist, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_stats, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    set_error(p, e, "create/stream");
    if (p->side_stream) cudaStreamDestroy(p->side_stream);
    if (p->ev_join) cudaEventDestroy(p->ev_join);
    if (p->ev_pool) cudaEventDestroy(p->ev_pool);
    if (p->stat_stream) cudaStreamDestroy(p->stat_stream);
    if (p->ev_cdist) cudaEventDestroy(p->ev_cdist);
    if (p->ev_stats) cudaEventDestroy(p->ev_stats);
    delete p;
    return LAPL_ERR_CUDA;
  }
  *out = p;
  return LAPL_OK;
}
}  // namespace
}  // namespace lapl

extern "C" {

lapl_status lapl_attn_workspace_size(lapl_attn_handle h, size_t* bytes) {
  if (!h || !bytes) return LAPL_ERR_INVALID_ARG;
  *bytes = h->ws.total;
  return LAPL_OK;
}

// min_workspace: the workspace size the caller must provide (0: lapl_attn_workspace_size).
static lapl_status run_forward(lapl_attn_handle p, const void* q, const void* k, const void* v,
                               const float* bias, void* out, void* workspace,
                               size_t workspace_bytes, cudaStream_t st,
                               const lapl_attn_debug* dbg, bool keep = false,
                               size_t min_workspace = 0) {
  if (!p) return LAPL_ERR_INVALID_ARG;
  if (p->geo.bh == 0) return LAPL_OK;   // empty batch
  if (!q || !k || !v || !out || !workspace) return LAPL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      !aligned16(workspace) || (bias && ((uintptr_t)bias & 3u)))
    return LAPL_ERR_ALIGNMENT;
  if (keep || min_workspace == 0) min_workspace = p->ws.total;
  if (workspace_bytes < min_workspace) return LAPL_ERR_WORKSPACE;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_error(p, e, "forward/device");
    return LAPL_ERR_CUDA;
  }
  if (dev != p->device) return LAPL_ERR_INVALID_ARG;

  char* ws = static_cast<char*>(workspace);
  float* L = reinterpret_cast<float*>(ws + p->ws.landmarks);
  float* X = reinterpret_cast<float*>(ws + p->ws.x);
  // The Newton-Schulz iterates, kept only for a backward pass.
  float* Xs = keep ? reinterpret_cast<float*>(ws + p->ws.xs) : nullptr;
  float* At = reinterpret_cast<float*>(ws + p->ws.at);
  float* Bt = reinterpret_cast<float*>(ws + p->ws.bt);
  float* mu = reinterpret_cast<float*>(ws + p->ws.mu);
  float* rstd = reinterpret_cast<float*>(ws + p->ws.rstd);
  float* bvp = reinterpret_cast<float*>(ws + p->ws.bvp);

  float* M = reinterpret_cast<float*>(ws + p->ws.mmat);

  const lapl_attn_debug none = {};
  const lapl_attn_debug& D = dbg ? *dbg : none;

#define LAPL_TRY(call, where)        \
  do {                               \
    cudaError_t err_ = (call);       \
    if (err_ != cudaSuccess) {       \
      set_error(p, err_, where);     \
      return LAPL_ERR_CUDA;          \
    }                                \
  } while (0)

  const bool tm = p->timing;
#define LAPL_MARK(i, s)                                              \
  if (tm) LAPL_TRY(cudaEventRecord(p->ev_stage[i], s), "forward/timing")

  cudaStream_t side = p->side_stream;
  auto launch_solve = [&](cudaStream_t s) {
    return p->geo.ns_tc ? launch_ns_tc(*p, L, X, D.d_ll, D.w, D.x, Xs, s)
                        : launch_ns(*p, L, X, D.d_ll, D.w, D.x, Xs, s);
  };
  LAPL_MARK(kMarkStart, st);
  if (p->geo.cg) {
    // Conjugate gradient: pooling -> distances -> B V -> CG (which builds W itself) -> output,
    // all on the launching stream; the CG kernel is a programmatic dependent of the B V kernel
    // and the output kernel of the CG kernel.  The solve marks are recorded back to back.
    LAPL_TRY(launch_pool(*p, k, L, D.landmarks, st), "forward/pool");
    LAPL_MARK(kMarkPoolDone, st);
    LAPL_MARK(kMarkNsStart, st);
    LAPL_MARK(kMarkNsDone, st);
    LAPL_MARK(kMarkCdistStart, st);
    LAPL_TRY(launch_cdist(*p, q, k, v, L, At, Bt, D.d_ql, D.d_lk, D.a, st), "forward/cdist");
    LAPL_MARK(kMarkCdistDone, st);
    LAPL_TRY(launch_bv(*p, Bt, v, bvp, At, mu, rstd, D.mu, D.rstd, st), "forward/bv");
    LAPL_MARK(kMarkBvDone, st);
    LAPL_TRY(launch_cg(*p, L, bvp, M, D.d_ll, D.w, D.bv, D.m, st), "forward/cg");
    LAPL_MARK(kMarkMixDone, st);
    LAPL_TRY(launch_output(*p, At, M, mu, rstd, bias, out, st), "forward/output");
    LAPL_MARK(kMarkOutputDone, st);
    if (tm) p->timed_once = true;
    return LAPL_OK;
  }
  if (p->geo.ns_exclusive) {
    // The solve is the longest chain: pooling -> solve -> M -> output on the launching stream;
    // the solve's CTAs are placed the moment pooling ends.  The distance kernel and
    // B V run next to it on the side stream, which is done long before the solve.
    LAPL_TRY(launch_pool(*p, k, L, D.landmarks, st), "forward/pool");
    LAPL_MARK(kMarkPoolDone, st);
    LAPL_TRY(cudaEventRecord(p->ev_pool, st), "forward/pooled");
    LAPL_MARK(kMarkNsStart, st);
    LAPL_TRY(launch_solve(st), "forward/newton-schulz");
    LAPL_MARK(kMarkNsDone, st);
    LAPL_TRY(cudaStreamWaitEvent(side, p->ev_pool, 0), "forward/pooled-wait");
    LAPL_MARK(kMarkCdistStart, side);
    LAPL_TRY(launch_cdist(*p, q, k, v, L, At, Bt, D.d_ql, D.d_lk, D.a, side),
             "forward/cdist");
    LAPL_MARK(kMarkCdistDone, side);
    LAPL_TRY(launch_bv(*p, Bt, v, bvp, At, mu, rstd, D.mu, D.rstd, side), "forward/bv");
    LAPL_MARK(kMarkBvDone, side);
    LAPL_TRY(cudaEventRecord(p->ev_join, side), "forward/join");
  } else {
    // Pooling -> distances -> B V is the longest chain and runs on the launching stream; the
    // solve runs next to it on the side stream.
    LAPL_TRY(launch_pool(*p, k, L, D.landmarks, st), "forward/pool");
    LAPL_MARK(kMarkPoolDone, st);
    LAPL_TRY(cudaEventRecord(p->ev_pool, st), "forward/pooled");
    LAPL_TRY(cudaStreamWaitEvent(side, p->ev_pool, 0), "forward/pooled-wait");
    LAPL_MARK(kMarkNsStart, side);
    LAPL_TRY(launch_solve(side), "forward/newton-schulz");
    LAPL_MARK(kMarkNsDone, side);
    LAPL_TRY(cudaEventRecord(p->ev_join, side), "forward/join");
    LAPL_MARK(kMarkCdistStart, st);
    LAPL_TRY(launch_cdist(*p, q, k, v, L, At, Bt, D.d_ql, D.d_lk, D.a, st),
             "forward/cdist");
    LAPL_MARK(kMarkCdistDone, st);
    if (p->geo.stats_beside) {
      // B V is launched first, so that its CTAs (one per SM, most of the shared memory) are
      // placed before the statistics CTAs take the remaining thread slots.
      LAPL_TRY(cudaEventRecord(p->ev_cdist, st), "forward/distances");
      LAPL_TRY(launch_bv_tc(*p, Bt, v, bvp, st, false), "forward/bv");
      LAPL_TRY(cudaStreamWaitEvent(p->stat_stream, p->ev_cdist, 0), "forward/distances-wait");
      LAPL_TRY(launch_col_stats(*p, At, mu, rstd, D.mu, D.rstd, p->stat_stream),
               "forward/statistics");
      LAPL_TRY(cudaEventRecord(p->ev_stats, p->stat_stream), "forward/statistics-done");
      LAPL_TRY(cudaStreamWaitEvent(st, p->ev_stats, 0), "forward/statistics-wait");
    } else {
      LAPL_TRY(launch_bv(*p, Bt, v, bvp, At, mu, rstd, D.mu, D.rstd, st), "forward/bv");
    }
    LAPL_MARK(kMarkBvDone, st);
  }
  LAPL_TRY(cudaStreamWaitEvent(st, p->ev_join, 0), "forward/join-wait");
  float* bv_keep = keep ? reinterpret_cast<float*>(ws + p->ws.bv) : nullptr;
  LAPL_TRY(launch_mix(*p, X, bvp, M, bv_keep, D.bv, D.m, st), "forward/mix");
  LAPL_MARK(kMarkMixDone, st);
  LAPL_TRY(launch_output(*p, At, M, mu, rstd, bias, out, st), "forward/output");
  LAPL_MARK(kMarkOutputDone, st);
  if (tm) p->timed_once = true;
#undef LAPL_MARK
#undef LAPL_TRY
  return LAPL_OK;
}

lapl_status lapl_attn_backward_workspace_size(lapl_attn_handle h, size_t* bytes) {
  if (!h || !bytes) return LAPL_ERR_INVALID_ARG;
  if (h->geo.cg) return LAPL_ERR_UNSUPPORTED;
  *bytes = bwd_layout(*h).total;
  return LAPL_OK;
}

lapl_status lapl_attn_backward(lapl_attn_handle h, const void* q, const void* k, const void* v,
                               const float* bias, const float* dout, float* dq, float* dk,
                               float* dv, float* dbias, const void* fwd_workspace,
                               size_t fwd_workspace_bytes, void* bwd_workspace,
                               size_t bwd_workspace_bytes, void* stream) {
  if (!h) return LAPL_ERR_INVALID_ARG;
  if (h->geo.cg) return LAPL_ERR_UNSUPPORTED;
  if (h->geo.bh == 0) return LAPL_OK;
  if (!q || !k || !v || !dout || !dq || !dk || !dv || !fwd_workspace || !bwd_workspace)
    return LAPL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || !aligned16(fwd_workspace) ||
      !aligned16(bwd_workspace) || (bias && ((uintptr_t)bias & 3u)) ||
      (dbias && ((uintptr_t)dbias & 3u)))
    return LAPL_ERR_ALIGNMENT;
  if (fwd_workspace_bytes < h->ws.total || bwd_workspace_bytes < bwd_layout(*h).total)
    return LAPL_ERR_WORKSPACE;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_error(h, e, "backward/device");
    return LAPL_ERR_CUDA;
  }
  if (dev != h->device) return LAPL_ERR_INVALID_ARG;
  e = launch_backward(*h, q, k, v, bias, dout, dq, dk, dv, dbias,
                      static_cast<const char*>(fwd_workspace), static_cast<char*>(bwd_workspace),
                      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    set_error(h, e, "backward");
    return LAPL_ERR_CUDA;
  }
  return LAPL_OK;
}

int lapl_attn_backward_kernels(lapl_attn_handle h) {
  return (h && h->geo.bh > 0 && !h->geo.cg) ? 8 : 0;
}

lapl_status lapl_attn_forward(lapl_attn_handle h, const void* q, const void* k, const void* v,
                              const float* bias, void* out, void* workspace,
                              size_t workspace_bytes, void* stream) {
  return run_forward(h, q, k, v, bias, out, workspace, workspace_bytes,
                     static_cast<cudaStream_t>(stream), nullptr);
}

lapl_status lapl_attn_forward_train(lapl_attn_handle h, const void* q, const void* k,
                                    const void* v, const float* bias, void* out,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  if (h && h->geo.cg) return LAPL_ERR_UNSUPPORTED;
  return run_forward(h, q, k, v, bias, out, workspace, workspace_bytes,
                     static_cast<cudaStream_t>(stream), nullptr, true);
}

lapl_status lapl_attn_forward_debug(lapl_attn_handle h, const void* q, const void* k,
                                    const void* v, const float* bias, void* out,
                                    void* workspace, size_t workspace_bytes, void* stream,
                                    const lapl_attn_debug* dbg) {
  if (!dbg) return LAPL_ERR_INVALID_ARG;
  return run_forward(h, q, k, v, bias, out, workspace, workspace_bytes,
                     static_cast<cudaStream_t>(stream), dbg);
}

namespace {
struct StagingLayout {
  size_t q, k, v, out, bias, ws, total;
};

StagingLayout staging_layout(const lapl_attn_plan* p);

// Bytes of the host entry point's staging buffer: one forward's inputs, output and workspace,
// or, with half-batch plans, the two halves' regions one after the other.
size_t staging_bytes(const lapl_attn_plan* p) {
  if (p->half[0])
    return align_up(staging_layout(p->half[0]).total, kAlign) + staging_layout(p->half[1]).total;
  return staging_layout(p).total;
}

StagingLayout staging_layout(const lapl_attn_plan* p) {
  StagingLayout s;
  const size_t elems = (size_t)p->geo.bh * p->geo.n * p->geo.d;
  const size_t in_b = elems * elem_bytes(p->cfg.in_dtype);
  const size_t out_b = elems * elem_bytes(p->cfg.out_dtype);
  size_t off = 0;
  s.q = off; off = align_up(off + in_b, kAlign);
  s.k = off; off = align_up(off + in_b, kAlign);
  s.v = off; off = align_up(off + in_b, kAlign);
  s.out = off; off = align_up(off + out_b, kAlign);
  s.bias = off; off = align_up(off + (size_t)p->cfg.heads * p->geo.m * sizeof(float), kAlign);
  s.ws = off; off = align_up(off + p->ws.total, kAlign);
  s.total = off;
  return s;
}
}  // namespace

lapl_status lapl_attn_host_staging_size(lapl_attn_handle h, size_t* bytes) {
  if (!h || !bytes) return LAPL_ERR_INVALID_ARG;
  *bytes = staging_bytes(h);
  return LAPL_OK;
}

}  // extern "C"

namespace lapl {
namespace {
// One forward of plan h from host buffers through the staging region `base` (laid out by
// staging_layout(h)), enqueued on st.  Arguments already checked.
lapl_status forward_host_one(lapl_attn_handle h, const void* q, const void* k, const void* v,
                             const float* bias, void* out, char* base, cudaStream_t st) {
  const StagingLayout s = staging_layout(h);
  const size_t elems = (size_t)h->geo.bh * h->geo.n * h->geo.d;
  const size_t in_b = elems * elem_bytes(h->cfg.in_dtype);
  const size_t out_b = elems * elem_bytes(h->cfg.out_dtype);
  const bool side_copies = h->geo.ns_exclusive && !h->geo.cg;
  cudaError_t e = cudaSuccess;
  // After the side stream has been given copies, every exit joins it back into the launching
  // stream, so that a caller who synchronises that stream also waits for those copies before
  // it frees or reuses the host inputs or the staging buffer.
  auto fail = [&](lapl_status r, cudaError_t err, const char* where) {
    if (err != cudaSuccess) set_error(h, err, where);
    if (side_copies && cudaEventRecord(h->ev_join, h->side_stream) == cudaSuccess)
      cudaStreamWaitEvent(st, h->ev_join, 0);
    return r;
  };
  if (side_copies) {
    // The solve chain (pooling first) needs K only; Q and V are first read by the distance and
    // B V kernels, which run on the side stream.  So the side stream copies K, Q, V in that
    // order (after everything enqueued on the launching stream so far) and the launching
    // stream waits for K alone: pooling and the solve start one copy after the call instead of
    // three, and Q and V land while they run.
    cudaStream_t side = h->side_stream;
    e = cudaEventRecord(h->ev_pool, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side, h->ev_pool, 0);
    if (e != cudaSuccess) {
      set_error(h, e, "forward_host/h2d");
      return LAPL_ERR_CUDA;
    }
    e = cudaMemcpyAsync(base + s.k, k, in_b, cudaMemcpyHostToDevice, side);
    if (e == cudaSuccess) e = cudaEventRecord(h->ev_join, side);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, h->ev_join, 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(base + s.q, q, in_b, cudaMemcpyHostToDevice, side);
    if (e == cudaSuccess) e = cudaMemcpyAsync(base + s.v, v, in_b, cudaMemcpyHostToDevice, side);
  } else {
    e = cudaMemcpyAsync(base + s.k, k, in_b, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(base + s.q, q, in_b, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(base + s.v, v, in_b, cudaMemcpyHostToDevice, st);
  }
  float* dbias = nullptr;
  if (e == cudaSuccess && bias) {
    dbias = reinterpret_cast<float*>(base + s.bias);
    e = cudaMemcpyAsync(dbias, bias, (size_t)h->cfg.heads * h->geo.m * sizeof(float),
                        cudaMemcpyHostToDevice, st);
  }
  if (e != cudaSuccess) return fail(LAPL_ERR_CUDA, e, "forward_host/h2d");
  lapl_status r = run_forward(h, base + s.q, base + s.k, base + s.v, dbias, base + s.out,
                              base + s.ws, h->ws.total, st, nullptr);
  if (r != LAPL_OK) return fail(r, cudaSuccess, "");
  e = cudaMemcpyAsync(out, base + s.out, out_b, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return fail(LAPL_ERR_CUDA, e, "forward_host/d2h");
  return LAPL_OK;
}
}  // namespace
}  // namespace lapl

extern "C" {

lapl_status lapl_attn_forward_host(lapl_attn_handle h, const void* q, const void* k,
                                   const void* v, const float* bias, void* out, void* staging,
                                   size_t staging_bytes_given, void* stream) {
  if (!h) return LAPL_ERR_INVALID_ARG;
  if (h->geo.bh == 0) return LAPL_OK;
  if (!q || !k || !v || !out || !staging) return LAPL_ERR_INVALID_ARG;
  if (!aligned16(staging)) return LAPL_ERR_ALIGNMENT;
  if (staging_bytes_given < staging_bytes(h)) return LAPL_ERR_WORKSPACE;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_error(h, e, "forward_host/device");
    return LAPL_ERR_CUDA;
  }
  if (dev != h->device) return LAPL_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(staging);
  if (!h->half[0]) return forward_host_one(h, q, k, v, bias, out, base, st);

  // Two half-batch forwards: the first on the launching stream, the second on the pipe stream
  // (after everything enqueued on the launching stream so far), joined back at the end.  Each
  // half's slices are computed exactly as by the full plan (same kernels, the B V partition
  // forced to the full plan's), so the output is the same bit for bit.
  lapl_attn_plan* h0 = h->half[0];
  lapl_attn_plan* h1 = h->half[1];
  const size_t in0 = (size_t)h0->geo.bh * h0->geo.n * h0->geo.d * elem_bytes(h->cfg.in_dtype);
  const size_t out0 = (size_t)h0->geo.bh * h0->geo.n * h0->geo.d * elem_bytes(h->cfg.out_dtype);
  char* base1 = base + align_up(staging_layout(h0).total, kAlign);
  e = cudaEventRecord(h->ev_pipe_start, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(h->pipe_stream, h->ev_pipe_start, 0);
  if (e != cudaSuccess) {
    set_error(h, e, "forward_host/fork");
    return LAPL_ERR_CUDA;
  }
  lapl_status r = forward_host_one(h0, q, k, v, bias, out, base, st);
  if (r != LAPL_OK) {
    snprintf(h->last_error, sizeof(h->last_error), "%s", h0->last_error);
    return r;
  }
  r = forward_host_one(h1, static_cast<const char*>(q) + in0, static_cast<const char*>(k) + in0,
                       static_cast<const char*>(v) + in0, bias, static_cast<char*>(out) + out0,
                       base1, h->pipe_stream);
  if (r != LAPL_OK) snprintf(h->last_error, sizeof(h->last_error), "%s", h1->last_error);
  // The launching stream waits for the second half whatever happened to it.
  e = cudaEventRecord(h->ev_pipe_join, h->pipe_stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, h->ev_pipe_join, 0);
  if (r == LAPL_OK && e != cudaSuccess) {
    set_error(h, e, "forward_host/join");
    return LAPL_ERR_CUDA;
  }
  return r;
}

lapl_status lapl_attn_set_timing(lapl_attn_handle h, int enable) {
  if (!h) return LAPL_ERR_INVALID_ARG;
  if (enable && !h->ev_stage[0]) {
    for (int i = 0; i < kMarks; ++i) {
      cudaError_t e = cudaEventCreate(&h->ev_stage[i]);
      if (e != cudaSuccess) {
        set_error(h, e, "set_timing");
        return LAPL_ERR_CUDA;
      }
    }
  }
  h->timing = enable != 0;
  h->timed_once = false;
  return LAPL_OK;
}

static cudaError_t wait_marks(lapl_attn_handle h) {
  cudaError_t e = cudaEventSynchronize(h->ev_stage[kMarkOutputDone]);
  if (e == cudaSuccess) e = cudaEventSynchronize(h->ev_stage[kMarkNsDone]);
  return e;
}

lapl_status lapl_attn_stage_times(lapl_attn_handle h, float* ms) {
  if (!h || !ms || !h->timing || !h->timed_once) return LAPL_ERR_INVALID_ARG;
  cudaError_t e = wait_marks(h);
  const int pairs[6][2] = {{kMarkStart, kMarkPoolDone},     {kMarkNsStart, kMarkNsDone},
                           {kMarkCdistStart, kMarkCdistDone}, {kMarkCdistDone, kMarkBvDone},
                           {kMarkBvDone, kMarkMixDone},       {kMarkMixDone, kMarkOutputDone}};
  for (int i = 0; i < 6 && e == cudaSuccess; ++i)
    e = cudaEventElapsedTime(&ms[i], h->ev_stage[pairs[i][0]], h->ev_stage[pairs[i][1]]);
  if (e != cudaSuccess) {
    set_error(h, e, "stage_times");
    return LAPL_ERR_CUDA;
  }
  return LAPL_OK;
}

lapl_status lapl_attn_stage_marks(lapl_attn_handle h, float* ms) {
  if (!h || !ms || !h->timing || !h->timed_once) return LAPL_ERR_INVALID_ARG;
  cudaError_t e = wait_marks(h);
  for (int i = 0; i < kMarks && e == cudaSuccess; ++i)
    e = cudaEventElapsedTime(&ms[i], h->ev_stage[kMarkStart], h->ev_stage[i]);
  if (e != cudaSuccess) {
    set_error(h, e, "stage_marks");
    return LAPL_ERR_CUDA;
  }
  return LAPL_OK;
}

int lapl_attn_kernels_per_forward(lapl_attn_handle h) {
  if (!h || h->geo.bh == 0) return 0;
  // The tensor-core B V runs after a statistics launch of its own.
  const int stats = (h->geo.bv_tc && h->geo.stat_ctas > 0) ? 1 : 0;
  return (h->geo.cg ? 5 : 6) + stats;
}

lapl_status lapl_attn_device_errors(lapl_attn_handle h, void* stream, unsigned* flags) {
  if (!h || !flags) return LAPL_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, h->dev_err, sizeof(word), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(h->dev_err, 0, sizeof(word), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    set_error(h, e, "device_errors");
    return LAPL_ERR_CUDA;
  }
  *flags = word;
  if (word) {
    snprintf(h->last_error, sizeof(h->last_error),
             "device error flags 0x%x: a bounded barrier wait gave up in:%s%s%s", word,
             (word & kErrBitCdist) ? " the distance kernel;" : "",
             (word & kErrBitSolve) ? " the tensor-core Newton-Schulz solve;" : "",
             (word & kErrBitChain) ? " a tensor-core kernel of the output chain;" : "");
    return LAPL_ERR_DEVICE_TIMEOUT;
  }
  return LAPL_OK;
}

lapl_status lapl_attn_set_fault_injection(lapl_attn_handle h, unsigned long long wait_ns,
                                          int skip_last_copy) {
  if (!h || skip_last_copy < 0 || skip_last_copy > 3) return LAPL_ERR_INVALID_ARG;
  h->cd_wait_ns = wait_ns ? wait_ns : 1000000000ull;
  h->cd_skip_last_copy = skip_last_copy;
  for (int i = 0; i < 2; ++i)
    if (h->half[i]) lapl_attn_set_fault_injection(h->half[i], wait_ns, skip_last_copy);
  return LAPL_OK;
}

lapl_status lapl_attn_plan_info_get(lapl_attn_handle h, lapl_attn_plan_info* info) {
  if (!h || !info) return LAPL_ERR_INVALID_ARG;
  const Geometry& g = h->geo;
  info->cdist_tma = g.cd_gtc ? 3 : g.cd_l1 ? 2 : (g.cd_tma ? 1 : 0);
  info->cdist_ctas = g.cd_part.ctas;
  info->cdist_threads = g.cd_threads;
  info->ns_cluster = g.ns_cluster;
  info->ns_tensor_core = g.ns_tc ? 1 : 0;
  info->ns_exclusive = g.ns_exclusive ? 1 : 0;
  info->bv_splits = g.bv_splits;
  info->bv_tensor_core = g.bv_tc ? 1 : 0;
  info->out_tensor_core = g.out_tc ? 1 : 0;
  return LAPL_OK;
}

lapl_status lapl_attn_destroy(lapl_attn_handle h) {
  if (!h) return LAPL_OK;
  for (int i = 0; i < 2; ++i) lapl_attn_destroy(h->half[i]);
  if (h->ev_pipe_start) cudaEventDestroy(h->ev_pipe_start);
  if (h->ev_pipe_join) cudaEventDestroy(h->ev_pipe_join);
  if (h->pipe_stream) cudaStreamDestroy(h->pipe_stream);
  for (int i = 0; i < kMarks; ++i)
    if (h->ev_stage[i]) cudaEventDestroy(h->ev_stage[i]);
  if (h->ev_join) cudaEventDestroy(h->ev_join);
  if (h->ev_pool) cudaEventDestroy(h->ev_pool);
  if (h->side_stream) cudaStreamDestroy(h->side_stream);
  if (h->ev_cdist) cudaEventDestroy(h->ev_cdist);
  if (h->ev_stats) cudaEventDestroy(h->ev_stats);
  if (h->stat_stream) cudaStreamDestroy(h->stat_stream);
  delete h;
  return LAPL_OK;
}

}  // extern "C"

namespace lapl {
// Internal: the plain forward on a caller-chosen workspace of at least ws.fwd_total bytes
// (used by noalloc.cu; the regions only the training forward writes are not needed).
lapl_status forward_on_workspace(lapl_attn_handle p, const void* q, const void* k, const void* v,
                                 const float* bias, void* out, void* workspace,
                                 size_t workspace_bytes, cudaStream_t st) {
  return run_forward(p, q, k, v, bias, out, workspace, workspace_bytes, st, nullptr, false,
                     p ? p->ws.fwd_total : 0);
}

void record_error(lapl_attn_handle p, const char* text) {
  snprintf(p->last_error, sizeof(p->last_error), "%s", text);
}
}  // namespace lapl
