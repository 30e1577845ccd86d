// pool.cu -- landmark pooling.
//
// Landmarks are average-pooled keys ("LaplacianFormer: Rethinking Linear Attention with
// Laplacian Kernel", English explainer page, 2.C.1): L[j] is the mean of K over the
// non-overlapping (grid_h/s) x (grid_w/s) window j = jr*s + jc of the token grid.
//
// A lane owns 16 bytes of channels (4 fp32 or 8 bf16) of every tlw-th token of a window row,
// so a warp load covers tlw consecutive tokens of one grid row, and each lane issues its loads
// in batches of 8 before summing.  Two CTA shapes, chosen per plan by the window size:
//   windows of >= 64 tokens: one CTA of 4 warps (8 from 1024 tokens) per (head, landmark),
//     warp w takes the window rows w, w + 4, ... (w, w + 8, ...);
//   smaller windows: one CTA per (head, landmark row jr), warp w takes all of window jc = w.
// The (warp, token lane) partials meet in shared memory and are summed in a fixed order.
// HBM-bound: K is read exactly once.
#include "common.cuh"

namespace lapl {
namespace {

constexpr int kPoolWarps = kMaxS;   // 8: one warp per window of a landmark row
constexpr int kPoolThreads = 32 * kPoolWarps;

template <bool kBf16>
__global__ void __launch_bounds__(kPoolThreads)
pool_landmarks_kernel(const void* __restrict__ kin, float* __restrict__ landmarks,
                      float* __restrict__ dbg, int grid_w, int n, int d, int s, int ph, int pw,
                      int per_row) {
  constexpr int CH = kBf16 ? 8 : 4;          // channels per lane (16 bytes)
  __shared__ float part[kPoolWarps][32][CH];
  // A programmatic dependent (the Newton-Schulz solve on this stream) may be placed now: it
  // sets up its tensor memory and barriers, then waits for this grid before it reads L.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = s * s;
  long bh;
  int jr, jc, row0, rstep;
  if (per_row) {
    bh = blockIdx.x / s;
    jr = (int)(blockIdx.x % s);
    jc = warp;
    row0 = 0;
    rstep = 1;
  } else {
    bh = blockIdx.x / m;
    const int j = (int)(blockIdx.x % m);
    jr = j / s;
    jc = j % s;
    row0 = warp;
    rstep = (int)(blockDim.x >> 5);
  }
  const bool active = jc < s;                // per_row: warps beyond the s windows idle
  const int lpt = d / CH;                    // lanes per token
  const int tlw = 32 / lpt;                  // token lanes of the warp
  const int tl = lane / lpt, piece = lane % lpt;
  float acc[CH];
#pragma unroll
  for (int c = 0; c < CH; ++c) acc[c] = 0.f;
  if (active && tl < tlw) {
    const size_t row_bytes = (size_t)d * (kBf16 ? 2 : 4);
    const char* base = reinterpret_cast<const char*>(kin) +
                       ((size_t)bh * n + (size_t)(jr * ph) * grid_w + (size_t)jc * pw) * row_bytes +
                       piece * 16;
    // This lane's tokens of the window: rows row0, row0 + rstep, ..., per_lane_row of them per
    // row (columns tl, tl + tlw, ...).  Loads are issued in batches of kBatch before any is
    // summed.
    constexpr int kBatch = 8;
    const int per_lane_row = (pw - tl + tlw - 1) / tlw;
    const int rows = (ph - row0 + rstep - 1) / rstep;
    const int total = rows * per_lane_row;
    for (int i0 = 0; i0 < total; i0 += kBatch) {
      uint4 raw[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = i0 + u;
        raw[u] = make_uint4(0u, 0u, 0u, 0u);          // zero bits: +0.0 in fp32 and bf16
        if (i < total) {
          const int ri = i / per_lane_row, c = tl + (i - ri * per_lane_row) * tlw;
          const int r = row0 + ri * rstep;
          raw[u] = *reinterpret_cast<const uint4*>(base + ((size_t)r * grid_w + c) * row_bytes);
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if constexpr (kBf16) {
          acc[0] += bf16_lo(raw[u].x); acc[1] += bf16_hi(raw[u].x);
          acc[2] += bf16_lo(raw[u].y); acc[3] += bf16_hi(raw[u].y);
          acc[4] += bf16_lo(raw[u].z); acc[5] += bf16_hi(raw[u].z);
          acc[6] += bf16_lo(raw[u].w); acc[7] += bf16_hi(raw[u].w);
        } else {
          acc[0] += __uint_as_float(raw[u].x); acc[1] += __uint_as_float(raw[u].y);
          acc[2] += __uint_as_float(raw[u].z); acc[3] += __uint_as_float(raw[u].w);
        }
      }
    }
  }
#pragma unroll
  for (int c = 0; c < CH; ++c) part[warp][lane][c] = acc[c];
  __syncthreads();
  // Combiner lanes: per_row, lanes 0..lpt-1 of every active warp (its own window); otherwise
  // threads 0..lpt-1 (all warps' partials of the CTA's window).
  const int w_lo = per_row ? warp : 0, w_hi = per_row ? warp + 1 : (int)(blockDim.x >> 5);
  if (active && (per_row ? lane : (int)threadIdx.x) < lpt) {
    const int piece0 = per_row ? lane : (int)threadIdx.x;
    float sum[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) sum[c] = 0.f;
    for (int w = w_lo; w < w_hi; ++w)
      for (int t = 0; t < tlw; ++t)
#pragma unroll
        for (int c = 0; c < CH; ++c) sum[c] += part[w][t * lpt + piece0][c];
    // The mean as a product with 1 / (window size): the same value as the division when the
    // window size is a power of two (every workload's), within an ulp otherwise, without a
    // division per value.
    const float inv_cnt = 1.f / (float)(ph * pw);
    const size_t o = ((size_t)bh * m + jr * s + jc) * d + piece0 * CH;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const float val = sum[c] * inv_cnt;
      landmarks[o + c] = val;
      if (dbg) dbg[o + c] = val;
    }
  }
}

}  // namespace

cudaError_t launch_pool(const lapl_attn_plan& p, const void* k, float* landmarks,
                        float* dbg_landmarks, cudaStream_t st) {
  const Geometry& g = p.geo;
  const int s = g.s;
  const int ph = p.cfg.grid_h / s, pw = p.cfg.grid_w / s;
  const int per_row = ph * pw < 64 ? 1 : 0;
  const unsigned grid = (unsigned)(g.bh * (per_row ? s : g.m));
  // Windows of 1024 tokens or more take 8 warps per CTA (twice the loads in flight per SM):
  // N = 65536 sweeps (32 x 32 windows) 35.6 -> 30.7 us fp32, 22.5 -> 20.5 us bf16; at 16 x 16
  // windows 8 warps measured slower (high-resolution shape 20.5 -> 22.7 us).
  const int threads = per_row ? kPoolThreads : (ph * pw >= 1024 ? 256 : 128);
  if (p.cfg.in_dtype == LAPL_BF16)
    pool_landmarks_kernel<true><<<grid, threads, 0, st>>>(
        k, landmarks, dbg_landmarks, p.cfg.grid_w, g.n, g.d, s, ph, pw, per_row);
  else
    pool_landmarks_kernel<false><<<grid, threads, 0, st>>>(
        k, landmarks, dbg_landmarks, p.cfg.grid_w, g.n, g.d, s, ph, pw, per_row);
  return cudaGetLastError();
}

}  // namespace lapl
