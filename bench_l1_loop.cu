// bench_l1_loop.cu -- microbenchmark of the L1-distance inner loop on the FP32 and ALU pipes.
//
// Each thread accumulates sum_c |x_c - l_c| for 4 tokens x C landmarks over 32 channels per
// step, with tokens read from a 128-byte-swizzled shared tile (as the distance kernels stage
// them) and landmarks as shared-memory broadcasts: the distance kernels' loop without their
// pipeline.  Forms of one element term:
//   scalar   sub.f32, then add.f32 with the absolute value as an operand modifier (2 FP32-pipe
//            instructions)
//   sub2abs  sub.f32x2 for two channels, then two abs-adds (1.5 instructions, all FP32 pipe)
//   min2     |q - l| = q + l - 2 min(q, l): two min.f32 (ALU pipe) and one add.f32x2 (1.5
//            instructions; the q + l part is a per-row constant, added once outside the loop)
//   mix      the first NS landmarks of a warp as sub2abs, the others as min2 (both pipes)
//   ffma     one fma.f32 per term (a control: the loop's own ceiling with one instruction)
// Per-SM throughput: every CTA records (%smid, start clock, end clock); an SM's time is the
// span of its CTAs.  Output: one line per (form, CTAs per SM) with elements / clock / SM (min,
// mean, max over SMs).  No global memory traffic inside the timed loop.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <vector>

namespace {

constexpr int DH = 32;    // channels
constexpr int R = 4;      // tokens per thread

__device__ __forceinline__ void acc_scalar(float& t, float x, float l) {
  asm("{\n\t.reg .f32 dd;\n\tsub.f32 dd, %1, %2;\n\tabs.f32 dd, dd;\n\tadd.f32 %0, %0, dd;\n\t}"
      : "+f"(t)
      : "f"(x), "f"(l));
}
__device__ __forceinline__ void acc_sub2abs(float& t, float x0, float x1, float l0, float l1) {
  asm("{\n\t.reg .b64 a, b, d;\n\t.reg .f32 d0, d1;\n\t"
      "mov.b64 a, {%1, %2};\n\tmov.b64 b, {%3, %4};\n\t"
      "sub.f32x2 d, a, b;\n\tmov.b64 {d0, d1}, d;\n\t"
      "abs.f32 d0, d0;\n\tabs.f32 d1, d1;\n\tadd.f32 %0, %0, d0;\n\tadd.f32 %0, %0, d1;\n\t}"
      : "+f"(t)
      : "f"(x0), "f"(x1), "f"(l0), "f"(l1));
}
__device__ __forceinline__ void acc_min2(float& t0, float& t1, float x0, float x1, float l0,
                                         float l1) {
  asm("{\n\t.reg .b64 a, m;\n\t.reg .f32 m0, m1;\n\t"
      "min.f32 m0, %2, %4;\n\tmin.f32 m1, %3, %5;\n\t"
      "mov.b64 m, {m0, m1};\n\tmov.b64 a, {%0, %1};\n\t"
      "add.f32x2 a, a, m;\n\tmov.b64 {%0, %1}, a;\n\t}"
      : "+f"(t0), "+f"(t1)
      : "f"(x0), "f"(x1), "f"(l0), "f"(l1));
}

enum Form { kScalar = 0, kSub2Abs = 1, kMin2 = 2, kMix = 3, kFfma = 4 };

template <int F, int C, int NS, int MINB>
__global__ void __launch_bounds__(256, MINB)
loop_kernel(const float* __restrict__ in, float* __restrict__ out, int iters,
            long long* __restrict__ rec) {
  __shared__ __align__(16) float qs[32 * R * DH];
  __shared__ __align__(16) float ls[8 * C * DH];
  for (int i = threadIdx.x; i < 32 * R * DH; i += blockDim.x) qs[i] = in[i & 4095];
  for (int i = threadIdx.x; i < 8 * C * DH; i += blockDim.x) ls[i] = in[(i * 7) & 4095];
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float* lrow = ls + (warp & 7) * C * DH;
  const char* rowp = reinterpret_cast<const char*>(qs) + lane * 128;
  const int sw = lane & 7;
  float a0[R][C], a1[R][C];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int j = 0; j < C; ++j) a0[r][j] = a1[r][j] = 0.f;
  unsigned smid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll 2
    for (int c4 = 0; c4 < DH / 4; ++c4) {
      const char* pc = rowp + (((c4 & 7) ^ sw) << 4);
      float4 x[R];
#pragma unroll
      for (int r = 0; r < R; ++r) x[r] = *reinterpret_cast<const float4*>(pc + r * 32 * 128);
#pragma unroll
      for (int j = 0; j < C; ++j) {
        const float4 l = *reinterpret_cast<const float4*>(lrow + j * DH + 4 * c4);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          if (F == kScalar) {
            acc_scalar(a0[r][j], x[r].x, l.x); acc_scalar(a0[r][j], x[r].y, l.y);
            acc_scalar(a0[r][j], x[r].z, l.z); acc_scalar(a0[r][j], x[r].w, l.w);
          } else if (F == kFfma) {
            a0[r][j] = fmaf(x[r].x, l.x, a0[r][j]); a0[r][j] = fmaf(x[r].y, l.y, a0[r][j]);
            a0[r][j] = fmaf(x[r].z, l.z, a0[r][j]); a0[r][j] = fmaf(x[r].w, l.w, a0[r][j]);
          } else if (F == kSub2Abs || (F == kMix && j < NS)) {
            acc_sub2abs(a0[r][j], x[r].x, x[r].y, l.x, l.y);
            acc_sub2abs(a0[r][j], x[r].z, x[r].w, l.z, l.w);
          } else {
            acc_min2(a0[r][j], a1[r][j], x[r].x, x[r].y, l.x, l.y);
            acc_min2(a0[r][j], a1[r][j], x[r].z, x[r].w, l.z, l.w);
          }
        }
      }
    }
  }
  const long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int j = 0; j < C; ++j) s += a0[r][j] + a1[r][j];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) {
    rec[3 * blockIdx.x] = smid;
    rec[3 * blockIdx.x + 1] = t0;
    rec[3 * blockIdx.x + 2] = t1;
  }
}

template <int F, int C, int NS, int MINB>
void run(const char* name, const float* in, float* out, long long* rec, int sms, int per_sm) {
  auto k = loop_kernel<F, C, NS, MINB>;
  int occ = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, 256, 0);
  if (occ < per_sm) return;
  cudaFuncAttributes fa;
  cudaFuncGetAttributes(&fa, k);
  const int blocks = sms * per_sm, iters = 400 / per_sm;
  k<<<blocks, 256>>>(in, out, iters, rec);   // warm
  k<<<blocks, 256>>>(in, out, iters, rec);
  const cudaError_t err = cudaDeviceSynchronize();
  if (err != cudaSuccess) {
    printf("%s: %s\n", name, cudaGetErrorString(err));
    exit(1);
  }
  std::vector<long long> h(3 * blocks);
  cudaMemcpy(h.data(), rec, h.size() * sizeof(long long), cudaMemcpyDeviceToHost);
  std::vector<long long> lo(sms, -1), hi(sms, 0);
  std::vector<int> cnt(sms, 0);
  for (int b = 0; b < blocks; ++b) {
    const int s = (int)h[3 * b];
    if (s < 0 || s >= sms) continue;
    if (lo[s] < 0 || h[3 * b + 1] < lo[s]) lo[s] = h[3 * b + 1];
    hi[s] = std::max(hi[s], h[3 * b + 2]);
    cnt[s]++;
  }
  const double per_cta = 256.0 * iters * DH * R * C;
  double mn = 1e30, mx = 0, sum = 0;
  int nsm = 0;
  for (int s = 0; s < sms; ++s)
    if (cnt[s]) {
      const double r = cnt[s] * per_cta / (double)(hi[s] - lo[s]);
      mn = std::min(mn, r);
      mx = std::max(mx, r);
      sum += r;
      ++nsm;
    }
  printf("%s C=%d ctas_per_sm=%d regs=%d elem_per_clk_per_sm min=%.1f mean=%.1f max=%.1f\n", name,
         C, per_sm, fa.numRegs, mn, sum / nsm, mx);
}

}  // namespace

int main() {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  float *in, *out;
  long long* rec;
  cudaMalloc(&in, 4096 * sizeof(float));
  cudaMalloc(&out, (size_t)sms * 2 * 256 * sizeof(float));
  cudaMalloc(&rec, (size_t)sms * 2 * 3 * sizeof(long long));
  std::vector<float> hin(4096);
  for (int i = 0; i < 4096; ++i) hin[i] = (float)((i * 37) % 101) / 17.f - 3.f;
  cudaMemcpy(in, hin.data(), hin.size() * sizeof(float), cudaMemcpyHostToDevice);
  printf("sms=%d\n", sms);
  for (int p = 1; p <= 2; ++p) {
    run<kScalar, 7, 0, 2>("scalar", in, out, rec, sms, p);
    run<kSub2Abs, 7, 0, 2>("sub2abs", in, out, rec, sms, p);
    run<kMin2, 7, 0, 1>("min2", in, out, rec, sms, p);
    run<kMix, 7, 3, 2>("mix", in, out, rec, sms, p);
    run<kMix, 8, 4, 2>("mix", in, out, rec, sms, p);
    run<kFfma, 7, 0, 2>("ffma", in, out, rec, sms, p);
  }
  return 0;
}
