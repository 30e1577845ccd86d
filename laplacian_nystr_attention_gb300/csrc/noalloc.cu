// noalloc.cu -- a forward pass that allocates nothing, not even the workspace.
//
// Some callers cannot allocate device memory at all: code running inside a host that owns every
// allocation and hands out only its own tensors, plugins loaded into a process whose allocator
// must not be bypassed, or environments where cudaMalloc is forbidden after start-up.
// lapl_attn_forward_noalloc serves them: it runs the same kernels as lapl_attn_forward, with the
// workspace placed in a fixed-size array in the library's own device memory instead of a
// caller-provided buffer.
//
// The array is a file-scope __device__ variable: every GPU that loads this library holds it
// (kNoAllocScratchBytes) until the process exits.  Host code cannot use the array's name as a
// device address, so the address is looked up once per device with cudaGetSymbolAddress, on the
// first call made while that device is current, and cached for the life of the process.  A
// cudaDeviceReset unloads the module, after which the cached address is stale: this entry
// point must not be used on a device after it has been reset.
//
// Only the plain forward's regions are placed in the array (WorkspaceLayout::fwd_total): the
// regions a training forward keeps for the backward pass lie past that offset and are never
// touched here.
#include <mutex>
#include <stdio.h>

#include "common.cuh"

namespace lapl {
lapl_status forward_on_workspace(lapl_attn_handle p, const void* q, const void* k, const void* v,
                                 const float* bias, void* out, void* workspace,
                                 size_t workspace_bytes, cudaStream_t st);
void record_error(lapl_attn_handle p, const char* text);
}  // namespace lapl

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];   // device address of g_noalloc_scratch, per device

}  // namespace

extern "C" lapl_status lapl_attn_forward_noalloc(lapl_attn_handle h, const void* q,
                                                 const void* k, const void* v,
                                                 const float* bias, void* out, void* stream) {
  if (!h) return LAPL_ERR_INVALID_ARG;
  if (h->ws.fwd_total > kNoAllocScratchBytes) {
    char msg[160];
    snprintf(msg, sizeof(msg),
             "forward_noalloc: this configuration needs %zu workspace bytes, the static scratch "
             "holds %zu",
             h->ws.fwd_total, kNoAllocScratchBytes);
    lapl::record_error(h, msg);
    return LAPL_ERR_WORKSPACE;
  }
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    lapl::record_error(h, "forward_noalloc: no usable current device");
    return LAPL_ERR_CUDA;
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
      void* addr = nullptr;
      e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
      if (e != cudaSuccess || !addr) {
        char msg[160];
        snprintf(msg, sizeof(msg), "forward_noalloc: cudaGetSymbolAddress failed: %s",
                 cudaGetErrorString(e));
        lapl::record_error(h, msg);
        return LAPL_ERR_CUDA;
      }
      g_scratch_addr[dev] = addr;
    }
    scratch = g_scratch_addr[dev];
  }
  // Every workspace region is fully written before it is read, so the previous call's
  // leftovers in the array need no clearing.
  return lapl::forward_on_workspace(h, q, k, v, bias, out, scratch, kNoAllocScratchBytes,
                                    static_cast<cudaStream_t>(stream));
}
