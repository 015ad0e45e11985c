// attn_bwd_noalloc: the backward pass for callers that cannot allocate device memory.
//
// attn_bwd needs a caller-provided workspace (the fp32 dQ accumulator and two per-row
// vectors).  Some callers cannot produce one: code running inside another runtime's
// plugin or callback interface, where device memory belongs to that runtime's pool, or
// a latency-critical loop in which a cudaMalloc would implicitly synchronise the device.
// For them this entry point takes the workspace from a fixed array that lives in the
// library itself, so the call allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU that loads the library holds
// kNoallocScratchBytes of it until the process exits.  In host code its name is only a
// host-side stand-in, so its device address is looked up per device with
// cudaGetSymbolAddress (on the first call made on that device, again on the next call if
// that lookup failed) and passed on as an ordinary pointer.  All calls share the one array: calls that overlap on the GPU (for
// example on two streams) race on it.  It keeps the previous call's contents; the
// backward's own first kernel clears everything that must start at zero.
#include <cstdio>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/attn.h"

namespace attn {
void set_last_error(const char* msg);  // api.cu: the message attn_last_error() returns
}

namespace {

constexpr size_t kNoallocScratchBytes = size_t(64) << 20;  // 64 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
// The array's device address per device, once looked up.  Only a successful lookup is
// kept: a call whose lookup failed (a sticky error left by an earlier launch, or a first
// call made during stream capture) reports it, and the next call tries again.
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu[kMaxDevices];

}  // namespace

extern "C" {

int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                     void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                     int deterministic, void* stream) {
  const size_t need = attn_bwd_workspace_size(B, Hq, Hkv, N, d, deterministic);
  if (need == (size_t)-1) return ATTN_ERR_INVALID_ARG;  // attn_last_error() has the reason
  char msg[256];
  if (need > kNoallocScratchBytes) {
    snprintf(msg, sizeof msg,
             "attn_bwd_noalloc: these sizes need %zu bytes of workspace, more than its built-in %zu "
             "(64 MiB); call attn_bwd with a workspace instead",
             need, kNoallocScratchBytes);
    attn::set_last_error(msg);
    return ATTN_ERR_WORKSPACE;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    snprintf(msg, sizeof msg, "attn_bwd_noalloc: no usable current device (%s)", cudaGetErrorString(e));
    attn::set_last_error(msg);
    return ATTN_ERR_CUDA;
  }
  // With that device current: the array's device address, looked up until it succeeds.
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu[dev]);
    if (g_scratch_ptr[dev] == nullptr) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || p == nullptr) {
        snprintf(msg, sizeof msg, "attn_bwd_noalloc: cudaGetSymbolAddress failed (%s)", cudaGetErrorString(e));
        attn::set_last_error(msg);
        return ATTN_ERR_CUDA;
      }
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }
  return attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, causal, scale, deterministic, scratch,
                  kNoallocScratchBytes, stream);
}

}  // extern "C"
