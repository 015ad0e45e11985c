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
// host-side stand-in, so its device address is looked up once per device with
// cudaGetSymbolAddress (on the first call made on that device) and passed on as an
// ordinary pointer.  All calls share the one array: calls that overlap on the GPU (for
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
void* g_scratch_ptr[kMaxDevices];
cudaError_t g_scratch_err[kMaxDevices];
std::once_flag g_scratch_once[kMaxDevices];

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
  // Once per device, with that device current: the array's device address.
  std::call_once(g_scratch_once[dev], [dev] {
    void* p = nullptr;
    g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    g_scratch_ptr[dev] = p;
  });
  if (g_scratch_err[dev] != cudaSuccess || g_scratch_ptr[dev] == nullptr) {
    snprintf(msg, sizeof msg, "attn_bwd_noalloc: cudaGetSymbolAddress failed (%s)",
             cudaGetErrorString(g_scratch_err[dev]));
    attn::set_last_error(msg);
    return ATTN_ERR_CUDA;
  }
  return attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, N, d, causal, scale, deterministic,
                  g_scratch_ptr[dev], kNoallocScratchBytes, stream);
}

}  // extern "C"
