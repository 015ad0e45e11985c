// Backward kernels (placeholder launcher until the tcgen05 backward lands).
#include "kernels.h"

namespace attn {

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d, int deterministic) {
  (void)Hkv;
  const size_t rows = (size_t)B * Hq * N;
  const size_t nq = (size_t)B * Hq * ((N + 127) / 128);
  size_t n = align256(rows * d * 4) + 2 * align256(rows * 4);
  if (deterministic) n += align256(nq * 4);
  return n;
}

void bwd_workspace_carve(void* ws, int B, int Hq, int Hkv, int N, int d, int deterministic, BwdParams* p) {
  (void)Hkv;
  char* b = static_cast<char*>(ws);
  const size_t rows = (size_t)B * Hq * N;
  p->dq_acc = reinterpret_cast<float*>(b);
  b += align256(rows * d * 4);
  p->delta = reinterpret_cast<float*>(b);
  b += align256(rows * 4);
  p->lse2 = reinterpret_cast<float*>(b);
  b += align256(rows * 4);
  p->sem = deterministic ? reinterpret_cast<int*>(b) : nullptr;
}

cudaError_t launch_bwd(const BwdMaps&, const BwdParams&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace attn
