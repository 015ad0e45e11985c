// C-ABI entry points (declared in include/attn.h): argument checks, TMA tensor maps,
// kernel selection and launch.  No allocation on any call path; every launch goes on
// the caller's stream.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/attn.h"
#include "kernels.h"

namespace attn {

// Status word written by kernels that give up on a bounded wait, and the optional
// rescale counter.  One copy per device; the host reaches them through their device
// addresses (cudaGetSymbolAddress, cached per device).
__device__ int g_dev_status;
__device__ unsigned long long g_rescale_count;

namespace {

thread_local char t_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof t_err, fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(ATTN_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

std::atomic<float> g_tau{8.0f};
std::atomic<int> g_poly{0};
std::atomic<long long> g_wait_ns{2000000000LL};
std::atomic<int> g_sync_check{0};
std::atomic<int> g_count_rescales{0};
std::atomic<int> g_test_skip_kv{0};
std::atomic<int> g_varlen_lpt{1};
std::atomic<int> g_one_tile_d128{0};
std::atomic<int> g_persistent{0};
std::atomic<int> g_decode_one_tile{1};    // grouped decode at d = 128 through the one-tile kernel (fwd_wide.cu)
std::atomic<int> g_bwd_tile_rows{128};   // d <= 128 backward: 128-row (bwd.cu) or 64-row (bwd_wide.cu) query tiles

struct DevSyms {
  int* status = nullptr;
  unsigned long long* rescale = nullptr;
  int sms = 0;
  cudaError_t err = cudaSuccess;
};
constexpr int kMaxDev = 64;
DevSyms g_syms[kMaxDev];
std::once_flag g_syms_once[kMaxDev];

const DevSyms* dev_syms(int* dev_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    static DevSyms bad;
    bad.err = e;
    return &bad;
  }
  if (dev_out) *dev_out = dev;
  DevSyms& s = g_syms[dev % kMaxDev];
  std::call_once(g_syms_once[dev % kMaxDev], [&] {
    void* p = nullptr;
    s.err = cudaGetSymbolAddress(&p, g_dev_status);
    s.status = static_cast<int*>(p);
    if (s.err == cudaSuccess) {
      s.err = cudaGetSymbolAddress(&p, g_rescale_count);
      s.rescale = static_cast<unsigned long long*>(p);
    }
    if (s.err == cudaSuccess) s.err = cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, dev);
  });
  return &s;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link-time
// dependency on libcuda).
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeFn g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

EncodeFn get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess) g_encode = reinterpret_cast<EncodeFn>(fn);
  });
  return g_encode;
}

// [BH, rows, d] bf16 tensor, boxes of 128 rows x 64 columns, 128-byte swizzle.
// box_rows x box_planes: 128 x 1 for ordinary tiles; N x g to gather the g query heads of
// a group (rows h * N + q) into one tile in grouped decode mode.
int make_map(CUtensorMap* m, const void* base, int d, int rows, long long bh, const char* name, int box_rows = 128,
             int box_planes = 1) {
  EncodeFn enc = get_encode();
  if (!enc) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(g_encode_err));
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)bh};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)rows * (cuuint64_t)d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_planes};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "tensor map for %s: CUresult %d", name, (int)r);
  return ATTN_OK;
}

// [BH, rows, 128] e4m3 tensor (one byte per element), boxes of 128 rows x 128 bytes,
// 128-byte swizzle: one box is a whole 128 x 128 tile.
int make_map_e4m3(CUtensorMap* m, const void* base, int rows, long long bh, const char* name) {
  EncodeFn enc = get_encode();
  if (!enc) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(g_encode_err));
  cuuint64_t dims[3] = {128, (cuuint64_t)rows, (cuuint64_t)bh};
  cuuint64_t strides[2] = {128, (cuuint64_t)rows * 128};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "tensor map for %s: CUresult %d", name, (int)r);
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// wide: the forward also takes d = 192 and 256 (one-tile kernel, fwd_wide.cu).
int check_shape(int B, int Hq, int Hkv, int N, int d, float scale, bool wide = false) {
  if (B < 0 || N < 0) return fail(ATTN_ERR_INVALID_ARG, "B=%d and N=%d must be >= 0", B, N);
  if (Hq <= 0 || Hkv <= 0) return fail(ATTN_ERR_INVALID_ARG, "Hq=%d and Hkv=%d must be >= 1", Hq, Hkv);
  if (Hq % Hkv != 0) return fail(ATTN_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
  if (wide && (d == 192 || d == 256)) {
  } else if (d != 64 && d != 128) {
    return fail(ATTN_ERR_UNSUPPORTED, wide ? "head dim d=%d (supported: 64, 128, 192, 256)"
                                           : "head dim d=%d (supported here: 64, 128)", d);
  }
  if (!(scale > 0.0f) || !std::isfinite(scale)) return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
  if ((long long)B * Hq > 0x7fffffffLL) return fail(ATTN_ERR_INVALID_ARG, "B*Hq too large");
  return ATTN_OK;
}

// The error a non-zero device status word stands for.
int status_fail(int v) {
  if (v == DEV_BAD_OFFSETS)
    return fail(ATTN_ERR_INVALID_ARG, "packed-sequence offsets failed the device check (device status %d)", v);
  return fail(ATTN_ERR_TIMEOUT, "a kernel gave up on a bounded wait (device status %d)", v);
}

int post_launch(const DevSyms* s, cudaStream_t st) {
  if (!g_sync_check.load()) return ATTN_OK;
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int v = 0;
  e = cudaMemcpy(&v, s->status, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (v != 0) return status_fail(v);
  return ATTN_OK;
}

}  // namespace

void set_last_error(const char* msg) { snprintf(t_err, sizeof t_err, "%s", msg); }

}  // namespace attn

using namespace attn;

extern "C" {

const char* attn_last_error(void) { return t_err; }

const char* attn_version(void) { return "attn-gb300 0.1 (sm_103a)"; }

int attn_set_debug_knobs(float tau, int poly_per_16, long long wait_limit_ns, int sync_check) {
  if (!(tau >= 0.0f) || !std::isfinite(tau)) return fail(ATTN_ERR_INVALID_ARG, "tau must be finite and >= 0");
  if (poly_per_16 != 0 && poly_per_16 != 4 && poly_per_16 != 16)
    return fail(ATTN_ERR_UNSUPPORTED, "poly_per_16=%d (supported: 0, 4, 16)", poly_per_16);
  if (wait_limit_ns <= 0) return fail(ATTN_ERR_INVALID_ARG, "wait limit must be > 0");
  g_tau.store(tau);
  g_poly.store(poly_per_16);
  g_wait_ns.store(wait_limit_ns);
  g_sync_check.store(sync_check ? 1 : 0);
  return ATTN_OK;
}

int attn_set_test_hooks(int skip_first_kv_load) {
  g_test_skip_kv.store(skip_first_kv_load ? 1 : 0);
  return ATTN_OK;
}

int attn_get_debug_knobs(float* tau, int* poly_per_16, long long* wait_limit_ns, int* sync_check) {
  if (tau) *tau = g_tau.load();
  if (poly_per_16) *poly_per_16 = g_poly.load();
  if (wait_limit_ns) *wait_limit_ns = g_wait_ns.load();
  if (sync_check) *sync_check = g_sync_check.load();
  return ATTN_OK;
}

int attn_device_status(int clear) {
  const DevSyms* s = dev_syms(nullptr);
  if (s->err != cudaSuccess) return cuda_fail(s->err, "device symbols");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "device synchronize");
  int v = 0;
  e = cudaMemcpy(&v, s->status, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (clear) {
    const int z = 0;
    e = cudaMemcpy(s->status, &z, sizeof z, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
  }
  if (v != 0) return status_fail(v);
  return ATTN_OK;
}

int attn_rescale_counter(int enable, unsigned long long* value_out) {
  const DevSyms* s = dev_syms(nullptr);
  if (s->err != cudaSuccess) return cuda_fail(s->err, "device symbols");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "device synchronize");
  unsigned long long v = 0;
  e = cudaMemcpy(&v, s->rescale, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "counter read");
  if (value_out) *value_out = v;
  const unsigned long long z = 0;
  e = cudaMemcpy(s->rescale, &z, sizeof z, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "counter clear");
  g_count_rescales.store(enable ? 1 : 0);
  return ATTN_OK;
}

// Grouped decode plan for N queries after Nk keys: used when a group's g query heads x N
// queries fit one 128-row tile (g >= 2); the keys are split so that the grid about fills
// the GPU once.  pack = 0 means the ordinary path.
struct KvPlan {
  int pack, splits, blocks_per_split;
  size_t ws_bytes;
};
static size_t al256(size_t x) { return (x + 255) & ~size_t(255); }
static KvPlan kv_plan(int B, int Hq, int Hkv, int N, int Nk, int d, int sms) {
  KvPlan k{0, 1, 0, 0};
  const int g = Hq / Hkv;
  if (B <= 0 || N <= 0 || Nk <= 0 || g < 2 || (long long)g * N > 128 || d > 128) return k;
  const int nkv = (Nk + 127) / 128;
  const long long units = (long long)B * Hkv;
  long long sp = std::min<long long>(nkv, std::max<long long>(1, sms / units));
  const int bps = (int)((nkv + sp - 1) / sp);
  sp = (nkv + bps - 1) / bps;   // every split holds at least one key block
  k.pack = 1;
  k.splits = (int)sp;
  k.blocks_per_split = bps;
  k.ws_bytes = al256((size_t)sp * units * 128 * d * 4) + al256((size_t)sp * units * 128 * 4);
  return k;
}

// The forward for N queries against Nk keys (query i at key position i + Nk - N).
static int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                    int N, int Nk, int d, int causal, float scale, void* workspace, size_t ws_bytes,
                    void* stream) {
  int rc = check_shape(B, Hq, Hkv, N, d, scale, true);
  if (rc != ATTN_OK) return rc;
  if (Nk < 0) return fail(ATTN_ERR_INVALID_ARG, "Nk=%d must be >= 0", Nk);
  if (B == 0 || N == 0) return ATTN_OK;
  if (Nk == 0) return fail(ATTN_ERR_INVALID_ARG, "Nk=0 with N=%d queries: the softmax has no keys", N);
  if (causal && N > Nk)
    return fail(ATTN_ERR_INVALID_ARG, "causal needs N <= Nk (got N=%d, Nk=%d): the first queries would see no key",
                N, Nk);
  if (!q || !k || !v || !o || !lse) return fail(ATTN_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(ATTN_ERR_MISALIGNED, "q, k, v, o and lse must be 16-byte aligned");
  int dev = 0;
  const DevSyms* s = dev_syms(&dev);
  if (s->err != cudaSuccess) return cuda_fail(s->err, "device setup");
  const KvPlan plan = kv_plan(B, Hq, Hkv, N, Nk, d, std::max(1, s->sms));
  const bool pack = plan.pack && workspace != nullptr && ws_bytes >= plan.ws_bytes && aligned16(workspace);

  FwdMaps maps;
  if (pack) {
    if ((rc = make_map(&maps.q, q, d, N, (long long)B * Hq, "q", N, Hq / Hkv)) != ATTN_OK) return rc;
  } else if ((rc = make_map(&maps.q, q, d, N, (long long)B * Hq, "q")) != ATTN_OK) {
    return rc;
  }
  if ((rc = make_map(&maps.k, k, d, Nk, (long long)B * Hkv, "k")) != ATTN_OK) return rc;
  if ((rc = make_map(&maps.v, v, d, Nk, (long long)B * Hkv, "v")) != ATTN_OK) return rc;
  if ((rc = make_map(&maps.o, o, d, N, (long long)B * Hq, "o")) != ATTN_OK) return rc;

  FwdParams p{};
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = N; p.g = Hq / Hkv;
  p.Nk = Nk; p.koff = Nk - N;
  p.causal = causal ? 1 : 0;
  p.pair_heads = (p.g >= 2 && p.g % 2 == 0) ? 1 : 0;
  p.n_qblk = (N + 127) / 128;
  p.n_kvblk = (Nk + 127) / 128;
  p.n_rowslots = p.pair_heads ? p.n_qblk : (p.n_qblk + 1) / 2;
  p.units_per_row = p.pair_heads ? B * (Hq / 2) : B * Hq;
  p.c = scale * 1.4426950408889634f;
  p.tau = g_tau.load();
  p.lse = lse;
  p.wait_ns = (unsigned long long)g_wait_ns.load();
  p.status = s->status;
  p.rescale_count = g_count_rescales.load() ? s->rescale : nullptr;
  p.test_skip_first_kv = g_test_skip_kv.load();
  // Units of two tiles, one CTA each.  When the last wave would hold few units (at most
  // half the SMs) they are split into one-tile CTAs, so that the last wave takes one tile's
  // time instead of two tiles' (non-causal only: causal units come longest first, so the
  // last ones are short already).
  const long long units = (long long)p.n_rowslots * p.units_per_row;
  p.split_from = (int)std::min<long long>(units, 0x7fffffffLL);
  if (!p.causal) {
    const long long sms = std::max(1, s->sms);
    const long long rem = units % sms;
    if (units >= sms && rem > 0 && 2 * rem <= sms) p.split_from = (int)(units - rem);
    else if (units < sms && 2 * units <= sms) p.split_from = 0;
  }
  long long grid = p.split_from + 2 * (units - p.split_from);
  p.prefetch_ahead = std::max(1, s->sms);
  p.q_tile_bytes = (unsigned)((d / 64) * 128 * 128);
  // One query tile per CTA (fwd_wide.cu): always for d > 128, and for d = 128 when chosen.
  const bool wide = d > 128 || (d == 128 && !pack && g_one_tile_d128.load());
  if (wide) grid = (long long)B * Hq * p.n_qblk;
  if (pack) {
    p.pack = 1;
    p.kv_splits = plan.splits;
    p.blocks_per_split = plan.blocks_per_split;
    p.q_tile_bytes = (unsigned)((d / 64) * 128 * N * p.g);   // NCH boxes of 64 columns x N rows x g heads
    char* w = static_cast<char*>(workspace);
    p.part_o = reinterpret_cast<float*>(w);
    p.part_lse = reinterpret_cast<float*>(w + al256((size_t)plan.splits * B * Hkv * 128 * d * 4));
    grid = (long long)B * Hkv * plan.splits;
  }
  if (grid > 0x7fffffffLL) return fail(ATTN_ERR_INVALID_ARG, "problem too large for one launch");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Persistent two-tile kernel (fwd_persist.cu): one CTA per SM walking the same work list.
  const bool persist = !wide && !pack && g_persistent.load() && g_poly.load() == 0;
  // Grouped decode at d = 128: the one-tile kernel (S of the next key block overlaps the
  // softmax of this one) unless the two-tile kernel is chosen.
  const bool pack_one_tile = pack && d == 128 && g_decode_one_tile.load();
  cudaError_t e;
  if (pack_one_tile) {
    e = launch_fwd_wide(maps, p, d, (int)grid, st);
  } else if (persist) {
    p.o_ptr = o;
    const long long entries = grid;
    const long long pgrid = std::min<long long>(entries, std::max(1, s->sms));
    e = launch_fwd_persistent(maps, p, d, (int)pgrid, (int)entries, st);
  } else {
    e = wide ? launch_fwd_wide(maps, p, d, (int)grid, st) : launch_fwd(maps, p, d, pack ? 0 : g_poly.load(), (int)grid, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  if (pack && (e = launch_fwd_merge(p, d, o, st)) != cudaSuccess) return cuda_fail(e, "forward merge launch");
  return post_launch(s, st);
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N,
             int d, int causal, float scale, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, N, N, d, causal, scale, nullptr, 0, stream);
}

size_t attn_fwd_kv_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int d) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Nq < 0 || Nk < 0 ||
      (d != 64 && d != 128 && d != 192 && d != 256)) {
    set_last_error("attn_fwd_kv_workspace_size: invalid sizes");
    return (size_t)-1;
  }
  const DevSyms* s = dev_syms(nullptr);
  const int sms = s->err == cudaSuccess ? std::max(1, s->sms) : 1;
  return kv_plan(B, Hq, Hkv, Nq, Nk, d, sms).ws_bytes;
}

int attn_fwd_kv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                int Nk, int d, int causal, float scale, void* workspace, size_t workspace_bytes, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, causal, scale, workspace, workspace_bytes, stream);
}

// Packed variable-length sequences.  The unit table's size is bounded from the packed
// length alone: sum_b ceil(nq_b / 128) <= floor(total_q / 128) + B tiles per head.
static long long varlen_cap(int B, int Hq, int Hkv, int total_q, int d) {
  const int g = Hq / Hkv;
  const bool pair = g >= 2 && g % 2 == 0;
  const long long tiles = (long long)total_q / 128 + B;
  if (d > 128) return tiles * Hq;   // one tile per record (the one-tile kernel)
  return pair ? tiles * (Hq / 2) : ((tiles + B + 1) / 2) * Hq;
}
static constexpr size_t kVarlenHeader = 256;   // [0] records, [1] offsets invalid

size_t attn_fwd_varlen_workspace_size(int B, int Hq, int Hkv, int total_q, int d) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || total_q < 0 ||
      (d != 64 && d != 128 && d != 192 && d != 256)) {
    set_last_error("attn_fwd_varlen_workspace_size: invalid sizes");
    return (size_t)-1;
  }
  if (B == 0 || total_q == 0) return 0;
  return kVarlenHeader + (size_t)varlen_cap(B, Hq, Hkv, total_q, d) * sizeof(int4);
}

int attn_set_fwd_persistent(int enable) {
  g_persistent.store(enable ? 1 : 0);
  return ATTN_OK;
}

int attn_set_decode_one_tile(int enable) {
  g_decode_one_tile.store(enable ? 1 : 0);
  return ATTN_OK;
}

int attn_set_fwd_one_tile(int enable) {
  g_one_tile_d128.store(enable ? 1 : 0);
  return ATTN_OK;
}

int attn_set_varlen_order(int longest_first) {
  g_varlen_lpt.store(longest_first ? 1 : 0);
  return ATTN_OK;
}

int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                    const int* cu_seqlens_k, int B, int Hq, int Hkv, int total_q, int total_k, int d, int causal,
                    float scale, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_shape(B, Hq, Hkv, total_q, d, scale, true);
  if (rc != ATTN_OK) return rc;
  if (total_k < 0) return fail(ATTN_ERR_INVALID_ARG, "total_k=%d must be >= 0", total_k);
  if (total_q > 0x7fffff00 || total_k > 0x7fffff00)
    return fail(ATTN_ERR_INVALID_ARG, "packed lengths must stay below 2^31 - 256 rows");
  if (Hq > 65535) return fail(ATTN_ERR_UNSUPPORTED, "Hq=%d: packed sequences support at most 65535 heads", Hq);
  if (B == 0 || total_q == 0) return ATTN_OK;
  if (total_k == 0) return fail(ATTN_ERR_INVALID_ARG, "total_k=0 with %d queries: the softmax has no keys", total_q);
  if (!q || !k || !v || !o || !lse || !cu_seqlens_q || !cu_seqlens_k)
    return fail(ATTN_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(ATTN_ERR_MISALIGNED, "q, k, v, o and lse must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(cu_seqlens_q) | reinterpret_cast<uintptr_t>(cu_seqlens_k)) & 3u)
    return fail(ATTN_ERR_MISALIGNED, "cu_seqlens_q and cu_seqlens_k must be 4-byte aligned");
  const long long cap = varlen_cap(B, Hq, Hkv, total_q, d);
  const size_t need = kVarlenHeader + (size_t)cap * sizeof(int4);
  if (!workspace || workspace_bytes < need)
    return fail(ATTN_ERR_WORKSPACE, "workspace of %zu bytes given, %zu needed", workspace_bytes, need);
  if (!aligned16(workspace)) return fail(ATTN_ERR_MISALIGNED, "workspace must be 16-byte aligned");
  if (cap > 0x7fffffffLL) return fail(ATTN_ERR_INVALID_ARG, "problem too large for one launch");
  int dev = 0;
  const DevSyms* s = dev_syms(&dev);
  if (s->err != cudaSuccess) return cuda_fail(s->err, "device setup");

  FwdMaps maps;
  if ((rc = make_map(&maps.q, q, d, total_q, Hq, "q")) != ATTN_OK) return rc;
  if ((rc = make_map(&maps.k, k, d, total_k, Hkv, "k")) != ATTN_OK) return rc;
  if ((rc = make_map(&maps.v, v, d, total_k, Hkv, "v")) != ATTN_OK) return rc;
  if ((rc = make_map(&maps.o, o, d, total_q, Hq, "o")) != ATTN_OK) return rc;

  char* w = static_cast<char*>(workspace);
  FwdParams p{};
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = total_q; p.g = Hq / Hkv;
  p.Nk = total_k; p.koff = 0;
  p.causal = causal ? 1 : 0;
  p.pair_heads = (p.g >= 2 && p.g % 2 == 0) ? 1 : 0;
  p.pack = 2;
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.vl_count = reinterpret_cast<const int*>(w);
  p.vl_units = reinterpret_cast<const int4*>(w + kVarlenHeader);
  p.o_ptr = o;
  p.q_tile_bytes = (unsigned)((d / 64) * 128 * 128);
  p.c = scale * 1.4426950408889634f;
  p.tau = g_tau.load();
  p.lse = lse;
  p.wait_ns = (unsigned long long)g_wait_ns.load();
  p.status = s->status;
  p.rescale_count = g_count_rescales.load() ? s->rescale : nullptr;
  p.test_skip_first_kv = g_test_skip_kv.load();

  VarlenSched sc{};
  sc.cu_q = cu_seqlens_q;
  sc.cu_k = cu_seqlens_k;
  const bool wide = d > 128;        // one query tile per CTA (the one-tile kernel)
  sc.backward = 0;
  sc.single = wide ? 1 : 0;
  sc.B = B; sc.Hq = Hq; sc.Hkv = Hkv; sc.pair_heads = wide ? 0 : p.pair_heads; sc.causal = p.causal;
  sc.total_q = total_q; sc.total_k = total_k;
  sc.nbins = (int)std::min<long long>((total_k + 127LL) / 128 + 1, 32768LL);   // classes: a sequence's key blocks
  sc.cap = (int)cap;
  sc.lpt = g_varlen_lpt.load();
  sc.header = reinterpret_cast<int*>(w);
  sc.units = reinterpret_cast<int4*>(w + kVarlenHeader);
  sc.status = s->status;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_varlen_schedule(sc, st);
  if (e != cudaSuccess) return cuda_fail(e, "unit table launch");
  e = wide ? launch_fwd_wide(maps, p, d, (int)cap, st) : launch_fwd(maps, p, d, 0, (int)cap, st);
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  return post_launch(s, st);
}

int attn_quantize_fp8(const void* x, void* x8, float* scales, int B, int H, int N, int d, void* stream) {
  if (B < 0 || H <= 0 || N < 0) return fail(ATTN_ERR_INVALID_ARG, "B=%d, H=%d, N=%d: need B, N >= 0 and H >= 1", B, H, N);
  if (d != 128) return fail(ATTN_ERR_UNSUPPORTED, "head dim d=%d (the FP8 path supports 128)", d);
  if (B == 0 || N == 0) return ATTN_OK;
  if ((long long)B * H * ((N + 127) / 128) > 0x7fffffffLL) return fail(ATTN_ERR_INVALID_ARG, "too many blocks");
  if (!x || !x8 || !scales) return fail(ATTN_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(x) || !aligned16(x8) || (reinterpret_cast<uintptr_t>(scales) & 3u))
    return fail(ATTN_ERR_MISALIGNED, "x and x8 must be 16-byte aligned, scales 4-byte aligned");
  cudaError_t e = launch_quantize_fp8(x, x8, scales, (long long)B * H, N, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantiser launch");
  return ATTN_OK;
}

int attn_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* q_scale, const float* k_scale,
                 const float* v_scale, void* o, float* lse, int B, int Hq, int Hkv, int N, int d, int causal,
                 float scale, void* stream) {
  int rc = check_shape(B, Hq, Hkv, N, d == 128 ? 128 : 0, scale);
  if (rc != ATTN_OK) {
    if (d != 128) return fail(ATTN_ERR_UNSUPPORTED, "head dim d=%d (the FP8 path supports 128)", d);
    return rc;
  }
  if (B == 0 || N == 0) return ATTN_OK;
  if (!q8 || !k8 || !v8 || !q_scale || !k_scale || !v_scale || !o || !lse)
    return fail(ATTN_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8) || !aligned16(o) || !aligned16(lse))
    return fail(ATTN_ERR_MISALIGNED, "q8, k8, v8, o and lse must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(q_scale) | reinterpret_cast<uintptr_t>(k_scale) |
       reinterpret_cast<uintptr_t>(v_scale)) & 3u)
    return fail(ATTN_ERR_MISALIGNED, "the scale arrays must be 4-byte aligned");
  int dev = 0;
  const DevSyms* s = dev_syms(&dev);
  if (s->err != cudaSuccess) return cuda_fail(s->err, "device setup");
  FwdMaps maps;
  if ((rc = make_map_e4m3(&maps.q, q8, N, (long long)B * Hq, "q8")) != ATTN_OK) return rc;
  if ((rc = make_map_e4m3(&maps.k, k8, N, (long long)B * Hkv, "k8")) != ATTN_OK) return rc;
  if ((rc = make_map_e4m3(&maps.v, v8, N, (long long)B * Hkv, "v8")) != ATTN_OK) return rc;
  if ((rc = make_map(&maps.o, o, 128, N, (long long)B * Hq, "o")) != ATTN_OK) return rc;
  FwdParams p{};
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = N; p.g = Hq / Hkv;
  p.Nk = N; p.koff = 0;
  p.causal = causal ? 1 : 0;
  p.pair_heads = (p.g >= 2 && p.g % 2 == 0) ? 1 : 0;
  p.n_qblk = (N + 127) / 128;
  p.n_kvblk = p.n_qblk;
  p.n_rowslots = p.pair_heads ? p.n_qblk : (p.n_qblk + 1) / 2;
  p.units_per_row = p.pair_heads ? B * (Hq / 2) : B * Hq;
  p.c = scale * 1.4426950408889634f;
  p.tau = g_tau.load();
  p.lse = lse;
  p.wait_ns = (unsigned long long)g_wait_ns.load();
  p.status = s->status;
  p.rescale_count = g_count_rescales.load() ? s->rescale : nullptr;
  p.test_skip_first_kv = g_test_skip_kv.load();
  // Two-tile units, the last partial wave split into one-tile CTAs (as attn_fwd).
  const long long units = (long long)p.n_rowslots * p.units_per_row;
  p.split_from = (int)std::min<long long>(units, 0x7fffffffLL);
  if (!p.causal) {
    const long long sms = std::max(1, s->sms);
    const long long rem = units % sms;
    if (units >= sms && rem > 0 && 2 * rem <= sms) p.split_from = (int)(units - rem);
    else if (units < sms && 2 * units <= sms) p.split_from = 0;
  }
  const long long grid = p.split_from + 2 * (units - p.split_from);
  if (grid > 0x7fffffffLL) return fail(ATTN_ERR_INVALID_ARG, "problem too large for one launch");
  p.prefetch_ahead = std::max(1, s->sms);
  const Fp8Scales sc{q_scale, k_scale, v_scale};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_fwd_fp8(maps, p, sc, (int)grid, st);
  if (e != cudaSuccess) return cuda_fail(e, "FP8 forward launch");
  return post_launch(s, st);
}

int attn_exp2_sw(const float* x, float* y, long long n, int variant, void* stream) {
  if (n < 0) return fail(ATTN_ERR_INVALID_ARG, "n must be >= 0");
  if (n > 0 && (!x || !y)) return fail(ATTN_ERR_INVALID_ARG, "null pointer");
  if (variant < 0 || variant > 2) return fail(ATTN_ERR_INVALID_ARG, "variant must be 0, 1 or 2");
  cudaError_t e = launch_exp2_test(x, y, n, variant, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "exp2 launch");
  return ATTN_OK;
}

}  // extern "C"

extern "C" {

size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int N, int d, int deterministic) {
  if (check_shape(B, Hq, Hkv, N, d, 1.0f, true) != ATTN_OK) return (size_t)-1;
  if (B == 0 || N == 0) return 0;
  if (d > 128) return bwd_wide_workspace_bytes(B, Hq, N, d, deterministic);
  // Enough for either query-tile choice (attn_set_bwd_query_tile), so that a workspace sized
  // once serves both.
  return std::max(bwd_workspace_bytes(B, Hq, Hkv, N, d, deterministic),
                  bwd_wide_workspace_bytes(B, Hq, N, d, deterministic));
}

int attn_set_bwd_query_tile(int rows) {
  if (rows != 64 && rows != 128) return fail(ATTN_ERR_INVALID_ARG, "query tile rows=%d (64 or 128)", rows);
  g_bwd_tile_rows.store(rows);
  return ATTN_OK;
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
             void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d, int causal, float scale,
             int deterministic, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_shape(B, Hq, Hkv, N, d, scale, true);
  if (rc != ATTN_OK) return rc;
  if (B == 0 || N == 0) return ATTN_OK;
  // 64-row query tiles (bwd_wide.cu): always for d = 192, 256; for d <= 128 when chosen.
  const bool wide = d > 128 || g_bwd_tile_rows.load() == 64;
  const size_t need = wide ? bwd_wide_workspace_bytes(B, Hq, N, d, deterministic)
                           : bwd_workspace_bytes(B, Hq, Hkv, N, d, deterministic);
  if (!workspace || workspace_bytes < need)
    return fail(ATTN_ERR_WORKSPACE, "workspace of %zu bytes given, %zu needed", workspace_bytes, need);
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return fail(ATTN_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace))
    return fail(ATTN_ERR_MISALIGNED, "every tensor and the workspace must be 16-byte aligned");
  int dev = 0;
  const DevSyms* s = dev_syms(&dev);
  if (s->err != cudaSuccess) return cuda_fail(s->err, "device setup");
  BwdMaps maps;
  const int qrows = wide ? 64 : 128;   // query tile rows of the kernel
  if ((rc = make_map(&maps.q, q, d, N, (long long)B * Hq, "q", qrows)) != ATTN_OK) return rc;
  if ((rc = make_map(&maps.k, k, d, N, (long long)B * Hkv, "k")) != ATTN_OK) return rc;
  if ((rc = make_map(&maps.v, v, d, N, (long long)B * Hkv, "v")) != ATTN_OK) return rc;
  if ((rc = make_map(&maps.dout, dout, d, N, (long long)B * Hq, "dout", qrows)) != ATTN_OK) return rc;
  if ((rc = make_map(&maps.dk, dk, d, N, (long long)B * Hkv, "dk")) != ATTN_OK) return rc;
  if ((rc = make_map(&maps.dv, dv, d, N, (long long)B * Hkv, "dv")) != ATTN_OK) return rc;
  BwdParams p{};
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = N; p.g = Hq / Hkv; p.D = d;
  p.causal = causal ? 1 : 0;
  p.deterministic = deterministic ? 1 : 0;
  p.scale = scale;
  p.c = scale * 1.4426950408889634f;
  p.q = q; p.k = k; p.v = v; p.o = o; p.dout = dout; p.lse = lse;
  p.dq = dq; p.dk = dk; p.dv = dv;
  if (wide) bwd_wide_workspace_carve(workspace, B, Hq, N, d, deterministic, &p);
  else bwd_workspace_carve(workspace, B, Hq, Hkv, N, d, deterministic, &p);
  p.wait_ns = (unsigned long long)g_wait_ns.load();
  p.status = s->status;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = wide ? launch_bwd_wide(maps, p, st) : launch_bwd(maps, p, st);
  if (e == cudaErrorNotSupported) return fail(ATTN_ERR_UNSUPPORTED, "backward not available for these arguments");
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  return post_launch(s, st);
}

}  // extern "C"

extern "C" {

size_t attn_bwd_varlen_workspace_size(int B, int Hq, int Hkv, int total_q, int total_k, int d, int deterministic) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || total_q < 0 || total_k < 0 || (d != 64 && d != 128)) {
    set_last_error("attn_bwd_varlen_workspace_size: invalid sizes");
    return (size_t)-1;
  }
  if (B == 0 || (total_q == 0 && total_k == 0)) return 0;
  return bwd_varlen_layout(B, Hq, Hkv, total_q, total_k, d, deterministic).total;
}

int attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                    void* dq, void* dk, void* dv, const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int Hq,
                    int Hkv, int total_q, int total_k, int d, int causal, float scale, int deterministic,
                    void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_shape(B, Hq, Hkv, total_q, d, scale);
  if (rc != ATTN_OK) return rc;
  if (total_k < 0) return fail(ATTN_ERR_INVALID_ARG, "total_k=%d must be >= 0", total_k);
  if (total_q > 0x7fffff00 || total_k > 0x7fffff00)
    return fail(ATTN_ERR_INVALID_ARG, "packed lengths must stay below 2^31 - 256 rows");
  if (B == 0 || (total_q == 0 && total_k == 0)) return ATTN_OK;
  if (total_k == 0) return fail(ATTN_ERR_INVALID_ARG, "total_k=0 with %d queries: the softmax has no keys", total_q);
  const BwdVarlenLayout L = bwd_varlen_layout(B, Hq, Hkv, total_q, total_k, d, deterministic);
  if (!workspace || workspace_bytes < L.total)
    return fail(ATTN_ERR_WORKSPACE, "workspace of %zu bytes given, %zu needed", workspace_bytes, L.total);
  // With no queries at all the query-side tensors are empty and may be NULL.
  if (total_q == 0) {
    q = o = dout = k;
    dq = const_cast<void*>(k);
    lse = static_cast<const float*>(k);
  }
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !cu_seqlens_q || !cu_seqlens_k)
    return fail(ATTN_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace))
    return fail(ATTN_ERR_MISALIGNED, "every tensor and the workspace must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(cu_seqlens_q) | reinterpret_cast<uintptr_t>(cu_seqlens_k)) & 3u)
    return fail(ATTN_ERR_MISALIGNED, "cu_seqlens_q and cu_seqlens_k must be 4-byte aligned");
  if (L.cap > 0x7fffffffLL || (long long)Hq * L.sem_stride > 0x7fffffffLL)
    return fail(ATTN_ERR_INVALID_ARG, "problem too large for one launch");
  int dev = 0;
  const DevSyms* s = dev_syms(&dev);
  if (s->err != cudaSuccess) return cuda_fail(s->err, "device setup");
  // Tensor maps over the packed views (with no queries, one-row maps that are never read).
  BwdMaps maps;
  const int tq = std::max(total_q, 1), tk = total_k;
  if ((rc = make_map(&maps.q, q, d, tq, Hq, "q")) != ATTN_OK) return rc;
  if ((rc = make_map(&maps.dout, dout, d, tq, Hq, "dout")) != ATTN_OK) return rc;
  if ((rc = make_map(&maps.k, k, d, tk, Hkv, "k")) != ATTN_OK) return rc;
  if ((rc = make_map(&maps.v, v, d, tk, Hkv, "v")) != ATTN_OK) return rc;
  if ((rc = make_map(&maps.dk, dk, d, tk, Hkv, "dk")) != ATTN_OK) return rc;
  if ((rc = make_map(&maps.dv, dv, d, tk, Hkv, "dv")) != ATTN_OK) return rc;

  char* w = static_cast<char*>(workspace);
  BwdParams p{};
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = total_q; p.g = Hq / Hkv; p.D = d;
  p.causal = causal ? 1 : 0;
  p.deterministic = deterministic ? 1 : 0;
  p.scale = scale;
  p.c = scale * 1.4426950408889634f;
  p.q = q; p.k = k; p.v = v; p.o = o; p.dout = dout; p.lse = lse;
  p.dq = dq; p.dk = dk; p.dv = dv;
  p.dq_acc = reinterpret_cast<float*>(w + L.dq_acc);
  p.delta = reinterpret_cast<float*>(w + L.delta);
  p.lse2 = reinterpret_cast<float*>(w + L.lse2);
  p.sem = deterministic ? reinterpret_cast<int*>(w + L.sem) : nullptr;
  p.wait_ns = (unsigned long long)g_wait_ns.load();
  p.status = s->status;
  p.varlen = 1;
  p.total_k = total_k;
  p.sem_stride = L.sem_stride;
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.vl_count = reinterpret_cast<const int*>(w + L.table);
  p.vl_units = reinterpret_cast<const int4*>(w + L.table + kVarlenHeader);

  VarlenSched sc{};
  sc.cu_q = cu_seqlens_q;
  sc.cu_k = cu_seqlens_k;
  sc.backward = 1;
  sc.B = B; sc.Hq = Hq; sc.Hkv = Hkv; sc.pair_heads = 0; sc.causal = p.causal;
  sc.total_q = total_q; sc.total_k = total_k;
  sc.nbins = (int)std::min<long long>((total_k + 127LL) / 128 + 1, 32768LL);   // classes: a sequence's key blocks
  sc.cap = (int)L.cap;
  sc.lpt = g_varlen_lpt.load();
  sc.header = reinterpret_cast<int*>(w + L.table);
  sc.units = reinterpret_cast<int4*>(w + L.table + kVarlenHeader);
  sc.status = s->status;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_varlen_schedule(sc, st);
  if (e != cudaSuccess) return cuda_fail(e, "unit table launch");
  e = launch_bwd(maps, p, st);
  if (e == cudaErrorNotSupported) return fail(ATTN_ERR_UNSUPPORTED, "backward not available for these arguments");
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  return post_launch(s, st);
}

}  // extern "C"
