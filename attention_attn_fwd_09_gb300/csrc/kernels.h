// Launch interfaces shared between the host entry points (api.cu) and the kernel
// translation units.  Host-only types; no torch.
#pragma once
#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

// Launches `kernel` as a programmatic dependent of the stream's previous kernel: its CTAs
// may be scheduled once every CTA of that kernel has called pdl_trigger (or exited), and
// they must call pdl_wait before touching anything the previous kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Device status word codes (see attn_device_status).  Kernels never trap: a kernel that
// gives up on a bounded wait, or finds its device-side arguments invalid, writes one of
// these and returns.
enum : int { DEV_OK = 0, DEV_TIMEOUT = 1, DEV_BAD_OFFSETS = 2 };

struct FwdParams {
  int B, Hq, Hkv, N, g;      // N: query length
  int Nk, koff;              // key length and Nk - N (query i stands at key position i + koff)
  int causal;
  int pair_heads;          // 1: a CTA's two tiles are query heads 2p, 2p+1 of one KV group
  int n_qblk, n_kvblk;     // ceil(N / 128), ceil(Nk / 128)
  int units_per_row;       // CTAs per query-row slot (see fwd.cu unit mapping)
  int n_rowslots;          // query-row slots per head (pair) sequence
  int split_from;          // units >= split_from run as two one-tile CTAs (the last, partial wave)
  int prefetch_ahead;      // > 0: a CTA prefetches into L2 the first tiles of CTA blockIdx + this
  // Grouped decode mode (queries after a key cache, g * N <= 128): one CTA per (K/V head,
  // key split) with one tile holding the group's g query heads x N queries; each CTA writes
  // a normalised partial O and LSE for its key range, merged by launch_fwd_merge.
  int pack;                // 0 ordinary, 1 grouped decode, 2 packed variable-length sequences
  int kv_splits, blocks_per_split;
  unsigned q_tile_bytes;   // bytes one Q tile load delivers (a full tile, or g * N rows of it)
  float* part_o;           // [kv_splits][B * Hkv][128][D] fp32
  float* part_lse;         // [kv_splits][B * Hkv][128] fp32, natural log
  // Packed variable-length mode (pack == 2): Q/O [Hq, N, D], K/V [Hkv, Nk, D] with N and Nk
  // the packed lengths; each CTA takes one record of the unit table written by
  // launch_varlen_schedule (CTAs past *vl_count have no record and exit at once).
  const int* cu_q;         // [B + 1] query row offsets (device)
  const int* cu_k;         // [B + 1] key row offsets (device)
  const int* vl_count;     // records in the table
  const int4* vl_units;    // {b, hq0 | hq1 << 16, r0, r1}: rows r0, r1 of sequence b (r1 < 0: one tile)
  void* o_ptr;             // O, for tiles that end inside their sequence (plain stores)
  float c;                 // scale * log2(e)
  float tau;               // conditional-rescale threshold, log2 units
  float* lse;              // [B, Hq, N] fp32, natural log
  unsigned long long wait_ns;
  int* status;
  unsigned long long* rescale_count;  // optional counter (nullptr = off)
  int test_skip_first_kv;             // test hook: never load ring index 0 (exercises timeouts)
};

struct FwdMaps {
  CUtensorMap q, k, v, o;
};

// Forward: D in {64, 128}; poly_per_16 in {0, 4, 16} elements of every 16 computed by
// the FMA polynomial instead of MUFU.EX2.
cudaError_t launch_fwd(const FwdMaps& maps, const FwdParams& p, int D, int poly_per_16, int grid,
                       cudaStream_t stream);
// Grouped decode mode: combine the kv_splits partial results into o [B,Hq,N,D] bf16 and
// lse [B,Hq,N] fp32.
cudaError_t launch_fwd_merge(const FwdParams& p, int D, void* o, cudaStream_t stream);

// Packed variable-length mode: the unit table.  One CTA validates the offsets and writes
// one record per CTA, longest sequence first: for the forward two 128-row query tiles of
// one sequence, for the backward one 128-key block of one sequence and K/V head.
struct VarlenSched {
  const int* cu_q;
  const int* cu_k;
  int backward;            // 0: forward records; 1: backward records {b, hkv, key block, 0}
  int single;              // forward: one query tile per record (the one-tile kernel, d > 128)
  int B, Hq, Hkv, pair_heads, causal, total_q, total_k;
  int nbins;               // work classes (a sequence's key blocks, clamped to nbins - 1)
  int cap;                 // records the table can hold
  int lpt;                 // 1: longest first; 0: every record in one class (arrival order)
  int* header;             // [0] records written; [1] 0, or 1 when the offsets were invalid
  int4* units;             // [cap] records
  int* status;             // device status word (DEV_BAD_OFFSETS on invalid offsets)
};
cudaError_t launch_varlen_schedule(const VarlenSched& s, cudaStream_t stream);
size_t fwd_smem_bytes(int D);
// Persistent two-tile forward (fwd_persist.cu), d = 64 or 128, ordinary mode, MUFU
// exponentials: grid CTAs walk entries 0 .. n_entries - 1 of the work list (units below
// p.split_from whole, then one-tile halves) in steps of grid; O is written through p.o_ptr.
cudaError_t launch_fwd_persistent(const FwdMaps& maps, const FwdParams& p, int D, int grid, int n_entries,
                                  cudaStream_t stream);
// One-tile forward (fwd_wide.cu) for d = 128, 192 or 256: one 128-row query tile per CTA,
// grid = B * Hq * ceil(N / 128); same parameters as launch_fwd.  pack == 1 (grouped decode,
// d = 128: grid = B * Hkv * kv_splits, then launch_fwd_merge) and pack == 2 (packed
// sequences, d = 192, 256: grid = the table's bound) as for launch_fwd.
cudaError_t launch_fwd_wide(const FwdMaps& maps, const FwdParams& p, int D, int grid, cudaStream_t stream);

// FP8 forward (fwd_fp8.cu), d = 128, ordinary tiling: Q/K/V maps over e4m3 bytes (boxes
// of 128 rows x 128 bytes), O map as for launch_fwd; block scales per 128 rows of a head.
struct Fp8Scales {
  const float* q;   // [B, Hq, ceil(N / 128)]
  const float* k;   // [B, Hkv, ceil(N / 128)]
  const float* v;   // [B, Hkv, ceil(N / 128)]
};
cudaError_t launch_fwd_fp8(const FwdMaps& maps, const FwdParams& p, const Fp8Scales& sc, int grid, cudaStream_t stream);
size_t fwd_fp8_smem_bytes();
// Block quantiser: x bf16 [heads, N, 128] -> x8 e4m3 [heads, N, 128], scales [heads, ceil(N / 128)].
cudaError_t launch_quantize_fp8(const void* x, void* x8, float* scales, long long heads, int N, cudaStream_t stream);

// Software exp2 accuracy / throughput test entry: variant 0 = production polynomial,
// 1 = full-range polynomial, 2 = MUFU ex2.approx.
cudaError_t launch_exp2_test(const float* x, float* y, long long n, int variant, cudaStream_t s);

// Backward.
struct BwdParams {
  int B, Hq, Hkv, N, g, D;
  int causal, deterministic;
  float scale, c;            // softmax scale; scale * log2(e)
  const void *q, *k, *v, *o, *dout;
  const float* lse;
  void *dq, *dk, *dv;
  float* dq_acc;             // [B, Hq, ceil(N/128)*128, D] fp32 workspace (rows padded to whole tiles)
  float* delta;              // [B, Hq, N] fp32 workspace (rowsum(dO o O))
  float* lse2;               // [B, Hq, N] fp32 workspace (LSE * log2 e)
  int* sem;                  // deterministic-order counters
  float* dq_acc2;            // deterministic, d <= 128, not packed: the second accumulator
                             // (shaped as dq_acc); null otherwise
  unsigned long long wait_ns;
  int* status;
  // Packed sequences (varlen = 1): N is total_q, Q/O/dO/dQ [Hq, total_q, D], K/V/dK/dV
  // [Hkv, total_k, D]; dq_acc is [Hq, total_q + 128 B, D] with sequence b's rows starting
  // at cu_q[b] + 128 b (room for its last tile's padding), sem [Hq][sem_stride].
  int varlen, total_k, sem_stride;
  const int* cu_q;
  const int* cu_k;
  const int* vl_count;
  const int4* vl_units;      // {b, hkv, key block n, 0}
};
struct BwdMaps {
  CUtensorMap q, k, v, dout, dk, dv;
};
cudaError_t launch_bwd(const BwdMaps& maps, const BwdParams& p, cudaStream_t stream);
size_t bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d, int deterministic);
// Packed sequences: workspace layout (dq_acc, delta, lse2, sem, then the unit table).
struct BwdVarlenLayout {
  size_t dq_acc, delta, lse2, sem, table, total;
  long long rows_pad, cap;
  int sem_stride;
};
BwdVarlenLayout bwd_varlen_layout(int B, int Hq, int Hkv, int total_q, int total_k, int d, int deterministic);
// Points p->dq_acc, delta, lse2, sem (and, deterministic, dq_acc2) into the caller's
// workspace.
void bwd_workspace_carve(void* ws, int B, int Hq, int Hkv, int N, int d, int deterministic, BwdParams* p);
// Backward for d = 192, 256 (bwd_wide.cu): maps as launch_bwd except q and dout, whose
// boxes are 64 rows; workspace: dQacc [B, Hq, ceil(N/64)*64, d], D and LSE2 [B, Hq, N],
// counters [B, Hq, ceil(N/64), 2] when deterministic.
size_t bwd_wide_workspace_bytes(int B, int Hq, int N, int d, int deterministic);
void bwd_wide_workspace_carve(void* ws, int B, int Hq, int N, int d, int deterministic, BwdParams* p);
cudaError_t launch_bwd_wide(const BwdMaps& maps, const BwdParams& p, cudaStream_t stream);

}  // namespace attn
