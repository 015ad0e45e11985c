// The unit table for packed variable-length sequences: which two 128-row query tiles
// each CTA of the forward takes, or which key block each CTA of the backward takes,
// longest first.
//
// "FlashAttention-4 explained", section 06 (scheduling): sequences of different lengths
// give CTAs of very different amounts of work, and starting the largest first keeps short
// ones from leaving the last wave to a few long CTAs.  The order is longest sequence
// first (by its key blocks), and within a sequence its heaviest CTAs first: for the
// forward the tiles with the most visible keys (causal: the last rows), for the backward
// the key blocks seen by the most query tiles (causal: the first blocks).  The CTAs of a
// sequence and head then run side by side and share its K/V (forward) or Q/dO (backward)
// tiles in L2; ordering every CTA by its own work instead spread them over many heads and
// measured 23 % slower for the causal backward.  The lengths are known only once the
// offsets are on the device, so one CTA builds the order there: a counting sort over
// work classes, without a host round trip.
//
// Forward records: {b, hq0 | hq1 << 16, r0, r1}: tiles starting at rows r0 and r1 of
// sequence b (query heads hq0 and hq1; r1 < 0 when the sequence's last tile has no
// partner).  The pairing is the ordinary forward's: two query heads of one K/V group on
// the same rows when the group size is even, otherwise two consecutive row tiles of one
// head; with `single` (the one-tile kernel of wide heads) a record is one tile of one
// head, {b, hq | hq << 16, r0, -1}.  Backward records: {b, hkv, n, 0}: key block n of
// sequence b and K/V head hkv.
#include <cstdint>
#include <mutex>

#include "kernels.h"

namespace attn {
namespace {

constexpr int kSchedThreads = 1024;

// One pass over every (sequence, slot): PHASE 0 counts the records of each class (the
// sequence's key blocks), PHASE 1 reserves their places (hist then holds each class's
// next free index) and writes them.  Warps take sequences, lanes take a sequence's slots
// (forward: row slots, last first, one record per query head or head pair; backward: key
// blocks, first first, one record per K/V head).  A sequence's slots share its class; the
// lanes of a warp take consecutive places in lane order, one atomic per round, and a
// warp's rounds follow one another, so a sequence's records keep the slot order.  The
// deterministic backward relies on this: its key block n waits for block n - 1's
// additions, so block n - 1 must never be placed after block n.
template <int PHASE>
__device__ void visit_slots(const VarlenSched& s, int* hist) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = s.backward ? s.Hkv : (s.pair_heads ? s.Hq / 2 : s.Hq);
  const bool one_row = s.single || s.pair_heads;   // a slot is one row tile
  for (int b = warp; b < s.B; b += kSchedThreads / 32) {
    const int q0 = s.cu_q[b], nq = s.cu_q[b + 1] - q0;
    const int nk = s.cu_k[b + 1] - s.cu_k[b];
    const int tiles = (nq + 127) / 128;
    const int slots = s.backward ? (nk + 127) / 128 : (one_row ? tiles : (tiles + 1) / 2);
    const int work = s.lpt ? min((nk + 127) / 128, s.nbins - 1) : 0;
    for (int base = 0; base < slots; base += 32) {
      const int i = base + lane;
      const bool act = i < slots;
      const int sl = s.backward ? i : slots - 1 - i;
      int r0 = 0, r1 = -1;
      if (s.backward) {
        r0 = sl;
      } else if (s.single) {
        r0 = sl * 128;
      } else {
        r0 = s.pair_heads ? sl * 128 : sl * 256;
        r1 = s.pair_heads ? r0 : (r0 + 128 < nq ? r0 + 128 : -1);
      }
      const int bin = act ? s.nbins - 1 - work : -1;   // ascending bins = descending work
      const unsigned grp = __match_any_sync(0xffffffffu, bin);
      const int leader = __ffs(grp) - 1;
      const int rank = __popc(grp & ((1u << lane) - 1u));
      int first = 0;
      if (act && lane == leader) first = atomicAdd(&hist[bin], __popc(grp) * per);
      first = __shfl_sync(0xffffffffu, first, leader);
      if constexpr (PHASE == 1) {
        if (act) {
          const int pos = first + rank * per;
          for (int u = 0; u < per; ++u) {
            if (pos + u >= s.cap) break;
            if (s.backward) {
              s.units[pos + u] = make_int4(b, u, r0, 0);
            } else {
              const int hq0 = s.pair_heads ? 2 * u : u;
              const int hq1 = s.pair_heads ? 2 * u + 1 : u;
              s.units[pos + u] = make_int4(b, hq0 | (hq1 << 16), r0, r1);
            }
          }
        }
      }
      __syncwarp();
    }
  }
}

__global__ void __launch_bounds__(kSchedThreads, 1) varlen_schedule_kernel(const VarlenSched s) {
  extern __shared__ int hist[];                 // [nbins]
  __shared__ int bad;
  __shared__ int warp_sum[kSchedThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) bad = 0;
  for (int i = tid; i < s.nbins; i += kSchedThreads) hist[i] = 0;
  __syncthreads();

  // Offsets: start at 0, never decrease, end at the packed lengths; a sequence with
  // queries has keys, and a causal one at least as many keys as queries.  Together these
  // keep every row the forward touches inside the packed tensors.
  for (int b = tid; b < s.B; b += kSchedThreads) {
    const int q0 = s.cu_q[b], q1 = s.cu_q[b + 1], k0 = s.cu_k[b], k1 = s.cu_k[b + 1];
    bool ok = q1 >= q0 && k1 >= k0 && (q1 == q0 || k1 > k0) && (!s.causal || k1 - k0 >= q1 - q0);
    if (b == 0) ok = ok && q0 == 0 && k0 == 0;
    if (b == s.B - 1) ok = ok && q1 == s.total_q && k1 == s.total_k;
    if (!ok) bad = 1;
  }
  __syncthreads();
  if (bad) {
    if (tid == 0) {
      s.header[0] = 0;
      s.header[1] = 1;
      atomicExch(s.status, DEV_BAD_OFFSETS);
    }
    return;
  }

  visit_slots<0>(s, hist);
  __syncthreads();

  // Exclusive scan of the class counts: thread t owns bins [t*C, (t+1)*C).
  const int C = (s.nbins + kSchedThreads - 1) / kSchedThreads;
  const int lo = min(tid * C, s.nbins), hi = min(lo + C, s.nbins);
  int mine = 0;
  for (int i = lo; i < hi; ++i) mine += hist[i];
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    warp_sum[lane] = w;                          // inclusive over warps
  }
  __syncthreads();
  int run = incl - mine + (warp > 0 ? warp_sum[warp - 1] : 0);
  const int total = warp_sum[kSchedThreads / 32 - 1];
  for (int i = lo; i < hi; ++i) {
    const int c = hist[i];
    hist[i] = run;
    run += c;
  }
  __syncthreads();

  visit_slots<1>(s, hist);
  if (tid == 0) {
    s.header[0] = min(total, s.cap);
    s.header[1] = 0;
  }
}

}  // namespace

cudaError_t launch_varlen_schedule(const VarlenSched& s, cudaStream_t stream) {
  const size_t smem = (size_t)s.nbins * sizeof(int);
  static std::once_flag flags[64];
  static cudaError_t attr_err[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::call_once(flags[dev & 63], [&] {
    attr_err[dev & 63] = cudaFuncSetAttribute(varlen_schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              128 * 1024);
  });
  if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
  if (smem > 128 * 1024) return cudaErrorInvalidValue;
  varlen_schedule_kernel<<<1, kSchedThreads, smem, stream>>>(s);
  return cudaGetLastError();
}

}  // namespace attn
