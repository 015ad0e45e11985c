// Fused exact attention backward for sm_103a: preprocess, main (tcgen05) and dQ convert.
//
// Stages ("Hotelren FA4 summary" section 4.2, the five-stage backward pipeline; the
// reverse-engineering page: P is recomputed, never stored):
//   preprocess  D_i = sum_d dO_id O_id, LSE2_i = LSE_i * log2(e), dQacc = 0, counters = 0
//               (dQacc rows are padded to whole 128-query tiles per head; the padding
//               rows take the zero dQ of the queries past N and are never read)
//   main        per CTA one key block of one K/V head, looping over the query tiles of
//               every query head of the group:
//                 S^T  = K Q^T                 (tcgen05, TMEM)
//                 dP^T = V dO^T                (tcgen05, TMEM)
//                 P^T  = exp2(S^T c - LSE2)    (exact probabilities, written back as bf16)
//                 dV  += P^T dO                (A = P^T from TMEM)
//                 dS^T = P^T o (dP^T - D)      (bf16, to shared memory)
//                 dK  += dS^T Q                (A = dS^T, K-major view of the tile)
//                 dQ^T = K^T dS^T              (both operands MN-major views of the K and
//                                               dS^T tiles: TMEM lane i holds column i of dQ)
//                 dQacc += dQ                  (fp32 red.global.add straight from TMEM
//                                               registers, one 128-byte line of a dQacc row
//                                               per warp instruction; in key-block order
//                                               when deterministic)
//               The transposed orientation (keys on TMEM lanes) makes every result land in
//               the layout its consumer reads ("FlashAttention-4 explained" section 05).
//   convert     dq = bf16(scale * dQacc)
// dK is scaled by `scale` in the main kernel's epilogue.
#include <algorithm>
#include <cstdint>
#include <mutex>
#include <type_traits>
#include <utility>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Deterministic mode splits a tile's contributions into up to this many classes, each with
// its own counter and accumulator (see the kernel).
constexpr int kDetMaxClasses = 4;
// Classes used for a non-causal head of nq query tiles (causal heads use one).  Measured on
// GB300 (B2 H16 d128, deterministic): four classes instead of two take N = 8192 from 3.27 to
// 3.08 ms and N = 16384 from 6.00 to 5.85 ms, but N = 2048 from 0.472 to 0.496 ms (the two
// extra accumulators' zeroing and reading weigh more on a short call).
static int det_classes(int nq) { return nq >= 64 ? 4 : 2; }

// Layout: dQacc [B, Hq, ceil(N/128)*128, d] fp32, delta and LSE2 [B, Hq, N] fp32, and when
// deterministic the counters [kDetMaxClasses][B, Hq, ceil(N/128)] and det_classes - 1 more
// accumulators shaped as dQacc, each starting on a 256-byte boundary.
size_t bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d, int deterministic) {
  (void)Hkv;
  const size_t rows = (size_t)B * Hq * N;
  const int tiles = (N + 127) / 128;
  const size_t nq = (size_t)B * Hq * tiles;
  size_t n = align256(nq * 128 * d * 4) + 2 * align256(rows * 4);
  if (deterministic) n += align256(kDetMaxClasses * nq * 4) + (det_classes(tiles) - 1) * align256(nq * 128 * d * 4);
  return n;
}

BwdVarlenLayout bwd_varlen_layout(int B, int Hq, int Hkv, int total_q, int total_k, int d, int deterministic) {
  BwdVarlenLayout L{};
  // Sequence b's accumulator rows start at cu_q[b] + 128 b: its last tile's padding fits
  // before the next sequence.  A tile id floor((cu_q[b] + 128 b) / 128) + m is unique per
  // (sequence, tile) and at most rows_pad / 128.
  L.rows_pad = (long long)total_q + 128LL * B;
  L.sem_stride = (int)(L.rows_pad / 128 + 1);
  L.cap = (long long)Hkv * ((long long)total_k / 128 + B);   // >= Hkv * sum_b ceil(nk_b / 128)
  size_t off = 0;
  L.dq_acc = off;
  off += align256((size_t)Hq * L.rows_pad * d * 4);
  L.delta = off;
  off += align256((size_t)Hq * total_q * 4);
  L.lse2 = off;
  off += align256((size_t)Hq * total_q * 4);
  L.sem = off;
  if (deterministic) off += align256((size_t)Hq * L.sem_stride * 4);
  L.table = off;
  off += 256 + (size_t)L.cap * 16;
  L.total = off;
  return L;
}

void bwd_workspace_carve(void* ws, int B, int Hq, int Hkv, int N, int d, int deterministic, BwdParams* p) {
  (void)Hkv;
  char* b = static_cast<char*>(ws);
  const size_t rows = (size_t)B * Hq * N;
  const size_t nq = (size_t)B * Hq * ((N + 127) / 128);
  p->dq_acc = reinterpret_cast<float*>(b);
  b += align256(nq * 128 * d * 4);
  p->delta = reinterpret_cast<float*>(b);
  b += align256(rows * 4);
  p->lse2 = reinterpret_cast<float*>(b);
  b += align256(rows * 4);
  p->sem = deterministic ? reinterpret_cast<int*>(b) : nullptr;
  b += deterministic ? align256(kDetMaxClasses * nq * 4) : 0;
  p->dq_acc2 = deterministic ? reinterpret_cast<float*>(b) : nullptr;
}

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Packed sequences: the sequence holding packed row r (0 <= r < cu[B]): the b with
// cu[b] <= r < cu[b + 1] (empty sequences are skipped).  Always in [0, B - 1].
__device__ __forceinline__ int seq_of(const int* __restrict__ cu, int B, int r) {
  int lo = 1, hi = B;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(cu + mid) > r) hi = mid;
    else lo = mid + 1;
  }
  return lo - 1;
}

// ------------------------------------------------------------------------------------
// Preprocess: one 16-thread group per row (d = 128: 8 bf16 per thread; d = 64: 4); the
// grid's y index walks the heads (bh), x the head's rows in groups of 16, so that no
// thread divides by N.
// ------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const uint16_t* __restrict__ o,
                                                              const uint16_t* __restrict__ dout,
                                                              const float* __restrict__ lse, float* __restrict__ delta,
                                                              float* __restrict__ lse2, float* __restrict__ dq_acc,
                                                              float* __restrict__ dq_extra, int n_extra,
                                                              long long extra_stride,
                                                              int* __restrict__ sem, long long rows, int N, int npad,
                                                              int n_sem, const int* __restrict__ cu_q, int nseq,
                                                              long long rows_pad) {
  constexpr int PER = D / 16;  // elements per thread
  // Launched as a programmatic dependent (of the forward, say): wait for the previous
  // kernel's writes (O, LSE, dO), then let the main kernel be scheduled.
  pdl_wait();
  pdl_trigger();
  const long long nthreads = (long long)gridDim.x * gridDim.y * blockDim.x;
  for (long long g = ((long long)blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x; g < n_sem;
       g += nthreads)
    sem[g] = 0;
  // Rows past N (the last group of a head) take part in the shuffles below with zeros and
  // store nothing.
  const int r = blockIdx.x * 16 + (threadIdx.x >> 4);   // row within the head
  const bool valid = r < N;
  const int sub = threadIdx.x & 15;
  const long long n_heads = rows / N;
  for (long long bh = blockIdx.y; bh < n_heads; bh += gridDim.y) {
  const long long row = bh * N + (valid ? r : 0);
  const uint16_t* orow = o + row * D + sub * PER;
  const uint16_t* drow = dout + row * D + sub * PER;
  float acc = 0.f;
  if constexpr (PER == 8) {
    const uint4 a = valid ? *reinterpret_cast<const uint4*>(orow) : make_uint4(0u, 0u, 0u, 0u);
    const uint4 b = valid ? *reinterpret_cast<const uint4*>(drow) : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = fmaf(__uint_as_float(av[i] << 16), __uint_as_float(bv[i] << 16), acc);
      acc = fmaf(__uint_as_float(av[i] & 0xffff0000u), __uint_as_float(bv[i] & 0xffff0000u), acc);
    }
  } else {
    const uint2 a = valid ? *reinterpret_cast<const uint2*>(orow) : make_uint2(0u, 0u);
    const uint2 b = valid ? *reinterpret_cast<const uint2*>(drow) : make_uint2(0u, 0u);
    const uint32_t av[2] = {a.x, a.y}, bv[2] = {b.x, b.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      acc = fmaf(__uint_as_float(av[i] << 16), __uint_as_float(bv[i] << 16), acc);
      acc = fmaf(__uint_as_float(av[i] & 0xffff0000u), __uint_as_float(bv[i] & 0xffff0000u), acc);
    }
  }
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, 16);
  if (!valid) continue;
  // Packed sequences (cu_q set): row r of sequence b sits at r + 128 b of its head's rows.
  const long long zrow = cu_q ? bh * rows_pad + r + 128LL * seq_of(cu_q, nseq, r) : bh * npad + r;
  float4* z = reinterpret_cast<float4*>(dq_acc + zrow * D + sub * PER);
#pragma unroll
  for (int i = 0; i < PER / 4; ++i) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int x = 0; x < n_extra; ++x) {
    float4* z2 = reinterpret_cast<float4*>(dq_extra + x * extra_stride + zrow * D + sub * PER);
#pragma unroll
    for (int i = 0; i < PER / 4; ++i) z2[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (sub == 0) {
    delta[row] = acc;
    lse2[row] = lse[row] * kLog2e;
  }
  }
}

// ------------------------------------------------------------------------------------
// Convert: dq = bf16(scale * dQacc), 8 elements per thread (dQacc rows padded per head);
// with more accumulators, dq = bf16(scale * (((dQacc + dQacc_1) + dQacc_2) + ...)), always in
// that order.  The grid's y index walks the heads, x the head's N x D / 8 groups of 8.
// ------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) bwd_convert_kernel(const float* __restrict__ acc,
                                                           const float* __restrict__ extra, int n_extra,
                                                           long long extra_stride, uint16_t* __restrict__ dq,
                                                           float scale, long long n8, int N, int npad,
                                                           const int* __restrict__ cu_q, int nseq, long long rows_pad) {
  pdl_wait();   // launched as a programmatic dependent of the main kernel
  constexpr int G8 = D / 8;                  // groups of 8 per row (a power of two)
  const long long n_heads = n8 / ((long long)N * G8);
  const int per_head = N * G8;
  for (long long bh = blockIdx.y; bh < n_heads; bh += gridDim.y)
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < per_head; e += gridDim.x * blockDim.x) {
    const int rr = e / G8, c8 = e & (G8 - 1);
    const long long i = bh * per_head + e;
    const long long arow = cu_q ? bh * rows_pad + rr + 128LL * seq_of(cu_q, nseq, rr) : bh * npad + rr;
    const long long src = arow * G8 + c8;
    float4 a = reinterpret_cast<const float4*>(acc)[2 * src];
    float4 b = reinterpret_cast<const float4*>(acc)[2 * src + 1];
    for (int x = 0; x < n_extra; ++x) {
      const float4* acc2 = reinterpret_cast<const float4*>(extra + x * extra_stride);
      const float4 a2 = acc2[2 * src];
      const float4 b2 = acc2[2 * src + 1];
      a = make_float4(a.x + a2.x, a.y + a2.y, a.z + a2.z, a.w + a2.w);
      b = make_float4(b.x + b2.x, b.y + b2.y, b.z + b2.z, b.w + b2.w);
    }
    uint4 r;
    r.x = pack_bf16x2(a.x * scale, a.y * scale);
    r.y = pack_bf16x2(a.z * scale, a.w * scale);
    r.z = pack_bf16x2(b.x * scale, b.y * scale);
    r.w = pack_bf16x2(b.z * scale, b.w * scale);
    reinterpret_cast<uint4*>(dq)[i] = r;
  }
}


// ------------------------------------------------------------------------------------
// Main backward kernel.
// Warps: 0 TMA producer, 1 MMA issuer, 2 TMEM allocator, 3 -LSE2/-D prefetch,
//        4-7 and 8-11 "compute" (P^T, dS^T; keys on TMEM lanes; queries 0-63 and 64-127),
//        12-15 "drain" (dQ^T -> dQacc).
// TMEM columns: S^T/P^T [0,128), dP^T then dQ^T [128,256), dV [256,256+D), dK [256+D,256+2D).
// ------------------------------------------------------------------------------------
constexpr int kBwdThreads = 512;

template <int D>
struct BwdCfg {
  static constexpr int NCH = D / 64;
  static constexpr uint32_t CHUNK = 128 * 128;        // 128 rows x 64 bf16
  static constexpr uint32_t TILE = CHUNK * NCH;       // 128 x D bf16
  static constexpr uint32_t DS_TILE = 2 * CHUNK;      // 128 keys x 128 queries bf16
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = TILE;
  static constexpr uint32_t OFF_STAGE = 2 * TILE;     // 2 stages x (Q tile, dO tile)
  static constexpr uint32_t OFF_DS = OFF_STAGE + 4 * TILE;
  static constexpr uint32_t OFF_VEC = OFF_DS + DS_TILE;   // lse2[128], delta[128]
  static constexpr uint32_t OFF_CTRL = OFF_VEC + 1024;
  static constexpr uint32_t SMEM = 1024 + OFF_CTRL + 256;
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 128, false, false);   // S^T, dP^T
  static constexpr uint32_t IDESC_KB = idesc_bf16_f32(128, D, false, true);     // dV, dK
  // dQ^T: M = 128 rows of K^T (for D = 64 the upper 64 read the V tile that follows K in
  // shared memory: padding that the drain ignores), N = 128 queries.
  static constexpr uint32_t IDESC_DQT = idesc_bf16_f32(128, 128, true, true);
};

enum {
  W_KV = 0, W_FULL = 1 /* +stage */, W_EMPTY = 3 /* +stage */, W_S = 5, W_DP = 6, W_P = 7, W_DS = 8, W_DQ = 9,
  W_DQFREE = 10, W_DSFREE = 11, W_DONE = 12, W_EPI = 13,
  W_VFULL = 14,   // -LSE2 and -D of the next tile are in shared memory (32 arrivals, warp 3)
  W_GD = 15,
  W_VFREE = 16,   // both compute warpgroups are done with those vectors (256 arrivals)
  W_ADDED = 17,   // deterministic: the drain has issued a tile's additions (128 arrivals)
  W_RELEASED = 18,  // deterministic: the releaser has passed that tile's counter on (1)
  W_COUNT = 19
};

// Bounded barrier for one warpgroup (128 threads) built on an mbarrier: every thread
// arrives, then waits for the phase to complete.  Unlike bar.sync it gives up (and
// reports) if some warp of the group has left early.
__device__ __forceinline__ bool group_sync(uint32_t bar, int& phase, const WaitCtl& w) {
  mbar_arrive(bar);
  const bool ok = mbar_wait(bar, phase & 1, w);
  ++phase;
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ bool warp_wait_b(uint32_t bar, uint32_t parity, const WaitCtl& w) {
  const bool ok = mbar_wait(bar, parity, w);
  return __all_sync(0xffffffffu, ok);
}

template <int N>
__device__ __forceinline__ void reg_fence_b(uint32_t (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i])::"memory");
}

// Adds x at base + OFF bytes: one instruction with an immediate offset.
template <int OFF>
__device__ __forceinline__ void red_add_f32_at(float* base, float x) {
  asm volatile("red.global.add.f32 [%0+%1], %2;" ::"l"(base), "n"(OFF), "f"(x) : "memory");
}
// Pause after each 16 reductions of the drain (ns), per kernel instantiation.  The drain has
// slack; spread out, its reductions leave room in the load/store path for the compute warps'
// shared-memory traffic.  Measured on GB300: 0 -> 100 ns gave +1 to +4 % across the
// training, long, causal and deterministic shapes at d = 128; with the L2 prefetch of the
// next wave in place, 150 ns against 100 gives the atomic d = 128 kernel a further 1.4 to
// 1.7 % (B4 H16 N2048, N = 8192 both masks) but costs d = 64 14 % and the deterministic
// kernel 8 %, whose additions wait for their turn and do best with 50 ns (-0.9 %).
template <int D, bool DET>
__host__ __device__ constexpr unsigned drain_pause_ns() {
  return DET ? 50u : (D == 128 ? 150u : 100u);
}
// Rows J0 .. J0 + 15 of a tile (row stride D floats), column = this lane.
template <int D, int J0, int... J>
__device__ __forceinline__ void red_add_chunk(float* base, const float (&v)[128], std::integer_sequence<int, J...>) {
  (red_add_f32_at<(J0 + J) * D * 4>(base, v[J0 + J]), ...);
}
// All 128 rows in chunks of 16, with a pause after each chunk so that the reductions
// do not hold the load/store path while the compute warps need it.
template <int D, unsigned PAUSE, int... C>
__device__ __forceinline__ void red_add_rows(float* base, const float (&v)[128], std::integer_sequence<int, C...>) {
  ((red_add_chunk<D, C * 16>(base, v, std::make_integer_sequence<int, 16>{}),
    __nanosleep(PAUSE)), ...);
}
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

struct BwdKernelArgs {
  int B, Hq, Hkv, N, g, nq, nkb, causal, deterministic;
  int det_rotate;   // deterministic with the rotating per-tile order (see the kernel)
  int det_k;        // deterministic: contribution classes (1, 2 or 4), one accumulator each
  int det_releaser; // deterministic: warp 2 passes the counters on (else the drain leader)
  int prefetch_ahead;  // > 0: the producer prefetches into L2 the first tiles of CTA blockIdx + this
  float c, scale;
  const float* lse2;
  const float* delta;
  float* dq_acc;
  float* dq_extra;  // deterministic: accumulators 1 .. det_k - 1, extra_stride floats apart
  long long extra_stride;
  int* sem;
  unsigned long long wait_ns;
  int* status;
};
// Packed sequences (the VL kernels): N = total_q; see BwdParams.  A separate type, so that
// the other kernels' parameters stay as they are.
struct BwdKernelArgsVL : BwdKernelArgs {
  int total_k, sem_stride;
  long long rows_pad;
  const int* cu_q;
  const int* cu_k;
  const int* vl_count;
  const int4* vl_units;
  uint16_t* dk;          // for key blocks that end past their sequence (row stores)
  uint16_t* dv;
};

// VL: packed sequences; the CTA's key block, sequence and K/V head come from its record
// of the unit table, rows count from the sequence's start, keys past its end are masked
// and a block that runs past the end stores dK and dV row by row.  DET: the deterministic
// dQ order (a kernel of its own, so that the atomic kernel carries none of its code).
template <int D, bool VL, bool DET>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                    const std::conditional_t<VL, BwdKernelArgsVL, BwdKernelArgs> a) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint8_t* ctrl = smem + C::OFF_CTRL;
  const uint32_t bar0 = smem_u32(ctrl);
  auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 8 * W_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* vec_lse = reinterpret_cast<float*>(smem + C::OFF_VEC);
  float* vec_d = vec_lse + 128;

  const int warp = warp_id(), lane = lane_id();
  // Launched (atomic mode) as a programmatic dependent of the preprocess kernel, whose
  // outputs (-LSE2, -D, the zeroed dQ accumulators and counters) are read only after
  // pdl_wait: by the vector loader, the drain and the releaser.  Everything else (barriers,
  // TMEM, the K, V, Q and dO loads, the first products) overlaps the preprocess's end.
  // Packed sequences wait here (the unit table comes from an earlier kernel).
  pdl_trigger();
  if constexpr (VL) pdl_wait();
  // The sequence: first query row q0, nqs queries in nqt tiles, first key row k0, nks keys,
  // koff = nks - nqs (query i stands at key i + koff).  Constants of the launch unless VL.
  int b, hkv, n, bkv, q0 = 0, nqs = a.N, k0 = 0, nks = a.N, koff = 0, nqt = a.nq;
  if constexpr (VL) {
    // CTAs past the table's records have no work: they leave before touching barriers or
    // tensor memory.
    if ((int)blockIdx.x >= __ldg(a.vl_count)) return;
    const int4 u = a.vl_units[blockIdx.x];
    b = u.x;
    hkv = u.y;
    n = u.z;
    q0 = a.cu_q[b];
    nqs = a.cu_q[b + 1] - q0;
    k0 = a.cu_k[b];
    nks = a.cu_k[b + 1] - k0;
    koff = nks - nqs;
    nqt = (nqs + 127) / 128;
    bkv = hkv;                                     // K/V plane of the packed tensor maps
  } else {
    // Causal: key block n has nq - n query tiles, so blocks are launched in order of n
    // across all heads (longest first).  Otherwise the blocks of one head run together
    // and share its Q and dO tiles in L2.
    const int nbkv = a.B * a.Hkv;
    bkv = a.causal ? blockIdx.x % nbkv : blockIdx.x / a.nkb;
    n = a.causal ? blockIdx.x / nbkv : blockIdx.x % a.nkb;
    b = bkv / a.Hkv;
    hkv = bkv % a.Hkv;
  }
  // First query tile that sees the block (causal: query i sees keys <= i + koff).
  const int m0 = a.causal ? (VL ? max(0, n * 128 - koff) / 128 : n) : 0;
  const int n_m = nqt - m0;
  const int n_iter = a.g * n_m;
  WaitCtl wc{a.wait_ns, a.status, abort_flag};

  if (threadIdx.x == 0) {
    for (int i = 0; i < W_COUNT; ++i)
      mbar_init(BAR(i), (i == W_P || i == W_DS || i == W_VFREE) ? 256
                        : (i == W_DQFREE || i == W_EPI || i == W_GD || i == W_ADDED) ? 128
                        : (i == W_VFULL) ? 32 : 1);
    // W_EMPTY: released by a commit once the stage's last MMA (dK) has finished.
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tdP = tmem + 128u, tdV = tmem + 256u, tdK = tmem + 256u + D;

  // Query tiles are visited in a staggered order: key block n starts at query tile n, so
  // the CTAs of one head add into different dQ rows at any moment (they would otherwise
  // all hit the same rows together).  Causal CTAs already start at their diagonal tile.
  // Deterministic mode fixes, for every tile, the order in which key blocks add into it:
  //  - rotating (non-causal, when every key block of a head fits on the GPU at once): the
  //    staggered order above, with tile m taking blocks m, m - 1, m - 2, ... (mod nq) —
  //    the order in which they reach it, each one iteration after the previous, so a
  //    block waits only for an add made an iteration earlier.  A block waits on a block
  //    with a higher index, so the whole head must be resident: the host enables it only
  //    when a head's blocks take at most half the SMs.
  //  - otherwise: one descending tile order shared by all key blocks of a head (causal
  //    blocks end at their diagonal), tile m taking blocks 0, 1, 2, ...; block n reaches
  //    each tile in the same iteration as block n - 1 and waits for that block's adds.
  //  Packed sequences use the shared order when deterministic; otherwise non-causal
  //  blocks start at tile n mod nqt and causal ones at their first tile.
  const bool shared_order = DET && !a.det_rotate;
  const int m_start = shared_order ? nqt - 1 : (VL ? (a.causal ? m0 : (nqt > 0 ? n % nqt : 0)) : n);
  const int m_step = shared_order ? -1 : 1;
  auto iter_head_row = [&](int it, int& bh, int& m) {
    const int r = it / n_m;
    m = m_start + m_step * (it - r * n_m);
    if (m >= nqt) m -= nqt;                          // non-causal rotation wraps around
    bh = (VL ? 0 : b * a.Hq) + hkv * a.g + r;
  };
  // Deterministic: iteration it's counter, accumulator and turn.  A block's place among a
  // tile's contributions (its iteration with the rotating order, its index with the shared
  // one) splits them into det_k classes, place mod det_k, each added into its own
  // accumulator in its own order (the convert kernel sums the accumulators in a fixed
  // order).  A block then waits for the contribution det_k places before its own instead
  // of the one just before: with the rotating order det_k iterations of slack, with the
  // shared order a chain det_k times shorter, so the round trip of one addition (poll,
  // adds, fence, counter) sets the pace less.  Packed sequences: one class; the counters
  // of a sequence's tiles start at (q0 + 128 b) / 128.
  auto det_slot = [&](int it, int*& sem, float*& acc, int& turn) {
    int bh, m;
    iter_head_row(it, bh, m);
    const int place = a.det_rotate ? it - (it / n_m) * n_m : n;
    const int cls = place & (a.det_k - 1);
    turn = place / a.det_k;
    acc = cls ? a.dq_extra + (size_t)(cls - 1) * a.extra_stride : a.dq_acc;
    if constexpr (VL) sem = a.sem + (size_t)bh * a.sem_stride + (q0 + 128 * b) / 128 + m;
    else sem = a.sem + (size_t)cls * a.B * a.Hq * a.nq + (size_t)bh * a.nq + m;
  };

  // Register split (per thread): warpgroup 0 (producer, MMA) 88, the two compute
  // warpgroups 136 each, drain 152: 88 + 2 x 136 + 152 = 512 = 4 x 128, the launch's
  // 128 x 512 threads, and no role spills.  Each role's code sits inside its own branch
  // so that its limit covers it.
  const int wg = warp >> 2;
  if (wg == 0) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 88;");
  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(BAR(W_KV), 2 * C::TILE);
      for (int c = 0; c < C::NCH; ++c) {
        tma_load_3d(sbase + C::OFF_K + c * C::CHUNK, &tm_k, c * 64, k0 + n * 128, bkv, BAR(W_KV));
        tma_load_3d(sbase + C::OFF_V + c * C::CHUNK, &tm_v, c * 64, k0 + n * 128, bkv, BAR(W_KV));
      }
      int next = 0;
      bool ok = true;
      for (int it = 0; it < n_iter; ++it) {
        const int st = it & 1, round = it >> 1;
        if (round > 0 && !mbar_wait(BAR(W_EMPTY + st), (round - 1) & 1, wc)) { ok = false; break; }
        int bh, m;
        iter_head_row(it, bh, m);
        const uint32_t qs = sbase + C::OFF_STAGE + st * 2 * C::TILE;
        mbar_arrive_expect_tx(BAR(W_FULL + st), 2 * C::TILE);
        for (int c = 0; c < C::NCH; ++c) {
          tma_load_3d(qs + c * C::CHUNK, &tm_q, c * 64, q0 + m * 128, bh, BAR(W_FULL + st));
          tma_load_3d(qs + C::TILE + c * C::CHUNK, &tm_do, c * 64, q0 + m * 128, bh, BAR(W_FULL + st));
        }
        next = it + 1;
      }
      // The CTA one wave later (blockIdx + the SM count) starts about when this one ends:
      // bring its K and V tiles and its first Q and dO tiles into L2 now.  Measured on GB300
      // (atomic): B4 H16 N2048 0.3746 -> 0.3697 ms, d = 64 -0.9 %, N = 8192 unchanged; the
      // deterministic kernels lost 0.6 to 1.2 %, so they do without.
      if constexpr (!VL && !DET) {
        const int nxt = (int)blockIdx.x + a.prefetch_ahead;
        if (ok && a.prefetch_ahead > 0 && nxt < (int)gridDim.x) {
          const int nbkv = a.B * a.Hkv;
          const int bkv2 = a.causal ? nxt % nbkv : nxt / a.nkb;
          const int n2 = a.causal ? nxt / nbkv : nxt % a.nkb;
          const int bh2 = (bkv2 / a.Hkv) * a.Hq + (bkv2 % a.Hkv) * a.g;
          const int m2 = shared_order ? a.nq - 1 : n2;
          for (int c = 0; c < C::NCH; ++c) {
            tma_prefetch_l2_3d(&tm_k, c * 64, n2 * 128, bkv2);
            tma_prefetch_l2_3d(&tm_v, c * 64, n2 * 128, bkv2);
            tma_prefetch_l2_3d(&tm_q, c * 64, m2 * 128, bh2);
            tma_prefetch_l2_3d(&tm_do, c * 64, m2 * 128, bh2);
          }
        }
      }
      if (!ok) {
        const unsigned long long t0 = globaltimer_ns();
        for (int it = max(0, next - 2); it < next; ++it)
          while (!mbar_try_wait(BAR(W_FULL + (it & 1)), (it >> 1) & 1) && globaltimer_ns() - t0 < a.wait_ns) {
          }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(BAR(W_KV), 0, wc);
      tc_fence_after();
      // Matrix descriptors as low words (start address and leading byte offset) advanced by
      // (offset / 16), with one constant high word: one add per operand per MMA.
      constexpr uint32_t HI = sdesc_sw128_hi(1024);
      const uint32_t k_lo = sdesc_sw128_lo(sbase + C::OFF_K, 16);            // K, K-major
      const uint32_t kt_lo = sdesc_sw128_lo(sbase + C::OFF_K, C::CHUNK);     // K^T, MN-major
      const uint32_t v_lo = sdesc_sw128_lo(sbase + C::OFF_V, 16);
      const uint32_t ds_lo = sdesc_sw128_lo(sbase + C::OFF_DS, 16);          // dS^T, K-major
      const uint32_t dst_lo = sdesc_sw128_lo(sbase + C::OFF_DS, C::CHUNK);   // dS^T, MN-major
      // S^T = K Q^T for tile `it`, once its Q/dO stage has landed.
      auto issue_s = [&](int it) -> bool {
        const int st = it & 1;
        if (!mbar_wait(BAR(W_FULL + st), (it >> 1) & 1, wc)) return false;
        tc_fence_after();
        const uint32_t q_lo = sdesc_sw128_lo(sbase + C::OFF_STAGE + st * 2 * C::TILE, 16);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
          if constexpr (DET) {
            const uint32_t a = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
            mma_ss(tS, sdesc_sw128(sbase + C::OFF_K + a, 16, 1024),
                   sdesc_sw128(sbase + C::OFF_STAGE + st * 2 * C::TILE + a, 16, 1024), C::IDESC_S, kk > 0);
          } else {
            mma_ss_w(tS, k_lo + off, HI, q_lo + off, HI, C::IDESC_S, kk > 0);
          }
        }
        mma_commit(BAR(W_S));
        return true;
      };
      if (ok && n_iter > 0) ok = issue_s(0);
      for (int it = 0; it < n_iter && ok; ++it) {
        const int st = it & 1;
        const uint32_t qs = sbase + C::OFF_STAGE + st * 2 * C::TILE, dos = qs + C::TILE;
        // dP^T = V dO^T, once the previous dQ^T has left those columns
        if (it > 0 && !mbar_wait(BAR(W_DQFREE), (it - 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t do_lo = sdesc_sw128_lo(dos, 16), dot_lo = sdesc_sw128_lo(dos, C::CHUNK);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
          if constexpr (DET) {
            const uint32_t a = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
            mma_ss(tdP, sdesc_sw128(sbase + C::OFF_V + a, 16, 1024), sdesc_sw128(dos + a, 16, 1024), C::IDESC_S, kk > 0);
          } else {
            mma_ss_w(tdP, v_lo + off, HI, do_lo + off, HI, C::IDESC_S, kk > 0);
          }
        }
        mma_commit(BAR(W_DP));
        // dV += P^T dO
        if (!mbar_wait(BAR(W_P), it & 1, wc)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          if constexpr (DET)
            mma_ts(tdV, tS + (kk >> 2) * 64 + (kk & 3) * 8, sdesc_sw128(dos + kk * 2048, C::CHUNK, 1024), C::IDESC_KB,
                   (it > 0 || kk > 0));
          else
            mma_ts_w(tdV, tS + (kk >> 2) * 64 + (kk & 3) * 8, dot_lo + kk * (2048 >> 4), HI, C::IDESC_KB,
                     (it > 0 || kk > 0));
        // The next tile's S^T goes ahead of this tile's dK and dQ, so that its
        // probabilities are computed while they run.  MMAs of one thread execute in issue
        // order: S^T lands in the columns of P^T only after dV has read them.
        if (it + 1 < n_iter && !issue_s(it + 1)) { ok = false; break; }
        // dK += dS^T Q and dQ^T = K^T dS^T.  At d = 64 dQ^T goes first, so that the drain reads it
        // while dK runs (the next dP^T waits for that read): measured 2.6 % faster there, and
        // 9 % slower at d = 128, where the drain's reductions then overlap the compute warps'
        // shared-memory traffic.
        constexpr bool DQ_FIRST = D == 64;
        if (!mbar_wait(BAR(W_DS), it & 1, wc)) { ok = false; break; }
        tc_fence_after();
        auto issue_dqt = [&]() {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            if constexpr (DET)
              mma_ss(tdP, sdesc_sw128(sbase + C::OFF_K + kk * 2048, C::CHUNK, 1024),
                     sdesc_sw128(sbase + C::OFF_DS + kk * 2048, C::CHUNK, 1024), C::IDESC_DQT, kk > 0);
            else
              mma_ss_w(tdP, kt_lo + kk * (2048 >> 4), HI, dst_lo + kk * (2048 >> 4), HI, C::IDESC_DQT, kk > 0);
          mma_commit(BAR(W_DQ));
        };
        if constexpr (DQ_FIRST) issue_dqt();
        const uint32_t qt_lo = sdesc_sw128_lo(qs, C::CHUNK);   // Q, MN-major
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
          if constexpr (DET)
            mma_ss(tdK, sdesc_sw128(sbase + C::OFF_DS + (kk >> 2) * C::CHUNK + (kk & 3) * 32, 16, 1024),
                   sdesc_sw128(qs + kk * 2048, C::CHUNK, 1024), C::IDESC_KB, (it > 0 || kk > 0));
          else
            mma_ss_w(tdK, ds_lo + off, HI, qt_lo + kk * (2048 >> 4), HI, C::IDESC_KB, (it > 0 || kk > 0));
        }
        mma_commit(BAR(W_EMPTY + st));  // dK was the stage's last reader: the producer may refill it
        if constexpr (!DQ_FIRST) issue_dqt();
        mma_commit(BAR(W_DSFREE));      // dQ^T and dK, the readers of dS^T, are done
      }
      mma_commit(BAR(W_DONE));
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(BAR(W_DONE), 0) && globaltimer_ns() - t0 < a.wait_ns) {
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------------ vector loader
    // -LSE2 and -D of each tile's 128 queries (lane + 32u), fetched into registers one
    // tile ahead so that their global-memory latency hides behind the current tile, and
    // written to shared memory once both compute warpgroups are done with the previous
    // ones.  Queries past the sequence's end (past N, or the next packed sequence's) get
    // -inf / 0, which makes their probabilities and dS zero.
    pdl_wait();
    float nl[4], nd[4];
    auto fetch = [&](int it) {
      int bh, m;
      iter_head_row(it, bh, m);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int qj = m * 128 + u * 32 + lane;
        nl[u] = qj < nqs ? -a.lse2[(size_t)bh * a.N + q0 + qj] : -INFINITY;
        nd[u] = qj < nqs ? -a.delta[(size_t)bh * a.N + q0 + qj] : 0.f;
      }
    };
    if (n_iter > 0) fetch(0);
    for (int it = 0; it < n_iter; ++it) {
      if (it > 0 && !warp_wait_b(BAR(W_VFREE), (it - 1) & 1, wc)) break;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        vec_lse[u * 32 + lane] = nl[u];
        vec_d[u * 32 + lane] = nd[u];
      }
      mbar_arrive(BAR(W_VFULL));
      if (it + 1 < n_iter) fetch(it + 1);
    }
  } else if (DET && warp == 2) {
    // ------------------------------------------------------------------ releaser
    // Passes each tile's counter on once the drain has issued the tile's additions: the
    // drain's arrivals (release, CTA scope) order its additions before this thread's
    // gpu-scope fence, which is cumulative, and that fence before the increment.  The
    // fence waits for the additions to land; here it delays no TMEM read of the drain.
    if (a.det_releaser && lane == 0) {
      pdl_wait();
      for (int it = 0; it < n_iter; ++it) {
        if (!mbar_wait(BAR(W_ADDED), it & 1, wc) || *abort_flag) break;
        int* sem;
        float* acc;
        int turn;
        det_slot(it, sem, acc, turn);
        __threadfence();
        atomicAdd(sem, 1);
        mbar_arrive(BAR(W_RELEASED));
      }
    }
    __syncwarp();
  }
  } else if (wg == 1 || wg == 2) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 136;");
    // ------------------------------------------------------------------ compute: P^T, dS^T
    // Two warpgroups share the work column-wise: half h owns queries [64h, 64h + 64) of
    // every key row.  Its packed P goes to TMEM columns [64h, 64h + 32), inside its own
    // part of S, so neither half overwrites scores the other has not read yet.
    const int h = wg - 1;
    const int row = (warp & 3) * 32 + lane;          // key row within the block
    const int kr = n * 128 + row;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    uint8_t* ds_tile = smem + C::OFF_DS;
    bool ok = true;
    for (int it = 0; it < n_iter && ok; ++it) {
      int bh, m;
      iter_head_row(it, bh, m);
      // This tile's -LSE2 and -D (index = query within the tile), from the vector loader.
      if (!warp_wait_b(BAR(W_VFULL), it & 1, wc)) { ok = false; break; }
      if (!warp_wait_b(BAR(W_S), it & 1, wc)) { ok = false; break; }
      tc_fence_after();
      // Visible queries for this key row: qj + koff >= kr when causal, qj < nqs (through
      // the vectors), and the key itself < nks.
      const int qmin = (a.causal ? kr - koff - m * 128 : 0) - h * 64;   // this half's columns below qmin are masked
      const bool key_ok = kr < nks;
      const bool need_mask = qmin > 0 || !key_ok;
      const float4* nl4 = reinterpret_cast<const float4*>(vec_lse + h * 64);
      const float4* nd4 = reinterpret_cast<const float4*>(vec_d + h * 64);
      uint32_t pk[32];
      {
        // Two halves of 32 columns: the second half's load is in flight while the first
        // half's probabilities are computed, and the first half's P is stored meanwhile.
        uint32_t u[64];
        tmem_ld32(tS + lane_off + h * 64, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
        tmem_wait_ld();
        reg_fence_b(*reinterpret_cast<uint32_t(*)[32]>(&u[0]));
        tmem_ld32(tS + lane_off + h * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
#pragma unroll
        for (int i = 0; i < 64; i += 4) {
          if (i == 32) {
            tmem_st16(tS + lane_off + h * 64, *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]));
            tmem_wait_ld();
            reg_fence_b(*reinterpret_cast<uint32_t(*)[32]>(&u[32]));
          }
          const float4 nl = nl4[i >> 2];
          float x0, x1, x2, x3;
          ffma2(x0, x1, __uint_as_float(u[i]), __uint_as_float(u[i + 1]), a.c, a.c, nl.x, nl.y);
          ffma2(x2, x3, __uint_as_float(u[i + 2]), __uint_as_float(u[i + 3]), a.c, a.c, nl.z, nl.w);
          float p0 = ex2_mufu(x0), p1 = ex2_mufu(x1), p2 = ex2_mufu(x2), p3 = ex2_mufu(x3);
          if (need_mask) {
            if (i < qmin || !key_ok) p0 = 0.f;
            if (i + 1 < qmin || !key_ok) p1 = 0.f;
            if (i + 2 < qmin || !key_ok) p2 = 0.f;
            if (i + 3 < qmin || !key_ok) p3 = 0.f;
          }
          pk[i >> 1] = pack_bf16x2(p0, p1);
          pk[(i >> 1) + 1] = pack_bf16x2(p2, p3);
        }
      }
      tmem_st16(tS + lane_off + h * 64 + 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16]));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(BAR(W_P));
      // dS^T = P^T o (dP^T - D), bf16, into the shared tile (rows = keys, 128B swizzle),
      // once the previous dK/dQ products have finished reading it.
      if (it > 0 && !warp_wait_b(BAR(W_DSFREE), (it - 1) & 1, wc)) { ok = false; break; }
      if (!warp_wait_b(BAR(W_DP), it & 1, wc)) { ok = false; break; }
      tc_fence_after();
      {
        // As above: the second 32 columns of dP^T load while the first are turned into dS^T.
        uint32_t u[64];
        tmem_ld32(tdP + lane_off + h * 64, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
        tmem_wait_ld();
        reg_fence_b(*reinterpret_cast<uint32_t(*)[32]>(&u[0]));
        tmem_ld32(tdP + lane_off + h * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          if (cc == 1) {
            tmem_wait_ld();
            reg_fence_b(*reinterpret_cast<uint32_t(*)[32]>(&u[32]));
          }
          uint32_t out[16];
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const int l0 = cc * 32 + i;
            const float4 nd = nd4[l0 >> 2];
            const uint32_t pa = pk[l0 >> 1], pb = pk[(l0 >> 1) + 1];
            float e0, e1, e2, e3;
            fadd2(e0, e1, __uint_as_float(u[l0]), __uint_as_float(u[l0 + 1]), nd.x, nd.y);
            fadd2(e2, e3, __uint_as_float(u[l0 + 2]), __uint_as_float(u[l0 + 3]), nd.z, nd.w);
            fmul2(e0, e1, e0, e1, __uint_as_float(pa << 16), __uint_as_float(pa & 0xffff0000u));
            fmul2(e2, e3, e2, e3, __uint_as_float(pb << 16), __uint_as_float(pb & 0xffff0000u));
            out[i >> 1] = pack_bf16x2(e0, e1);
            out[(i >> 1) + 1] = pack_bf16x2(e2, e3);
          }
          // Query columns [64h + 32cc, +32) are 16-byte chunks 4cc..4cc+3 of box h.
#pragma unroll
          for (int uu = 0; uu < 4; ++uu) {
            const uint32_t off = h * C::CHUNK + row * 128 + ((((cc * 4) + uu) ^ (row & 7)) * 16);
            *reinterpret_cast<uint4*>(ds_tile + off) =
                make_uint4(out[4 * uu], out[4 * uu + 1], out[4 * uu + 2], out[4 * uu + 3]);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(BAR(W_DS));
      mbar_arrive(BAR(W_VFREE));
    }
    // Epilogue: dV and scale * dK -> bf16 -> stage 0 buffers -> TMA store, once every MMA
    // has completed (the last loads into the stage buffers have then been consumed).
    // Packed sequences: a block that runs past its sequence's last key is written row by
    // row from registers (a TMA store would overwrite the next sequence's first rows), and
    // a block no query sees (a sequence with keys but no queries) writes zeros.
    if (h == 0 && ok && warp_wait_b(BAR(W_DONE), 0, wc)) {
      tc_fence_after();
      uint8_t* sv = smem + C::OFF_STAGE;
      uint8_t* sk = sv + C::TILE;
      const bool direct = VL && n * 128 + 128 > nks;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        const uint32_t tsrc = (which ? tdK : tdV) + lane_off;
        const float mul = which ? a.scale : 1.f;
        uint8_t* dst = which ? sk : sv;
        uint16_t* grow = nullptr;
        if constexpr (VL) grow = (which ? a.dk : a.dv) + ((size_t)bkv * a.total_k + k0 + kr) * D;
#pragma unroll 1
        for (int q = 0; q < D / 32; ++q) {
          uint32_t r[32];
          if (VL && n_iter == 0) {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
          } else {
            tmem_ld32(tsrc + q * 32, r);
            tmem_wait_ld();
            reg_fence_b(r);
          }
          uint32_t pkk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pkk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * mul, __uint_as_float(r[2 * i + 1]) * mul);
          if (direct) {
            if (kr < nks) {
#pragma unroll
              for (int u = 0; u < 4; ++u)
                *reinterpret_cast<uint4*>(grow + q * 32 + u * 8) =
                    make_uint4(pkk[4 * u], pkk[4 * u + 1], pkk[4 * u + 2], pkk[4 * u + 3]);
            }
            continue;
          }
          const int box = q >> 1, j0 = (q & 1) * 4;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t off = box * C::CHUNK + row * 128 + (((j0 + u) ^ (row & 7)) * 16);
            *reinterpret_cast<uint4*>(dst + off) = make_uint4(pkk[4 * u], pkk[4 * u + 1], pkk[4 * u + 2], pkk[4 * u + 3]);
          }
        }
      }
      if (!direct) {
        fence_proxy_async_smem();
        mbar_arrive(BAR(W_EPI));
        if (warp == 4 && lane == 0 && mbar_wait(BAR(W_EPI), 0, wc)) {
          for (int c = 0; c < C::NCH; ++c) {
            tma_store_3d(&tm_dv, sbase + C::OFF_STAGE + c * C::CHUNK, c * 64, k0 + n * 128, bkv);
            tma_store_3d(&tm_dk, sbase + C::OFF_STAGE + C::TILE + c * C::CHUNK, c * 64, k0 + n * 128, bkv);
          }
          tma_store_commit();
          tma_store_wait_read();   // the CTA may exit once the stores have read shared memory
        }
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 152;");
    // ------------------------------------------------------------------ drain: dQ -> dQacc
    // dQ is formed transposed, so TMEM lane i holds column i of dQ for the tile's 128
    // queries.  Lane i of a warp adds element i of one query row: each red.global.add of a
    // warp covers 32 consecutive floats (one 128-byte line) of a dQacc row.  The drain
    // reads TMEM and writes L2 only; it never touches shared memory, which the MMAs need.
    const int dcol = (warp & 3) * 32 + lane;         // dQ column = TMEM lane
    const bool has_col = (warp & 3) * 32 < D;        // D = 64: lanes 64-127 hold padding
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const bool leader = warp == 12 && lane == 0;
    pdl_wait();   // the accumulators and counters are the preprocess kernel's
    // The tile's dQ from TMEM into registers; frees the columns for the next dP^T.
    auto read_dq = [&](int it, float (&v)[128]) -> bool {
      if (!warp_wait_b(BAR(W_DQ), it & 1, wc)) return false;
      tc_fence_after();
      if (has_col) {
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32(tdP + lane_off + q * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[q * 32]));
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 128; ++i) asm volatile("" : "+f"(v[i])::"memory");
      }
      tc_fence_before();
      mbar_arrive(BAR(W_DQFREE));
      return true;
    };
    // Rows are padded to whole tiles, so queries past N (or past the sequence) add into
    // padding rows, which are never read.  Packed sequences: a sequence's rows start at
    // q0 + 128 b of its head's rows.
    auto add_dq = [&](float* acc, int bh, int m, const float (&v)[128]) {
      if (!has_col) return;
      size_t arow;
      if constexpr (VL) arow = (size_t)bh * a.rows_pad + q0 + 128 * (size_t)b + (size_t)m * 128;
      else arow = (size_t)bh * a.nq * 128 + (size_t)m * 128;
      red_add_rows<D, drain_pause_ns<D, DET>()>(acc + arow * D + dcol, v, std::make_integer_sequence<int, 8>{});
    };
    if constexpr (!DET) {
      for (int it = 0; it < n_iter; ++it) {
        int bh, m;
        iter_head_row(it, bh, m);
        float v[128];
        if (!read_dq(it, v)) break;
        add_dq(a.dq_acc, bh, m, v);
      }
    } else {
      int gphase = 0;
      for (int it = 0; it < n_iter; ++it) {
        int bh, m;
        iter_head_row(it, bh, m);
        int* sem;
        float* acc;
        int turn;
        det_slot(it, sem, acc, turn);
        // The leader waits for the turn before the tile's dQ is ready, so the poll's round
        // trip stays off the critical path (a turn depends only on other blocks' earlier
        // additions).
        if (leader) {
          const unsigned long long t0 = globaltimer_ns();
          while (ld_acquire(sem) != turn) {
            if (*abort_flag) break;
            if (globaltimer_ns() - t0 > a.wait_ns) {
              *abort_flag = 1;
              atomicExch(a.status, DEV_TIMEOUT);
              break;
            }
          }
        }
        float v[128];
        if (!read_dq(it, v)) break;
        // Every drain thread learns that the turn has come (the leader's acquire, passed on
        // through the group barrier).
        if (!group_sync(BAR(W_GD), gphase, wc) || *abort_flag) break;
        add_dq(acc, bh, m, v);
        if (a.det_releaser) {
          // Hand the tile to the releaser (warp 2), at most one tile ahead of it.
          if (it > 0 && !warp_wait_b(BAR(W_RELEASED), (it - 1) & 1, wc)) break;
          mbar_arrive(BAR(W_ADDED));
        } else {
          // Release here: the group barrier (its arrival releases at CTA scope) orders
          // every drain thread's additions before the leader's gpu-scope fence, which is
          // cumulative, and that fence before the counter's increment.
          if (!group_sync(BAR(W_GD), gphase, wc)) break;
          if (leader) {
            __threadfence();
            atomicAdd(sem, 1);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

template <int D, bool VL, bool DET>
static cudaError_t launch_bwd_t(const BwdMaps& m, const BwdParams& p, cudaStream_t s) {
  // Packed sequences: N is total_q and B the number of sequences, so a head has N rows.
  const long long rows = VL ? (long long)p.Hq * p.N : (long long)p.B * p.Hq * p.N;
  const int nq = (p.N + 127) / 128;
  const int n_sem = !p.deterministic ? 0 : VL ? p.Hq * p.sem_stride : kDetMaxClasses * p.B * p.Hq * nq;
  const long long rows_pad = VL ? (long long)p.N + 128LL * p.B : 0;
  const int* cu_q = VL ? p.cu_q : nullptr;
  int dev = 0, sms = 152;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // The rotating deterministic order (see the kernel) needs every key block of a head on
  // the GPU at once: enabled when a head's blocks take at most half the SMs.
  const bool rotate = !VL && DET && !p.causal && 2 * nq <= sms;
  // Deterministic, measured on GB300 (B2 H16 d128): two classes (four from N = 8192 on, see
  // det_classes) cut the non-causal cost
  // (N = 8192, rotating: 3.60 -> 3.27 ms; N = 16384, shared: 6.77 -> 6.00 ms, both with the
  // releaser; four classes gained at most 6 % more and lost 5 % at N = 2048) but not the
  // causal one, whose second accumulator only costs its zeroing and reading; the releaser
  // helps wherever it is used here (causal N = 8192: 1.71 -> 1.49 ms) but, with one class,
  // not the non-causal shared order (N = 16384: 6.77 -> 7.47 ms).
  const int det_k = DET && !VL && !p.causal ? det_classes(nq) : 1;
  const int det_rel = DET && (det_k > 1 || p.causal) ? 1 : 0;
  float* const extra = det_k > 1 ? p.dq_acc2 : nullptr;
  const long long extra_stride = (long long)(align256((size_t)p.B * p.Hq * nq * 128 * D * 4) / 4);
  {
    const long long n_heads = p.N > 0 ? rows / p.N : 0;
    const unsigned gx = (unsigned)((p.N + 15) / 16), gy = (unsigned)std::min<long long>(n_heads, 65535);
    if (rows > 0) {
      e = launch_pdl(bwd_preprocess_kernel<D>, dim3(gx, gy), dim3(256), 0, s,
                     static_cast<const uint16_t*>(p.o), static_cast<const uint16_t*>(p.dout), p.lse, p.delta, p.lse2,
                     p.dq_acc, extra, det_k - 1, extra_stride, p.sem, rows, p.N, nq * 128, n_sem, cu_q, p.B,
                     rows_pad);
      if (e != cudaSuccess) return e;
    }
  }
  {
    auto kern = attn_bwd_kernel<D, VL, DET>;
    constexpr uint32_t smem = BwdCfg<D>::SMEM;
    static std::once_flag flags[64];
    static cudaError_t attr_err[64];
    std::call_once(flags[dev & 63], [&] {
      attr_err[dev & 63] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
    std::conditional_t<VL, BwdKernelArgsVL, BwdKernelArgs> a{};
    a.B = p.B; a.Hq = p.Hq; a.Hkv = p.Hkv; a.N = p.N; a.g = p.g; a.nq = nq; a.nkb = nq;
    a.causal = p.causal; a.deterministic = p.deterministic;
    a.det_rotate = rotate ? 1 : 0;
    a.det_k = det_k;
    a.det_releaser = det_rel;
    a.prefetch_ahead = sms;
    a.c = p.c; a.scale = p.scale;
    a.lse2 = p.lse2; a.delta = p.delta; a.dq_acc = p.dq_acc; a.dq_extra = extra; a.extra_stride = extra_stride;
    a.sem = p.sem;
    a.wait_ns = p.wait_ns; a.status = p.status;
    long long grid = (long long)p.B * p.Hkv * nq;
    if constexpr (VL) {
      a.total_k = p.total_k; a.sem_stride = p.sem_stride; a.rows_pad = rows_pad;
      a.cu_q = p.cu_q; a.cu_k = p.cu_k; a.vl_count = p.vl_count; a.vl_units = p.vl_units;
      a.dk = static_cast<uint16_t*>(p.dk);
      a.dv = static_cast<uint16_t*>(p.dv);
      grid = (long long)p.Hkv * ((long long)p.total_k / 128 + p.B);   // the unit table's bound
    }
    if (grid > 0) {
      // Deterministic: a plain launch (as a programmatic dependent it measured 2 % slower at
      // B4 H16 N2048; the atomic kernel gains 0.6 %).
      if constexpr (DET) {
        kern<<<(unsigned)grid, kBwdThreads, smem, s>>>(m.q, m.k, m.v, m.dout, m.dk, m.dv, a);
        e = cudaGetLastError();
      } else {
        e = launch_pdl(kern, dim3((unsigned)grid), dim3(kBwdThreads), smem, s, m.q, m.k, m.v, m.dout, m.dk, m.dv, a);
      }
      if (e != cudaSuccess) return e;
    }
  }
  {
    const long long n8 = rows * D / 8;
    const long long n_heads = p.N > 0 ? rows / p.N : 0;
    const long long per_head = (long long)p.N * (D / 8);
    const unsigned gy = (unsigned)std::min<long long>(n_heads, 65535);
    const unsigned gx = (unsigned)std::max<long long>(1, std::min<long long>((per_head + 255) / 256,
                                                                             ((long long)sms * 16 + gy - 1) / gy));
    if (n8 > 0) {
      return launch_pdl(bwd_convert_kernel<D>, dim3(gx, gy), dim3(256), 0, s,
                        static_cast<const float*>(p.dq_acc), static_cast<const float*>(extra), det_k - 1,
                        extra_stride, static_cast<uint16_t*>(p.dq), p.scale, n8, p.N, nq * 128, cu_q, p.B,
                        rows_pad);
    }
    return cudaSuccess;
  }
}

template <int D, bool VL>
static cudaError_t launch_bwd_det(const BwdMaps& maps, const BwdParams& p, cudaStream_t stream) {
  return p.deterministic ? launch_bwd_t<D, VL, true>(maps, p, stream) : launch_bwd_t<D, VL, false>(maps, p, stream);
}

cudaError_t launch_bwd(const BwdMaps& maps, const BwdParams& p, cudaStream_t stream) {
  if (p.varlen) {
    if (p.D == 64) return launch_bwd_det<64, true>(maps, p, stream);
    if (p.D == 128) return launch_bwd_det<128, true>(maps, p, stream);
    return cudaErrorNotSupported;
  }
  if (p.D == 64) return launch_bwd_det<64, false>(maps, p, stream);
  if (p.D == 128) return launch_bwd_det<128, false>(maps, p, stream);
  return cudaErrorNotSupported;
}

}  // namespace attn
