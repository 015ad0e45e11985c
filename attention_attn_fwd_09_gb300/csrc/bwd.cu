// Fused exact attention backward for sm_103a: preprocess, main (tcgen05) and dQ convert.
//
// Stages ("Hotelren FA4 summary" section 4.2, the five-stage backward pipeline; the
// reverse-engineering page: P is recomputed, never stored):
//   preprocess  D_i = sum_d dO_id O_id, LSE2_i = LSE_i * log2(e), dQacc = 0, counters = 0
//   main        per CTA one key block of one K/V head, looping over the query tiles of
//               every query head of the group:
//                 S^T  = K Q^T                 (tcgen05, TMEM)
//                 dP^T = V dO^T                (tcgen05, TMEM)
//                 P^T  = exp2(S^T c - LSE2)    (exact probabilities, written back as bf16)
//                 dV  += P^T dO                (A = P^T from TMEM)
//                 dS^T = P^T o (dP^T - D)      (bf16, to shared memory)
//                 dK  += dS^T Q                (A = dS^T, K-major view of the tile)
//                 dQ   = dS K                  (A = dS, MN-major view of the same tile)
//                 dQacc += dQ                  (CTA pairs on adjacent key blocks swap dQ
//                                               halves through distributed shared memory;
//                                               each adds the pair's sum for its half with
//                                               fp32 TMA bulk reductions, in pair order when
//                                               deterministic)
//               The transposed orientation (keys on TMEM lanes) makes every result land in
//               the layout its consumer reads ("FlashAttention-4 explained" section 05).
//   convert     dq = bf16(scale * dQacc)
// dK is scaled by `scale` in the main kernel's epilogue.
#include <algorithm>
#include <cstdint>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d, int deterministic) {
  (void)Hkv;
  const size_t rows = (size_t)B * Hq * N;
  const size_t nq = (size_t)B * Hq * ((N + 127) / 128);
  size_t n = align256(rows * d * 4) + 2 * align256(rows * 4);
  if (deterministic) n += align256(nq * 2 * 4);   // one counter per (query tile, dQ half)
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

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------------------------
// Preprocess: one 16-thread group per row (d = 128: 8 bf16 per thread; d = 64: 4).
// ------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const uint16_t* __restrict__ o,
                                                              const uint16_t* __restrict__ dout,
                                                              const float* __restrict__ lse, float* __restrict__ delta,
                                                              float* __restrict__ lse2, float* __restrict__ dq_acc,
                                                              int* __restrict__ sem, long long rows, int n_sem) {
  constexpr int PER = D / 16;  // elements per thread
  const long long row = (long long)blockIdx.x * 16 + (threadIdx.x >> 4);
  const int sub = threadIdx.x & 15;
  const long long gtid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (sem != nullptr && gtid < n_sem) sem[gtid] = 0;
  if (row >= rows) return;
  const uint16_t* orow = o + row * D + sub * PER;
  const uint16_t* drow = dout + row * D + sub * PER;
  float acc = 0.f;
  if constexpr (PER == 8) {
    const uint4 a = *reinterpret_cast<const uint4*>(orow);
    const uint4 b = *reinterpret_cast<const uint4*>(drow);
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = fmaf(__uint_as_float(av[i] << 16), __uint_as_float(bv[i] << 16), acc);
      acc = fmaf(__uint_as_float(av[i] & 0xffff0000u), __uint_as_float(bv[i] & 0xffff0000u), acc);
    }
  } else {
    const uint2 a = *reinterpret_cast<const uint2*>(orow);
    const uint2 b = *reinterpret_cast<const uint2*>(drow);
    const uint32_t av[2] = {a.x, a.y}, bv[2] = {b.x, b.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      acc = fmaf(__uint_as_float(av[i] << 16), __uint_as_float(bv[i] << 16), acc);
      acc = fmaf(__uint_as_float(av[i] & 0xffff0000u), __uint_as_float(bv[i] & 0xffff0000u), acc);
    }
  }
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, 16);
  float4* z = reinterpret_cast<float4*>(dq_acc + row * D + sub * PER);
#pragma unroll
  for (int i = 0; i < PER / 4; ++i) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (sub == 0) {
    delta[row] = acc;
    lse2[row] = lse[row] * kLog2e;
  }
}

// ------------------------------------------------------------------------------------
// Convert: dq = bf16(scale * dQacc), 8 elements per thread.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) bwd_convert_kernel(const float* __restrict__ acc, uint16_t* __restrict__ dq,
                                                           float scale, long long n8) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (long long)gridDim.x * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
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
// Warps: 0 TMA producer, 1 MMA issuer, 2 TMEM allocator, 3 idle,
//        4-7 and 8-11 "compute" (P^T, dS^T; keys on TMEM lanes; queries 0-63 and 64-127),
//        12-15 "drain" (dQ rows -> dQacc).
// TMEM columns: S^T/P^T [0,128), dP^T then dQ [128,256), dV [256,256+D), dK [256+D,256+2D).
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
  static constexpr uint32_t IDESC_DQ = idesc_bf16_f32(128, D, true, true);      // dQ
};

enum {
  W_KV = 0, W_FULL = 1 /* +stage */, W_EMPTY = 3 /* +stage */, W_S = 5, W_DP = 6, W_P = 7, W_DS = 8, W_DQ = 9,
  W_DQFREE = 10, W_DSFREE = 11, W_DONE = 12, W_EPI = 13, W_GC = 14, W_GD = 15,
  W_DRAINED = 16, // the drain warpgroup has finished (one arrival)
  W_GC1 = 17,     // staging sync of the second compute warpgroup
  X_READY = 18,   // +stage: the partner CTA's stage buffer may receive our dQ half (1 remote arrival)
  X_RECV = 20,    // +stage: the partner's dQ half has landed in our stage buffer (128 remote arrivals)
  W_COUNT = 22
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

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

struct BwdKernelArgs {
  int B, Hq, Hkv, N, g, nq, nkb /* key blocks per head rounded up to even */, causal, deterministic;
  float c, scale;
  const float* lse2;
  const float* delta;
  float* dq_acc;
  int* sem;
  unsigned long long wait_ns;
  int* status;
};

template <int D>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kBwdThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                    const __grid_constant__ CUtensorMap tm_dqacc, const BwdKernelArgs a) {
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
  // The two CTAs of a cluster take adjacent key blocks n = 2p, 2p + 1 of one K/V head
  // and visit the same query tiles in the same order.  When the head has an odd number
  // of key blocks the last cluster's second CTA has no block ("dead"): it only joins the
  // cluster barriers, and its partner adds its whole dQ by itself ("unpaired").
  const int bkv = blockIdx.x / a.nkb, n = blockIdx.x % a.nkb;
  const int b = bkv / a.Hkv, hkv = bkv % a.Hkv;
  const uint32_t rank = cluster_ctarank();            // == n & 1
  const int pair = n >> 1;
  const bool live = n < a.nq;
  const bool paired = (n | 1) < a.nq;
  const int m0 = a.causal ? 2 * pair : 0;
  const int n_m = a.nq - m0;
  const int n_iter = live ? a.g * n_m : 0;
  WaitCtl wc{a.wait_ns, a.status, abort_flag};

  if (threadIdx.x == 0) {
    for (int i = 0; i < W_COUNT; ++i)
      mbar_init(BAR(i), (i == W_P || i == W_DS) ? 256
                        : (i == W_DQFREE || i == W_EPI || i == W_GC || i == W_GC1 || i == W_GD || i == X_RECV ||
                           i == X_RECV + 1) ? 128 : 1);
    // W_EMPTY: released by the drain's leader (one arrival), W_DRAINED: one arrival.
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync_all();   // both CTAs' barriers exist before either arrives on the other's
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tdP = tmem + 128u, tdV = tmem + 256u, tdK = tmem + 256u + D;

  // Query tiles are visited in a staggered order: pair p starts at query tile p, so the
  // pairs of one head add into different dQ rows at any moment (they would otherwise
  // all hit the same rows together).  Causal pairs start at the diagonal tile of their
  // first key block (for the second block that tile is fully masked).  In deterministic
  // mode each pair still trails its predecessor by about one iteration.
  auto iter_head_row = [&](int it, int& bh, int& m) {
    const int r = it / n_m;
    m = a.causal ? m0 + it % n_m : (it % n_m + pair) % n_m;
    bh = b * a.Hq + hkv * a.g + r;
  };

  // Register split (per thread): warpgroup 0 (producer, MMA) 56, two compute warpgroups
  // 152 each, drain 152: 56 + 3 x 152 = 512 = 4 x 128, the launch's 128 x 512 threads.  Each
  // role's code sits inside its own branch so that its limit covers it.
  const int wg = warp >> 2;
  if (!live) {
    // no key block: nothing to compute
  } else if (wg == 0) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 56;");
  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(BAR(W_KV), 2 * C::TILE);
      for (int c = 0; c < C::NCH; ++c) {
        tma_load_3d(sbase + C::OFF_K + c * C::CHUNK, &tm_k, c * 64, n * 128, bkv, BAR(W_KV));
        tma_load_3d(sbase + C::OFF_V + c * C::CHUNK, &tm_v, c * 64, n * 128, bkv, BAR(W_KV));
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
          tma_load_3d(qs + c * C::CHUNK, &tm_q, c * 64, m * 128, bh, BAR(W_FULL + st));
          tma_load_3d(qs + C::TILE + c * C::CHUNK, &tm_do, c * 64, m * 128, bh, BAR(W_FULL + st));
        }
        next = it + 1;
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
      const uint32_t kb = sbase + C::OFF_K, vb = sbase + C::OFF_V, dsb = sbase + C::OFF_DS;
      for (int it = 0; it < n_iter && ok; ++it) {
        const int st = it & 1;
        if (!mbar_wait(BAR(W_FULL + st), (it >> 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t qs = sbase + C::OFF_STAGE + st * 2 * C::TILE, dos = qs + C::TILE;
        // S^T = K Q^T
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
          mma_ss(tS, sdesc_sw128(kb + off, 16, 1024), sdesc_sw128(qs + off, 16, 1024), C::IDESC_S, kk > 0);
        }
        mma_commit(BAR(W_S));
        // dP^T = V dO^T, once the previous dQ has left those columns
        if (it > 0 && !mbar_wait(BAR(W_DQFREE), (it - 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
          mma_ss(tdP, sdesc_sw128(vb + off, 16, 1024), sdesc_sw128(dos + off, 16, 1024), C::IDESC_S, kk > 0);
        }
        mma_commit(BAR(W_DP));
        // dV += P^T dO
        if (!mbar_wait(BAR(W_P), it & 1, wc)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tdV, tS + (kk >> 2) * 64 + (kk & 3) * 8, sdesc_sw128(dos + kk * 2048, C::CHUNK, 1024), C::IDESC_KB,
                 (it > 0 || kk > 0));
        // dK += dS^T Q ; dQ = dS K
        if (!mbar_wait(BAR(W_DS), it & 1, wc)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
          mma_ss(tdK, sdesc_sw128(dsb + off, 16, 1024), sdesc_sw128(qs + kk * 2048, C::CHUNK, 1024), C::IDESC_KB,
                 (it > 0 || kk > 0));
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tdP, sdesc_sw128(dsb + kk * 2048, C::CHUNK, 1024), sdesc_sw128(kb + kk * 2048, C::CHUNK, 1024),
                 C::IDESC_DQ, kk > 0);
        mma_commit(BAR(W_DQ));          // the drain releases this Q/dO stage after staging dQ in it
        mma_commit(BAR(W_DSFREE));
      }
      mma_commit(BAR(W_DONE));
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(BAR(W_DONE), 0) && globaltimer_ns() - t0 < a.wait_ns) {
      }
    }
  }
  } else if (wg == 1 || wg == 2) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 152;");
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
    int gphase = 0;
    for (int it = 0; it < n_iter && ok; ++it) {
      int bh, m;
      iter_head_row(it, bh, m);
      // Stage this half's -LSE2 and -D (index = query within the tile); the first sync keeps
      // the previous tile's readers ahead of the overwrite.  Queries past N get -inf / 0,
      // which makes their probabilities and dS exactly zero.
      if (!group_sync(BAR(h ? W_GC1 : W_GC), gphase, wc)) { ok = false; break; }
      if (row < 64) {
        const int qc = h * 64 + row, qj = m * 128 + qc;
        vec_lse[qc] = qj < a.N ? -a.lse2[(size_t)bh * a.N + qj] : -INFINITY;
        vec_d[qc] = qj < a.N ? -a.delta[(size_t)bh * a.N + qj] : 0.f;
      }
      if (!group_sync(BAR(h ? W_GC1 : W_GC), gphase, wc)) { ok = false; break; }
      if (!warp_wait_b(BAR(W_S), it & 1, wc)) { ok = false; break; }
      tc_fence_after();
      // Visible queries for this key row: qj >= kr when causal, qj < N, and the key itself < N.
      const int qmin = (a.causal ? kr - m * 128 : 0) - h * 64;   // this half's columns below qmin are masked
      const bool key_ok = kr < a.N;
      const bool need_mask = qmin > 0 || !key_ok;
      const float4* nl4 = reinterpret_cast<const float4*>(vec_lse + h * 64);
      const float4* nd4 = reinterpret_cast<const float4*>(vec_d + h * 64);
      uint32_t pk[32];
      {
        uint32_t u[64];
        tmem_ld32(tS + lane_off + h * 64, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
        tmem_ld32(tS + lane_off + h * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
        tmem_wait_ld();
        reg_fence_b(u);
#pragma unroll
        for (int i = 0; i < 64; i += 4) {
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
      tmem_st32(tS + lane_off + h * 64, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(BAR(W_P));
      // dS^T = P^T o (dP^T - D), bf16, into the shared tile (rows = keys, 128B swizzle),
      // once the previous dK/dQ products have finished reading it.
      if (it > 0 && !warp_wait_b(BAR(W_DSFREE), (it - 1) & 1, wc)) { ok = false; break; }
      if (!warp_wait_b(BAR(W_DP), it & 1, wc)) { ok = false; break; }
      tc_fence_after();
      {
        uint32_t u[64];
        tmem_ld32(tdP + lane_off + h * 64, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
        tmem_ld32(tdP + lane_off + h * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
        tmem_wait_ld();
        reg_fence_b(u);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
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
    }
    // Epilogue: dV and scale * dK -> bf16 -> stage 0 buffers -> TMA store, once every MMA
    // has completed and the drain no longer stages dQ in the stage buffers.
    if (h == 0 && ok && warp_wait_b(BAR(W_DONE), 0, wc) && warp_wait_b(BAR(W_DRAINED), 0, wc)) {
      tc_fence_after();
      uint8_t* sv = smem + C::OFF_STAGE;
      uint8_t* sk = sv + C::TILE;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        const uint32_t tsrc = (which ? tdK : tdV) + lane_off;
        const float mul = which ? a.scale : 1.f;
        uint8_t* dst = which ? sk : sv;
#pragma unroll 1
        for (int q = 0; q < D / 32; ++q) {
          uint32_t r[32];
          tmem_ld32(tsrc + q * 32, r);
          tmem_wait_ld();
          reg_fence_b(r);
          uint32_t pkk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pkk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * mul, __uint_as_float(r[2 * i + 1]) * mul);
          const int box = q >> 1, j0 = (q & 1) * 4;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t off = box * C::CHUNK + row * 128 + (((j0 + u) ^ (row & 7)) * 16);
            *reinterpret_cast<uint4*>(dst + off) = make_uint4(pkk[4 * u], pkk[4 * u + 1], pkk[4 * u + 2], pkk[4 * u + 3]);
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(BAR(W_EPI));
      if (warp == 4 && lane == 0 && mbar_wait(BAR(W_EPI), 0, wc)) {
        for (int c = 0; c < C::NCH; ++c) {
          tma_store_3d(&tm_dv, sbase + C::OFF_STAGE + c * C::CHUNK, c * 64, n * 128, bkv);
          tma_store_3d(&tm_dk, sbase + C::OFF_STAGE + C::TILE + c * C::CHUNK, c * 64, n * 128, bkv);
        }
        tma_store_commit();
        tma_store_wait_all();
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 152;");
    // ------------------------------------------------------------------ drain: dQ -> dQacc
    // dQ leaves TMEM into registers (the columns are then free for the next dP).  A paired
    // CTA keeps dQ columns [rank * D/2, rank * D/2 + D/2) and stores the other half of
    // each row straight into its partner's stage buffer for this iteration (distributed
    // shared memory), once the partner reports that its MMAs are done with that buffer.
    // When the partner's half has arrived in ours, each thread adds its own half of its
    // row in place, and the sum goes into dQacc by TMA bulk reductions: every dQ element
    // crosses L2 once per pair instead of once per key block.  The stage buffer (its MMAs
    // are done; the producer refills it only for the iteration after next, once the
    // drain releases it) holds 128-row x 32-column fp32 boxes with 128-byte swizzle.
    const int row = (warp & 3) * 32 + lane;          // query row within the tile
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const bool leader = warp == 12 && lane == 0;
    const uint32_t peer = rank ^ 1u;
    constexpr int HB = D / 64;                       // 32-column boxes per half
    bool ok = true;
    int gphase = 0;
    for (int it = 0; it < n_iter && ok; ++it) {
      int bh, m;
      iter_head_row(it, bh, m);
      const int st = it & 1;
      uint8_t* stage = smem + C::OFF_STAGE + st * 2 * C::TILE;
      if (!warp_wait_b(BAR(W_DQ), it & 1, wc)) { ok = false; break; }
      tc_fence_after();
      float v[D];
#pragma unroll
      for (int q = 0; q < D / 32; ++q) tmem_ld32(tdP + lane_off + q * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[q * 32]));
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < D; ++i) asm volatile("" : "+f"(v[i])::"memory");
      tc_fence_before();
      mbar_arrive(BAR(W_DQFREE));
      int nbox, col0;
      if (paired) {
        // Our stage buffer may now receive the partner's half.
        if (leader) mbar_arrive_cluster(mapa_shared(BAR(X_READY + st), peer));
        const bool rdy = mbar_wait_cluster(BAR(X_READY + st), (it >> 1) & 1, wc);
        if (!__all_sync(0xffffffffu, rdy)) { ok = false; break; }
        const uint32_t dst = mapa_shared(smem_u32(stage), peer);
#pragma unroll
        for (int j = 0; j < HB; ++j)
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int i0 = j * 32 + 4 * c;            // column within a half
            const float s0 = rank ? v[i0] : v[D / 2 + i0], s1 = rank ? v[i0 + 1] : v[D / 2 + i0 + 1];
            const float s2 = rank ? v[i0 + 2] : v[D / 2 + i0 + 2], s3 = rank ? v[i0 + 3] : v[D / 2 + i0 + 3];
            st_cluster_f4(dst + j * 16384 + row * 128 + ((c ^ (row & 7)) << 4), s0, s1, s2, s3);
          }
        mbar_arrive_cluster(mapa_shared(BAR(X_RECV + st), peer));
        const bool got = mbar_wait_cluster(BAR(X_RECV + st), (it >> 1) & 1, wc);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
#pragma unroll
        for (int j = 0; j < HB; ++j)
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int i0 = j * 32 + 4 * c;
            float4* cell = reinterpret_cast<float4*>(stage + j * 16384 + row * 128 + ((c ^ (row & 7)) << 4));
            float4 x = *cell;
            x.x += rank ? v[D / 2 + i0] : v[i0];
            x.y += rank ? v[D / 2 + i0 + 1] : v[i0 + 1];
            x.z += rank ? v[D / 2 + i0 + 2] : v[i0 + 2];
            x.w += rank ? v[D / 2 + i0 + 3] : v[i0 + 3];
            *cell = x;
          }
        nbox = HB;
        col0 = int(rank) * (D / 2);
      } else {
#pragma unroll
        for (int bx = 0; bx < D / 32; ++bx) {
          const float* src = &v[bx * 32];
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<float4*>(stage + bx * 16384 + row * 128 + ((c ^ (row & 7)) << 4)) =
                make_float4(src[4 * c], src[4 * c + 1], src[4 * c + 2], src[4 * c + 3]);
        }
        nbox = D / 32;
        col0 = 0;
      }
      fence_proxy_async_smem();
      if (!group_sync(BAR(W_GD), gphase, wc)) { ok = false; break; }
      if (leader) {
        // Deterministic: the pairs add into each (query tile, half) in pair order 0, 1, 2, ...
        int* sem = a.deterministic ? a.sem + ((size_t)bh * a.nq + m) * 2 : nullptr;
        const int h_lo = paired ? int(rank) : 0, h_hi = paired ? int(rank) : 1;
        bool lok = true;   // leader only: a failure here stops the others at their next wait
        if (a.deterministic) {
          const unsigned long long t0 = globaltimer_ns();
          for (int hh = h_lo; hh <= h_hi && lok; ++hh)
            while (ld_acquire(sem + hh) != pair) {
              if (*abort_flag) { lok = false; break; }
              if (globaltimer_ns() - t0 > a.wait_ns) {
                *abort_flag = 1;
                atomicExch(a.status, DEV_TIMEOUT);
                lok = false;
                break;
              }
            }
        }
        if (lok) {
          for (int bx = 0; bx < nbox; ++bx)
            tma_reduce_add_3d(&tm_dqacc, smem_u32(stage + bx * 16384), col0 + bx * 32, m * 128, bh);
          tma_store_commit();
          if (a.deterministic) {
            tma_store_wait_all();                       // the adds have landed
            asm volatile("fence.proxy.async.global;" ::: "memory");
            __threadfence();
            for (int hh = h_lo; hh <= h_hi; ++hh) atomicAdd(sem + hh, 1);
          } else {
            tma_store_wait_read();                      // the stage buffer has been read
          }
          mbar_arrive(BAR(W_EMPTY + st));
        }
      }
    }
    if (leader) {
      tma_store_wait_all();
      mbar_arrive(BAR(W_DRAINED));
    }
  }

  tc_fence_before();
  __syncwarp();
  // Neither CTA leaves while the other may still store into its shared memory or
  // arrive on its barriers.
  cluster_sync_all();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

template <int D>
static cudaError_t launch_bwd_t(const BwdMaps& m, const BwdParams& p, cudaStream_t s) {
  const long long rows = (long long)p.B * p.Hq * p.N;
  const int nq = (p.N + 127) / 128;
  const int n_sem = p.deterministic ? p.B * p.Hq * nq * 2 : 0;
  {
    const long long blocks = std::max((rows + 15) / 16, ((long long)n_sem + 255) / 256);
    bwd_preprocess_kernel<D><<<(unsigned)blocks, 256, 0, s>>>(
        static_cast<const uint16_t*>(p.o), static_cast<const uint16_t*>(p.dout), p.lse, p.delta, p.lse2, p.dq_acc,
        p.sem, rows, n_sem);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  {
    auto kern = attn_bwd_kernel<D>;
    constexpr uint32_t smem = BwdCfg<D>::SMEM;
    static std::once_flag flags[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::call_once(flags[dev & 63], [&] {
      attr_err[dev & 63] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
    BwdKernelArgs a{};
    const int nkb = nq + (nq & 1);   // clusters of two CTAs: pad to an even count
    a.B = p.B; a.Hq = p.Hq; a.Hkv = p.Hkv; a.N = p.N; a.g = p.g; a.nq = nq; a.nkb = nkb;
    a.causal = p.causal; a.deterministic = p.deterministic;
    a.c = p.c; a.scale = p.scale;
    a.lse2 = p.lse2; a.delta = p.delta; a.dq_acc = p.dq_acc; a.sem = p.sem;
    a.wait_ns = p.wait_ns; a.status = p.status;
    const long long grid = (long long)p.B * p.Hkv * nkb;
    kern<<<(unsigned)grid, kBwdThreads, smem, s>>>(m.q, m.k, m.v, m.dout, m.dk, m.dv, m.dqacc, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  {
    const long long n8 = rows * D / 8;
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long blocks = std::min<long long>((n8 + 255) / 256, (long long)sms * 8);
    bwd_convert_kernel<<<(unsigned)blocks, 256, 0, s>>>(p.dq_acc, static_cast<uint16_t*>(p.dq), p.scale, n8);
    return cudaGetLastError();
  }
}

cudaError_t launch_bwd(const BwdMaps& maps, const BwdParams& p, cudaStream_t stream) {
  if (p.D == 64) return launch_bwd_t<64>(maps, p, stream);
  if (p.D == 128) return launch_bwd_t<128>(maps, p, stream);
  return cudaErrorNotSupported;
}

}  // namespace attn
