// Attention backward with 64-row query tiles: d = 192 and 256, and the same design for d = 64
// and 128 ("Hotelren FA4 summary" section 6.2, recommended head dims up to 256; the stages
// of section 4.2: S = K Q^T, dP = V dO^T, dV = P^T dO, dS = P o (dP - D), dK = dS^T Q,
// dQ = dS K; the reverse-engineering page: P is recomputed, never stored).
//
// Each CTA owns one 128-key block of one K/V head and one column block of dK, dV and dQ,
// and walks query tiles of 64 rows.  At d = 256 the dV and dK accumulators of a 128-key
// block would take all 512 TMEM columns and K, V, Q and dO tiles of 128 rows 256 KB of
// shared memory, so for d > 128 the columns are split in two halves over two CTAs (d = 256:
// columns 0-127 and 128-255; d = 192: 0-127 and 128-191); for d <= 128 one CTA owns all of
// them.
//   S^T   = K Q^T           M = 128 keys, N = 64 queries, all d columns
//   dP^T  = V dO^T          same shape
//   P^T   = exp2(S^T c - LSE2)         (bf16 into the S^T columns)
//   dV_h += P^T dO_h        N = the block's columns, A = P^T from TMEM
//   dS^T  = P^T o (dP^T - D)           (bf16 into shared memory)
//   dK_h += dS^T Q_h
//   dQ^T_h = K_h^T dS^T     M = the block's d rows (TMEM lane = dQ column), N = 64 queries
//   dQacc += dQ_h           fp32 red.global.add, one 128-byte line of a row per warp
//                           instruction (in key-block order when deterministic)
// Two halves both recompute S^T and dP^T (the price of the TMEM budget at d > 128).  TMEM:
// S^T [0,64), dP^T [64,128), dQ^T [128,192), dV_h, dK_h after (at most 448 columns).  dQ^T
// has columns of its own, so no product waits for the drain except the next dQ^T: the
// loop-carried chain of the 128-row-tile kernel (dP^T -> dS^T -> dQ^T -> drain -> next dP^T,
// with dQ^T aliasing dP^T) is gone.  Two threads issue the products: warp 1 dP^T, S^T and
// dV, warp 2 dK and dQ^T (with 64-row tiles a product is short, and one thread's issue rate
// would bound the tensor pipe).  Shared memory: K and V tiles resident; Q and dO tiles of
// 64 rows in three stages (d <= 128), two (d = 192) or one (d = 256, where a stage's dO is
// refilled after dV and its Q after dK); dS^T 16 KB.  With two or more stages the next
// tile's S^T and dP^T are issued ahead of this tile's dK and dQ^T.
#include <algorithm>
#include <cstdint>
#include <mutex>
#include <type_traits>
#include <utility>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {

namespace {

constexpr int kBwThreads = 512;
constexpr float kLog2eW = 1.4426950408889634f;

template <int D>
struct BwCfg {
  static constexpr int NCH = D / 64;                  // 64-column chunks of a row
  static constexpr uint32_t KCH = 128 * 128;          // 128 rows x 64 bf16
  static constexpr uint32_t KT = KCH * NCH;           // K or V tile, 128 x D
  static constexpr uint32_t QCH = 64 * 128;           // 64 rows x 64 bf16
  static constexpr uint32_t QT = QCH * NCH;           // Q or dO tile, 64 x D
  static constexpr int NHALF = D > 128 ? 2 : 1;       // column blocks of dK/dV/dQ (CTAs per key block)
  static constexpr int NST = D == 256 ? 1 : (D == 192 ? 2 : 3);   // Q/dO stages
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = KT;
  static constexpr uint32_t OFF_Q = 2 * KT;                    // NST x QT
  static constexpr uint32_t OFF_DO = OFF_Q + NST * QT;         // NST x QT
  static constexpr uint32_t OFF_DS = OFF_DO + NST * QT;        // 128 keys x 64 queries bf16
  static constexpr uint32_t OFF_VEC = OFF_DS + 128 * 128;      // -LSE2[64], -D[64]
  static constexpr uint32_t OFF_CTRL = OFF_VEC + 512;
  static constexpr uint32_t SMEM = 1024 + OFF_CTRL + 256;
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 64, false, false);     // S^T, dP^T
  static constexpr uint32_t IDESC_DQT = idesc_bf16_f32(128, 64, true, true);     // dQ^T
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(OFF_DS % 1024 == 0 && OFF_Q % 1024 == 0 && OFF_DO % 1024 == 0, "swizzle atoms aligned");
};

enum {
  X_KV = 0,
  X_QFULL = 1,      // +stage (up to 3)
  X_DOFULL = 4,     // +stage
  X_QFREE = 7,      // +stage: dK (the stage's last Q reader) done
  X_DOFREE = 10,    // +stage: dV (the stage's last dO reader) done
  X_S = 13,         // S^T complete
  X_DP = 14,        // dP^T complete
  X_P = 15,         // P^T written (256)
  X_DPFREE = 16,    // dP^T read by the compute warps (256)
  X_DS = 17,        // dS^T written (256)
  X_DSFREE = 18,    // dK and dQ^T (the readers of dS^T) done
  X_DQ = 19,        // dQ^T complete
  X_DQFREE = 20,    // dQ^T read by the drain (128)
  X_VFULL = 21,     // vectors of the next tile written (32)
  X_VFREE = 22,     // vectors read (256)
  X_GD = 23,        // drain group barrier (128)
  X_EPI = 24,       // epilogue staging written (128)
  X_DONE = 25,
  X_COUNT = 26
};
static_assert(X_COUNT * 8 + 8 <= 256, "barriers and the TMEM slot fit the control block");
static_assert(BwCfg<64>::NST <= 3 && BwCfg<128>::NST <= 3, "three stage barriers of each kind");

__device__ __forceinline__ bool w_wait(uint32_t bar, uint32_t parity, const WaitCtl& w) {
  const bool ok = mbar_wait(bar, parity, w);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ bool w_group_sync(uint32_t bar, int& phase, const WaitCtl& w) {
  mbar_arrive(bar);
  const bool ok = mbar_wait(bar, phase & 1, w);
  ++phase;
  return __all_sync(0xffffffffu, ok);
}

template <int N>
__device__ __forceinline__ void w_fence(uint32_t (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i])::"memory");
}

template <int OFF>
__device__ __forceinline__ void w_red_at(float* base, float x) {
  asm volatile("red.global.add.f32 [%0+%1], %2;" ::"l"(base), "n"(OFF), "f"(x) : "memory");
}
// Rows J0 .. J0 + 15 of a 64-row tile (row stride D floats), column = this lane, then a
// short pause so that the reductions leave the load/store path to the compute warps:
// 150 ns with atomic dQ (measured on GB300 against 100 ns: 64-row tiles at d = 128 -2 %,
// d = 256 -0.3 %, d = 192 unchanged), 100 ns when deterministic.
template <int D, unsigned PAUSE, int J0, int... J>
__device__ __forceinline__ void w_red_chunk(float* base, const float (&v)[64], std::integer_sequence<int, J...>) {
  (w_red_at<(J0 + J) * D * 4>(base, v[J0 + J]), ...);
  __nanosleep(PAUSE);
}
template <int D, unsigned PAUSE, int... C>
__device__ __forceinline__ void w_red_rows(float* base, const float (&v)[64], std::integer_sequence<int, C...>) {
  (w_red_chunk<D, PAUSE, C * 16>(base, v, std::make_integer_sequence<int, 16>{}), ...);
}

__device__ __forceinline__ int w_ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

struct BwArgs {
  int B, Hq, Hkv, N, g, nq64, nkb, causal;
  float c, scale;
  const float* lse2;
  const float* delta;
  float* dq_acc;      // [B, Hq, nq64 * 64, D]
  int* sem;           // [B, Hq, nq64, column blocks] when deterministic
  unsigned long long wait_ns;
  int* status;
  int prefetch_ahead;   // > 0: the producer prefetches into L2 the first tiles of CTA blockIdx + this
};

template <int D, bool DET>
__global__ void __launch_bounds__(kBwThreads, 1)
    attn_bwd_wide_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                         const BwArgs a) {
  using C = BwCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint8_t* ctrl = smem + C::OFF_CTRL;
  const uint32_t bar0 = smem_u32(ctrl);
  auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 8 * X_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* vec_l = reinterpret_cast<float*>(smem + C::OFF_VEC);   // -LSE2 of the tile's 64 queries
  float* vec_d = vec_l + 64;                                     // -D

  const int warp = warp_id(), lane = lane_id();
  // CTA -> (column half, key block, K/V head).  Causal grids launch key block 0 of every
  // head first (it sees the most query tiles); otherwise a head's blocks run together.
  const int half = C::NHALF == 2 ? (int)(blockIdx.x & 1) : 0;
  const int rest = C::NHALF == 2 ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int nbkv = a.B * a.Hkv;
  const int bkv = a.causal ? rest % nbkv : rest / a.nkb;
  const int n = a.causal ? rest / nbkv : rest % a.nkb;
  const int b = bkv / a.Hkv, hkv = bkv % a.Hkv;
  const int c0 = half * 128;                       // first dK/dV/dQ column of this CTA
  const int DH = min(128, D - c0);                 // 128, or 64 (second half at d = 192; d = 64)
  const int m0 = a.causal ? 2 * n : 0;             // first 64-row query tile that sees the block
  const int n_m = a.nq64 - m0;
  const int n_iter = a.g * max(n_m, 0);
  WaitCtl wc{a.wait_ns, a.status, abort_flag};

  if (threadIdx.x == 0) {
    for (int i = 0; i < X_COUNT; ++i) {
      uint32_t cnt = 1;
      if (i == X_P || i == X_DPFREE || i == X_DS || i == X_VFREE) cnt = 256;
      else if (i == X_DQFREE || i == X_GD || i == X_EPI) cnt = 128;
      else if (i == X_VFULL) cnt = 32;
      else if (i == X_DONE) cnt = 2;      // one commit from each MMA-issuing thread
      mbar_init(BAR(i), cnt);
    }
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
  const uint32_t tS = tmem, tdP = tmem + 64u, tdQ = tmem + 128u, tdV = tmem + 192u, tdK = tmem + 192u + DH;

  // Query tiles: non-causal blocks start at tile (2n mod nq64) so that the blocks of a head
  // add into different dQ rows at a time; causal blocks start at their first tile.  When
  // deterministic, every block of a head visits the tiles in the same descending order,
  // and tile m takes the blocks' additions in ascending block order (a counter per tile
  // and column half).
  const int m_start = DET ? a.nq64 - 1 : (a.causal ? m0 : (a.nq64 > 0 ? (2 * n) % a.nq64 : 0));
  const int m_step = DET ? -1 : 1;
  auto iter_head_row = [&](int it, int& bh, int& m) {
    const int r = it / n_m;
    m = m_start + m_step * (it - r * n_m);
    if (m >= a.nq64) m -= a.nq64;
    bh = b * a.Hq + hkv * a.g + r;
  };

  const int wg = warp >> 2;
  if (wg == 0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 88;");
    if (warp == 0) {
      // -------------------------------------------------------------- producer
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
        mbar_arrive_expect_tx(BAR(X_KV), 2 * C::KT);
        for (int c = 0; c < C::NCH; ++c) {
          tma_load_3d(sbase + C::OFF_K + c * C::KCH, &tm_k, c * 64, n * 128, bkv, BAR(X_KV));
          tma_load_3d(sbase + C::OFF_V + c * C::KCH, &tm_v, c * 64, n * 128, bkv, BAR(X_KV));
        }
        int q_next = 0, do_next = 0;   // loads issued (for the clean-up after a failed wait)
        bool ok = true;
        for (int it = 0; it < n_iter && ok; ++it) {
          const int st = it % C::NST, round = it / C::NST;
          int bh, m;
          iter_head_row(it, bh, m);
          // dO first: its stage frees earlier (after dV) than Q's (after dK).
          if (round > 0 && !mbar_wait(BAR(X_DOFREE + st), (round - 1) & 1, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(BAR(X_DOFULL + st), C::QT);
          for (int c = 0; c < C::NCH; ++c)
            tma_load_3d(sbase + C::OFF_DO + st * C::QT + c * C::QCH, &tm_do, c * 64, m * 64, bh, BAR(X_DOFULL + st));
          do_next = it + 1;
          if (round > 0 && !mbar_wait(BAR(X_QFREE + st), (round - 1) & 1, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(BAR(X_QFULL + st), C::QT);
          for (int c = 0; c < C::NCH; ++c)
            tma_load_3d(sbase + C::OFF_Q + st * C::QT + c * C::QCH, &tm_q, c * 64, m * 64, bh, BAR(X_QFULL + st));
          q_next = it + 1;
        }
        // The CTA one wave later (blockIdx + the SM count) starts about when this one ends:
        // bring its K and V tiles and its first dO and Q tiles into L2 now (atomic dQ only,
        // as in the 128-row kernel).
        if constexpr (!DET) {
          const int nxt = (int)blockIdx.x + a.prefetch_ahead;
          if (ok && a.prefetch_ahead > 0 && nxt < (int)gridDim.x) {
            const int rest2 = C::NHALF == 2 ? (nxt >> 1) : nxt;
            const int bkv2 = a.causal ? rest2 % nbkv : rest2 / a.nkb;
            const int n2 = a.causal ? rest2 / nbkv : rest2 % a.nkb;
            const int m2 = a.causal ? 2 * n2 : (a.nq64 > 0 ? (2 * n2) % a.nq64 : 0);
            const int bh2 = (bkv2 / a.Hkv) * a.Hq + (bkv2 % a.Hkv) * a.g;
            for (int c = 0; c < C::NCH; ++c) {
              tma_prefetch_l2_3d(&tm_k, c * 64, n2 * 128, bkv2);
              tma_prefetch_l2_3d(&tm_v, c * 64, n2 * 128, bkv2);
              tma_prefetch_l2_3d(&tm_do, c * 64, m2 * 64, bh2);
              tma_prefetch_l2_3d(&tm_q, c * 64, m2 * 64, bh2);
            }
          }
        }
        if (!ok) {
          const unsigned long long t0 = globaltimer_ns();
          for (int it = max(0, do_next - C::NST); it < do_next; ++it)
            while (!mbar_try_wait(BAR(X_DOFULL + it % C::NST), (it / C::NST) & 1) && globaltimer_ns() - t0 < a.wait_ns) {
            }
          for (int it = max(0, q_next - C::NST); it < q_next; ++it)
            while (!mbar_try_wait(BAR(X_QFULL + it % C::NST), (it / C::NST) & 1) && globaltimer_ns() - t0 < a.wait_ns) {
            }
        }
      }
    } else if (warp == 1) {
      // -------------------------------------------------------------- first MMA issuer: dP^T, S^T, dV
      if (lane == 0) {
        bool ok = mbar_wait(BAR(X_KV), 0, wc);
        tc_fence_after();
        constexpr uint32_t HI = sdesc_sw128_hi(1024);
        const uint32_t k_lo = sdesc_sw128_lo(sbase + C::OFF_K, 16), v_lo = sdesc_sw128_lo(sbase + C::OFF_V, 16);
        const uint32_t idesc_kv = idesc_bf16_f32(128, DH, false, true);
        // dP^T = V dO^T for tile `it`, once its dO has landed and the compute warps have read
        // the previous dP^T.
        auto issue_dp = [&](int it) -> bool {
          const int st = it % C::NST;
          const uint32_t do_lo = sdesc_sw128_lo(sbase + C::OFF_DO + st * C::QT, 16);
          if (!mbar_wait(BAR(X_DOFULL + st), (it / C::NST) & 1, wc)) return false;
          if (it > 0 && !mbar_wait(BAR(X_DPFREE), (it - 1) & 1, wc)) return false;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ka = ((kk >> 2) * C::KCH + (kk & 3) * 32) >> 4, qa = ((kk >> 2) * C::QCH + (kk & 3) * 32) >> 4;
            mma_ss_w(tdP, v_lo + ka, HI, do_lo + qa, HI, C::IDESC_S, kk > 0);
          }
          mma_commit(BAR(X_DP));
          return true;
        };
        // S^T = K Q^T for tile `it` (the previous dV, which read P^T from these columns, was
        // issued before it).
        auto issue_s = [&](int it) -> bool {
          const int st = it % C::NST;
          const uint32_t q_lo = sdesc_sw128_lo(sbase + C::OFF_Q + st * C::QT, 16);
          if (!mbar_wait(BAR(X_QFULL + st), (it / C::NST) & 1, wc)) return false;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ka = ((kk >> 2) * C::KCH + (kk & 3) * 32) >> 4, qa = ((kk >> 2) * C::QCH + (kk & 3) * 32) >> 4;
            mma_ss_w(tS, k_lo + ka, HI, q_lo + qa, HI, C::IDESC_S, kk > 0);
          }
          mma_commit(BAR(X_S));
          return true;
        };
        // With two or more stages the next tile's S^T and dP^T go ahead of this tile's dK
        // and dQ^T, so that its probabilities and dS^T are computed while they run; with one
        // stage (d = 256) the next tile's Q can only land after this tile's dK.
        constexpr bool PIPE = C::NST >= 2;
        if (PIPE && n_iter > 0) ok = ok && issue_dp(0) && issue_s(0);
        for (int it = 0; it < n_iter && ok; ++it) {
          const int st = it % C::NST;
          const uint32_t dot_lo = sdesc_sw128_lo(sbase + C::OFF_DO + st * C::QT + (c0 / 64) * C::QCH, C::QCH);
          if (!PIPE && !(issue_dp(it) && issue_s(it))) { ok = false; break; }
          // dV_h += P^T dO_h: P^T of queries 32 w .. 32 w + 31 sits in columns 32 w .. 32 w + 15.
          if (!mbar_wait(BAR(X_P), it & 1, wc)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts_w(tdV, tS + (kk >> 1) * 32 + (kk & 1) * 8, dot_lo + kk * (2048 >> 4), HI, idesc_kv,
                     (it > 0 || kk > 0));
          mma_commit(BAR(X_DOFREE + st));
          if (PIPE && it + 1 < n_iter && !(issue_s(it + 1) && issue_dp(it + 1))) { ok = false; break; }
        }
        mma_commit(BAR(X_DONE));
        const unsigned long long t0 = globaltimer_ns();
        while (!mbar_try_wait(BAR(X_DONE), 0) && globaltimer_ns() - t0 < a.wait_ns) {
        }
      }
    } else if (warp == 2) {
      // -------------------------------------------------------------- second MMA issuer: dK, dQ^T
      // Its accumulators (dK, dQ^T) are disjoint from the first issuer's (S^T, dP^T, dV), and
      // each thread's commits track only its own products, so the two streams only meet
      // through the barriers below.
      if (lane == 0) {
        bool ok = mbar_wait(BAR(X_KV), 0, wc);
        tc_fence_after();
        constexpr uint32_t HI = sdesc_sw128_hi(1024);
        const uint32_t kt_lo = sdesc_sw128_lo(sbase + C::OFF_K + (c0 / 64) * C::KCH, C::KCH);   // K_h^T, MN-major
        const uint32_t ds_lo = sdesc_sw128_lo(sbase + C::OFF_DS, 16);                           // dS^T, K-major
        const uint32_t dst_lo = sdesc_sw128_lo(sbase + C::OFF_DS, 16);                          // dS^T, MN-major
        const uint32_t idesc_kv = idesc_bf16_f32(128, DH, false, true);
        for (int it = 0; it < n_iter && ok; ++it) {
          const int st = it % C::NST;
          const uint32_t qt_lo = sdesc_sw128_lo(sbase + C::OFF_Q + st * C::QT + (c0 / 64) * C::QCH, C::QCH);
          // dK_h += dS^T Q_h
          if (!mbar_wait(BAR(X_DS), it & 1, wc)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss_w(tdK, ds_lo + kk * (32 >> 4), HI, qt_lo + kk * (2048 >> 4), HI, idesc_kv, (it > 0 || kk > 0));
          mma_commit(BAR(X_QFREE + st));
          // dQ^T_h = K_h^T dS^T into columns of its own, once the drain has read the last one
          if (it > 0 && !mbar_wait(BAR(X_DQFREE), (it - 1) & 1, wc)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss_w(tdQ, kt_lo + kk * (2048 >> 4), HI, dst_lo + kk * (2048 >> 4), HI, C::IDESC_DQT, kk > 0);
          mma_commit(BAR(X_DQ));
          mma_commit(BAR(X_DSFREE));
        }
        mma_commit(BAR(X_DONE));
        const unsigned long long t0 = globaltimer_ns();
        while (!mbar_try_wait(BAR(X_DONE), 0) && globaltimer_ns() - t0 < a.wait_ns) {
        }
      }
    } else if (warp == 3) {
      // -------------------------------------------------------------- vector loader
      // -LSE2 and -D of the tile's 64 queries (lane + 32 u), one tile ahead in registers;
      // queries past N get -inf / 0, which makes their P and dS zero.
      float nl[2], nd[2];
      auto fetch = [&](int it) {
        int bh, m;
        iter_head_row(it, bh, m);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int qj = m * 64 + u * 32 + lane;
          nl[u] = qj < a.N ? -a.lse2[(size_t)bh * a.N + qj] : -INFINITY;
          nd[u] = qj < a.N ? -a.delta[(size_t)bh * a.N + qj] : 0.f;
        }
      };
      if (n_iter > 0) fetch(0);
      for (int it = 0; it < n_iter; ++it) {
        if (it > 0 && !w_wait(BAR(X_VFREE), (it - 1) & 1, wc)) break;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          vec_l[u * 32 + lane] = nl[u];
          vec_d[u * 32 + lane] = nd[u];
        }
        mbar_arrive(BAR(X_VFULL));
        if (it + 1 < n_iter) fetch(it + 1);
      }
    }
  } else if (wg == 1 || wg == 2) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 136;");
    // ---------------------------------------------------------------- compute: P^T, dS^T
    // Thread = key row (TMEM lane); warpgroup w takes queries 32 w .. 32 w + 31 of the tile.
    const int w = wg - 1;
    const int row = (warp & 3) * 32 + lane;
    const int kr = n * 128 + row;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    uint8_t* ds_tile = smem + C::OFF_DS;
    bool ok = true;
    for (int it = 0; it < n_iter && ok; ++it) {
      int bh, m;
      iter_head_row(it, bh, m);
      if (!w_wait(BAR(X_VFULL), it & 1, wc)) { ok = false; break; }
      if (!w_wait(BAR(X_S), it & 1, wc)) { ok = false; break; }
      tc_fence_after();
      // query q = m * 64 + 32 w + i sees key kr when q >= kr (causal); keys past N are masked.
      const int qmin = (a.causal ? kr - m * 64 : 0) - 32 * w;
      const bool key_ok = kr < a.N;
      const bool need_mask = qmin > 0 || !key_ok;
      const float4* nl4 = reinterpret_cast<const float4*>(vec_l + 32 * w);
      const float4* nd4 = reinterpret_cast<const float4*>(vec_d + 32 * w);
      uint32_t pk[16];
      {
        uint32_t u[32];
        tmem_ld32(tS + lane_off + 32 * w, u);
        tmem_wait_ld();
        w_fence(u);
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
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
      tmem_st16(tS + lane_off + 32 * w, pk);   // inside this warpgroup's own S^T columns
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(BAR(X_P));
      // dS^T = P^T o (dP^T - D), once dK and dQ^T have finished reading the previous one.
      if (!w_wait(BAR(X_DP), it & 1, wc)) { ok = false; break; }
      tc_fence_after();
      uint32_t u[32];
      tmem_ld32(tdP + lane_off + 32 * w, u);
      tmem_wait_ld();
      w_fence(u);
      tc_fence_before();
      mbar_arrive(BAR(X_DPFREE));
      if (it > 0 && !w_wait(BAR(X_DSFREE), (it - 1) & 1, wc)) { ok = false; break; }
      uint32_t out[16];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float4 nd = nd4[i >> 2];
        const uint32_t pa = pk[i >> 1], pb = pk[(i >> 1) + 1];
        float e0, e1, e2, e3;
        fadd2(e0, e1, __uint_as_float(u[i]), __uint_as_float(u[i + 1]), nd.x, nd.y);
        fadd2(e2, e3, __uint_as_float(u[i + 2]), __uint_as_float(u[i + 3]), nd.z, nd.w);
        fmul2(e0, e1, e0, e1, __uint_as_float(pa << 16), __uint_as_float(pa & 0xffff0000u));
        fmul2(e2, e3, e2, e3, __uint_as_float(pb << 16), __uint_as_float(pb & 0xffff0000u));
        out[i >> 1] = pack_bf16x2(e0, e1);
        out[(i >> 1) + 1] = pack_bf16x2(e2, e3);
      }
      // dS^T row = key, 64 queries = one 128-byte swizzled row; queries 32 w .. are
      // 16-byte chunks 4 w .. 4 w + 3.
#pragma unroll
      for (int uu = 0; uu < 4; ++uu)
        *reinterpret_cast<uint4*>(ds_tile + row * 128 + (((4 * w + uu) ^ (row & 7)) * 16)) =
            make_uint4(out[4 * uu], out[4 * uu + 1], out[4 * uu + 2], out[4 * uu + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(BAR(X_DS));
      mbar_arrive(BAR(X_VFREE));
    }
    // Epilogue (warpgroup 1): dV_h and scale * dK_h -> bf16 -> the K/V tiles' shared
    // memory (free once every MMA has completed) -> TMA store, 64 columns per box.
    if (w == 0 && ok && w_wait(BAR(X_DONE), 0, wc)) {
      tc_fence_after();
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        const uint32_t tsrc = (which ? tdK : tdV) + lane_off;
        const float mul = which ? a.scale : 1.f;
        uint8_t* dst = smem + C::OFF_K + which * (2 * C::KCH);
#pragma unroll 1
        for (int q = 0; q < DH / 32; ++q) {
          uint32_t r[32];
          if (n_iter == 0) {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
          } else {
            tmem_ld32(tsrc + q * 32, r);
            tmem_wait_ld();
            w_fence(r);
          }
          uint32_t pkk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pkk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * mul, __uint_as_float(r[2 * i + 1]) * mul);
          const int box = q >> 1, j0 = (q & 1) * 4;
#pragma unroll
          for (int uu = 0; uu < 4; ++uu) {
            const uint32_t off = box * C::KCH + row * 128 + (((j0 + uu) ^ (row & 7)) * 16);
            *reinterpret_cast<uint4*>(dst + off) = make_uint4(pkk[4 * uu], pkk[4 * uu + 1], pkk[4 * uu + 2], pkk[4 * uu + 3]);
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(BAR(X_EPI));
      if (warp == 4 && lane == 0 && mbar_wait(BAR(X_EPI), 0, wc)) {
        for (int c = 0; c < DH / 64; ++c) {
          tma_store_3d(&tm_dv, sbase + C::OFF_K + c * C::KCH, c0 + c * 64, n * 128, bkv);
          tma_store_3d(&tm_dk, sbase + C::OFF_K + 2 * C::KCH + c * C::KCH, c0 + c * 64, n * 128, bkv);
        }
        tma_store_commit();
        tma_store_wait_read();   // the CTA may exit once the stores have read shared memory
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 152;");
    // ---------------------------------------------------------------- drain: dQ_h -> dQacc
    // TMEM lane i holds dQ column c0 + i for the tile's 64 queries; lane i of a warp adds
    // element i of one query row, so each red.global.add of a warp is one 128-byte line.
    const int dcol = (warp & 3) * 32 + lane;
    const bool has_col = (warp & 3) * 32 < DH;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const bool leader = warp == 12 && lane == 0;
    auto read_dq = [&](int it, float (&v)[64]) -> bool {
      if (!w_wait(BAR(X_DQ), it & 1, wc)) return false;
      tc_fence_after();
      if (has_col) {
        tmem_ld32(tdQ + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tmem_ld32(tdQ + lane_off + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 64; ++i) asm volatile("" : "+f"(v[i])::"memory");
      }
      tc_fence_before();
      mbar_arrive(BAR(X_DQFREE));
      return true;
    };
    auto add_dq = [&](int bh, int m, const float (&v)[64]) {
      if (!has_col) return;
      const size_t arow = (size_t)bh * a.nq64 * 64 + (size_t)m * 64;
      w_red_rows<D, (DET ? 100u : 150u)>(a.dq_acc + arow * D + c0 + dcol, v, std::make_integer_sequence<int, 4>{});
    };
    if constexpr (!DET) {
      for (int it = 0; it < n_iter; ++it) {
        int bh, m;
        iter_head_row(it, bh, m);
        float v[64];
        if (!read_dq(it, v)) break;
        add_dq(bh, m, v);
      }
    } else {
      int gphase = 0;
      for (int it = 0; it < n_iter; ++it) {
        int bh, m;
        iter_head_row(it, bh, m);
        int* sem = a.sem + ((size_t)bh * a.nq64 + m) * C::NHALF + half;
        if (leader) {
          const unsigned long long t0 = globaltimer_ns();
          while (w_ld_acquire(sem) != n) {
            if (*abort_flag) break;
            if (globaltimer_ns() - t0 > a.wait_ns) {
              *abort_flag = 1;
              atomicExch(a.status, DEV_TIMEOUT);
              break;
            }
          }
        }
        float v[64];
        if (!read_dq(it, v)) break;
        if (!w_group_sync(BAR(X_GD), gphase, wc) || *abort_flag) break;
        add_dq(bh, m, v);
        // The group barrier orders every drain thread's additions before the leader's
        // gpu-scope fence (cumulative), and that fence before the counter's increment.
        if (!w_group_sync(BAR(X_GD), gphase, wc)) break;
        if (leader) {
          __threadfence();
          atomicAdd(sem, 1);
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

// Preprocess: 16 threads per row; D = rowsum(dO o O), LSE2 = LSE log2(e),
// the row's dQacc zeroed (rows padded to whole 64-row tiles), counters zeroed.
template <int D>
__global__ void __launch_bounds__(256) bwd_wide_preprocess_kernel(const uint16_t* __restrict__ o,
                                                                   const uint16_t* __restrict__ dout,
                                                                   const float* __restrict__ lse,
                                                                   float* __restrict__ delta, float* __restrict__ lse2,
                                                                   float* __restrict__ dq_acc, int* __restrict__ sem,
                                                                   long long rows, int N, int npad, long long n_sem) {
  constexpr int PER = D / 16;   // 4, 8, 12 or 16 elements per thread
  const long long row = (long long)blockIdx.x * 16 + (threadIdx.x >> 4);
  const int sub = threadIdx.x & 15;
  const long long gtid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (sem != nullptr && gtid < n_sem) sem[gtid] = 0;
  if (row >= rows) return;
  const uint16_t* orow = o + row * D + sub * PER;
  const uint16_t* drow = dout + row * D + sub * PER;
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < PER / 4; ++i) {
    const uint2 av = *reinterpret_cast<const uint2*>(orow + 4 * i);
    const uint2 bv = *reinterpret_cast<const uint2*>(drow + 4 * i);
    const uint32_t aw[2] = {av.x, av.y}, bw[2] = {bv.x, bv.y};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      acc = fmaf(__uint_as_float(aw[k] << 16), __uint_as_float(bw[k] << 16), acc);
      acc = fmaf(__uint_as_float(aw[k] & 0xffff0000u), __uint_as_float(bw[k] & 0xffff0000u), acc);
    }
  }
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, 16);
  const long long bh = row / N, r = row - bh * N;
  float4* z = reinterpret_cast<float4*>(dq_acc + (bh * npad + r) * D + sub * PER);
#pragma unroll
  for (int i = 0; i < PER / 4; ++i) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (sub == 0) {
    delta[row] = acc;
    lse2[row] = lse[row] * kLog2eW;
  }
}

// dq = bf16(scale * dQacc), 8 elements per thread (dQacc rows padded per head).
template <int D>
__global__ void __launch_bounds__(256) bwd_wide_convert_kernel(const float* __restrict__ acc, uint16_t* __restrict__ dq,
                                                                float scale, long long n8, int N, int npad) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / (D / 8), bh = row / N, rr = row - bh * N;
    const long long src = ((bh * npad + rr) * D) / 8 + i % (D / 8);
    const float4 x = reinterpret_cast<const float4*>(acc)[2 * src];
    const float4 y = reinterpret_cast<const float4*>(acc)[2 * src + 1];
    uint4 r;
    r.x = pack_bf16x2(x.x * scale, x.y * scale);
    r.y = pack_bf16x2(x.z * scale, x.w * scale);
    r.z = pack_bf16x2(y.x * scale, y.y * scale);
    r.w = pack_bf16x2(y.z * scale, y.w * scale);
    reinterpret_cast<uint4*>(dq)[i] = r;
  }
}

template <int D, bool DET>
cudaError_t launch_wide_t(const BwdMaps& m, const BwdParams& p, cudaStream_t s) {
  const long long rows = (long long)p.B * p.Hq * p.N;
  const int nq64 = (p.N + 63) / 64;
  const long long n_sem = DET ? (long long)p.B * p.Hq * nq64 * BwCfg<D>::NHALF : 0;
  {
    const long long blocks = std::max((rows + 15) / 16, (n_sem + 255) / 256);
    if (blocks > 0) {
      bwd_wide_preprocess_kernel<D><<<(unsigned)blocks, 256, 0, s>>>(
          static_cast<const uint16_t*>(p.o), static_cast<const uint16_t*>(p.dout), p.lse, p.delta, p.lse2, p.dq_acc,
          p.sem, rows, p.N, nq64 * 64, n_sem);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  int dev = 0, sms = 152;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  {
    auto kern = attn_bwd_wide_kernel<D, DET>;
    constexpr uint32_t smem = BwCfg<D>::SMEM;
    static std::once_flag flags[64];
    static cudaError_t attr_err[64];
    std::call_once(flags[dev & 63], [&] {
      attr_err[dev & 63] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
    BwArgs a{};
    a.B = p.B; a.Hq = p.Hq; a.Hkv = p.Hkv; a.N = p.N; a.g = p.g; a.nq64 = nq64; a.nkb = (p.N + 127) / 128;
    a.causal = p.causal;
    a.c = p.c; a.scale = p.scale;
    a.lse2 = p.lse2; a.delta = p.delta; a.dq_acc = p.dq_acc; a.sem = p.sem;
    a.wait_ns = p.wait_ns; a.status = p.status;
    a.prefetch_ahead = sms;
    const long long grid = (long long)p.B * p.Hkv * a.nkb * BwCfg<D>::NHALF;
    if (grid > 0) {
      kern<<<(unsigned)grid, kBwThreads, smem, s>>>(m.q, m.k, m.v, m.dout, m.dk, m.dv, a);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  const long long n8 = rows * D / 8;
  const long long blocks = std::min<long long>((n8 + 255) / 256, (long long)sms * 8);
  if (blocks > 0)
    bwd_wide_convert_kernel<D><<<(unsigned)blocks, 256, 0, s>>>(p.dq_acc, static_cast<uint16_t*>(p.dq), p.scale, n8,
                                                                p.N, nq64 * 64);
  return cudaGetLastError();
}

}  // namespace

size_t bwd_wide_workspace_bytes(int B, int Hq, int N, int d, int deterministic) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t rows = (size_t)B * Hq * N;
  const size_t nq64 = (size_t)(N + 63) / 64;
  size_t n = al((size_t)B * Hq * nq64 * 64 * d * 4) + 2 * al(rows * 4);
  if (deterministic) n += al((size_t)B * Hq * nq64 * (d > 128 ? 2 : 1) * 4);
  return n;
}

void bwd_wide_workspace_carve(void* ws, int B, int Hq, int N, int d, int deterministic, BwdParams* p) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  char* c = static_cast<char*>(ws);
  const size_t rows = (size_t)B * Hq * N;
  const size_t nq64 = (size_t)(N + 63) / 64;
  p->dq_acc = reinterpret_cast<float*>(c);
  c += al((size_t)B * Hq * nq64 * 64 * d * 4);
  p->delta = reinterpret_cast<float*>(c);
  c += al(rows * 4);
  p->lse2 = reinterpret_cast<float*>(c);
  c += al(rows * 4);
  p->sem = deterministic ? reinterpret_cast<int*>(c) : nullptr;
}

cudaError_t launch_bwd_wide(const BwdMaps& maps, const BwdParams& p, cudaStream_t stream) {
  if (p.D == 64) return p.deterministic ? launch_wide_t<64, true>(maps, p, stream) : launch_wide_t<64, false>(maps, p, stream);
  if (p.D == 128) return p.deterministic ? launch_wide_t<128, true>(maps, p, stream) : launch_wide_t<128, false>(maps, p, stream);
  if (p.D == 192) return p.deterministic ? launch_wide_t<192, true>(maps, p, stream) : launch_wide_t<192, false>(maps, p, stream);
  if (p.D == 256) return p.deterministic ? launch_wide_t<256, true>(maps, p, stream) : launch_wide_t<256, false>(maps, p, stream);
  return cudaErrorNotSupported;
}

}  // namespace attn
