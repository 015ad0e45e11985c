// FP8 forward for sm_103a: Q, K, V in e4m3 with one fp32 scale per 128-row block of each
// head ("Hotelren FA4 summary" section 6.3, future directions: FP8 inputs; the
// reverse-engineering page's FP8 path), and the block quantiser that produces them.
//
// What it computes: O = softmax(scale * Q~ K~^T [causal]) V~ and LSE, where X~ is the
// dequantised input (e4m3 value times its block's scale).  Block scales: q_scale
// [B, Hq, ceil(N/128)], k_scale and v_scale [B, Hkv, ceil(N/128)].
//
// How: the two-tile pipeline of fwd.cu (TMA producer warp, one MMA-issuing thread, two
// softmax warpgroups in ping-pong, a correction warpgroup that rescales O only when a row
// maximum grows by more than tau, TMA-store epilogue), with these changes:
//   * S = Q8 K8^T runs on the 8-bit tensor path (tcgen05.mma kind::f8f6f4, e4m3 x e4m3 ->
//     fp32): a 128 x 128 tile is four K = 32 steps instead of eight K = 16 steps;
//   * the scales enter the softmax: the exponent of block j uses c_j = scale * log2(e) *
//     sq * sk_j, and log2(sv_j) is added to it, so the exponential unit returns p * sv_j
//     directly; the row sum l accumulates p itself (the block sum divided by sv_j);
//   * P * sv_j is stored to tensor memory as fp16 (11-bit significand, finer than bf16), and
//     V8 is widened to fp16 in shared memory by the correction warpgroup, which is idle
//     between its rare rescales (e4m3 -> fp16 is exact), so O += P V~ runs on the 16-bit
//     path (kind::f16 with f16 operands).  Keeping P at 16
//     bits keeps the forward's error within the bf16 path's bounds against the exact
//     attention of the dequantised inputs; an e4m3 P (3 mantissa bits) would not be;
//   * O accumulates sum_j (p sv_j) V8_j = sum_j p V~_j in fp32, and the epilogue divides by l.
//
// Shared memory (d = 128): Q8 2 x 16 KB, K8 ring 2 x 16 KB, V8 staging 3 x 16 KB, V16
// (converted) 2 x 32 KB, which also stages O for the TMA store at the end.
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512); P_t (f16 pairs)
// overwrites the first 64 columns of S_t.
#include <cstdint>
#include <mutex>

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kF8Threads = 512;
constexpr float kLn2F8 = 0.6931471805599453f;

struct F8Cfg {
  static constexpr uint32_t T8 = 128 * 128;        // 128 rows x 128 e4m3 bytes (one swizzled box)
  static constexpr uint32_t CH16 = 128 * 128;      // 128 rows x 64 fp16 (one swizzled box)
  static constexpr uint32_t T16 = 2 * CH16;        // 128 x 128 fp16
  static constexpr int NK = 2;                     // K8 ring (released by the MMA group commits)
  static constexpr int NV8 = 3;                    // V8 staging slots (released by the converters)
  static constexpr int NV16 = 2;                   // converted V slots (released by the group commits)
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + 2 * T8;
  static constexpr uint32_t OFF_V8 = OFF_K + NK * T8;
  static constexpr uint32_t OFF_V16 = OFF_V8 + NV8 * T8;
  static constexpr uint32_t OFF_CTRL = OFF_V16 + NV16 * T16;
  static constexpr uint32_t CTRL_BYTES = 256 + 6 * 256 * 4 + 64;
  static constexpr uint32_t SMEM = 1024 + OFF_CTRL + CTRL_BYTES;
  static constexpr uint32_t IDESC_QK = idesc_f32acc(128, 128, FMT_E4M3, FMT_E4M3, false, false);
  static constexpr uint32_t IDESC_PV = idesc_f32acc(128, 128, FMT_F16, FMT_F16, false, true);
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(idesc_f32acc(128, 128, FMT_BF16, FMT_BF16, false, true) == idesc_bf16_f32(128, 128, false, true),
                "descriptor encodings agree");
};

enum {
  E_Q = 0,
  E_SFULL = 1,     // +t: S_t of the current block complete
  E_PFULL = 3,     // +t: P written (softmax, 128) and O rescaled (correction, 128)
  E_STATS = 5,     // +t: row statistics of the block written (128)
  E_REL = 7,       // +(group & 1): group j's MMAs done: K8 slot of block j, V16 slot of block j - 1 free
  E_OFULL = 9,     // +t: the tile's last PV complete
  E_DONE = 11,
  E_KFULL = 12,    // +slot (2)
  E_V8FULL = 14,   // +slot (3)
  E_V8EMPTY = 17,  // +slot (3): the correction warpgroup has read the slot (128 arrivals)
  E_V16FULL = 20,  // +slot (2): the correction warpgroup has written the slot (128 arrivals)
  E_EPI = 22,      // +t
  E_FIN = 24,      // +t
  E_COUNT = 26
};
static_assert(E_COUNT * 8 <= 256, "barriers fit the control block's first 256 bytes");

__device__ __forceinline__ bool f8_warp_wait(uint32_t bar, uint32_t parity, const WaitCtl& w) {
  const bool ok = mbar_wait(bar, parity, w);
  return __all_sync(0xffffffffu, ok);
}

template <int N>
__device__ __forceinline__ void f8_fence(uint32_t (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i])::"memory");
}

// The CTA's work: up to two 128-row query tiles sharing one K/V head.  The mapping of the
// bf16 forward: for grouped heads with even g, rows rs of query heads 2p and 2p + 1;
// otherwise two consecutive row tiles of one head.  Causal grids start the longest rows;
// non-causal grids run a head's row slots back to back.  Units past split_from run as
// two one-tile CTAs (the last, partial wave).
struct F8Tiles {
  int n[2], row0[2], bh[2], bkv;
};
__device__ __forceinline__ F8Tiles f8_unit(const FwdParams& p, int unit) {
  F8Tiles T;
  int hu, rs;
  if (p.causal) {
    rs = p.n_rowslots - 1 - unit / p.units_per_row;
    hu = unit % p.units_per_row;
  } else {
    hu = unit / p.n_rowslots;
    rs = unit % p.n_rowslots;
  }
  int b, hq0, hq1, r0, r1;
  if (p.pair_heads) {
    const int pairs = p.Hq / 2;
    b = hu / pairs;
    hq0 = 2 * (hu % pairs);
    hq1 = hq0 + 1;
    r0 = r1 = rs * 128;
  } else {
    b = hu / p.Hq;
    hq0 = hq1 = hu % p.Hq;
    r0 = 2 * rs * 128;
    r1 = r0 + 128;
  }
  const int rows[2] = {r0, r1}, hqs[2] = {hq0, hq1};
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    T.row0[t] = rows[t];
    T.bh[t] = b * p.Hq + hqs[t];
    if (rows[t] >= p.N) T.n[t] = 0;
    else if (p.causal) T.n[t] = min(rows[t] + 127, p.N - 1) / 128 + 1;
    else T.n[t] = p.n_kvblk;
  }
  T.bkv = b * p.Hkv + hq0 / p.g;
  return T;
}

// V8 block j (128 keys x 128 e4m3, 128-byte swizzled rows as TMA lands them) -> fp16 in the
// layout the PV product reads (two 64-column boxes with 128-byte swizzle, the layout TMA
// gives a bf16 V tile).  128 threads; a 16-byte piece (r, u) is columns 16u .. 16u + 15 of
// key row r.  Each quarter-warp takes half of two adjacent rows, (r, u in 0..3) with
// (r + 1, u in 4..7) or the other way round, so that its eight 16-byte loads and each of
// its two rounds of 16-byte stores fall on eight distinct bank groups.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t pair) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(pair));   // low byte -> low half
  return r;
}
__device__ __forceinline__ void widen_v_tile(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int ct) {
  const int w = ct >> 5, l = ct & 31;
  const int quarter = l >> 3, lq = l & 7;
  const int half = lq >> 2;                                  // which row of the pair
  const int u = (lq & 3) + 4 * (half ^ (quarter & 1));
  // Rows r = 16 it + r0 (it = 0..7); r & 7 = r0 & 7 for every it, so each address is a
  // per-thread base plus an immediate.
  const int r0 = 4 * w + 2 * (quarter >> 1) + half, sw = r0 & 7;
  const uint8_t* s_base = src + r0 * 128 + ((u ^ sw) << 4);
  uint8_t* d_base = dst + (u >> 2) * F8Cfg::CH16 + r0 * 128;
  const int d0 = ((2 * (u & 3)) ^ sw) << 4, d1 = ((2 * (u & 3) + 1) ^ sw) << 4;
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const uint4 v = *reinterpret_cast<const uint4*>(s_base + it * 2048);
    const uint32_t in[4] = {v.x, v.y, v.z, v.w};
    uint32_t h[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint16_t lo, hi;
      asm("mov.b32 {%0, %1}, %2;" : "=h"(lo), "=h"(hi) : "r"(in[i]));
      h[2 * i] = e4m3x2_to_f16x2(lo);
      h[2 * i + 1] = e4m3x2_to_f16x2(hi);
    }
    *reinterpret_cast<uint4*>(d_base + it * 2048 + d0) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(d_base + it * 2048 + d1) = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

__global__ void __launch_bounds__(kF8Threads, 1)
    attn_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                        const FwdParams p, const Fp8Scales sc) {
  using C = F8Cfg;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint8_t* ctrl = smem + C::OFF_CTRL;
  const uint32_t bar0 = smem_u32(ctrl);
  auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * i; };
  float* alpha_buf = reinterpret_cast<float*>(ctrl + 256);   // [2][128]
  float* m_fin = alpha_buf + 256;                            // [2][128]
  float* l_fin = m_fin + 256;                                // [2][128]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(l_fin + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  const int wg = warp >> 2;
  auto f8_cta = [&](int cta) -> F8Tiles {
    if (cta < p.split_from) return f8_unit(p, cta);
    const int k = cta - p.split_from;
    F8Tiles U = f8_unit(p, p.split_from + k / 2);
    if (k & 1) {
      U.n[0] = U.n[1];
      U.row0[0] = U.row0[1];
      U.bh[0] = U.bh[1];
    }
    U.n[1] = 0;
    return U;
  };
  const F8Tiles T = f8_cta(blockIdx.x);
  const int nmax = max(T.n[0], T.n[1]);
  WaitCtl wc{p.wait_ns, p.status, abort_flag};

  if (threadIdx.x == 0) {
    mbar_init(BAR(E_Q), 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(BAR(E_SFULL + t), 1);
      mbar_init(BAR(E_PFULL + t), 256);
      mbar_init(BAR(E_STATS + t), 128);
      mbar_init(BAR(E_REL + t), 1);
      mbar_init(BAR(E_OFULL + t), 1);
      mbar_init(BAR(E_EPI + t), 128);
      mbar_init(BAR(E_FIN + t), 128);
      mbar_init(BAR(E_KFULL + t), 1);
      mbar_init(BAR(E_V16FULL + t), 128);
    }
    mbar_init(BAR(E_DONE), 1);
    for (int s = 0; s < C::NV8; ++s) {
      mbar_init(BAR(E_V8FULL + s), 1);
      mbar_init(BAR(E_V8EMPTY + s), 128);
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

  // Register split against the launch's 128 x 512: producer and MMA 64; softmax 184 each;
  // correction (and V widening) 80.
  if (wg == 0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 64;");
    if (warp == 0) {
      // ---------------------------------------------------------------- producer
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_o);
        mbar_arrive_expect_tx(BAR(E_Q), (T.n[0] > 0 ? C::T8 : 0) + (T.n[1] > 0 ? C::T8 : 0));
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (T.n[t] > 0) tma_load_3d(sbase + C::OFF_Q + t * C::T8, &tm_q, 0, T.row0[t], T.bh[t], BAR(E_Q));
        // Loads issued so far (for the clean-up after a failed wait).
        int k_issued = 0, v_issued = 0;
        bool ok = true;
        for (int j = 0; j < nmax && ok; ++j) {
          const int ks = j % C::NK;
          // K8 slot ks last held block j - 2, released with group j - 2.
          if (j >= C::NK && !mbar_wait(BAR(E_REL + ((j - C::NK) & 1)), ((j - C::NK) >> 1) & 1, wc)) {
            ok = false;
            break;
          }
          if (j != 0 || !p.test_skip_first_kv) {
            mbar_arrive_expect_tx(BAR(E_KFULL + ks), C::T8);
            tma_load_3d(sbase + C::OFF_K + ks * C::T8, &tm_k, 0, j * 128, T.bkv, BAR(E_KFULL + ks));
          }
          k_issued = j + 1;
          const int vs = j % C::NV8;
          if (j >= C::NV8 && !mbar_wait(BAR(E_V8EMPTY + vs), ((j / C::NV8) - 1) & 1, wc)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(BAR(E_V8FULL + vs), C::T8);
          tma_load_3d(sbase + C::OFF_V8 + vs * C::T8, &tm_v, 0, j * 128, T.bkv, BAR(E_V8FULL + vs));
          v_issued = j + 1;
        }
        // The CTA one wave later (blockIdx + the SM count) starts about when this one ends:
        // bring its Q tiles and first K, V tiles into L2 now.
        const int nxt = (int)blockIdx.x + p.prefetch_ahead;
        if (ok && p.prefetch_ahead > 0 && nxt < (int)gridDim.x) {
          const F8Tiles U = f8_cta(nxt);
#pragma unroll
          for (int t = 0; t < 2; ++t)
            if ((t ? U.n[1] : U.n[0]) > 0) tma_prefetch_l2_3d(&tm_q, 0, t ? U.row0[1] : U.row0[0], t ? U.bh[1] : U.bh[0]);
          if (max(U.n[0], U.n[1]) > 0) {
            tma_prefetch_l2_3d(&tm_k, 0, 0, U.bkv);
            tma_prefetch_l2_3d(&tm_v, 0, 0, U.bkv);
          }
        }
        if (!ok) {
          // Let the copies still in flight land before the shared memory goes away.
          const unsigned long long t0 = globaltimer_ns();
          for (int j = max(0, k_issued - C::NK); j < k_issued; ++j) {
            if (j == 0 && p.test_skip_first_kv) continue;
            while (!mbar_try_wait(BAR(E_KFULL + j % C::NK), (j / C::NK) & 1) && globaltimer_ns() - t0 < p.wait_ns) {
            }
          }
          for (int j = max(0, v_issued - C::NV8); j < v_issued; ++j)
            while (!mbar_try_wait(BAR(E_V8FULL + j % C::NV8), (j / C::NV8) & 1) && globaltimer_ns() - t0 < p.wait_ns) {
            }
        }
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------------- MMA issuer
      if (lane == 0) {
        bool ok = mbar_wait(BAR(E_Q), 0, wc);
        tc_fence_after();
        for (int j = 0; j <= nmax && ok; ++j) {
          const int ks = j % C::NK, vs = (j + C::NV16 - 1) % C::NV16;
          if (j < nmax && !mbar_wait(BAR(E_KFULL + ks), (j / C::NK) & 1, wc)) { ok = false; break; }
          if (j >= 1 && !mbar_wait(BAR(E_V16FULL + vs), ((j - 1) / C::NV16) & 1, wc)) { ok = false; break; }
          tc_fence_after();
          constexpr uint32_t HI = sdesc_sw128_hi(1024);
          const uint32_t k_lo = sdesc_sw128_lo(sbase + C::OFF_K + ks * C::T8, 16);
          const uint32_t v_lo = sdesc_sw128_lo(sbase + C::OFF_V16 + vs * C::T16, C::CH16);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (!ok) break;
            const uint32_t tS = tmem + uint32_t(t * 128), tO = tmem + 256u + uint32_t(t * 128);
            if (j >= 1 && j <= T.n[t]) {
              // O_t += (P_t sv) V16_(j-1), A = P from tensor memory (f16 pairs)
              if (!mbar_wait(BAR(E_PFULL + t), (j - 1) & 1, wc)) { ok = false; break; }
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_ts_w(tO, tS + kk * 8, v_lo + kk * (2048 >> 4), HI, C::IDESC_PV, (j > 1 || kk > 0) ? 1u : 0u);
              if (j == T.n[t]) mma_commit(BAR(E_OFULL + t));
            }
            if (j < T.n[t]) {
              // S_t = Q8_t K8_j^T: four K = 32 steps within the 128-byte swizzled rows
              const uint32_t q_lo = sdesc_sw128_lo(sbase + C::OFF_Q + t * C::T8, 16);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ss_f8_w(tS, q_lo + kk * (32 >> 4), HI, k_lo + kk * (32 >> 4), HI, C::IDESC_QK, kk > 0 ? 1u : 0u);
              mma_commit(BAR(E_SFULL + t));
            }
          }
          if (!ok) break;
          mma_commit(BAR(E_REL + (j & 1)));   // K8 slot of block j and V16 slot of block j - 1
        }
        mma_commit(BAR(E_DONE));
        const unsigned long long t0 = globaltimer_ns();
        while (!mbar_try_wait(BAR(E_DONE), 0) && globaltimer_ns() - t0 < p.wait_ns) {
        }
      }
    }
  } else if (wg == 1 || wg == 2) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 184;");
    // ------------------------------------------------------------------ softmax
    const int t = wg - 1;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t tS = tmem + (uint32_t((warp & 3) * 32) << 16) + uint32_t(t * 128);
    const int row0_t = t ? T.row0[1] : T.row0[0];
    const int grow = row0_t + row;
    const int n_t = t ? T.n[1] : T.n[0];
    const int bh_t = t ? T.bh[1] : T.bh[0];
    const float c_t = n_t > 0 ? p.c * __ldg(sc.q + (size_t)bh_t * p.n_qblk + row0_t / 128) : 0.f;
    const float* skp = sc.k + (size_t)T.bkv * p.n_kvblk;
    const float* svp = sc.v + (size_t)T.bkv * p.n_kvblk;
    float sk_next = n_t > 0 ? __ldg(skp) : 1.f, sv_next = n_t > 0 ? __ldg(svp) : 1.f;
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j < n_t; ++j) {
      const float sk_j = sk_next, sv_j = sv_next;
      if (j + 1 < n_t) {
        sk_next = __ldg(skp + j + 1);
        sv_next = __ldg(svp + j + 1);
      }
      const float cj = c_t * sk_j;
      if (!f8_warp_wait(BAR(E_SFULL + t), j & 1, wc)) break;
      tc_fence_after();
      uint32_t u[128];
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, *reinterpret_cast<uint32_t(*)[32]>(&u[q * 32]));
      tmem_wait_ld();
      f8_fence(u);
      float* s = reinterpret_cast<float*>(u);
      const int kb = j * 128;
      if ((kb + 127 >= p.N) || (p.causal && kb + 127 > row0_t)) {
        const int lim = (p.causal ? min(grow, p.N - 1) : p.N - 1) - kb;   // last visible column
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i > lim) s[i] = -INFINITY;
      }
      float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
      for (int i = 4; i < 124; i += 8) {
        mx[0] = fmax3(mx[0], s[i], s[i + 1]);
        mx[1] = fmax3(mx[1], s[i + 2], s[i + 3]);
        mx[2] = fmax3(mx[2], s[i + 4], s[i + 5]);
        mx[3] = fmax3(mx[3], s[i + 6], s[i + 7]);
      }
      mx[0] = fmax3(mx[0], s[124], s[125]);
      mx[1] = fmax3(mx[1], s[126], s[127]);
      const float rmax = fmax3(fmaxf(mx[0], mx[1]), mx[2], mx[3]);
      const float m_cand = fmaxf(m, rmax * cj);
      float alpha = 1.f;
      if (j == 0) {
        m = m_cand;
      } else if (m_cand - m > p.tau) {
        alpha = ex2_mufu(m - m_cand);
        m = m_cand;
      }
      alpha_buf[t * 128 + row] = alpha;
      mbar_arrive(BAR(E_STATS + t));
      // p' = 2^(s cj - m + log2 sv_j) = p * sv_j; l sums p = p' / sv_j.
      const float off = __log2f(sv_j) - m;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[64];
#pragma unroll
      for (int i = 0; i < 128; i += 2) {
        float x0, x1;
        ffma2_bc(x0, x1, s[i], s[i + 1], cj, off);
        const float e0 = ex2_mufu(x0), e1 = ex2_mufu(x1);
        pk[i >> 1] = pack_f16x2(e0, e1);
        const int a2 = ((i >> 1) & 1) * 2;
        fadd2(acc[a2], acc[a2 + 1], acc[a2], acc[a2 + 1], e0, e1);
      }
      l = l * alpha + ((acc[0] + acc[1]) + (acc[2] + acc[3])) / sv_j;
      tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(BAR(E_PFULL + t));
    }
    m_fin[t * 128 + row] = m;
    l_fin[t * 128 + row] = l;
    mbar_arrive(BAR(E_FIN + t));
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 80;");
    // ------------------------------------------------------------------ correction + epilogue
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const int ct = (int)threadIdx.x - 384;
    // Widen V8 block jj into V16 slot jj % 2 once it has landed and the slot's previous
    // block (jj - 2) has been read by its PV products (released with group jj - 1).
    auto widen = [&](int jj) -> bool {
      const int vs8 = jj % C::NV8, vs16 = jj % C::NV16;
      if (!f8_warp_wait(BAR(E_V8FULL + vs8), (jj / C::NV8) & 1, wc)) return false;
      if (jj >= C::NV16 && !f8_warp_wait(BAR(E_REL + ((jj - 1) & 1)), ((jj - 1) >> 1) & 1, wc)) return false;
      widen_v_tile(smem + C::OFF_V8 + vs8 * C::T8, smem + C::OFF_V16 + vs16 * C::T16, ct);
      fence_proxy_async_smem();   // generic writes -> tensor-core reads
      mbar_arrive(BAR(E_V16FULL + vs16));
      mbar_arrive(BAR(E_V8EMPTY + vs8));
      return true;
    };
    bool ok = nmax == 0 || widen(0);
    for (int j = 0; j < nmax && ok; ++j) {
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (!ok || j >= T.n[t]) continue;
        if (!f8_warp_wait(BAR(E_STATS + t), j & 1, wc)) { ok = false; break; }
        const float alpha = alpha_buf[t * 128 + row];
        const bool any = __any_sync(0xffffffffu, alpha != 1.f);
        if (p.rescale_count != nullptr && j > 0) {
          const unsigned bal = __ballot_sync(0xffffffffu, alpha != 1.f);
          if (lane == 0 && bal) atomicAdd(p.rescale_count, (unsigned long long)__popc(bal));
        }
        if (j > 0 && any) {
          // S_t(j) complete => PV_t(j-1), issued before it, is complete too.
          if (!f8_warp_wait(BAR(E_SFULL + t), j & 1, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t tO = tmem + lane_off + 256u + uint32_t(t * 128);
          uint32_t r[32];
#pragma unroll 1
          for (int q = 0; q < 4; ++q) {
            tmem_ld32(tO + q * 32, r);
            tmem_wait_ld();
            f8_fence(r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(tO + q * 32, r);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(BAR(E_PFULL + t));
      }
      // The next block's V, needed by the PV products two MMA iterations from now.
      if (ok && j + 1 < nmax && !widen(j + 1)) ok = false;
    }
    // Epilogue: once every product of both tiles has completed (the V16 slots, which stage
    // O, are then free), per tile O / l -> bf16 -> V16 slot t -> TMA store, and the LSE.
#pragma unroll
    for (int t = 0; t < 2; ++t)
      if (ok && T.n[t] > 0 && !f8_warp_wait(BAR(E_OFULL + t), 0, wc)) ok = false;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (!ok || T.n[t] == 0) continue;
      if (!f8_warp_wait(BAR(E_FIN + t), 0, wc)) { ok = false; break; }
      tc_fence_after();
      const float mrow = m_fin[t * 128 + row], lrow = l_fin[t * 128 + row];
      const float inv = 1.f / lrow;
      const uint32_t tO = tmem + lane_off + 256u + uint32_t(t * 128);
      uint8_t* stage = smem + C::OFF_V16 + t * C::T16;
      uint32_t r[32];
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        tmem_ld32(tO + q * 32, r);
        tmem_wait_ld();
        f8_fence(r);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * inv, __uint_as_float(r[2 * i + 1]) * inv);
        const int box = (q * 32) / 64, j0 = ((q * 32) % 64) / 8;
#pragma unroll
        for (int uu = 0; uu < 4; ++uu) {
          const uint32_t off = box * C::CH16 + row * 128 + (((j0 + uu) ^ (row & 7)) * 16);
          *reinterpret_cast<uint4*>(stage + off) =
              make_uint4(pk[4 * uu], pk[4 * uu + 1], pk[4 * uu + 2], pk[4 * uu + 3]);
        }
      }
      const int grow = T.row0[t] + row;
      if (grow < p.N) p.lse[(size_t)T.bh[t] * p.N + grow] = (mrow + __log2f(lrow)) * kLn2F8;
      fence_proxy_async_smem();
      mbar_arrive(BAR(E_EPI + t));
      if (warp == 12 && lane == 0 && mbar_wait(BAR(E_EPI + t), 0, wc)) {
        for (int c = 0; c < 2; ++c)
          tma_store_3d(&tm_o, sbase + C::OFF_V16 + t * C::T16 + c * C::CH16, c * 64, T.row0[t], T.bh[t]);
        tma_store_commit();
      }
    }
    if (warp == 12 && lane == 0) tma_store_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------------------------
// Block quantiser: one CTA per 128-row block of one head (d = 128).  Thread t holds
// row t / 2, columns 64 (t & 1) .. + 63.  amax over the block, s = amax / 448 (1 when the
// block is all zero), codes = e4m3(x / s) rounded to nearest even, saturating.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quantize_fp8_kernel(const uint16_t* __restrict__ x, uint8_t* __restrict__ x8,
                                                           float* __restrict__ scales, int N, int nblk) {
  __shared__ float red[8];
  const int blk = blockIdx.x % nblk;
  const long long head = blockIdx.x / nblk;
  const int r = blk * 128 + (threadIdx.x >> 1);
  const int c0 = (threadIdx.x & 1) * 64;
  const bool live = r < N;
  const uint16_t* src = x + ((size_t)head * N + r) * 128 + c0;
  uint4 v[8];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[i] = live ? *reinterpret_cast<const uint4*>(src + 8 * i) : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
      amax = fmax3(amax, fabsf(__uint_as_float(w[k] << 16)), fabsf(__uint_as_float(w[k] & 0xffff0000u)));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  if (threadIdx.x == 0) scales[blockIdx.x] = s;
  if (!live) return;
  uint8_t* dst = x8 + ((size_t)head * N + r) * 128 + c0;
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    uint32_t outw[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t w[4] = {v[i + h].x, v[i + h].y, v[i + h].z, v[i + h].w};
#pragma unroll
      for (int k = 0; k < 4; k += 2) {
        const float2 a = make_float2(__fdiv_rn(__uint_as_float(w[k] << 16), s),
                                     __fdiv_rn(__uint_as_float(w[k] & 0xffff0000u), s));
        const float2 b = make_float2(__fdiv_rn(__uint_as_float(w[k + 1] << 16), s),
                                     __fdiv_rn(__uint_as_float(w[k + 1] & 0xffff0000u), s));
        const uint32_t lo = __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E4M3);
        const uint32_t hi = __nv_cvt_float2_to_fp8x2(b, __NV_SATFINITE, __NV_E4M3);
        outw[h * 2 + k / 2] = (lo & 0xffffu) | (hi << 16);
      }
    }
    *reinterpret_cast<uint4*>(dst + 8 * i) = make_uint4(outw[0], outw[1], outw[2], outw[3]);
  }
}

}  // namespace

size_t fwd_fp8_smem_bytes() { return F8Cfg::SMEM; }

cudaError_t launch_fwd_fp8(const FwdMaps& m, const FwdParams& p, const Fp8Scales& sc, int grid, cudaStream_t s) {
  static std::once_flag flags[64];
  static cudaError_t attr_err[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::call_once(flags[dev & 63], [&] {
    attr_err[dev & 63] =
        cudaFuncSetAttribute(attn_fwd_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, F8Cfg::SMEM);
  });
  if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
  attn_fwd_fp8_kernel<<<grid, kF8Threads, F8Cfg::SMEM, s>>>(m.q, m.k, m.v, m.o, p, sc);
  return cudaGetLastError();
}

cudaError_t launch_quantize_fp8(const void* x, void* x8, float* scales, long long heads, int N, cudaStream_t s) {
  const int nblk = (N + 127) / 128;
  const long long grid = heads * nblk;
  if (grid <= 0) return cudaSuccess;
  quantize_fp8_kernel<<<(unsigned)grid, 256, 0, s>>>(static_cast<const uint16_t*>(x), static_cast<uint8_t*>(x8),
                                                     scales, N, nblk);
  return cudaGetLastError();
}

}  // namespace attn
