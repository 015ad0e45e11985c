// Persistent variant of the two-tile forward (d = 64, 128): one CTA per SM, each looping
// over a static share of the work units (pairs of 128-row query tiles), with the next
// unit's loads and first products overlapping the current unit's end.
//
// Same arithmetic as attn_fwd_kernel in fwd.cu (the FlashAttention-4 forward pipeline,
// "Hotelren FA4 summary" section 3; the longest work first for causal grids,
// "FlashAttention-4 explained" section 06) and the same roles; what changes is the life of
// a CTA.  In fwd.cu every unit pays a fixed cost: its Q and first K/V tiles arrive from
// memory before the first S, its pipeline fills and drains, and its epilogue runs after the
// last PV with the tensor core idle, ≈ 6.5 µs per unit measured against ≈ 1.8 µs per key
// block, so 18 % of a 16-block unit.  Here:
//   * the K/V ring and the MMA issue stream run on from one unit's key blocks into the
//     next unit's without a break (the first S of unit u+1 is issued with the last PV of
//     unit u), so barrier phases count over the CTA's whole life;
//   * warp 3 loads the next unit's Q tiles as soon as the last S of the current unit has
//     read them (one more barrier pair: Q loaded, Q free);
//   * the epilogue writes O straight from registers to global memory (no staging in the Q
//     buffer, which the next unit's Q is already filling) while the tensor core computes
//     the next unit's first S; the next unit's first PV waits for it through the P-ready
//     barrier, which the correction group joins only after its epilogue.
// Measured on GB300 it beats the per-unit kernel only for the shortest units (N = 512:
// +7 %, N = 1024: +1 %) and trails it from N = 2048 on (-4 to -8 %; causal -10 to -15 %,
// where a static share of units is also less even than the hardware's CTA-by-CTA
// dispatch), so it is opt-in (attn_set_fwd_persistent).  Same DRAM traffic and L2 hit
// rate as the per-unit kernel, but less tensor-pipe activity in the steady state, for a
// reason not found: neither the register split (the per-unit kernel runs the same one)
// nor local memory (none) nor the Q loader's polling (paced) explains it.
#include <cstdint>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kPThreads = 512;
constexpr float kLn2p = 0.6931471805599453f;

template <int D>
struct PCfg {
  static constexpr int NCH = D / 64;
  static constexpr uint32_t CHUNK = 128 * 128;
  static constexpr uint32_t TILE = CHUNK * NCH;
  static constexpr int NS = (D == 128) ? 4 : 8;                 // K/V ring slots
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_RING = 2 * TILE;
  static constexpr uint32_t OFF_CTRL = OFF_RING + NS * TILE;
  static constexpr uint32_t CTRL_BYTES = 256 + 8 * 128 * 4 + 64;
  static constexpr uint32_t SMEM = 1024 + OFF_CTRL + CTRL_BYTES;
  static constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 128, false, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, false, true);
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

enum {
  P_Q = 0,        // the unit's Q tiles landed (phase: the CTA's unit count)
  P_QFREE = 1,    // every S of the unit completed: the Q buffers may be refilled
  P_SFULL = 2,    // +t
  P_PFULL = 4,    // +t: P written (softmax) and O rescaled (correction)
  P_STATS = 6,    // +t
  P_REL = 8,      // +(group & 1): K/V slots of release group g (K_g, V_(g-1)) are free
  P_OFULL = 10,   // +t: the tile's last PV of the unit completed
  P_FIN = 12,     // +t: the unit's final row statistics written
  P_DONE = 14,
  P_FULL = 15,    // +slot (up to 8)
  P_COUNT = 23
};
static_assert(P_COUNT * 8 <= 256, "barriers fit the control block's first 256 bytes");

__device__ __forceinline__ bool pwait(uint32_t bar, uint32_t parity, const WaitCtl& w) {
  const bool ok = mbar_wait(bar, parity, w);
  return __all_sync(0xffffffffu, ok);
}

template <int N>
__device__ __forceinline__ void pfence(uint32_t (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i])::"memory");
}

// A unit: up to two 128-row query tiles sharing one K/V head (the mapping of fwd.cu:
// causal grids longest rows first, others all row slots of a head back to back; units
// from split_from on are split into one-tile entries).
struct PTiles {
  int n[2], row0[2], bh[2], bkv;
};
__device__ __forceinline__ PTiles punit(const FwdParams& p, int unit) {
  PTiles T;
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
    else if (p.causal) T.n[t] = (min(rows[t] + 127, p.N - 1) + p.koff) / 128 + 1;
    else T.n[t] = p.n_kvblk;
  }
  T.bkv = b * p.Hkv + hq0 / p.g;
  return T;
}
// Entry e of the work list: units below split_from whole, the rest as one-tile halves.
__device__ __forceinline__ PTiles pentry(const FwdParams& p, int e) {
  if (e < p.split_from) return punit(p, e);
  const int k = e - p.split_from;
  PTiles T = punit(p, p.split_from + k / 2);
  if (k & 1) {
    T.n[0] = T.n[1];
    T.row0[0] = T.row0[1];
    T.bh[0] = T.bh[1];
  }
  T.n[1] = 0;
  return T;
}

template <int D>
__global__ void __launch_bounds__(kPThreads, 1)
    attn_fwd_persist_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const FwdParams p, int n_entries) {
  using C = PCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint8_t* ctrl = smem + C::OFF_CTRL;
  const uint32_t bar0 = smem_u32(ctrl);
  auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * i; };
  float* alpha_buf = reinterpret_cast<float*>(ctrl + 256);   // [2][128]
  float* m_fin = alpha_buf + 256;                            // [2][128]
  float* l_fin = m_fin + 256;                                // [2][128]
  float* lq_fin = l_fin + 256;                               // [2][128]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(lq_fin + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  const int wg = warp >> 2;
  const int e0 = blockIdx.x, estep = gridDim.x;
  WaitCtl wc{p.wait_ns, p.status, abort_flag};

  if (threadIdx.x == 0) {
    mbar_init(BAR(P_Q), 1);
    mbar_init(BAR(P_QFREE), 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(BAR(P_SFULL + t), 1);
      mbar_init(BAR(P_PFULL + t), 256);
      mbar_init(BAR(P_STATS + t), 128);
      mbar_init(BAR(P_REL + t), 1);
      mbar_init(BAR(P_OFULL + t), 1);
      mbar_init(BAR(P_FIN + t), 128);
    }
    mbar_init(BAR(P_DONE), 1);
    for (int s = 0; s < C::NS; ++s) mbar_init(BAR(P_FULL + s), 1);
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

  // Register split: warpgroup 0 (producers, MMA) 64, softmax 184 + 184, correction 80:
  // 64 + 2 x 184 + 80 = 512 = 4 x 128, the launch's 128 x 512 threads (no spills).
  if (wg == 0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 64;");
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------------- K/V producer
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      // Ring position 2G holds K of the CTA's G-th key block, 2G + 1 its V; the blocks of
      // consecutive units follow one another.
      const int skip_pos = p.test_skip_first_kv ? 0 : -1;
      int next_pos = 0, G = 0;
      bool ok = true;
      for (int e = e0; e < n_entries && ok; e += estep) {
        const PTiles T = pentry(p, e);
        const int nmax = max(T.n[0], T.n[1]);   // 0: an empty half of a split unit, skipped by every role
        for (int j = 0; j < nmax && ok; ++j, ++G) {
          for (int which = 0; which < 2; ++which) {
            const int pos = 2 * G + which, slot = pos % C::NS;
            if (pos >= C::NS) {
              const int g = (pos - C::NS + 1) / 2;
              if (!mbar_wait(BAR(P_REL + (g & 1)), (g >> 1) & 1, wc)) {
                ok = false;
                break;
              }
            }
            next_pos = pos + 1;
            if (pos == skip_pos) continue;
            mbar_arrive_expect_tx(BAR(P_FULL + slot), C::TILE);
            const CUtensorMap* tm = which ? &tm_v : &tm_k;
            for (int c = 0; c < C::NCH; ++c)
              tma_load_3d(sbase + C::OFF_RING + slot * C::TILE + c * C::CHUNK, tm, c * 64, j * 128, T.bkv,
                          BAR(P_FULL + slot));
          }
        }
      }
      if (!ok) {
        const unsigned long long t0 = globaltimer_ns();
        for (int pos = max(0, next_pos - C::NS); pos < next_pos; ++pos) {
          if (pos == skip_pos) continue;
          const uint32_t bar = BAR(P_FULL + pos % C::NS), par = (pos / C::NS) & 1;
          while (!mbar_try_wait(bar, par) && globaltimer_ns() - t0 < p.wait_ns) {
          }
        }
      }
    } else if (warp == 3 && lane == 0) {
      // ---------------------------------------------------------------- Q loader
      tma_prefetch_desc(&tm_q);
      int u = 0;
      bool ok = true;
      for (int e = e0; e < n_entries; e += estep) {
        const PTiles T = pentry(p, e);
        if (max(T.n[0], T.n[1]) == 0) continue;
        // The wait spans a whole unit and is not latency-critical at the microsecond
        // scale: poll with pauses, so as not to take issue slots from the softmax and
        // correction warps that share this warp's scheduler.
        if (u > 0) {
          const unsigned long long t0 = globaltimer_ns();
          while (!mbar_try_wait(BAR(P_QFREE), (u - 1) & 1)) {
            if (*abort_flag) { ok = false; break; }
            if (globaltimer_ns() - t0 > p.wait_ns) {
              *abort_flag = 1;
              atomicExch(p.status, DEV_TIMEOUT);
              ok = false;
              break;
            }
            __nanosleep(256);
          }
          if (!ok) break;
        }
        mbar_arrive_expect_tx(BAR(P_Q), (T.n[0] > 0 ? C::TILE : 0) + (T.n[1] > 0 ? C::TILE : 0));
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (T.n[t] == 0) continue;
          for (int c = 0; c < C::NCH; ++c)
            tma_load_3d(sbase + C::OFF_Q + t * C::TILE + c * C::CHUNK, &tm_q, c * 64, T.row0[t], T.bh[t], BAR(P_Q));
        }
        ++u;
      }
      (void)ok;
      if (u > 0) {
        // The last Q load must land before the CTA's shared memory goes away.
        const unsigned long long t0 = globaltimer_ns();
        while (!mbar_try_wait(BAR(P_Q), (u - 1) & 1) && globaltimer_ns() - t0 < p.wait_ns) {
        }
      }
    } else if (warp == 1 && lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      // Iteration G (the CTA's G-th key block): for each tile, PV of the previous block
      // (the previous unit's last block when G opens a unit) then S of block G; a commit
      // then releases K_G and V_(G-1).
      int G = 0, u = 0;
      // PV products issued per tile (their P-ready phases); scalars, so that nothing of
      // the issuing thread's state lives in local memory.
      int pvc0 = 0, pvc1 = 0;
      int prev_n0 = 0, prev_n1 = 0, prev_nmax = 0;
      bool ok = true;
      const uint32_t qb = sbase + C::OFF_Q;
      constexpr uint32_t HI = sdesc_sw128_hi(1024);
      const uint32_t q0_lo = sdesc_sw128_lo(qb, 16), q1_lo = sdesc_sw128_lo(qb + C::TILE, 16);
      // PV_t of the block at ring position vpos: O_t (+)= P_t V; `last` marks the tile's
      // last block of its unit (its completion is what the epilogue waits for).
#define PV_ISSUE(t, pvc, vpos, first, last)                                                              \
  if (ok) {                                                                                               \
    if (!mbar_wait(BAR(P_PFULL + (t)), (pvc) & 1, wc)) {                                                  \
      ok = false;                                                                                         \
    } else {                                                                                              \
      tc_fence_after();                                                                                   \
      const uint32_t vlo_ = sdesc_sw128_lo(sbase + C::OFF_RING + ((vpos) % C::NS) * C::TILE, C::CHUNK);   \
      const uint32_t tS_ = tmem + uint32_t((t) * 128), tO_ = tmem + 256u + uint32_t((t) * D);            \
      _Pragma("unroll") for (int kk = 0; kk < 8; ++kk)                                                    \
        mma_ts_w(tO_, tS_ + kk * 8, vlo_ + kk * (2048 >> 4), HI, C::IDESC_PV,                           \
                 (!(first) || kk > 0) ? 1u : 0u);                                                         \
      ++(pvc);                                                                                            \
      if (last) mma_commit(BAR(P_OFULL + (t)));                                                           \
    }                                                                                                     \
  }
      for (int e = e0; e < n_entries && ok; e += estep) {
        const PTiles T = pentry(p, e);
        const int nmax = max(T.n[0], T.n[1]);
        if (nmax == 0) continue;
        for (int j = 0; j < nmax && ok; ++j, ++G) {
          const int kpos = 2 * G, vpos = 2 * G - 1;
          if (!mbar_wait(BAR(P_FULL + kpos % C::NS), (kpos / C::NS) & 1, wc)) { ok = false; break; }
          if (G > 0 && !mbar_wait(BAR(P_FULL + vpos % C::NS), (vpos / C::NS) & 1, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t k_lo = sdesc_sw128_lo(sbase + C::OFF_RING + (kpos % C::NS) * C::TILE, 16);
          // Tile 0: PV of its previous block (if any), the unit's Q (before its first S;
          // tile 0 always has one at j = 0), S of block j.  Then the same for tile 1.
          do {
            if (j == 0) {
              if (prev_n0 > 0 && prev_n0 == prev_nmax) PV_ISSUE(0, pvc0, vpos, prev_n0 == 1, true);
            } else if (j - 1 < T.n[0]) {
              PV_ISSUE(0, pvc0, vpos, j == 1, j == T.n[0]);
            }
            if (!ok) break;
            if (j == 0) {
              if (!mbar_wait(BAR(P_Q), u & 1, wc)) { ok = false; break; }
              tc_fence_after();
            }
            if (j < T.n[0]) {
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
                mma_ss_w(tmem, q0_lo + off, HI, k_lo + off, HI, C::IDESC_QK, kk > 0 ? 1u : 0u);
              }
              mma_commit(BAR(P_SFULL + 0));
            }
          } while (0);
          if (!ok) break;
          do {
            if (j == 0) {
              if (prev_n1 > 0 && prev_n1 == prev_nmax) PV_ISSUE(1, pvc1, vpos, prev_n1 == 1, true);
            } else if (j - 1 < T.n[1]) {
              PV_ISSUE(1, pvc1, vpos, j == 1, j == T.n[1]);
            }
            if (!ok) break;
            if (j < T.n[1]) {
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
                mma_ss_w(tmem + 128u, q1_lo + off, HI, k_lo + off, HI, C::IDESC_QK, kk > 0 ? 1u : 0u);
              }
              mma_commit(BAR(P_SFULL + 1));
            }
          } while (0);
          if (!ok) break;
          if (j == nmax - 1) mma_commit(BAR(P_QFREE));   // every S of the unit issued before this
          mma_commit(BAR(P_REL + (G & 1)));
        }
        prev_n0 = T.n[0];
        prev_n1 = T.n[1];
        prev_nmax = nmax;
        ++u;
      }
      // The last unit's last PVs.
      if (ok && G > 0) {
        const int vpos = 2 * G - 1;
        if (mbar_wait(BAR(P_FULL + vpos % C::NS), (vpos / C::NS) & 1, wc)) {
          tc_fence_after();
          do {
            if (prev_n0 > 0 && prev_n0 == prev_nmax) PV_ISSUE(0, pvc0, vpos, prev_n0 == 1, true);
            if (prev_n1 > 0 && prev_n1 == prev_nmax) PV_ISSUE(1, pvc1, vpos, prev_n1 == 1, true);
          } while (0);
        }
      }
#undef PV_ISSUE
      mma_commit(BAR(P_DONE));
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(BAR(P_DONE), 0) && globaltimer_ns() - t0 < p.wait_ns) {
      }
    }
  } else if (wg == 1 || wg == 2) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 184;");
    // ------------------------------------------------------------------ softmax of tile t
    const int t = wg - 1;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t tS = tmem + (uint32_t((warp & 3) * 32) << 16) + uint32_t(t * 128);
    const float c = p.c;
    int cnt = 0;      // the tile's key blocks so far (S-ready / P-ready phases)
    int un = 0;       // units in which the tile was present (final-statistics phases)
    bool ok = true;
    for (int e = e0; e < n_entries && ok; e += estep) {
      const PTiles T = pentry(p, e);
      // Select, not index: t is not a compile-time constant, and an indexed struct would
      // live in local memory.
      const int n_t = t ? T.n[1] : T.n[0];
      if (n_t == 0) continue;
      const int row0_t = t ? T.row0[1] : T.row0[0];
      const int grow = row0_t + row;
      float m = -INFINITY, l = 0.f, lq = 0.f;
      for (int j = 0; j < n_t; ++j, ++cnt) {
        if (!pwait(BAR(P_SFULL + t), cnt & 1, wc)) { ok = false; break; }
        tc_fence_after();
        uint32_t u[128];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, *reinterpret_cast<uint32_t(*)[32]>(&u[q * 32]));
        tmem_wait_ld();
        pfence(u);
        float* s = reinterpret_cast<float*>(u);
        const int kb = j * 128;
        const bool need_mask = (kb + 127 >= p.Nk) || (p.causal && kb + 127 > row0_t + p.koff);
        if (need_mask) {
          const int lim = (p.causal ? min(grow + p.koff, p.Nk - 1) : p.Nk - 1) - kb;   // last visible column
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
        const float m_cand = fmaxf(m, rmax * c);
        float alpha = 1.f;
        if (j == 0) {
          m = m_cand;
        } else if (m_cand - m > p.tau) {
          alpha = ex2_mufu(m - m_cand);
          m = m_cand;
        }
        alpha_buf[t * 128 + row] = alpha;
        mbar_arrive(BAR(P_STATS + t));
        const float neg_m = -m;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[64];
#pragma unroll
        for (int i = 0; i < 128; i += 2) {
          float x0, x1;
          ffma2_bc(x0, x1, s[i], s[i + 1], c, neg_m);
          const float e0v = ex2_mufu(x0), e1v = ex2_mufu(x1);
          pk[i >> 1] = pack_bf16x2(e0v, e1v);
          const int a2 = ((i >> 1) & 1) * 2;
          fadd2(acc[a2], acc[a2 + 1], acc[a2], acc[a2 + 1], e0v, e1v);
        }
        {
          const float pmax = ex2_mufu(fmaf(rmax, c, neg_m));
          const float pmax_q = __uint_as_float(pack_bf16x2(pmax, 0.f) << 16);
          const float blk = (acc[0] + acc[1]) + (acc[2] + acc[3]);
          l = l * alpha + blk;
          lq = lq * alpha + (blk - (pmax - pmax_q));
        }
        tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
        tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(BAR(P_PFULL + t));
      }
      if (!ok) break;
      m_fin[t * 128 + row] = m;
      l_fin[t * 128 + row] = l;
      lq_fin[t * 128 + row] = lq;
      mbar_arrive(BAR(P_FIN + t));
      ++un;
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 80;");
    // ------------------------------------------------------------------ correction + epilogue
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    int cnt[2] = {0, 0}, un[2] = {0, 0};
    bool ok = true;
    uint16_t* obase = static_cast<uint16_t*>(p.o_ptr);
    for (int e = e0; e < n_entries && ok; e += estep) {
      const PTiles T = pentry(p, e);
      const int nmax = max(T.n[0], T.n[1]);
      if (nmax == 0) continue;
      for (int j = 0; j < nmax && ok; ++j) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!ok || j >= T.n[t]) continue;
          if (!pwait(BAR(P_STATS + t), cnt[t] & 1, wc)) { ok = false; break; }
          const float alpha = alpha_buf[t * 128 + row];
          const bool any = __any_sync(0xffffffffu, alpha != 1.f);
          if (p.rescale_count != nullptr && j > 0) {
            const unsigned bal = __ballot_sync(0xffffffffu, alpha != 1.f);
            if (lane == 0 && bal) atomicAdd(p.rescale_count, (unsigned long long)__popc(bal));
          }
          if (j > 0 && any) {
            // S_t of this block complete => PV_t of the previous block (issued before it)
            // is complete too.
            if (!pwait(BAR(P_SFULL + t), cnt[t] & 1, wc)) { ok = false; break; }
            tc_fence_after();
            const uint32_t tO = tmem + lane_off + 256u + uint32_t(t * D);
            uint32_t r[32];
#pragma unroll 1
            for (int q = 0; q < D / 32; ++q) {
              tmem_ld32(tO + q * 32, r);
              tmem_wait_ld();
              pfence(r);
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
              tmem_st32(tO + q * 32, r);
            }
            tmem_wait_st();
          }
          tc_fence_before();
          mbar_arrive(BAR(P_PFULL + t));
          ++cnt[t];
        }
      }
      // Epilogue of the unit: O / lq -> bf16 -> global memory, row by row (each thread
      // its row), and the LSE.  The next unit's first PV of this tile waits for this
      // group's P-ready arrival, which comes after these reads of O.
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (!ok || T.n[t] == 0) continue;
        if (!pwait(BAR(P_FIN + t), un[t] & 1, wc)) { ok = false; break; }
        if (!pwait(BAR(P_OFULL + t), un[t] & 1, wc)) { ok = false; break; }
        ++un[t];
        tc_fence_after();
        const float mrow = m_fin[t * 128 + row], lrow = l_fin[t * 128 + row];
        const float inv = 1.f / lq_fin[t * 128 + row];
        const int grow = T.row0[t] + row;
        const bool real = grow < p.N;
        uint16_t* orow = obase + ((size_t)T.bh[t] * p.N + grow) * D;
        const uint32_t tO = tmem + lane_off + 256u + uint32_t(t * D);
        uint32_t r[32];
#pragma unroll 1
        for (int q = 0; q < D / 32; ++q) {
          tmem_ld32(tO + q * 32, r);
          tmem_wait_ld();
          pfence(r);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * inv, __uint_as_float(r[2 * i + 1]) * inv);
          if (real) {
#pragma unroll
            for (int w = 0; w < 4; ++w)
              *reinterpret_cast<uint4*>(orow + q * 32 + w * 8) = make_uint4(pk[4 * w], pk[4 * w + 1], pk[4 * w + 2],
                                                                             pk[4 * w + 3]);
          }
        }
        if (real) p.lse[(size_t)T.bh[t] * p.N + grow] = (mrow + __log2f(lrow)) * kLn2p;
        tc_fence_before();
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

template <int D>
cudaError_t launch_persist_t(const FwdMaps& m, const FwdParams& p, int grid, int n_entries, cudaStream_t s) {
  auto kern = attn_fwd_persist_kernel<D>;
  constexpr uint32_t smem = PCfg<D>::SMEM;
  static std::once_flag flags[64];
  static cudaError_t attr_err[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::call_once(flags[dev & 63], [&] {
    attr_err[dev & 63] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
  kern<<<grid, kPThreads, smem, s>>>(m.q, m.k, m.v, p, n_entries);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_persistent(const FwdMaps& maps, const FwdParams& p, int D, int grid, int n_entries,
                                  cudaStream_t s) {
  if (D == 64) return launch_persist_t<64>(maps, p, grid, n_entries, s);
  if (D == 128) return launch_persist_t<128>(maps, p, grid, n_entries, s);
  return cudaErrorInvalidValue;
}

}  // namespace attn
