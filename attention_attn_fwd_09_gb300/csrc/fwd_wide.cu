// Fused exact attention forward for wide heads (d = 192, 256) on sm_103a.
//
// Same result as the forward in fwd.cu: O = softmax(scale * Q K^T [causal]) V and LSE,
// with the scores never leaving the SM.  The pages recommend head dimensions 128 and 256
// ("Hotelren FA4 summary", section 6.2, item 1; the reverse-engineering page's kernel
// launch parameters name 256 as the largest).
//
// Why a kernel of its own: the two-tile ping-pong of fwd.cu needs two S buffers and two O
// accumulators in tensor memory, 2 * 128 + 2 * d columns, which is more than the 512
// columns of an SM once d > 128.  Here a CTA owns ONE 128-row query tile and the ping-pong
// runs over key blocks instead: S of block j + 1 is computed into the second S buffer
// while the softmax works on block j, so the tensor core alternates S_(j+1) and PV_j
// ("Hotelren FA4 summary" section 3.1: softmax of one block overlapped with the MMAs of
// another).  TMEM: S buffers [0,128) and [128,256) (P overwrites the first 64 columns of
// its buffer as bf16 pairs), O [256, 256+d).
//
// The same kernel serves d = 128 when one query tile per CTA is chosen, and grouped decode at
// d = 128 (the group's query heads x a few queries in one tile, keys split over CTAs): there a
// CTA has only one tile anyway, and the overlap of S_(j+1) with the softmax of block j is what
// keeps the tensor core busy.
//
// Warp roles: warp 0 TMA producer (Q once, K and V tiles through a ring), warp 1 MMA
// issuer, warp 2 TMEM allocator, warpgroup 1 softmax (one row per thread), warpgroups 2
// and 3 correction and epilogue (each owns half of O's columns: the conditional rescale
// of "Hotelren FA4 summary" section 3.3, tau = 8 in log2 units).
#include <cstdint>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kWideThreads = 512;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct WideCfg {
  // d = 128 (SPLIT): a key block's S product takes only 1024 tensor-core cycles, less than
  // one warpgroup's softmax of it, so two softmax warpgroups split each block by columns
  // (64 keys each, exchanging their row maxima) and one warpgroup does the correction.
  // d = 192, 256: one softmax warpgroup, two correction warpgroups (half of O each).
  static constexpr bool SPLIT = D == 128;
  static constexpr int NCH = D / 64;                    // 64-column (128-byte) chunks
  static constexpr uint32_t CHUNK = 128 * 128;          // one 128 x 64 bf16 box
  static constexpr uint32_t TILE = CHUNK * NCH;         // one 128 x D bf16 tile
  static constexpr int NS = D == 256 ? 2 : D == 192 ? 3 : 5;   // K/V ring slots (one tile each)
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_RING = TILE;
  static constexpr uint32_t OFF_CTRL = OFF_RING + NS * TILE;
  // control block: barriers, alpha[2][128], half maxima [2][2][128], m[128], l[2][128],
  // lq[2][128], TMEM address, abort flag
  static constexpr uint32_t CTRL_BYTES = 256 + (256 + 512 + 128 + 256 + 256) * 4 + 64;
  static constexpr uint32_t SMEM = 1024 + OFF_CTRL + CTRL_BYTES;
  static constexpr int OCOLS = SPLIT ? D : D / 2;       // O columns per correction warpgroup
  static constexpr int FIRST_CORR_WG = SPLIT ? 3 : 2;
  static constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 128, false, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, false, true);
  static_assert(D == 128 || D == 192 || D == 256, "one-tile forward: d = 128, 192 or 256");
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(OCOLS % 32 == 0, "correction columns in 32-column loads");
};

// Barriers (8 bytes each).  Per-block barriers come in pairs indexed by the block's parity,
// so that a waiter can never see two phases of one barrier complete at once.
enum {
  V_Q = 0,
  V_FULL = 1,    // +slot: a K or V tile landed (up to 5 slots)
  V_SFULL = 6,   // +parity: S of the block complete (also frees the block's K slot)
  V_STATS = 8,   // +parity: the block's rescale factors are in shared memory (128)
  V_PFULL = 10,  // +parity: P written and O rescaled (384)
  V_PVD = 12,    // +parity: the block's PV product complete (also frees its V slot)
  V_FIN = 14,    // final row statistics written (by every softmax thread)
  V_EPI = 15,    // O staged in shared memory (by every correction thread)
  V_DONE = 16,
  V_XCH = 17,    // +2 quarter + parity (SPLIT): both halves' row maxima of a 32-row quarter (64)
  V_COUNT = 25
};
static_assert(V_COUNT * 8 <= 256, "barriers fit the control block's first 256 bytes");

__device__ __forceinline__ bool warp_wait_w(uint32_t bar, uint32_t parity, const WaitCtl& w) {
  const bool ok = mbar_wait(bar, parity, w);
  return __all_sync(0xffffffffu, ok);
}

template <int N>
__device__ __forceinline__ void reg_fence_w(uint32_t (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i])::"memory");
}

// Load order through the ring: K_0, K_1, V_0, K_2, V_1, ..., K_(n-1), V_(n-2), V_(n-1).
// K runs one block ahead of V because S_(j+1) is issued before PV_j; with one tile per
// slot, a plain K_j, V_j order would hold K_(j+2) back until PV_j had freed V_j's slot.
__device__ __forceinline__ int pos_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int pos_v(int j, int n) { return min(2 * j + 2, 2 * n - 1); }
// The tile at ring position pos: sets j and returns true for V_j, false for K_j.
__device__ __forceinline__ bool item_at(int pos, int n, int& j) {
  if (pos == 0) { j = 0; return false; }
  if (pos == 2 * n - 1) { j = n - 1; return true; }
  if (pos & 1) { j = (pos + 1) >> 1; return false; }
  j = (pos - 2) >> 1;
  return true;
}

// CTA -> (b * Hq + hq, 128-row block).  Causal grids run the longest rows first; others
// run the row blocks of a head back to back (its K and V stay hot in L2).  The sequence
// fields (first query row qs, one past the last qend, first key row krow0, keys nk,
// nk - nq = koff) are constants of the launch except for packed sequences.
struct WideTile {
  int n, row0, bh, bkv;
  int qs, qend, krow0, nk, koff;
  int j0;         // first key block (grouped decode: the start of this CTA's key split)
};
__device__ __forceinline__ WideTile map_wide(const FwdParams& p, int cta) {
  WideTile T;
  const int heads = p.B * p.Hq;
  int rb;
  if (p.causal) {
    rb = p.n_qblk - 1 - cta / heads;
    T.bh = cta % heads;
  } else {
    T.bh = cta / p.n_qblk;
    rb = cta % p.n_qblk;
  }
  T.row0 = rb * 128;
  const int b = T.bh / p.Hq, hq = T.bh % p.Hq;
  T.bkv = b * p.Hkv + hq / p.g;
  T.n = p.causal ? (min(T.row0 + 127, p.N - 1) + p.koff) / 128 + 1 : p.n_kvblk;
  T.qs = 0; T.qend = p.N; T.krow0 = 0; T.nk = p.Nk; T.koff = p.koff;
  T.j0 = 0;
  return T;
}

// Grouped decode (d = 128): CTA = (K/V head, key split); its tile holds the group's g query
// heads x N queries as rows h * N + q (rows past g * N are padding and never written).
__device__ __forceinline__ WideTile map_wide_grouped(const FwdParams& p, int cta) {
  WideTile T;
  const int unit = cta / p.kv_splits, sp = cta % p.kv_splits;
  const int b = unit / p.Hkv, hkv = unit % p.Hkv;
  T.bkv = unit;
  T.bh = b * p.Hq + hkv * p.g;
  T.row0 = 0;
  T.j0 = sp * p.blocks_per_split;
  T.n = min(p.n_kvblk, T.j0 + p.blocks_per_split) - T.j0;
  T.qs = 0; T.qend = p.N; T.krow0 = 0; T.nk = p.Nk; T.koff = p.koff;
  return T;
}

// Packed sequences: the CTA's record of the unit table (varlen.cu, one tile per record)
// names the sequence, the query head and the tile's first row within the sequence.
__device__ __forceinline__ WideTile map_wide_varlen(const FwdParams& p, const int4 u) {
  WideTile T;
  const int b = u.x, hq = u.y & 0xffff, r0 = u.z;
  const int q0 = p.cu_q[b], nq = p.cu_q[b + 1] - q0;
  const int k0 = p.cu_k[b], nk = p.cu_k[b + 1] - k0;
  T.qs = q0; T.qend = q0 + nq; T.krow0 = k0; T.nk = nk; T.koff = nk - nq;
  T.row0 = q0 + r0;
  T.bh = hq;
  T.bkv = hq / p.g;
  T.n = p.causal ? (min(r0 + 127, nq - 1) + T.koff) / 128 + 1 : (nk + 127) / 128;
  T.j0 = 0;
  return T;
}

// MODE 0: the standard forward; MODE 1: grouped decode (d = 128; partial results to the
// workspace, merged by launch_fwd_merge); MODE 2: packed variable-length sequences (d = 192,
// 256; one unit-table record per CTA).
template <int D, int MODE>
__global__ void __launch_bounds__(kWideThreads, 1)
    attn_fwd_wide_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                         const FwdParams p) {
  using C = WideCfg<D>;
  constexpr bool VL = MODE == 2;
  constexpr bool GRP = MODE == 1;
  static_assert(!GRP || C::SPLIT, "grouped decode through the one-tile kernel at d = 128 only");
  static_assert(V_FULL + C::NS <= V_SFULL, "every ring slot needs its own barrier below the next group");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint8_t* ctrl = smem + C::OFF_CTRL;
  const uint32_t bar0 = smem_u32(ctrl);
  auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * i; };
  float* alpha_buf = reinterpret_cast<float*>(ctrl + 256);   // [2][128]
  float* pm_buf = alpha_buf + 256;                           // [2][2][128] (SPLIT)
  float* m_fin = pm_buf + 512;                               // [128]
  float* l_fin = m_fin + 128;                                // [2][128]
  float* lq_fin = l_fin + 256;                               // [2][128]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(lq_fin + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  const int wg = warp >> 2;
  // A kernel launched after this one as a programmatic dependent (the decode merge, the
  // backward's preprocess) may be scheduled now; it waits for this grid's completion before
  // reading what it writes.
  pdl_trigger();
  WideTile T;
  if constexpr (VL) {
    // CTAs past the table's records have no work: they leave before touching barriers or
    // tensor memory.
    if ((int)blockIdx.x >= __ldg(p.vl_count)) return;
    T = map_wide_varlen(p, p.vl_units[blockIdx.x]);
  } else if constexpr (GRP) {
    T = map_wide_grouped(p, blockIdx.x);
  } else {
    T = map_wide(p, blockIdx.x);
  }
  const int n = T.n;
  WaitCtl wc{p.wait_ns, p.status, abort_flag};

  if (threadIdx.x == 0) {
    mbar_init(BAR(V_Q), 1);
    for (int s = 0; s < C::NS; ++s) mbar_init(BAR(V_FULL + s), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(BAR(V_SFULL + b), 1);
      mbar_init(BAR(V_STATS + b), 128);
      mbar_init(BAR(V_PFULL + b), 384);
      mbar_init(BAR(V_PVD + b), 1);
    }
    mbar_init(BAR(V_FIN), C::SPLIT ? 256 : 128);
    mbar_init(BAR(V_EPI), C::SPLIT ? 128 : 256);
    mbar_init(BAR(V_DONE), 1);
    for (int i = 0; i < 8; ++i) mbar_init(BAR(V_XCH + i), 64);
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

  // Register split (per thread), against the launch's 128 x 512 threads:
  //   d = 192, 256: warpgroup 0 (producer, MMA) 64, softmax 224, two correction
  //                 warpgroups 112 each: 64 + 224 + 2 x 112 = 512 = 4 x 128;
  //   d = 128:      warpgroup 0 64, two softmax halves 152 each, correction 144:
  //                 64 + 2 x 152 + 144 = 512.
  const bool softmax_wg = C::SPLIT ? (wg == 1 || wg == 2) : (wg == 1);
  if (wg == 0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 64;");
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------------- producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_o);
      mbar_arrive_expect_tx(BAR(V_Q), GRP ? p.q_tile_bytes : C::TILE);
      for (int c = 0; c < C::NCH; ++c) tma_load_3d(sbase + C::OFF_Q + c * C::CHUNK, &tm_q, c * 64, T.row0, T.bh, BAR(V_Q));
      // A slot is refilled once its previous occupant's reader completed: S_i for K_i,
      // PV_i for V_i.
      int next_idx = 0;
      bool ok = true;
      for (int pos = 0; pos < 2 * n; ++pos) {
        const int slot = pos % C::NS;
        if (pos >= C::NS) {
          int i;
          const bool was_v = item_at(pos - C::NS, n, i);
          const uint32_t bar = was_v ? BAR(V_PVD + (i & 1)) : BAR(V_SFULL + (i & 1));
          if (!mbar_wait(bar, (i >> 1) & 1, wc)) {
            ok = false;
            break;
          }
        }
        int j;
        const bool is_v = item_at(pos, n, j);
        next_idx = pos + 1;
        mbar_arrive_expect_tx(BAR(V_FULL + slot), C::TILE);
        const CUtensorMap* tm = is_v ? &tm_v : &tm_k;
        for (int c = 0; c < C::NCH; ++c)
          tma_load_3d(sbase + C::OFF_RING + slot * C::TILE + c * C::CHUNK, tm, c * 64, T.krow0 + (T.j0 + j) * 128,
                      T.bkv, BAR(V_FULL + slot));
      }
      // The CTA one wave later (blockIdx + the SM count) starts about when this one ends:
      // bring its Q tile and first K, V tiles into L2 now.
      if constexpr (MODE == 0) {
        const int nxt = (int)blockIdx.x + p.prefetch_ahead;
        if (ok && p.prefetch_ahead > 0 && nxt < (int)gridDim.x) {
          const WideTile U = map_wide(p, nxt);
          for (int c = 0; c < C::NCH; ++c) {
            tma_prefetch_l2_3d(&tm_q, c * 64, U.row0, U.bh);
            if (U.n > 0) {
              tma_prefetch_l2_3d(&tm_k, c * 64, U.krow0, U.bkv);
              tma_prefetch_l2_3d(&tm_v, c * 64, U.krow0, U.bkv);
            }
          }
        }
      }
      if (!ok) {
        // Let the copies still in flight land before the CTA's shared memory goes away.
        const unsigned long long t0 = globaltimer_ns();
        for (int idx = max(0, next_idx - C::NS); idx < next_idx; ++idx) {
          const uint32_t bar = BAR(V_FULL + idx % C::NS), par = (idx / C::NS) & 1;
          while (!mbar_try_wait(bar, par) && globaltimer_ns() - t0 < p.wait_ns) {
          }
        }
      }
    } else if (warp == 1 && lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      // Issue order: S_0, then per block j: S_(j+1), PV_j.  S_(j+1) lands in the buffer
      // of P_(j-1), which PV_(j-1) (issued earlier) has read: MMAs execute in issue order.
      bool ok = mbar_wait(BAR(V_Q), 0, wc);
      tc_fence_after();
      // Matrix descriptors as low words advanced by (offset / 16), one constant high word.
      constexpr uint32_t HI = sdesc_sw128_hi(1024);
      const uint32_t q_lo = sdesc_sw128_lo(sbase + C::OFF_Q, 16);
      auto issue_s = [&](int j) -> bool {
        const int idx = pos_k(j), slot = idx % C::NS;
        if (!mbar_wait(BAR(V_FULL + slot), (idx / C::NS) & 1, wc)) return false;
        tc_fence_after();
        const uint32_t k_lo = sdesc_sw128_lo(sbase + C::OFF_RING + slot * C::TILE, 16);
        const uint32_t tS = tmem + uint32_t((j & 1) * 128);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
          mma_ss_w(tS, q_lo + off, HI, k_lo + off, HI, C::IDESC_QK, kk > 0 ? 1u : 0u);
        }
        mma_commit(BAR(V_SFULL + (j & 1)));
        return true;
      };
      if (ok && n > 0) ok = issue_s(0);
      for (int j = 0; j < n && ok; ++j) {
        if (j + 1 < n && !issue_s(j + 1)) {
          ok = false;
          break;
        }
        // O += P_j V_j, once P_j is written and O rescaled for block j.
        if (!mbar_wait(BAR(V_PFULL + (j & 1)), (j >> 1) & 1, wc)) {
          ok = false;
          break;
        }
        const int vidx = pos_v(j, n), vslot = vidx % C::NS;
        if (!mbar_wait(BAR(V_FULL + vslot), (vidx / C::NS) & 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t v_lo = sdesc_sw128_lo(sbase + C::OFF_RING + vslot * C::TILE, C::CHUNK);
        const uint32_t tS = tmem + uint32_t((j & 1) * 128), tO = tmem + 256u;
        // P of keys 16kk .. 16kk + 15: columns 8kk .. of the buffer; with SPLIT the second
        // half's keys sit at columns 64 .. 95 (each half writes inside its own scores).
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_w(tO, tS + (C::SPLIT && kk >= 4 ? 32 : 0) + kk * 8, v_lo + kk * (2048 >> 4), HI, C::IDESC_PV,
                   (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(BAR(V_PVD + (j & 1)));
      }
      // Drain: every MMA issued above completes before TMEM is released.
      mma_commit(BAR(V_DONE));
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(BAR(V_DONE), 0) && globaltimer_ns() - t0 < p.wait_ns) {
      }
    }
  } else if (softmax_wg && C::SPLIT) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 152;");
    // ------------------------------------------------------------------ softmax, one half
    // Half h owns keys [64h, 64h + 64) of every block.  The two halves of a row exchange
    // their maxima, so both keep the same running maximum and rescale factor; each keeps
    // its own sums, added in the epilogue.
    const int h = wg - 1, q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    const int grow = T.row0 + row;
    const float c = p.c;
    float m = -INFINITY, l = 0.f, lq = 0.f;
    for (int j = 0; j < n; ++j) {
      if (!warp_wait_w(BAR(V_SFULL + (j & 1)), (j >> 1) & 1, wc)) break;
      tc_fence_after();
      const uint32_t tS = tmem + lane_off + uint32_t((j & 1) * 128 + h * 64);
      uint32_t u[64];
      tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
      tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
      tmem_wait_ld();
      reg_fence_w(u);
      float* s = reinterpret_cast<float*>(u);
      const int kb = (T.j0 + j) * 128 + h * 64;
      // Grouped decode: row = hq * N + q holds query q (rows past g * N are padding).
      const int qrow = GRP ? row % p.N : grow - T.qs;
      const bool need_mask = GRP || (kb + 63 >= T.nk) || (p.causal && kb + 63 > T.row0 - T.qs + T.koff);
      if (need_mask) {
        const int lim = (p.causal ? min(qrow + T.koff, T.nk - 1) : T.nk - 1) - kb;   // last visible column
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (i > lim) s[i] = -INFINITY;
      }
      float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
      for (int i = 4; i < 60; i += 8) {
        mx[0] = fmax3(mx[0], s[i], s[i + 1]);
        mx[1] = fmax3(mx[1], s[i + 2], s[i + 3]);
        mx[2] = fmax3(mx[2], s[i + 4], s[i + 5]);
        mx[3] = fmax3(mx[3], s[i + 6], s[i + 7]);
      }
      mx[0] = fmax3(mx[0], s[60], s[61]);
      mx[1] = fmax3(mx[1], s[62], s[63]);
      const float own = fmax3(fmaxf(mx[0], mx[1]), mx[2], mx[3]);
      float* pm = pm_buf + (j & 1) * 256;
      pm[h * 128 + row] = own;
      mbar_arrive(BAR(V_XCH + q4 * 2 + (j & 1)));
      if (!warp_wait_w(BAR(V_XCH + q4 * 2 + (j & 1)), (j >> 1) & 1, wc)) break;
      const float other = pm[(1 - h) * 128 + row];
      const float rmax = fmaxf(own, other);
      const float m_cand = fmaxf(m, rmax * c);
      float alpha = 1.f;
      if (j == 0) {
        m = m_cand;
      } else if (m_cand - m > p.tau) {
        alpha = ex2_mufu(m - m_cand);
        m = m_cand;
      }
      if (h == 0) {
        alpha_buf[(j & 1) * 128 + row] = alpha;
        mbar_arrive(BAR(V_STATS + (j & 1)));
      }
      // Grouped decode: a row may see no key of this CTA's split yet (m = -inf); its
      // probabilities are then 0, not 2^(-inf + inf).
      const float neg_m = (GRP && m == -INFINITY) ? 0.f : -m;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 64; i += 2) {
        float x0, x1;
        ffma2_bc(x0, x1, s[i], s[i + 1], c, neg_m);
        const float e0 = ex2_mufu(x0), e1 = ex2_mufu(x1);
        pk[i >> 1] = pack_bf16x2(e0, e1);
        const int a2 = ((i >> 1) & 1) * 2;
        fadd2(acc[a2], acc[a2 + 1], acc[a2], acc[a2 + 1], e0, e1);
      }
      {
        // The bf16 rounding of the block's largest p is taken off lq once per row, by
        // the half that holds that maximum (the first one on a tie).
        const bool holds_max = own == rmax && (h == 0 || other != rmax);
        const float pmax = ex2_mufu(fmaf(rmax, c, neg_m));
        const float pmax_q = __uint_as_float(pack_bf16x2(pmax, 0.f) << 16);
        const float blk = (acc[0] + acc[1]) + (acc[2] + acc[3]);
        l = l * alpha + blk;
        lq = lq * alpha + (holds_max ? blk - (pmax - pmax_q) : blk);
      }
      tmem_st32(tS, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(BAR(V_PFULL + (j & 1)));
    }
    if (h == 0) m_fin[row] = m;
    l_fin[h * 128 + row] = l;
    lq_fin[h * 128 + row] = lq;
    mbar_arrive(BAR(V_FIN));
  } else if (softmax_wg) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 224;");
    // ------------------------------------------------------------------ softmax
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const int grow = T.row0 + row;
    const float c = p.c;
    float m = -INFINITY, l = 0.f, lq = 0.f;
    for (int j = 0; j < n; ++j) {
      if (!warp_wait_w(BAR(V_SFULL + (j & 1)), (j >> 1) & 1, wc)) break;
      tc_fence_after();
      const uint32_t tS = tmem + lane_off + uint32_t((j & 1) * 128);
      uint32_t u[128];
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, *reinterpret_cast<uint32_t(*)[32]>(&u[q * 32]));
      tmem_wait_ld();
      reg_fence_w(u);
      float* s = reinterpret_cast<float*>(u);
      // Packed sequences: keys count from the sequence's start; those past its end (the
      // next sequence's) are masked like those past the tensor's end.
      const int kb = j * 128;
      const bool need_mask = (kb + 127 >= T.nk) || (p.causal && kb + 127 > T.row0 - T.qs + T.koff);
      if (need_mask) {
        const int lim = (p.causal ? min(grow - T.qs + T.koff, T.nk - 1) : T.nk - 1) - kb;   // last visible column
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
      alpha_buf[(j & 1) * 128 + row] = alpha;
      mbar_arrive(BAR(V_STATS + (j & 1)));
      // p = 2^(s*c - m); l sums the fp32 p, lq the same minus each block's bf16 rounding
      // of its largest p (the PV product multiplies bf16(p)), as in fwd.cu.
      const float neg_m = -m;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[64];
#pragma unroll
      for (int i = 0; i < 128; i += 2) {
        float x0, x1;
        ffma2_bc(x0, x1, s[i], s[i + 1], c, neg_m);
        const float e0 = ex2_mufu(x0), e1 = ex2_mufu(x1);
        pk[i >> 1] = pack_bf16x2(e0, e1);
        const int a2 = ((i >> 1) & 1) * 2;
        fadd2(acc[a2], acc[a2 + 1], acc[a2], acc[a2 + 1], e0, e1);
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
      mbar_arrive(BAR(V_PFULL + (j & 1)));
    }
    m_fin[row] = m;
    l_fin[row] = l;
    lq_fin[row] = lq;
    mbar_arrive(BAR(V_FIN));
  } else {
    if constexpr (C::SPLIT) asm volatile("setmaxnreg.inc.sync.aligned.u32 144;");
    else asm volatile("setmaxnreg.dec.sync.aligned.u32 112;");
    // ------------------------------------------------------------------ correction + epilogue
    const int half = wg - C::FIRST_CORR_WG;              // O columns [half * OCOLS, +OCOLS)
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tO = tmem + lane_off + 256u + uint32_t(half * C::OCOLS);
    bool ok = true;
    for (int j = 0; j < n && ok; ++j) {
      if (!warp_wait_w(BAR(V_STATS + (j & 1)), (j >> 1) & 1, wc)) {
        ok = false;
        break;
      }
      const float alpha = alpha_buf[(j & 1) * 128 + row];
      const bool any = __any_sync(0xffffffffu, alpha != 1.f);
      if (half == 0 && p.rescale_count != nullptr && j > 0) {
        const unsigned bal = __ballot_sync(0xffffffffu, alpha != 1.f);
        if (lane == 0 && bal) atomicAdd(p.rescale_count, (unsigned long long)__popc(bal));
      }
      if (j > 0 && any) {
        // O holds PV_(j-1) once that product completed.
        if (!warp_wait_w(BAR(V_PVD + ((j - 1) & 1)), ((j - 1) >> 1) & 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t r[32];
#pragma unroll 1
        for (int q = 0; q < C::OCOLS / 32; ++q) {
          tmem_ld32(tO + q * 32, r);
          tmem_wait_ld();
          reg_fence_w(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(tO + q * 32, r);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      mbar_arrive(BAR(V_PFULL + (j & 1)));
    }
    // Epilogue: O / lq -> bf16 -> swizzled shared memory (the Q tile, free once the last
    // S product completed, which it did before the last PV) -> TMA store; LSE to global.
    // Grouped decode: this key split's partial result, O / lq (0 where the row saw no key)
    // and LSE in fp32, for rows h * N + q of the group, to the workspace.
    if (GRP && ok && n > 0 && warp_wait_w(BAR(V_FIN), 0, wc) &&
        warp_wait_w(BAR(V_PVD + ((n - 1) & 1)), ((n - 1) >> 1) & 1, wc)) {
      tc_fence_after();
      const int unit = blockIdx.x / p.kv_splits, sp = blockIdx.x % p.kv_splits;
      const size_t slot = (size_t)sp * (p.B * p.Hkv) + unit;
      const bool real = row < p.g * p.N;
      const float lrow = l_fin[row] + l_fin[128 + row];
      const float lqr = lq_fin[row] + lq_fin[128 + row];
      const float invp = lqr > 0.f ? 1.f / lqr : 0.f;
      float* dst = p.part_o + (slot * 128 + row) * D;
      uint32_t r[32];
#pragma unroll 1
      for (int q = 0; q < D / 32; ++q) {
        tmem_ld32(tO + q * 32, r);   // warp-collective: every lane loads its row
        tmem_wait_ld();
        reg_fence_w(r);
        if (real) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(dst + q * 32 + i) =
                make_float4(__uint_as_float(r[i]) * invp, __uint_as_float(r[i + 1]) * invp,
                            __uint_as_float(r[i + 2]) * invp, __uint_as_float(r[i + 3]) * invp);
        }
      }
      if (real) p.part_lse[slot * 128 + row] = lrow > 0.f ? (m_fin[row] + __log2f(lrow)) * kLn2 : -INFINITY;
    } else if (!GRP && ok && n > 0 && warp_wait_w(BAR(V_FIN), 0, wc) &&
        warp_wait_w(BAR(V_PVD + ((n - 1) & 1)), ((n - 1) >> 1) & 1, wc)) {
      tc_fence_after();
      const float lrow = C::SPLIT ? l_fin[row] + l_fin[128 + row] : l_fin[row];
      const float inv = 1.f / (C::SPLIT ? lq_fin[row] + lq_fin[128 + row] : lq_fin[row]);
      uint8_t* stage = smem + C::OFF_Q;
      const int grow = T.row0 + row;
      // Packed sequences: a tile that runs past its sequence's last row is written row by
      // row (a TMA store would overwrite the next sequence's first rows).
      const bool direct = VL && T.row0 + 128 > T.qend;
      uint16_t* orow = static_cast<uint16_t*>(p.o_ptr) + ((size_t)T.bh * p.N + grow) * D;
      uint32_t r[32];
#pragma unroll 1
      for (int q = 0; q < C::OCOLS / 32; ++q) {
        tmem_ld32(tO + q * 32, r);
        tmem_wait_ld();
        reg_fence_w(r);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * inv, __uint_as_float(r[2 * i + 1]) * inv);
        const int col = half * C::OCOLS + q * 32;
        if (direct) {
          if (grow < T.qend) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
              *reinterpret_cast<uint4*>(orow + col + u * 8) =
                  make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          }
          continue;
        }
        const int box = col / 64, j0 = (col % 64) / 8;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t off = box * C::CHUNK + row * 128 + (((j0 + u) ^ (row & 7)) * 16);
          *reinterpret_cast<uint4*>(stage + off) = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
      if (half == 0 && grow < T.qend)
        p.lse[(size_t)T.bh * p.N + grow] = (m_fin[row] + __log2f(lrow)) * kLn2;
      if (!direct) {
        fence_proxy_async_smem();
        mbar_arrive(BAR(V_EPI));
        if (warp == 4 * C::FIRST_CORR_WG && lane == 0 && mbar_wait(BAR(V_EPI), 0, wc)) {
          for (int c = 0; c < C::NCH; ++c)
            tma_store_3d(&tm_o, sbase + C::OFF_Q + c * C::CHUNK, c * 64, T.row0, T.bh);
          tma_store_commit();
          tma_store_wait_all();
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

template <int D, int MODE>
cudaError_t launch_wide_t(const FwdMaps& m, const FwdParams& p, int grid, cudaStream_t s) {
  auto kern = attn_fwd_wide_kernel<D, MODE>;
  constexpr uint32_t smem = WideCfg<D>::SMEM;
  static std::once_flag flags[64];
  static cudaError_t attr_err[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::call_once(flags[dev & 63], [&] {
    attr_err[dev & 63] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
  kern<<<grid, kWideThreads, smem, s>>>(m.q, m.k, m.v, m.o, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_wide(const FwdMaps& maps, const FwdParams& p, int D, int grid, cudaStream_t s) {
  if (p.pack == 2) {   // packed sequences (d = 192, 256)
    if (D == 192) return launch_wide_t<192, 2>(maps, p, grid, s);
    if (D == 256) return launch_wide_t<256, 2>(maps, p, grid, s);
    return cudaErrorInvalidValue;
  }
  if (p.pack == 1) {   // grouped decode (d = 128)
    if (D == 128) return launch_wide_t<128, 1>(maps, p, grid, s);
    return cudaErrorInvalidValue;
  }
  if (D == 128) return launch_wide_t<128, 0>(maps, p, grid, s);
  if (D == 192) return launch_wide_t<192, 0>(maps, p, grid, s);
  if (D == 256) return launch_wide_t<256, 0>(maps, p, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace attn
