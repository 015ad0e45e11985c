// Fused exact attention forward for sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes: O = softmax(scale * Q K^T [causal]) V and LSE (natural log), with the
// N x N scores never leaving the SM ("Algorithm analysis" page, section 4: tiling so
// the N x N matrix is never formed).
//
// How (the FlashAttention-4 forward pipeline, "Hotelren FA4 summary" section 3.1 and
// "FlashAttention-4 explained" figure 3, re-laid out for this GPU):
//   * one CTA owns two 128-row query tiles ("high/low" tiles, section 3.1 item 1): two
//     row blocks of one head, or, for grouped heads, the same row block of two query
//     heads that share one K/V head, so every K/V tile loaded serves both (the MQA K/V
//     reuse of the reverse-engineering page);
//   * warp 0 is the TMA producer (Q tiles once, K and V tiles through rings of their own,
//     then an L2 prefetch of the first tiles of the CTA one wave later);
//   * warp 1 issues tcgen05.mma: S_t = Q_t K_j^T into TMEM, O_t += P_t V_j with P read
//     from TMEM (S and P share columns, "Hotelren FA4 summary" section 4.2 item 1);
//   * warpgroups 1 and 2 are the softmax of tile 0 and tile 1: while one does its
//     exponentials the tensor core works on the other tile (section 3.1 item 2);
//   * warpgroup 3 is the correction group: it rescales O in TMEM only when a row's
//     running maximum grew by more than tau (section 3.3, tau = 8 in log2 units), and
//     does the epilogue: O / l -> bf16 -> shared memory -> TMA store, plus the LSE;
//   * exponentials: each softmax thread can send a fixed subset of its elements through
//     the FMA-pipe cubic (exp2poly.cuh) and the rest through MUFU.EX2 (section 3.2,
//     mixed execution); the default (POLY = 0) sends all of them to MUFU.EX2, which
//     measured faster on this GPU.
//
// TMEM (512 columns, fp32): S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [256+D, 256+2D).
// P_t (bf16 pairs) overwrites the first 64 columns of S_t.
#include <cstdint>
#include <mutex>

#include "exp2poly.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kThreads = 512;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct FwdCfg {
  static constexpr int NCH = D / 64;                          // 64-column (128-byte) chunks
  static constexpr uint32_t CHUNK = 128 * 128;                // bytes of one 128 x 64 bf16 box
  static constexpr uint32_t TILE = CHUNK * NCH;               // one 128 x D bf16 tile
  // K and V tiles through rings of their own: K_j is last read by S_1(j), at the end of
  // block j, and first read by S_0(j) after PV_0(j - 1), so with one ring of four slots its
  // load could start only one block ahead and (≈ 2800 cycles from L2 under load, traced)
  // arrived late; three K slots start it two blocks ahead.  V_j is read one block after
  // its load can start with two slots.
  static constexpr int NK = (D == 128) ? 3 : 4;               // K ring slots
  static constexpr int NV = (D == 128) ? 2 : 4;               // V ring slots
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_KRING = 2 * TILE;
  static constexpr uint32_t OFF_VRING = OFF_KRING + NK * TILE;
  static constexpr uint32_t OFF_CTRL = OFF_VRING + NV * TILE;
  // control block: barriers, then alpha[2][128], then the TMEM address and abort flag
  static constexpr uint32_t CTRL_BYTES = 256 + 2 * 128 * 4 + 64;
  static constexpr uint32_t SMEM = 1024 + OFF_CTRL + CTRL_BYTES;
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 128, false, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, false, true);
};

// Barrier indices inside the control block (8 bytes each).
enum {
  B_Q = 0,
  B_SFULL = 1,    // +t
  B_PFULL = 3,    // +t
  B_STATS = 5,    // +t
  B_REL = 7,      // +(group & 1): K/V slots of release group j (K_j, V_(j-1)) are free
  B_OFULL = 9,    // +t: the tile's last PV product has completed (one phase)
  B_DONE = 11,
  B_KFULL = 12,   // +K slot (up to 4)
  B_VFULL = 16,   // +V slot (up to 4)
  B_EPI = 28,     // +t: the tile's O rows are staged in shared memory
  B_FIN = 30,     // +t: final row statistics (m, l, lq) in TMEM (one phase only)
  B_COUNT = 32
};

// A wait whose outcome is the same for all 32 lanes (the lanes then run .sync.aligned
// tcgen05 instructions together).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtl& w) {
  const bool ok = mbar_wait(bar, parity, w);
  return __all_sync(0xffffffffu, ok);
}

template <int N>
__device__ __forceinline__ void reg_fence(uint32_t (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i])::"memory");
}

// Which of a row's 128 elements go through the FMA polynomial: POLY of every 16, spread
// evenly (i = 16/POLY - 1, 2*16/POLY - 1, ...), so both pipes stay busy along the row.
template <int POLY>
__device__ __forceinline__ constexpr bool poly_lane(int i) {
  if constexpr (POLY <= 0) {
    return false;
  } else if constexpr (POLY >= 16) {
    return true;
  } else {
    constexpr int stride = 16 / POLY;
    return (i % stride) == stride - 1;
  }
}

struct Tiles {
  int n[2];       // key blocks per tile (0 = tile absent)
  int row0[2];    // first query row of each tile (packed sequences: row of the packed tensor)
  int bh[2];      // b * Hq + hq of each tile (grouped decode: the group's first head)
  int bkv;        // b * Hkv + hkv
  int j0;         // first key block (grouped decode: the start of this CTA's key split)
  // The sequence the tiles belong to: its first query row (qs), one past its last (qend),
  // its first key row (krow0), its number of keys (nk) and nk - nq (koff).  Constants of
  // the launch except for packed sequences.
  int qs, qend, krow0, nk, koff;
};

// Grouped decode mode: CTA = (K/V head, key split); its one tile holds the group's
// g query heads x N queries as rows h * N + q.
__device__ __forceinline__ Tiles map_unit_grouped(const FwdParams& p, int cta) {
  Tiles T;
  const int unit = cta / p.kv_splits, sp = cta % p.kv_splits;
  const int b = unit / p.Hkv, hkv = unit % p.Hkv;
  T.bkv = unit;
  T.bh[0] = T.bh[1] = b * p.Hq + hkv * p.g;
  T.row0[0] = T.row0[1] = 0;
  T.j0 = sp * p.blocks_per_split;
  T.n[0] = min(p.n_kvblk, T.j0 + p.blocks_per_split) - T.j0;
  T.n[1] = 0;
  T.qs = 0; T.qend = p.N; T.krow0 = 0; T.nk = p.Nk; T.koff = p.koff;
  return T;
}

// Packed sequences: the CTA's record of the unit table (varlen.cu) names the sequence,
// the two query heads and the two tiles' first rows within the sequence.
__device__ __forceinline__ Tiles map_unit_varlen(const FwdParams& p, const int4 u) {
  Tiles T;
  const int b = u.x;
  const int q0 = p.cu_q[b], nq = p.cu_q[b + 1] - q0;
  const int k0 = p.cu_k[b], nk = p.cu_k[b + 1] - k0;
  T.j0 = 0;
  T.qs = q0; T.qend = q0 + nq; T.krow0 = k0; T.nk = nk; T.koff = nk - nq;
  const int rows[2] = {u.z, u.w};
  const int hqs[2] = {u.y & 0xffff, u.y >> 16};
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    T.row0[t] = q0 + max(rows[t], 0);
    T.bh[t] = hqs[t];
    if (rows[t] < 0) T.n[t] = 0;
    else if (p.causal) T.n[t] = (min(rows[t] + 127, nq - 1) + T.koff) / 128 + 1;
    else T.n[t] = (nk + 127) / 128;
  }
  T.bkv = hqs[0] / p.g;
  return T;
}

__device__ __forceinline__ Tiles map_unit(const FwdParams& p, int unit) {
  Tiles T;
  T.j0 = 0;
  T.qs = 0; T.qend = p.N; T.krow0 = 0; T.nk = p.Nk; T.koff = p.koff;
  int hu, rs;
  if (p.causal) {  // longest rows first
    rs = p.n_rowslots - 1 - unit / p.units_per_row;
    hu = unit % p.units_per_row;
  } else {         // all row slots of a head back to back: K/V stay hot in L2
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
  const int rows[2] = {r0, r1};
  const int hqs[2] = {hq0, hq1};
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    T.row0[t] = rows[t];
    T.bh[t] = b * p.Hq + hqs[t];
    if (rows[t] >= p.N) {
      T.n[t] = 0;
    } else if (p.causal) {
      // the last key visible to the tile's last query
      const int last = min(rows[t] + 127, p.N - 1) + p.koff;
      T.n[t] = last / 128 + 1;
    } else {
      T.n[t] = p.n_kvblk;
    }
  }
  T.bkv = b * p.Hkv + hq0 / p.g;
  return T;
}

// MODE 0: the standard forward; MODE 1: grouped decode (partial results to the workspace);
// MODE 2: packed variable-length sequences (one unit-table record per CTA).
template <int D, int POLY, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint8_t* ctrl = smem + C::OFF_CTRL;
  const uint32_t bar0 = smem_u32(ctrl);
  auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * i; };
  float* alpha_buf = reinterpret_cast<float*>(ctrl + 256);        // [2][128]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(alpha_buf + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  const int wg = warp >> 2;
  // A kernel launched after this one as a programmatic dependent (the decode merge, the
  // backward's preprocess) may be scheduled now; it waits for this grid's completion before
  // reading what it writes.
  pdl_trigger();
  // CTAs past split_from each take one tile of a unit (the other half of the unit goes to
  // the next CTA); the lone tile always sits in slot 0.
  auto cta_tiles = [&](int cta) -> Tiles {
    if (cta < p.split_from) return map_unit(p, cta);
    const int k = cta - p.split_from;
    Tiles U = map_unit(p, p.split_from + k / 2);
    if (k & 1) {
      U.n[0] = U.n[1];
      U.row0[0] = U.row0[1];
      U.bh[0] = U.bh[1];
    }
    U.n[1] = 0;
    return U;
  };
  Tiles T;
  if constexpr (MODE == 2) {
    // CTAs past the table's records have no work: they leave before touching barriers or
    // tensor memory.
    if ((int)blockIdx.x >= __ldg(p.vl_count)) return;
    T = map_unit_varlen(p, p.vl_units[blockIdx.x]);
  } else if constexpr (MODE == 1) {
    T = map_unit_grouped(p, blockIdx.x);
  } else {
    T = cta_tiles(blockIdx.x);
  }
  const int nmax = max(T.n[0], T.n[1]);
  WaitCtl wc{p.wait_ns, p.status, abort_flag};

  if (threadIdx.x == 0) {
    mbar_init(BAR(B_Q), 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(BAR(B_SFULL + t), 1);
      mbar_init(BAR(B_PFULL + t), 256);   // softmax (P written) + correction (O rescaled)
      mbar_init(BAR(B_STATS + t), 128);
      mbar_init(BAR(B_REL + t), 1);
      mbar_init(BAR(B_OFULL + t), 1);
    }
    mbar_init(BAR(B_DONE), 1);
    mbar_init(BAR(B_EPI + 0), 128);
    mbar_init(BAR(B_EPI + 1), 128);
    mbar_init(BAR(B_FIN + 0), 128);
    mbar_init(BAR(B_FIN + 1), 128);
    for (int s = 0; s < C::NK; ++s) mbar_init(BAR(B_KFULL + s), 1);
    for (int s = 0; s < C::NV; ++s) mbar_init(BAR(B_VFULL + s), 1);
    *abort_flag = 0;
    fence_mbar_init();
    // Thread 0 is also the producer: its first loads (the Q tiles, K_0 and V_0, which need no
    // free slot) go out before the CTA-wide barrier, overlapping the TMEM allocation.
    const uint32_t qtile = MODE == 1 ? p.q_tile_bytes : C::TILE;
    mbar_arrive_expect_tx(BAR(B_Q), (T.n[0] > 0 ? qtile : 0) + (T.n[1] > 0 ? qtile : 0));
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (T.n[t] == 0) continue;
      for (int c = 0; c < C::NCH; ++c)
        tma_load_3d(sbase + C::OFF_Q + t * C::TILE + c * C::CHUNK, &tm_q, c * 64, T.row0[t], T.bh[t], BAR(B_Q));
    }
    if (nmax > 0 && !p.test_skip_first_kv) {
      for (int which = 0; which < 2; ++which) {
        const uint32_t bar = BAR(which ? B_VFULL : B_KFULL);
        mbar_arrive_expect_tx(bar, C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_3d(sbase + (which ? C::OFF_VRING : C::OFF_KRING) + c * C::CHUNK, which ? &tm_v : &tm_k, c * 64,
                      T.krow0 + T.j0 * 128, T.bkv, bar);
      }
    }
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Register split (per thread), against the launch's 128 x 512 threads: warpgroup 0
  // (producer, MMA), two softmax warpgroups, correction: d = 128 64 + 184 + 184 + 80, d = 64
  // 56 + 192 + 192 + 72, both 512 = 4 x 128 (measured on GB300: the d = 128 split is ~1 %
  // faster than the d = 64 one there, and ~2 % slower at d = 64).  Each role's code sits
  // inside its own branch so that the raised limit covers it.
  if (wg == 0) {
  if constexpr (D == 128) asm volatile("setmaxnreg.dec.sync.aligned.u32 64;");
  else asm volatile("setmaxnreg.dec.sync.aligned.u32 56;");
  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_o);
      // The Q tiles, K_0 and V_0 were issued before the CTA-wide barrier.  K_k goes to K slot
      // k mod NK once release k - NK (the end of block k - NK) has freed it; V_k to V slot
      // k mod NV once release k - NV + 1 has (V_(k-NV)'s last reader is the PV issued in block
      // k - NV + 1).  The loads go out in the order of the releases they wait for.  The test
      // hook skips K_0 and V_0 (the bounded-wait path).
      const bool skip0 = p.test_skip_first_kv;
      int nk = nmax > 0 ? 1 : 0, nv = nk;
      bool ok = true;
      while (ok && (nk < nmax || nv < nmax)) {
        const int gk = nk < nmax ? (nk >= C::NK ? nk - C::NK : -1) : 0x7fffffff;
        const int gv = nv < nmax ? (nv >= C::NV ? nv - C::NV + 1 : -1) : 0x7fffffff;
        const bool is_k = gk <= gv;
        const int g = is_k ? gk : gv;
        if (g >= 0 && !mbar_wait(BAR(B_REL + (g & 1)), (g >> 1) & 1, wc)) {
          ok = false;
          break;
        }
        const int k = is_k ? nk : nv;
        const uint32_t bar = is_k ? BAR(B_KFULL + k % C::NK) : BAR(B_VFULL + k % C::NV);
        const uint32_t dst = sbase + (is_k ? C::OFF_KRING + (k % C::NK) * C::TILE : C::OFF_VRING + (k % C::NV) * C::TILE);
        mbar_arrive_expect_tx(bar, C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_3d(dst + c * C::CHUNK, is_k ? &tm_k : &tm_v, c * 64, T.krow0 + (T.j0 + k) * 128, T.bkv, bar);
        if (is_k) ++nk;
        else ++nv;
      }
      // The CTA one wave later (blockIdx + the SM count) starts about when this one ends:
      // bring its Q tiles and first K, V tiles into L2 now, so that its first loads do not
      // wait on HBM.
      if constexpr (MODE == 0) {
        const int nxt = (int)blockIdx.x + p.prefetch_ahead;
        if (ok && p.prefetch_ahead > 0 && nxt < (int)gridDim.x) {
          const Tiles U = cta_tiles(nxt);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if ((t ? U.n[1] : U.n[0]) == 0) continue;
            for (int c = 0; c < C::NCH; ++c)
              tma_prefetch_l2_3d(&tm_q, c * 64, t ? U.row0[1] : U.row0[0], t ? U.bh[1] : U.bh[0]);
          }
          if (max(U.n[0], U.n[1]) > 0) {
            for (int c = 0; c < C::NCH; ++c) {
              tma_prefetch_l2_3d(&tm_k, c * 64, U.krow0 + U.j0 * 128, U.bkv);
              tma_prefetch_l2_3d(&tm_v, c * 64, U.krow0 + U.j0 * 128, U.bkv);
            }
          }
        }
      }
      if (!ok) {
        // Let the copies still in flight land before the CTA's shared memory goes away:
        // only the last NK K loads and NV V loads can be outstanding.
        const unsigned long long t0 = globaltimer_ns();
        for (int k = max(0, nk - C::NK); k < nk; ++k) {
          if (skip0 && k == 0) continue;
          while (!mbar_try_wait(BAR(B_KFULL + k % C::NK), (k / C::NK) & 1) && globaltimer_ns() - t0 < p.wait_ns) {
          }
        }
        for (int k = max(0, nv - C::NV); k < nv; ++k) {
          if (skip0 && k == 0) continue;
          while (!mbar_try_wait(BAR(B_VFULL + k % C::NV), (k / C::NV) & 1) && globaltimer_ns() - t0 < p.wait_ns) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(BAR(B_Q), 0, wc);
      tc_fence_after();
      for (int j = 0; j <= nmax && ok; ++j) {
        const int kslot = j % C::NK, vslot = (j + C::NV - 1) % C::NV;   // K_j, V_(j-1)
        if (j < nmax && !mbar_wait(BAR(B_KFULL + kslot), (j / C::NK) & 1, wc)) { ok = false; break; }
        if (j >= 1 && !mbar_wait(BAR(B_VFULL + vslot), ((j - 1) / C::NV) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        // Descriptor low words built once per block and advanced by (offset / 16); the high
        // words are constants.
        const uint32_t klo = sdesc_sw128_lo(sbase + C::OFF_KRING + kslot * C::TILE, 16);
        const uint32_t vlo = sdesc_sw128_lo(sbase + C::OFF_VRING + vslot * C::TILE, C::CHUNK);
        constexpr uint32_t HI = sdesc_sw128_hi(1024);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!ok) break;
          const uint32_t tS = tmem + uint32_t(t * 128), tO = tmem + 256u + uint32_t(t * D);
          if (j >= 1 && j <= T.n[t]) {
            // O_t += P_t(j-1) V_(j-1): the P barrier also carries the correction group's
            // arrival (O rescaled, or no rescale needed).
            if (!mbar_wait(BAR(B_PFULL + t), (j - 1) & 1, wc)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts_w(tO, tS + kk * 8, vlo + kk * (2048 >> 4), HI, C::IDESC_PV, (j > 1 || kk > 0) ? 1u : 0u);
            // Only the tile's last PV is signalled here (for the epilogue).  The correction
            // group learns that PV_t(j-1) finished from S_t(j)'s completion instead: MMAs
            // complete in issue order.
            if (j == T.n[t]) mma_commit(BAR(B_OFULL + t));
          }
          if (j < T.n[t]) {
            // S_t = Q_t K_j^T
            const uint32_t qlo = sdesc_sw128_lo(sbase + C::OFF_Q + t * C::TILE, 16);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
              mma_ss_w(tS, qlo + off, HI, klo + off, HI, C::IDESC_QK, kk > 0 ? 1u : 0u);
            }
            mma_commit(BAR(B_SFULL + t));
          }
        }
        if (!ok) break;
        mma_commit(BAR(B_REL + (j & 1)));   // release j: K_j's and V_(j-1)'s slots
      }
      // Drain: every MMA issued above completes before TMEM is released.
      mma_commit(BAR(B_DONE));
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(BAR(B_DONE), 0) && globaltimer_ns() - t0 < p.wait_ns) {
      }
    }
  }
  } else if (wg == 1 || wg == 2) {
    if constexpr (D == 128) asm volatile("setmaxnreg.inc.sync.aligned.u32 184;");
    else asm volatile("setmaxnreg.inc.sync.aligned.u32 192;");
    // ------------------------------------------------------------------ softmax
    const int t = wg - 1;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t tS = tmem + (uint32_t((warp & 3) * 32) << 16) + uint32_t(t * 128);
    const int row0_t = t ? T.row0[1] : T.row0[0];
    const int grow = row0_t + row;
    const float c = p.c;
    float m = -INFINITY, l = 0.f, lq = 0.f;
    const int n_t = t ? T.n[1] : T.n[0];
    for (int j = 0; j < n_t; ++j) {
      if (!warp_wait(BAR(B_SFULL + t), j & 1, wc)) break;
      tc_fence_after();
      // The whole 128-column row in one batch of TMEM loads and a single wait.
      uint32_t u[128];
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, *reinterpret_cast<uint32_t(*)[32]>(&u[q * 32]));
      tmem_wait_ld();
      reg_fence(u);
      float* s = reinterpret_cast<float*>(u);
      const int kb = (T.j0 + j) * 128;
      // Grouped decode: row = h * N + q holds query q (rows past g * N are padding).  Packed
      // sequences: rows and keys count from the sequence's start; the keys past its end
      // (the next sequence's) are masked like those past the tensor's end.
      const int qrow = MODE == 1 ? row % p.N : grow - T.qs;
      const bool need_mask =
          MODE == 1 || (kb + 127 >= T.nk) || (p.causal && kb + 127 > row0_t - T.qs + T.koff);
      if (need_mask) {
        const int lim = (p.causal ? min(qrow + T.koff, T.nk - 1) : T.nk - 1) - kb;  // last visible column
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i > lim) s[i] = -INFINITY;
      }
      // Row maximum over exactly the 128 columns: 4 seeds, 15 steps of 8, a last step of 4.
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
      mbar_arrive(BAR(B_STATS + t));
      // p = 2^(s*c - m).  l sums the fp32 p (it gives LSE).  O is divided by lq = l minus
      // the bf16 rounding error of each block's largest p: when a row's weight sits on one
      // key and the maximum is stale (that p is not exactly 1), the PV product uses
      // bf16(p), and dividing by the matching sum makes O exact up to the output rounding.
      // Grouped decode: a row may see no key of this CTA's key range yet (m = -inf); its
      // probabilities are then 0, not 2^(-inf + inf).
      const float neg_m = (MODE == 1 && m == -INFINITY) ? 0.f : -m;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[64];
#pragma unroll
      for (int i = 0; i < 128; i += 2) {
        float x0, x1;
        ffma2_bc(x0, x1, s[i], s[i + 1], c, neg_m);
        const float e0 = poly_lane<POLY>(i) ? exp2_poly(x0) : ex2_mufu(x0);
        const float e1 = poly_lane<POLY>(i + 1) ? exp2_poly(x1) : ex2_mufu(x1);
        pk[i >> 1] = pack_bf16x2(e0, e1);
        const int a2 = ((i >> 1) & 1) * 2;
        fadd2(acc[a2], acc[a2 + 1], acc[a2], acc[a2 + 1], e0, e1);
      }
      {
        const float pmax = ex2_mufu(fmaf(rmax, c, neg_m));   // bit-identical to that element's p above
        const float pmax_q = __uint_as_float(pack_bf16x2(pmax, 0.f) << 16);
        const float blk = (acc[0] + acc[1]) + (acc[2] + acc[3]);
        l = l * alpha + blk;
        lq = lq * alpha + (blk - (pmax - pmax_q));
      }
      tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(BAR(B_PFULL + t));
    }
    // The row's final statistics go to TMEM columns 64-67 of this tile's S, dead once the
    // last P (columns 0-63) is written, for the correction group's epilogue.  A barrier of
    // its own: arriving on B_STATS again here could complete that barrier's last two phases
    // before the correction group waits on the first.
    {
      const uint32_t st[4] = {__float_as_uint(m), __float_as_uint(l), __float_as_uint(lq), 0u};
      tmem_st4(tS + 64, st);
      tmem_wait_st();
    }
    tc_fence_before();
    mbar_arrive(BAR(B_FIN + t));
  } else {
    if constexpr (D == 128) asm volatile("setmaxnreg.dec.sync.aligned.u32 80;");
    else asm volatile("setmaxnreg.dec.sync.aligned.u32 72;");
    // ------------------------------------------------------------------ correction + epilogue
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    bool ok = true;
    for (int j = 0; j < nmax && ok; ++j) {
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (!ok || j >= T.n[t]) continue;
        if (!warp_wait(BAR(B_STATS + t), j & 1, wc)) { ok = false; break; }
        const float alpha = alpha_buf[t * 128 + row];
        const bool any = __any_sync(0xffffffffu, alpha != 1.f);
        if (p.rescale_count != nullptr && j > 0) {
          const unsigned bal = __ballot_sync(0xffffffffu, alpha != 1.f);
          if (lane == 0 && bal) atomicAdd(p.rescale_count, (unsigned long long)__popc(bal));
        }
        if (j > 0 && any) {
          // S_t(j) complete => PV_t(j-1), issued before it, is complete too.
          if (!warp_wait(BAR(B_SFULL + t), j & 1, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t tO = tmem + lane_off + 256u + uint32_t(t * D);
          uint32_t r[32];
#pragma unroll 1
          for (int q = 0; q < D / 32; ++q) {
            tmem_ld32(tO + q * 32, r);
            tmem_wait_ld();
            reg_fence(r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(tO + q * 32, r);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(BAR(B_PFULL + t));
      }
    }
    // Epilogue per tile: O / l -> bf16 -> swizzled shared memory (the tile's Q buffer,
    // free once its last MMA completed) -> TMA store; LSE straight to global memory.
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int n_t = T.n[t];
      if (!ok || n_t == 0) continue;
      if (!warp_wait(BAR(B_FIN + t), 0, wc)) { ok = false; break; }
      if (!warp_wait(BAR(B_OFULL + t), 0, wc)) { ok = false; break; }
      tc_fence_after();
      uint32_t fin[4];
      tmem_ld4(tmem + lane_off + uint32_t(t * 128) + 64u, fin);
      tmem_wait_ld();
      reg_fence(fin);
      const float mrow = __uint_as_float(fin[0]), lrow = __uint_as_float(fin[1]), lq_row = __uint_as_float(fin[2]);
      const float inv = 1.f / lq_row;
      const uint32_t tO = tmem + lane_off + 256u + uint32_t(t * D);
      if constexpr (MODE == 1) {
        // This key split's partial result: O / lq (0 where the row saw no key) and LSE, fp32,
        // for rows h * N + q of the group; rows past g * N are padding and not written.
        const int unit = blockIdx.x / p.kv_splits, sp = blockIdx.x % p.kv_splits;
        const size_t slot = (size_t)sp * (p.B * p.Hkv) + unit;
        const bool real = row < p.g * p.N;
        const float lqr = lq_row;
        const float invp = lqr > 0.f ? 1.f / lqr : 0.f;
        float* dst = p.part_o + (slot * 128 + row) * D;
        uint32_t r[32];
#pragma unroll 1
        for (int q = 0; q < D / 32; ++q) {
          tmem_ld32(tO + q * 32, r);   // warp-collective: every lane loads its row
          tmem_wait_ld();
          reg_fence(r);
          if (real) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(dst + q * 32 + i) =
                  make_float4(__uint_as_float(r[i]) * invp, __uint_as_float(r[i + 1]) * invp,
                              __uint_as_float(r[i + 2]) * invp, __uint_as_float(r[i + 3]) * invp);
          }
        }
        if (real) p.part_lse[slot * 128 + row] = lrow > 0.f ? (mrow + __log2f(lrow)) * kLn2 : -INFINITY;
        continue;
      }
      uint8_t* stage = smem + C::OFF_Q + t * C::TILE;
      const int grow = T.row0[t] + row;
      // Packed sequences: a tile that ends inside the packed tensor but past its sequence's
      // last row is written row by row (a TMA store would overwrite the next sequence).
      const bool direct = MODE == 2 && T.row0[t] + 128 > T.qend;
      uint16_t* orow = static_cast<uint16_t*>(p.o_ptr) + ((size_t)T.bh[t] * p.N + grow) * D;
      uint32_t r[32];
#pragma unroll 1
      for (int q = 0; q < D / 32; ++q) {
        tmem_ld32(tO + q * 32, r);
        tmem_wait_ld();
        reg_fence(r);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * inv, __uint_as_float(r[2 * i + 1]) * inv);
        if (direct) {
          if (grow < T.qend) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
              *reinterpret_cast<uint4*>(orow + q * 32 + u * 8) =
                  make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          }
          continue;
        }
        const int box = (q * 32) / 64, j0 = ((q * 32) % 64) / 8;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t off = box * C::CHUNK + row * 128 + (((j0 + u) ^ (row & 7)) * 16);
          *reinterpret_cast<uint4*>(stage + off) = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
      if (grow < T.qend) p.lse[(size_t)T.bh[t] * p.N + grow] = (mrow + __log2f(lrow)) * kLn2;
      if (direct) continue;
      fence_proxy_async_smem();
      mbar_arrive(BAR(B_EPI + t));
      if (warp == 12 && lane == 0 && mbar_wait(BAR(B_EPI + t), 0, wc)) {
        for (int c = 0; c < C::NCH; ++c)
          tma_store_3d(&tm_o, sbase + C::OFF_Q + t * C::TILE + c * C::CHUNK, c * 64, T.row0[t], T.bh[t]);
        tma_store_commit();
      }
    }
    if (warp == 12 && lane == 0) tma_store_wait_read();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int POLY, int MODE = 0>
cudaError_t launch_t(const FwdMaps& m, const FwdParams& p, int grid, cudaStream_t s) {
  auto kern = attn_fwd_kernel<D, POLY, MODE>;
  constexpr uint32_t smem = FwdCfg<D>::SMEM;
  static std::once_flag flags[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static cudaError_t attr_err[64];
  std::call_once(flags[dev & 63], [&] {
    attr_err[dev & 63] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
  kern<<<grid, kThreads, smem, s>>>(m.q, m.k, m.v, m.o, p);
  return cudaGetLastError();
}

}  // namespace

size_t fwd_smem_bytes(int D) { return D == 64 ? FwdCfg<64>::SMEM : FwdCfg<128>::SMEM; }

cudaError_t launch_fwd(const FwdMaps& maps, const FwdParams& p, int D, int poly, int grid, cudaStream_t s) {
  if (p.pack == 2) {   // packed sequences: the MUFU exponential only
    if (D == 64) return launch_t<64, 0, 2>(maps, p, grid, s);
    if (D == 128) return launch_t<128, 0, 2>(maps, p, grid, s);
    return cudaErrorInvalidValue;
  }
  if (p.pack) {   // grouped decode: the MUFU exponential only
    if (D == 64) return launch_t<64, 0, 1>(maps, p, grid, s);
    if (D == 128) return launch_t<128, 0, 1>(maps, p, grid, s);
    return cudaErrorInvalidValue;
  }
  if (D == 64) {
    if (poly == 0) return launch_t<64, 0>(maps, p, grid, s);
    if (poly == 4) return launch_t<64, 4>(maps, p, grid, s);
    if (poly == 16) return launch_t<64, 16>(maps, p, grid, s);
  } else if (D == 128) {
    if (poly == 0) return launch_t<128, 0>(maps, p, grid, s);
    if (poly == 4) return launch_t<128, 4>(maps, p, grid, s);
    if (poly == 16) return launch_t<128, 16>(maps, p, grid, s);
  }
  return cudaErrorInvalidValue;
}

// ------------------------------------------------------------------------------------
// Grouped decode: merge the key splits.  One warp per (K/V head, row h * N + q); lane i
// holds columns [D/32 i, D/32 (i + 1)).  LSE = ln sum_s e^LSE_s, O = sum_s e^(LSE_s - LSE) O_s.
// ------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) fwd_merge_kernel(const FwdParams p, uint16_t* __restrict__ o) {
  constexpr int PER = D / 32;
  // Launched as a programmatic dependent of the split kernel: wait until that grid has
  // completed and its partial results are visible.
  pdl_wait();
  const int gN = p.g * p.N, units = p.B * p.Hkv;
  const long long wid = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (wid >= (long long)units * gN) return;
  const int lane = threadIdx.x & 31;
  const int unit = (int)(wid / gN), r = (int)(wid % gN);
  float mx = -INFINITY;
  for (int sp = 0; sp < p.kv_splits; ++sp)
    mx = fmaxf(mx, p.part_lse[((size_t)sp * units + unit) * 128 + r]);
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  float wsum = 0.f;
  for (int sp = 0; sp < p.kv_splits; ++sp) {
    const size_t slot = (size_t)sp * units + unit;
    const float ls = p.part_lse[slot * 128 + r];
    if (ls == -INFINITY) continue;          // this split held no key visible to the row
    const float w = __expf(ls - mx);
    wsum += w;
    const float* src = p.part_o + (slot * 128 + r) * D + lane * PER;
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] += w * src[i];
  }
  const float inv = 1.f / wsum;
  const int b = unit / p.Hkv, hkv = unit % p.Hkv;
  const int h = hkv * p.g + r / p.N, q = r % p.N;
  const size_t orow = ((size_t)(b * p.Hq + h)) * p.N + q;
  uint32_t pk[PER / 2];
#pragma unroll
  for (int i = 0; i < PER / 2; ++i) pk[i] = pack_bf16x2(acc[2 * i] * inv, acc[2 * i + 1] * inv);
  if constexpr (PER == 4) {
    *reinterpret_cast<uint2*>(o + orow * D + lane * PER) = make_uint2(pk[0], pk[1]);
  } else {
    *reinterpret_cast<uint32_t*>(o + orow * D + lane * PER) = pk[0];
  }
  if (lane == 0) p.lse[orow] = mx + __logf(wsum);
}

cudaError_t launch_fwd_merge(const FwdParams& p, int D, void* o, cudaStream_t s) {
  const long long warps = (long long)p.B * p.Hkv * p.g * p.N;
  const unsigned blocks = (unsigned)((warps + 7) / 8);
  if (blocks == 0) return cudaSuccess;
  // Programmatic dependent launch: the merge's blocks are scheduled while the split kernel
  // still runs (on SMs it leaves free) and wait in pdl_wait for its completion, instead of
  // being launched after it.
  uint16_t* op = static_cast<uint16_t*>(o);
  if (D == 64) return launch_pdl(fwd_merge_kernel<64>, dim3(blocks), dim3(256), 0, s, p, op);
  if (D == 128) return launch_pdl(fwd_merge_kernel<128>, dim3(blocks), dim3(256), 0, s, p, op);
  return cudaErrorInvalidValue;
}

// ------------------------------------------------------------------------------------
// Software exp2 test kernel (grid-stride, plain loads/stores).
// ------------------------------------------------------------------------------------
__global__ void exp2_test_kernel(const float* __restrict__ x, float* __restrict__ y, long long n, int variant) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const float v = x[i];
    y[i] = variant == 0 ? exp2_poly(v) : (variant == 1 ? exp2_poly_full_range(v) : ex2_mufu(v));
  }
}

cudaError_t launch_exp2_test(const float* x, float* y, long long n, int variant, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long blocks = (n + 255) / 256;
  const int grid = (int)(blocks < (long long)sms * 8 ? blocks : (long long)sms * 8);
  exp2_test_kernel<<<grid, 256, 0, s>>>(x, y, n, variant);
  return cudaGetLastError();
}

}  // namespace attn
