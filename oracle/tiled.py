"""Step-by-step fp32 emulation of the tiled online softmax with the conditional rescale.

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle``).

It follows the algorithm in the order the FlashAttention-4 pages give it:

* "Algorithm analysis" page, section 4 (online-softmax pseudocode): loop over key tiles
  j, keep a running row maximum m and row sum l, rescale the running output by
  alpha = exp(m_old - m_new) when the maximum changes.  The pseudocode on that page
  forgets the final division by l; the standard reading divides once at the end.
* "Hotelren FA4 summary" page, section 3.3 (conditional softmax rescale): work in log2
  units; rescale only when the new maximum exceeds the running one by more than
  tau = log2(256) = 8.  Otherwise keep the stale maximum and accumulate exp2(x - m_stale)
  into both O and l, so that the single final division O / l stays exact (the
  "FlashAttention-4 explained" page, section 04, trick two, says the same in words).
  The printed function on that page returns ``new_max`` in the no-rescale branch and
  never forms ``new_sum``; here the stale maximum is kept and l is updated, which is the
  only reading under which the result is exact.

Everything is fp32 (numpy), with scores scaled into log2 units by c = scale * log2(e).
Returns O, LSE (natural log) and the rescale statistics.
"""
from __future__ import annotations

import numpy as np

LOG2E = 1.4426950408889634
LN2 = 0.6931471805599453


def _f32(t) -> np.ndarray:
    import torch
    if isinstance(t, np.ndarray):
        return t.astype(np.float32)
    return t.detach().cpu().to(torch.float32).numpy()


def tiled_head(q, k, v, causal: bool, scale: float, tau: float, block: int = 128):
    """One head: q [N,d], k [N,d], v [N,d] (values exactly representable in bf16).

    ``tau`` is the rescale threshold in log2 units (0 = rescale whenever the maximum
    grows).  Returns (O [N,d] fp32, LSE [N] fp32, n_rescale, n_max_grew, n_init) where
    n_rescale counts (row, key-tile) steps that rescaled after the first tile,
    n_max_grew counts steps in which the row maximum grew at all, and n_init the
    first-tile initialisations."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    N, d = q.shape
    c = np.float32(scale * LOG2E)
    O = np.zeros((N, d), np.float32)
    LSE = np.zeros((N,), np.float32)
    n_rescale = n_grew = n_init = 0
    for i0 in range(0, N, block):
        rows = np.arange(i0, min(i0 + block, N))
        qi = q[rows]
        m = np.full(len(rows), -np.inf, np.float32)
        l = np.zeros(len(rows), np.float32)
        acc = np.zeros((len(rows), d), np.float32)
        last_key = rows[-1] if causal else N - 1
        for j0 in range(0, last_key + 1, block):
            cols = np.arange(j0, min(j0 + block, N))
            s = (qi @ k[cols].T).astype(np.float32)            # S = Q_i K_j^T
            x = s * c                                          # log2 units
            if causal:
                x = np.where(cols[None, :] > rows[:, None], np.float32(-np.inf), x)
            m_tile = x.max(axis=1)
            m_cand = np.maximum(m, m_tile)
            first = np.isneginf(m)
            need = first | (m_cand - m > np.float32(tau))
            grew = (~first) & (m_cand > m)
            n_init += int(first.sum())
            n_rescale += int((need & ~first).sum())
            n_grew += int(grew.sum())
            m_new = np.where(need, m_cand, m)
            alpha = np.where(first, np.float32(0.0), np.exp2(m - m_new)).astype(np.float32)
            p = np.exp2(x - m_new[:, None]).astype(np.float32)
            l = alpha * l + p.sum(axis=1, dtype=np.float32)
            acc = alpha[:, None] * acc + (p @ v[cols]).astype(np.float32)
            m = m_new
        O[rows] = acc / l[:, None]
        LSE[rows] = (m + np.log2(l)) * np.float32(LN2)
    return O, LSE, n_rescale, n_grew, n_init


def tiled_attn(q, k, v, causal: bool, scale: float, tau: float, heads, block: int = 128):
    """Several heads of [B,H,N,d] inputs; ``heads`` lists (b, hq).  K/V head = hq // g."""
    Hq, Hkv = q.shape[1], k.shape[1]
    g = Hq // Hkv
    outs, lses, stats = [], [], np.zeros(3, np.int64)
    for b, h in heads:
        o, lse, r, gr, ini = tiled_head(q[b, h], k[b, h // g], v[b, h // g], causal, scale, tau, block)
        outs.append(o)
        lses.append(lse)
        stats += (r, gr, ini)
    return np.stack(outs), np.stack(lses), {"rescales": int(stats[0]), "max_grew": int(stats[1]),
                                            "inits": int(stats[2])}
