"""MLA attention over a latent cache, fp64 (oracle, test infrastructure only).

Notation (per head h, per cached token t):
  c_t in R^r       the shared latent (kv_lora_rank = r)
  kR_t in R^{d_R}  the shared rope key
  W_UK^h [d_n, r], W_UV^h [r, d_v]   the up-projections of kv_b_proj
  q~_h = [ (W_UK^h)^T qC_h ; qR_h ]  the absorbed query, length r + d_R

  s_{h,t}  = scale * (q~_h . [c_t ; kR_t])
  p_{h,.}  = softmax over visible t of s_{h,.}
  olat_h   = sum_t p_{h,t} c_t
  o_h      = (W_UV^h)^T olat_h
  lse_h    = ln sum_t exp(s_{h,t})          (natural log, of the scaled scores)

Source: "GLM-5.2 speculative drafting ... + opt-in MLA-latent KV cache", TL;DR
item 2 (absorb: cache the kv-latent + shared rope key, attention in latent
space) and "MLA model support (GLM-5.1 / DeepSeek-style)", maintainer reply
("per-head structure only re-emerges after the kv_b_proj up-projection").

Causal window (reading adopted for speculative verify, where the pages give only
acceptance rates): the q_len query rows of a sequence are its last q_len
positions, already in the cache, so query row i sees positions
0 .. L - q_len + i inclusive. With q_len = 1 that is the whole cache.

Every function here uses library matmul/einsum as its only building block and
follows the definition's order: scores, max-subtracted exponentials, sum, LSE,
normalised weights, latent output, up-projection.
"""
from __future__ import annotations

import numpy as np


def absorb_query(q_nope: np.ndarray, q_rope: np.ndarray, W_UK: np.ndarray) -> np.ndarray:
    """q~ = [ (W_UK^h)^T qC_h ; qR_h ] for every leading index.

    q_nope [..., H, d_n], q_rope [..., H, d_R], W_UK [H, d_n, r] -> [..., H, r + d_R].
    """
    q_lat = np.einsum("...hn,hnr->...hr", q_nope.astype(np.float64), W_UK.astype(np.float64))
    return np.concatenate([q_lat, q_rope.astype(np.float64)], axis=-1)


def causal_visible(q_len: int, L: int) -> np.ndarray:
    """[q_len, L] bool: query row i sees positions 0 .. L - q_len + i."""
    pos = np.arange(L)[None, :]
    last = (L - q_len + np.arange(q_len))[:, None]
    return pos <= last


def _softmax_stats(S: np.ndarray, visible: np.ndarray):
    """Max-subtracted softmax over the last axis restricted to ``visible``.

    Returns (P normalised, lse natural log). Rows with nothing visible give
    P = 0 and lse = -inf.
    """
    Sm = np.where(visible, S, -np.inf)
    m = Sm.max(axis=-1, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    E = np.where(visible, np.exp(Sm - m_safe), 0.0)
    l = E.sum(axis=-1, keepdims=True)
    with np.errstate(divide="ignore"):
        lse = (np.log(l) + m_safe)[..., 0]
    P = np.divide(E, l, out=np.zeros_like(E), where=l > 0)
    return P, lse


def absorbed(q: np.ndarray, C: np.ndarray, KR: np.ndarray, W_UV: np.ndarray, scale: float,
             return_latent: bool = False):
    """Absorbed attention for one sequence.

    q [q_len, H, r + d_R], C [L, r], KR [L, d_R], W_UV [H, r, d_v].
    Returns out [q_len, H, d_v], lse [q_len, H] (and olat [q_len, H, r]).
    """
    q = q.astype(np.float64)
    C = C.astype(np.float64)
    KR = KR.astype(np.float64)
    q_len, H, D = q.shape
    L, r = C.shape
    K = np.concatenate([C, KR], axis=1)                      # [L, r + d_R]
    S = scale * (q.reshape(q_len * H, D) @ K.T).reshape(q_len, H, L)
    vis = causal_visible(q_len, L)[:, None, :]
    P, lse = _softmax_stats(S, vis)
    olat = (P.reshape(q_len * H, L) @ C).reshape(q_len, H, r)   # latent-space output
    # per head: o_h = olat_h . W_UV^h
    out = np.matmul(olat.transpose(1, 0, 2), W_UV.astype(np.float64)).transpose(1, 0, 2)
    if return_latent:
        return out, lse, olat
    return out, lse


def full_head(q_nope: np.ndarray, q_rope: np.ndarray, C: np.ndarray, KR: np.ndarray,
              W_UK: np.ndarray, W_UV: np.ndarray, scale: float):
    """Non-absorbed attention: decompress per-head K/V, then standard attention.

    k^C_{h,t} = W_UK^h c_t,  v_{h,t} = (W_UV^h)^T c_t,
    s = scale (qC_h . k^C_{h,t} + qR_h . kR_t),  o_h = sum_t p v.
    q_nope [q_len, H, d_n], q_rope [q_len, H, d_R] -> out [q_len, H, d_v], lse [q_len, H].
    """
    C = C.astype(np.float64)
    KR = KR.astype(np.float64)
    KC = np.einsum("hnr,lr->hln", W_UK.astype(np.float64), C)     # [H, L, d_n]
    V = np.einsum("hrv,lr->hlv", W_UV.astype(np.float64), C)      # [H, L, d_v]
    q_len = q_nope.shape[0]
    L = C.shape[0]
    S = scale * (np.einsum("qhn,hln->qhl", q_nope.astype(np.float64), KC)
                 + np.einsum("qhd,ld->qhl", q_rope.astype(np.float64), KR))
    vis = causal_visible(q_len, L)[:, None, :]
    P, lse = _softmax_stats(S, vis)
    out = np.einsum("qhl,hlv->qhv", P, V)
    return out, lse


def softmax_weights(q: np.ndarray, C: np.ndarray, KR: np.ndarray, scale: float) -> np.ndarray:
    """The normalised weights p [q_len, H, L] of ``absorbed`` (for row-sum checks)."""
    q = q.astype(np.float64)
    K = np.concatenate([C.astype(np.float64), KR.astype(np.float64)], axis=1)
    S = scale * np.einsum("qhd,ld->qhl", q, K)
    vis = causal_visible(q.shape[0], C.shape[0])[:, None, :]
    P, _ = _softmax_stats(S, vis)
    return P


def decode_batch(q: np.ndarray, latents, ropes, W_UV: np.ndarray, scale: float, seqs=None):
    """Absorbed attention for each sequence b in ``seqs`` (all by default).

    q [B, q_len, H, r + d_R]; latents[b] [L_b, r]; ropes[b] [L_b, d_R].
    Returns dict b -> (out [q_len, H, d_v], lse [q_len, H]).
    """
    seqs = range(q.shape[0]) if seqs is None else seqs
    return {b: absorbed(q[b], latents[b], ropes[b], W_UV, scale) for b in seqs}


def row_subset(q: np.ndarray, C: np.ndarray, KR: np.ndarray, W_UV: np.ndarray, scale: float,
               rows):
    """Absorbed attention evaluated for selected (query row, head) pairs only.

    Used for spot checks at sizes where computing every row is slow. Each pair is
    computed on its own from the definition. Returns out [n, d_v], lse [n].
    """
    q_len = q.shape[0]
    L = C.shape[0]
    K = np.concatenate([C.astype(np.float64), KR.astype(np.float64)], axis=1)
    outs, lses = [], []
    for (i, h) in rows:
        last = L - q_len + i
        s = scale * (K[: last + 1] @ q[i, h].astype(np.float64))
        m = s.max()
        e = np.exp(s - m)
        l = e.sum()
        p = e / l
        olat = p @ C[: last + 1].astype(np.float64)
        outs.append(olat @ W_UV[h].astype(np.float64))
        lses.append(np.log(l) + m)
    return np.array(outs), np.array(lses)
