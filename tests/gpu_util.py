"""Helpers for the GPU parity tests: move a workload onto the device, fill the
paged cache through the library's own append, run decode / verify through the
C ABI, and the error measures the parity bar is written in."""
from __future__ import annotations

import numpy as np

import mla_latent_kv_08_gb300 as mla

# Parity bar for bf16 caches: max |gpu - oracle| / max |oracle| over each
# sequence's output rows, and absolute LSE error (natural log).
BF16_REL_TOL = 1e-2
BF16_LSE_TOL = 2e-3
# fp32 cache (tiny workload): fp32 arithmetic end to end.
FP32_REL_TOL = 1e-5
FP32_LSE_TOL = 1e-5


def torch_dtype(w):
    import torch
    return torch.float32 if w.dtype == "fp32" else torch.bfloat16


def shape_for(w, kind=None, impl=mla.MLA_IMPL_AUTO, splits=0, num_blocks=None) -> mla.Shape:
    if kind is None:
        kind = mla.MLA_KV_FP32 if w.dtype == "fp32" else mla.MLA_KV_BF16
    return mla.Shape(num_heads=w.H, kv_lora_rank=w.r, rope_dim=w.d_rope, v_head_dim=w.d_v,
                     block_size=w.block_size, num_blocks=num_blocks or w.num_blocks, kind=kind,
                     group_size=32, impl=impl, num_splits_hint=splits)


def dev(x, dtype=None, device="cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(device)


def append_tokens(cache, w, rows_c, rows_r, start_pos, R=None, T=None, device="cuda"):
    """Append per-sequence rows (lists of [n_b, r] / [n_b, d_R]) at start_pos[b]."""
    import torch
    dt = torch.float32 if cache.shape.kind == mla.MLA_KV_FP32 else torch.bfloat16
    counts = np.array([x.shape[0] for x in rows_c], dtype=np.int64)
    cu = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    c = dev(np.concatenate(rows_c).astype(np.float32), dt, device)
    kr = dev(np.concatenate(rows_r).astype(np.float32), dt, device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    mla.mla_latent_append(cache, dev(w.block_table, device=device), dev(np.asarray(start_pos, np.int32), device=device),
                          dev(cu, device=device), c, kr,
                          R=None if R is None else dev(R.astype(np.float32), device=device),
                          clip=None if T is None else dev(T.astype(np.float32), device=device),
                          status=status)
    return status


def fill_cache(w, shape, R=None, T=None, device="cuda"):
    cache = mla.Cache.allocate(shape, device)
    status = append_tokens(cache, w, w.latent, w.rope, np.zeros(w.B, np.int32), R, T, device)
    return cache, status


def attend(w, shape, cache, q, R=None, device="cuda", q_len=1):
    import torch
    dt = torch_dtype(w)
    qd = dev(q.astype(np.float32), dt, device)
    W = dev(w.W_UV.astype(np.float32), dt, device)
    out = torch.empty((w.B, q_len, w.H, w.d_v), dtype=dt, device=device)
    lse = torch.empty((w.B, q_len, w.H), dtype=torch.float32, device=device)
    ws = mla.alloc_workspace(shape, w.B, q_len, device)
    bt = dev(w.block_table, device=device)
    sl = dev(w.seq_lens.astype(np.int32), device=device)
    Rd = None if R is None else dev(R.astype(np.float32), device=device)
    if q_len == 1:
        mla.mla_decode(cache, bt, sl, qd, W, w.scale, out, lse, ws, R=Rd)
    else:
        mla.mla_verify(cache, bt, sl, qd, W, w.scale, out, lse, ws, R=Rd)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), ws


def rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))
