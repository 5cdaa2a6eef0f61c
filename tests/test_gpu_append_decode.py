"""mla_append_decode: appending a step's new tokens and decoding in one call gives the
results of mla_latent_append followed by mla_decode, bit for bit, on every cache kind
(the bf16 / fp32 copy of up to 4096 tokens runs inside the planner's launch; more
tokens, and the INT2 append, as a kernel of their own), and reports the append's flags
through its own status word."""
import numpy as np
import pytest

import workloads
from oracle import attention
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _int2_setup(B, H, len_range, seed=4):
    from oracle import int2 as oint2
    w = workloads.int2_rotated(seed, B=B, H=H, len_range=len_range, n_calib=8192)
    R, _ = oint2.fit_rotation(w.calib)
    T = oint2.clip_thresholds(w.calib, R)
    return w, R.astype(np.float32), T.astype(np.float32)


def _last_tokens(w, k=1):
    """Per sequence: its last k cached tokens (latent, rope) and their first position."""
    lat = [x[-k:] for x in w.latent]
    rope = [x[-k:] for x in w.rope]
    return lat, rope, (w.seq_lens - k).astype(np.int32)


# k new tokens a sequence: one (a decode step), three, and 6 x 700 = 4200, past the
# 4096 tokens that the planner's launch copies (the append then runs as its own kernel)
@pytest.mark.parametrize("kind_name,k", [("bf16", 1), ("fp32", 1), ("int2", 1), ("bf16", 3), ("bf16", 700)])
def test_append_decode_matches_append_then_decode(gpu_lib, kind_name, k):
    import mla_latent_kv_08_gb300 as mla
    import torch
    if kind_name == "fp32":
        w = workloads.tiny(0)
        q = np.stack([attention.absorb_query(w.q_nope[b], w.q_rope[b], w.W_UK) for b in range(w.B)])
        R = T = None
        shape = gu.shape_for(w)
    elif kind_name == "bf16":
        w = workloads.dsv3(31, B=6, H=128, len_range=(60, 400) if k < 700 else (800, 1000))
        q = w.q
        R = T = None
        shape = gu.shape_for(w)
    else:
        w, R, T = _int2_setup(B=4, H=128, len_range=(60, 300))
        q = w.q
        shape = gu.shape_for(w, kind=mla.MLA_KV_INT2_ROT)
    # cache A: every token appended beforehand; cache B: the same, but each sequence's
    # last slot overwritten with zeros, so that only the fused call's copy restores it
    cache_a, st_a = gu.fill_cache(w, shape, R, T)
    cache_b, st_b = gu.fill_cache(w, shape, R, T)
    lat, rope, pos = _last_tokens(w, k)
    zeros_c = [np.zeros_like(x) for x in lat]
    zeros_r = [np.zeros_like(x) for x in rope]
    gu.append_tokens(cache_b, w, zeros_c, zeros_r, pos, R, T)
    torch.cuda.synchronize()
    assert mla.mla_read_status_word(st_a)[0] == mla.MLA_OK and mla.mla_read_status_word(st_b)[0] == mla.MLA_OK

    out_a, lse_a, ws_a = gu.attend(w, shape, cache_a, q, R=R)

    dt = gu.torch_dtype(w)
    out_b = torch.empty((w.B, 1, w.H, w.d_v), dtype=dt, device="cuda")
    lse_b = torch.empty((w.B, 1, w.H), dtype=torch.float32, device="cuda")
    ws_b = mla.alloc_workspace(shape, w.B, 1)
    ast = torch.zeros(1, dtype=torch.int32, device="cuda")
    cu = (k * np.arange(w.B + 1)).astype(np.int32)
    mla.mla_append_decode(cache_b, gu.dev(w.block_table), gu.dev(pos), gu.dev(cu),
                          gu.dev(np.concatenate(lat).astype(np.float32), dt),
                          gu.dev(np.concatenate(rope).astype(np.float32), dt),
                          gu.dev(w.seq_lens.astype(np.int32)), gu.dev(q.astype(np.float32), dt),
                          gu.dev(w.W_UV.astype(np.float32), dt), w.scale, out_b, lse_b, ws_b,
                          R=None if R is None else gu.dev(R), clip=None if T is None else gu.dev(T),
                          append_status=ast)
    torch.cuda.synchronize()
    assert mla.mla_read_status_word(ast)[0] == mla.MLA_OK
    assert mla.mla_get_status(ws_b)[0] == mla.MLA_OK
    np.testing.assert_array_equal(out_b.float().cpu().numpy(), out_a)
    np.testing.assert_array_equal(lse_b.cpu().numpy(), lse_a)
    # and the cache now holds the true last tokens (cache bytes equal cache A's)
    for fa, fb in ((cache_a.latent, cache_b.latent), (cache_a.codes, cache_b.codes),
                   (cache_a.scale_zero, cache_b.scale_zero), (cache_a.rope, cache_b.rope)):
        if fa is not None:
            assert torch.equal(fa, fb)


def test_append_decode_reports_a_bad_position_on_its_own_status(gpu_lib):
    import mla_latent_kv_08_gb300 as mla
    import torch
    w = workloads.dsv3(32, B=3, H=128, len_range=(60, 200))
    shape = gu.shape_for(w)
    cache, _ = gu.fill_cache(w, shape)
    lat, rope, pos = _last_tokens(w)
    pos = pos.copy()
    pos[1] = w.block_table.shape[1] * w.block_size + 5          # past the block table
    dt = torch.bfloat16
    out = torch.empty((w.B, 1, w.H, w.d_v), dtype=dt, device="cuda")
    lse = torch.empty((w.B, 1, w.H), dtype=torch.float32, device="cuda")
    ws = mla.alloc_workspace(shape, w.B, 1)
    ast = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_append_decode(cache, gu.dev(w.block_table), gu.dev(pos), gu.dev(np.arange(w.B + 1, dtype=np.int32)),
                          gu.dev(np.concatenate(lat).astype(np.float32), dt),
                          gu.dev(np.concatenate(rope).astype(np.float32), dt),
                          gu.dev(w.seq_lens.astype(np.int32)), gu.dev(w.q.astype(np.float32), dt),
                          gu.dev(w.W_UV.astype(np.float32), dt), w.scale, out, lse, ws, append_status=ast)
    torch.cuda.synchronize()
    code, flags = mla.mla_read_status_word(ast)
    assert code != mla.MLA_OK and flags != 0
    # the decode itself ran on the cache as it stands (every slot already held its token)
    assert mla.mla_get_status(ws)[0] == mla.MLA_OK
    o = out.float().cpu().numpy()
    for b in range(w.B):
        ro, rl = attention.absorbed(w.q[b], w.latent[b], w.rope[b], w.W_UV, w.scale)
        assert gu.rel_err(o[b], ro) <= gu.BF16_REL_TOL
