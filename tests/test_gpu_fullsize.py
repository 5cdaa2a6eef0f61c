"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times (default planner, default implementation). Sequences are
checked whole where the oracle takes seconds, and on sampled sequences
otherwise."""
import numpy as np
import pytest

import workloads
from oracle import attention, layout
from oracle import int2 as oint2
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _check(out, lse, b, ro, rl):
    e = gu.rel_err(out[b], ro)
    le = float(np.max(np.abs(lse[b] - rl)))
    assert e <= gu.BF16_REL_TOL and le <= gu.BF16_LSE_TOL, (b, e, le)


def test_dsv3_full_all_sequences(gpu_lib):
    w = workloads.dsv3(1)
    shape = gu.shape_for(w)
    cache, _ = gu.fill_cache(w, shape)
    out, lse, ws = gu.attend(w, shape, cache, w.q)
    import mla_latent_kv_08_gb300 as mla
    assert mla.mla_get_status(ws)[0] == mla.MLA_OK
    for b in range(w.B):
        ro, rl = attention.absorbed(w.q[b], w.latent[b], w.rope[b], w.W_UV, w.scale)
        _check(out, lse, b, ro, rl)


def test_long_context_full(gpu_lib):
    w = workloads.long_context(2)
    shape = gu.shape_for(w)
    cache, _ = gu.fill_cache(w, shape)
    out, lse, _ = gu.attend(w, shape, cache, w.q)
    for b in range(w.B):
        ro, rl = attention.absorbed(w.q[b], w.latent[b], w.rope[b], w.W_UV, w.scale)
        _check(out, lse, b, ro, rl)


def test_verify_full_sampled(gpu_lib):
    w = workloads.verify(3)
    shape = gu.shape_for(w)
    cache, _ = gu.fill_cache(w, shape)
    out, lse, _ = gu.attend(w, shape, cache, w.q, q_len=w.q_len)
    longest = int(np.argmax(w.seq_lens))
    for b in sorted({0, 7, longest}):
        ro, rl = attention.absorbed(w.q[b], w.latent[b], w.rope[b], w.W_UV, w.scale)
        _check(out, lse, b, ro, rl)


def test_int2_full_codes_and_sampled_decode(gpu_lib):
    import mla_latent_kv_08_gb300 as mla
    import torch
    w = workloads.int2_rotated(4)
    R, _ = oint2.fit_rotation(w.calib)
    T = oint2.clip_thresholds(w.calib, R)
    R32, T32 = R.astype(np.float32), T.astype(np.float32)
    shape = gu.shape_for(w, kind=mla.MLA_KV_INT2_ROT)
    cache = mla.Cache.allocate(shape)
    gu.append_tokens(cache, w, w.latent, w.rope, np.zeros(w.B, np.int32), R32, T32)
    st = gu.append_tokens(cache, w, w.new_latent, w.new_rope, w.start_pos, R32, T32)   # the 1024-token append
    torch.cuda.synchronize()
    assert mla.mla_read_status_word(st)[0] == mla.MLA_OK
    # every appended token: codes and scale/zero bit-exact, read back through the block table
    codes_pool = cache.codes.cpu().numpy()
    sz_pool = cache.scale_zero.cpu().view(torch.int16).numpy().view(np.uint16)
    for b in range(w.B):
        rc, rsz = oint2.quantize(w.new_latent[b], R32, T32)
        rows = np.arange(w.start_pos[b], w.start_pos[b] + 32)
        got_c = np.stack([codes_pool[w.block_table[b, t // 64], t % 64] for t in rows])
        got_s = np.stack([sz_pool[w.block_table[b, t // 64], t % 64] for t in rows])
        np.testing.assert_array_equal(got_c, rc)
        np.testing.assert_array_equal(got_s, rsz)
    w.seq_lens = (w.seq_lens + 32).astype(np.int32)
    out, lse, _ = gu.attend(w, shape, cache, w.q, R=R32)
    for b in (0, int(np.argmin(w.seq_lens))):
        C = np.concatenate([w.latent[b], w.new_latent[b]])
        KR = np.concatenate([w.rope[b], w.new_rope[b]])
        codes, sz = oint2.quantize(C, R32, T32)
        ro, rl = oint2.attention_rotated(w.q[b], oint2.decode(codes, sz), KR, R32, w.W_UV, w.scale)
        _check(out, lse, b, ro, rl)
