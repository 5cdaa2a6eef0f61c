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


def test_prefill_chunk_full_sampled(gpu_lib):
    """One 512-token chunk at L = 8192, H = 128 (the benchmark's prefill workload), on
    the kernel and planner the benchmark times; sampled (row, head) pairs, each from the
    definition, across the chunk's causal window."""
    w = workloads.verify(5, B=1, q_len=512, len_range=(8192, 8192))
    shape = gu.shape_for(w)
    cache, _ = gu.fill_cache(w, shape)
    out, lse, ws = gu.attend(w, shape, cache, w.q, q_len=w.q_len)
    import mla_latent_kv_08_gb300 as mla
    assert mla.mla_get_status(ws)[0] == mla.MLA_OK
    pairs = [(i, h) for i in (0, 1, 127, 128, 255, 383, 510, 511) for h in (0, 63, 127)]
    ro, rl = attention.row_subset(w.q[0], w.latent[0], w.rope[0], w.W_UV, w.scale, pairs)
    got_o = np.stack([out[0, i, h] for i, h in pairs])
    got_l = np.array([lse[0, i, h] for i, h in pairs])
    assert gu.rel_err(got_o, ro) <= gu.BF16_REL_TOL
    assert float(np.max(np.abs(got_l - rl))) <= gu.BF16_LSE_TOL


def _int2_bench_cache(w, kind, R32, T):
    import mla_latent_kv_08_gb300 as mla
    shape = gu.shape_for(w, kind=kind)
    cache = mla.Cache.allocate(shape)
    st = gu.append_tokens(cache, w, w.latent, w.rope, np.zeros(w.B, np.int32), R32, T)
    return shape, cache, st


@pytest.mark.parametrize("q_rotated", [False, True])
def test_int2_full_library_calibration_folded(gpu_lib, q_rotated):
    """The rotated-INT2 workload as the benchmark runs it: R and the clip thresholds
    from the library's own calibration, W_UV folded (and, with q_rotated, the query
    given in the rotated basis, R not passed); sampled sequences against the oracle's
    attention over the cache the oracle's encoder builds from the same R and
    thresholds."""
    import mla_latent_kv_08_gb300 as mla
    import torch
    w = workloads.int2_rotated(4)
    R32, clip, _, _ = mla.calibrate_rotation(torch.from_numpy(np.asarray(w.calib)).cuda())
    R32 = np.asarray(R32, np.float32)
    clip = np.asarray(clip, np.float32)
    shape, cache, st = _int2_bench_cache(w, mla.MLA_KV_INT2_ROT, R32, clip)
    torch.cuda.synchronize()
    assert mla.mla_read_status_word(st)[0] == mla.MLA_OK
    Wf = torch.empty((w.H, w.r, w.d_v), dtype=torch.bfloat16, device="cuda")
    mla.mla_fold_rotation(shape, gu.dev(R32), gu.dev(w.W_UV, torch.bfloat16), Wf)
    fshape = gu.shape_for(w, kind=mla.MLA_KV_INT2_ROT)
    fshape.flags = mla.MLA_FLAG_WUV_FOLDED | (mla.MLA_FLAG_Q_ROTATED if q_rotated else 0)
    q_in = np.array(w.q, dtype=np.float64)
    q_ref = q_in
    if q_rotated:
        q_in[..., :w.r] = workloads.bf16_round((q_in[..., :w.r] @ R32.astype(np.float64)).astype(np.float32))
        q_ref = q_in.copy()
        q_ref[..., :w.r] = q_in[..., :w.r] @ R32.astype(np.float64).T
    out = torch.empty((w.B, 1, w.H, w.d_v), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, 1, w.H), dtype=torch.float32, device="cuda")
    ws = mla.alloc_workspace(fshape, w.B, 1)
    mla.mla_decode(cache, gu.dev(w.block_table), gu.dev(w.seq_lens.astype(np.int32)),
                   gu.dev(q_in.astype(np.float32), torch.bfloat16), Wf, w.scale, out, lse, ws,
                   R=None if q_rotated else gu.dev(R32), shape=fshape)
    torch.cuda.synchronize()
    assert mla.mla_get_status(ws)[0] == mla.MLA_OK
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    for b in (0, int(np.argmax(w.seq_lens)), int(np.argmin(w.seq_lens))):
        codes, sz = oint2.quantize(w.latent[b], R32, clip)
        ro, rl = oint2.attention_rotated(q_ref[b], oint2.decode(codes, sz), w.rope[b], R32, w.W_UV, w.scale)
        _check(o, l, b, ro, rl)


def test_int2_rope_full_library_calibration_folded(gpu_lib):
    """The rope-INT2 workload as the benchmark runs it (library calibration, rope-key
    thresholds from calibration rope keys, W_UV folded); sampled sequences."""
    import mla_latent_kv_08_gb300 as mla
    import torch
    w = workloads.int2_rotated(4)
    R32, clip, _, _ = mla.calibrate_rotation(torch.from_numpy(np.asarray(w.calib)).cuda())
    R32 = np.asarray(R32, np.float32)
    clip = np.asarray(clip, np.float32)
    rng = np.random.Generator(np.random.PCG64(11))
    KRcal = workloads.bf16_round(rng.standard_normal((w.calib.shape[0], w.d_rope)).astype(np.float32)).astype(np.float64)
    clip_r = np.asarray(mla.calib_thresholds(np.abs(KRcal), 32, 99.0), np.float32)
    T = np.concatenate([clip, clip_r])
    shape, cache, st = _int2_bench_cache(w, mla.MLA_KV_INT2_ROT_QR, R32, T)
    torch.cuda.synchronize()
    assert mla.mla_read_status_word(st)[0] == mla.MLA_OK
    Wf = torch.empty((w.H, w.r, w.d_v), dtype=torch.bfloat16, device="cuda")
    mla.mla_fold_rotation(shape, gu.dev(R32), gu.dev(w.W_UV, torch.bfloat16), Wf)
    fshape = gu.shape_for(w, kind=mla.MLA_KV_INT2_ROT_QR)
    fshape.flags = mla.MLA_FLAG_WUV_FOLDED
    out = torch.empty((w.B, 1, w.H, w.d_v), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, 1, w.H), dtype=torch.float32, device="cuda")
    ws = mla.alloc_workspace(fshape, w.B, 1)
    mla.mla_decode(cache, gu.dev(w.block_table), gu.dev(w.seq_lens.astype(np.int32)), gu.dev(w.q, torch.bfloat16),
                   Wf, w.scale, out, lse, ws, R=gu.dev(R32), shape=fshape)
    torch.cuda.synchronize()
    assert mla.mla_get_status(ws)[0] == mla.MLA_OK
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    for b in (0, int(np.argmax(w.seq_lens))):
        codes, sz = oint2.quantize_rope_int2(w.latent[b], w.rope[b], R32, clip, clip_r)
        Y = oint2.decode(codes, sz).astype(np.float64)
        ro, rl = oint2.attention_rope_int2(w.q[b], Y, R32, w.W_UV, w.scale)
        _check(o, l, b, ro, rl)
