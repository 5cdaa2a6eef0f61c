"""mla_decode_noalloc: the decode entry point for callers that cannot allocate
device memory when they call it (an engine plugin whose enqueue step must not
allocate, a server whose memory pool already owns the GPU). It must give the
same answer as mla_decode with a caller workspace, call after call, and refuse
problems too large for its fixed 32 MiB scratch without launching anything.

This file is named so that pytest collects it last."""
import numpy as np
import pytest

import workloads
from oracle import attention
from oracle import int2 as oint2
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_decode_twice(gpu_lib):
    import torch

    import mla_latent_kv_08_gb300 as mla
    w = workloads.dsv3(31, B=4, H=128, len_range=(100, 2500))
    shape = gu.shape_for(w)
    cache, _ = gu.fill_cache(w, shape)
    ref_out, ref_lse, ws = gu.attend(w, shape, cache, w.q)
    assert mla.mla_get_status(ws)[0] == mla.MLA_OK

    bf = torch.bfloat16
    bt = gu.dev(w.block_table)
    sl = gu.dev(w.seq_lens.astype(np.int32))
    q = gu.dev(w.q, bf)
    W = gu.dev(w.W_UV, bf)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full((w.B, 1, w.H, w.d_v), float("nan"), dtype=bf, device="cuda")
        lse = torch.full((w.B, 1, w.H), float("nan"), dtype=torch.float32, device="cuda")
        mla.mla_decode_noalloc(cache, bt, sl, q, W, w.scale, out, lse, status=status)
        torch.cuda.synchronize()
        assert mla.mla_read_status_word(status) == (mla.MLA_OK, 0), call
        o = out.float().cpu().numpy()
        l = lse.cpu().numpy()
        for b in range(w.B):
            assert gu.rel_err(o[b], ref_out[b]) <= gu.BF16_REL_TOL, (call, b)
            assert np.max(np.abs(l[b] - ref_lse[b])) <= gu.BF16_LSE_TOL, (call, b)
        # and the same bar against the CPU oracle
        for b in (0, w.B - 1):
            ro, rl = attention.absorbed(w.q[b], w.latent[b], w.rope[b], w.W_UV, w.scale)
            assert gu.rel_err(o[b], ro) <= gu.BF16_REL_TOL
            assert np.max(np.abs(l[b] - rl)) <= gu.BF16_LSE_TOL


def test_noalloc_rejects_oversized_problem(gpu_lib):
    import torch

    import mla_latent_kv_08_gb300 as mla
    # one split per sequence needs about B * H * kv_lora_rank * 4 bytes of
    # partials: 200 sequences x 128 heads x 512 x 4 B = 50 MiB > 32 MiB
    B, H = 200, 128
    shape = mla.Shape(num_heads=H, kv_lora_rank=512, rope_dim=64, v_head_dim=128, block_size=64, num_blocks=B)
    cache = mla.Cache.allocate(shape)
    bt = torch.arange(B, dtype=torch.int32, device="cuda").reshape(B, 1)
    sl = torch.full((B,), 64, dtype=torch.int32, device="cuda")
    q = torch.zeros((B, 1, H, 576), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((H, 512, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((B, 1, H, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((B, 1, H), dtype=torch.float32, device="cuda")
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_noalloc(cache, bt, sl, q, W, 0.1, out, lse)
    assert e.value.code == mla.MLA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int(out.float().abs().sum().item()) == 0      # nothing was launched


def _noalloc_twice(w, shape, cache, ref_out, ref_lse, R=None):
    """Two mla_decode_noalloc calls in a row, each checked against a caller-workspace
    decode of the same inputs; returns the outputs of the second call."""
    import torch

    import mla_latent_kv_08_gb300 as mla
    bf = torch.bfloat16
    bt = gu.dev(w.block_table)
    sl = gu.dev(w.seq_lens.astype(np.int32))
    q = gu.dev(w.q, bf)
    W = gu.dev(w.W_UV, bf)
    Rd = None if R is None else gu.dev(R.astype(np.float32))
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full((w.B, 1, w.H, w.d_v), float("nan"), dtype=bf, device="cuda")
        lse = torch.full((w.B, 1, w.H), float("nan"), dtype=torch.float32, device="cuda")
        mla.mla_decode_noalloc(cache, bt, sl, q, W, w.scale, out, lse, R=Rd, status=status)
        torch.cuda.synchronize()
        assert mla.mla_read_status_word(status) == (mla.MLA_OK, 0), call
        o = out.float().cpu().numpy()
        l = lse.cpu().numpy()
        for b in range(w.B):
            assert gu.rel_err(o[b], ref_out[b]) <= gu.BF16_REL_TOL, (call, b)
            assert np.max(np.abs(l[b] - ref_lse[b])) <= gu.BF16_LSE_TOL, (call, b)
    return o, l


def test_noalloc_rotated_int2_matches_workspace_decode(gpu_lib):
    """The rotated-INT2 cache routes its extra scratch (rotated query, merged rotated
    output, fp16 copy of R) through the fixed array as well."""
    import torch

    import mla_latent_kv_08_gb300 as mla
    w = workloads.int2_rotated(4, B=4, H=128, len_range=(100, 700), n_calib=8192)
    R, _ = oint2.fit_rotation(w.calib)
    T = oint2.clip_thresholds(w.calib, R)
    R32, T32 = R.astype(np.float32), T.astype(np.float32)
    shape = gu.shape_for(w, kind=mla.MLA_KV_INT2_ROT, impl=mla.MLA_IMPL_TCGEN05)
    assert mla.mla_resolve_impl(shape) == mla.MLA_IMPL_TCGEN05
    cache, st = gu.fill_cache(w, shape, R32, T32)
    torch.cuda.synchronize()
    assert mla.mla_read_status_word(st)[0] == mla.MLA_OK
    ref_out, ref_lse, ws = gu.attend(w, shape, cache, w.q, R=R32)
    assert mla.mla_get_status(ws)[0] == mla.MLA_OK
    o, l = _noalloc_twice(w, shape, cache, ref_out, ref_lse, R=R32)
    # and against the oracle's attention over its own dequantised codes
    for b in (0, w.B - 1):
        codes, sz = oint2.quantize(w.latent[b], R32, T32)
        ro, rl = oint2.attention_rotated(w.q[b], oint2.decode(codes, sz), w.rope[b], R32, w.W_UV, w.scale)
        assert gu.rel_err(o[b], ro) <= gu.BF16_REL_TOL
        assert np.max(np.abs(l[b] - rl)) <= gu.BF16_LSE_TOL


def test_noalloc_shrinks_the_split_count_to_fit(gpu_lib):
    """100 sequences x 128 heads: the planner's default split count needs about 46 MB
    of partial outputs, more than the 32 MiB array; one split per sequence needs 26 MB.
    The entry point picks the largest split count that fits and still matches."""
    import mla_latent_kv_08_gb300 as mla
    w = workloads.dsv3(33, B=100, H=128, len_range=(64, 600))
    shape = gu.shape_for(w)
    assert mla.mla_workspace_bytes(shape, w.B, 1) > (32 << 20)
    assert mla.mla_workspace_bytes(gu.shape_for(w, splits=1), w.B, 1) <= (32 << 20)
    cache, _ = gu.fill_cache(w, shape)
    ref_out, ref_lse, ws = gu.attend(w, shape, cache, w.q)
    assert mla.mla_get_status(ws)[0] == mla.MLA_OK
    o, l = _noalloc_twice(w, shape, cache, ref_out, ref_lse)
    for b in (0, 57, w.B - 1):
        ro, rl = attention.absorbed(w.q[b], w.latent[b], w.rope[b], w.W_UV, w.scale)
        assert gu.rel_err(o[b], ro) <= gu.BF16_REL_TOL
        assert np.max(np.abs(l[b] - rl)) <= gu.BF16_LSE_TOL


def test_noalloc_reports_the_same_codes_as_decode(gpu_lib):
    """A shape the tensor-core kernel cannot take, forced onto it, is refused with the
    code mla_decode gives (unsupported), not as an invalid argument."""
    import torch

    import mla_latent_kv_08_gb300 as mla
    shape = mla.Shape(num_heads=8, kv_lora_rank=256, rope_dim=64, v_head_dim=64, block_size=64, num_blocks=2,
                      impl=mla.MLA_IMPL_TCGEN05)
    cache = mla.Cache.allocate(shape)
    bt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    sl = torch.full((1,), 10, dtype=torch.int32, device="cuda")
    q = torch.zeros((1, 1, 8, 320), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((8, 256, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((1, 1, 8, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 1, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(mla.MlaError) as e:
        mla.mla_decode_noalloc(cache, bt, sl, q, W, 0.1, out, lse)
    assert e.value.code == mla.MLA_ERR_UNSUPPORTED
