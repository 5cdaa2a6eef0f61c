"""GPU parity: the library (through its C ABI) against the CPU oracle on the
same seeded inputs. bf16 caches: max relative error 1e-2 per sequence and LSE
absolute error 2e-3; fp32 cache: 1e-5 / 1e-5; cache bytes, INT2 codes, scales
and packing bit-exact."""
import math

import numpy as np
import pytest

import workloads
from oracle import attention, layout
from oracle import int2 as oint2
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _check_seq(out, lse, w, b, ref_out, ref_lse, rel_tol, lse_tol):
    e = gu.rel_err(out[b], ref_out)
    le = float(np.max(np.abs(lse[b] - ref_lse)))
    assert np.all(np.isfinite(out[b])), f"seq {b}: non-finite output"
    assert e <= rel_tol, f"seq {b}: rel err {e:.3e} > {rel_tol}"
    assert le <= lse_tol, f"seq {b}: lse err {le:.3e} > {lse_tol}"
    return e, le


# ------------------------------------------------------------------ tiny fp32

def test_tiny_fp32_matches_absorbed_and_full_head(gpu_lib):
    w = workloads.tiny(0)
    q = np.stack([attention.absorb_query(w.q_nope[b], w.q_rope[b], w.W_UK) for b in range(w.B)])
    shape = gu.shape_for(w)
    cache, status = gu.fill_cache(w, shape)
    out, lse, ws = gu.attend(w, shape, cache, q)
    import mla_latent_kv_08_gb300 as mla
    assert mla.mla_get_status(ws)[0] == mla.MLA_OK
    for b in range(w.B):
        ro, rl = attention.absorbed(q[b], w.latent[b], w.rope[b], w.W_UV, w.scale)
        _check_seq(out, lse, w, b, ro, rl, gu.FP32_REL_TOL, gu.FP32_LSE_TOL)
        fo, fl = attention.full_head(w.q_nope[b], w.q_rope[b], w.latent[b], w.rope[b], w.W_UK, w.W_UV, w.scale)
        _check_seq(out, lse, w, b, fo, fl, gu.FP32_REL_TOL, gu.FP32_LSE_TOL)


# ------------------------------------------------------------ append bytes

@pytest.mark.parametrize("kind", ["bf16", "fp32"])
def test_append_layout_bit_exact(gpu_lib, kind):
    import mla_latent_kv_08_gb300 as mla
    import torch
    w = workloads.dsv3(11, B=5, H=8, len_range=(1, 333))
    w.seq_lens[0] = 64        # exactly one block
    w.latent[0] = w.latent[0][:64] if w.latent[0].shape[0] >= 64 else np.resize(w.latent[0], (64, 512))
    w.rope[0] = np.resize(w.rope[0], (64, 64))
    tab, nb = workloads.make_paging(np.random.default_rng(5), w.seq_lens, 64, spare_blocks=3)
    w.block_table, w.num_blocks = tab, nb
    shape = gu.shape_for(w, kind=mla.MLA_KV_FP32 if kind == "fp32" else mla.MLA_KV_BF16)
    # split each sequence's tokens over two appends to exercise start_pos
    cache = mla.Cache.allocate(shape)
    half = [x.shape[0] // 2 for x in w.latent]
    gu.append_tokens(cache, w, [x[:h] for x, h in zip(w.latent, half)], [x[:h] for x, h in zip(w.rope, half)],
                     np.zeros(w.B, np.int32))
    st = gu.append_tokens(cache, w, [x[h:] for x, h in zip(w.latent, half)], [x[h:] for x, h in zip(w.rope, half)],
                          np.array(half, np.int32))
    torch.cuda.synchronize()
    assert mla.mla_read_status_word(st)[0] == mla.MLA_OK
    rows = [np.concatenate([w.latent[b], w.rope[b]], 1) for b in range(w.B)]
    ref = layout.write_paged(nb, 64, w.D, tab, rows, [0] * w.B)
    got = cache.latent.cpu()
    if kind == "fp32":
        np.testing.assert_array_equal(got.numpy().view(np.uint32), ref.astype(np.float32).view(np.uint32))
    else:
        np.testing.assert_array_equal(got.view(torch.int16).numpy().view(np.uint16), workloads.bf16_bits(ref))


@pytest.mark.parametrize("kind", ["bf16", "fp32"])
def test_index_key_layout_bit_exact(gpu_lib, kind):
    """The extra per-token key (64 elements: the 640-element row of a latent layer
    with an indexer key) lands after the rope key of each token's row."""
    import mla_latent_kv_08_gb300 as mla
    import torch
    w = workloads.dsv3(12, B=4, H=8, len_range=(1, 200))
    rng = np.random.default_rng(12)
    idx = [workloads.bf16_round(rng.standard_normal((int(L), 64)).astype(np.float32)) for L in w.seq_lens]
    shape = gu.shape_for(w, kind=mla.MLA_KV_FP32 if kind == "fp32" else mla.MLA_KV_BF16)
    shape.index_dim = 64
    assert mla.Cache.allocate(shape).bytes_per_token() == (4 if kind == "fp32" else 2) * 640
    cache = mla.Cache.allocate(shape)
    gu.append_tokens(cache, w, w.latent, w.rope, np.zeros(w.B, np.int32))
    dt = torch.float32 if kind == "fp32" else torch.bfloat16
    cu = np.concatenate([[0], np.cumsum(w.seq_lens)]).astype(np.int32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_latent_append_index(cache, gu.dev(w.block_table), gu.dev(np.zeros(w.B, np.int32)), gu.dev(cu),
                                gu.dev(np.concatenate(idx), dt), status=st)
    torch.cuda.synchronize()
    assert mla.mla_read_status_word(st)[0] == mla.MLA_OK
    rows = [np.concatenate([w.latent[b], w.rope[b], idx[b]], 1) for b in range(w.B)]
    ref = layout.write_paged(w.num_blocks, 64, 640, w.block_table, rows, [0] * w.B)
    got = cache.latent.cpu()
    if kind == "fp32":
        np.testing.assert_array_equal(got.numpy().view(np.uint32), ref.astype(np.float32).view(np.uint32))
    else:
        np.testing.assert_array_equal(got.view(torch.int16).numpy().view(np.uint16), workloads.bf16_bits(ref))


@pytest.mark.parametrize("impl_name", ["tcgen05", "simt"])
def test_index_key_is_never_read_by_attention(gpu_lib, impl_name):
    """With NaN extra keys in every row, decode equals the decode of the same tokens
    in a cache without the extra field, bit for bit (both follow the row stride)."""
    import mla_latent_kv_08_gb300 as mla
    w = workloads.dsv3(13, B=3, H=128, len_range=(70, 600))
    impl = mla.MLA_IMPL_SIMT if impl_name == "simt" else mla.MLA_IMPL_TCGEN05
    res = []
    for index_dim in (0, 64):
        shape = gu.shape_for(w, impl=impl)
        shape.index_dim = index_dim
        cache = mla.Cache.allocate(shape)
        if index_dim:
            cache.latent[..., 576:] = float("nan")
        gu.append_tokens(cache, w, w.latent, w.rope, np.zeros(w.B, np.int32))
        res.append(gu.attend(w, shape, cache, w.q)[:2])
    (o0, l0), (o1, l1) = res
    assert np.isfinite(o1).all()
    np.testing.assert_array_equal(o1, o0)
    np.testing.assert_array_equal(l1, l0)
    ro, rl = attention.absorbed(w.q[0], w.latent[0], w.rope[0], w.W_UV, w.scale)
    _check_seq(o1, l1, w, 0, ro, rl, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)


def test_append_empty_is_noop(gpu_lib):
    import mla_latent_kv_08_gb300 as mla
    import torch
    w = workloads.dsv3(12, B=2, H=8, len_range=(10, 20))
    shape = gu.shape_for(w)
    cache = mla.Cache.allocate(shape)
    gu.append_tokens(cache, w, [np.zeros((0, 512), np.float32)] * 2, [np.zeros((0, 64), np.float32)] * 2,
                     np.zeros(2, np.int32))
    torch.cuda.synchronize()
    assert int(cache.latent.abs().sum().item()) == 0


# ---------------------------------------------------------------- bf16 decode

def test_dsv3_small_bf16(gpu_lib):
    w = workloads.dsv3(1, B=6, H=128, len_range=(1, 900))
    w.seq_lens[1] = 1
    w.latent[1], w.rope[1] = w.latent[1][:1], w.rope[1][:1]
    shape = gu.shape_for(w)
    cache, _ = gu.fill_cache(w, shape)
    out, lse, _ = gu.attend(w, shape, cache, w.q)
    for b in range(w.B):
        ro, rl = attention.absorbed(w.q[b], w.latent[b], w.rope[b], w.W_UV, w.scale)
        _check_seq(out, lse, w, b, ro, rl, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)


def test_split_count_does_not_change_result(gpu_lib):
    w = workloads.dsv3(2, B=3, H=64, len_range=(2000, 3000))
    res = []
    for hint in (1, 7, 200):
        shape = gu.shape_for(w, splits=hint)
        cache, _ = gu.fill_cache(w, shape)
        res.append(gu.attend(w, shape, cache, w.q)[:2])
    for o, l in res[1:]:
        assert np.max(np.abs(l - res[0][1])) < 1e-5
        assert gu.rel_err(o, res[0][0]) < 8e-3      # bf16 output rounding of near-equal fp32 values
    ro, rl = attention.absorbed(w.q[0], w.latent[0], w.rope[0], w.W_UV, w.scale)
    _check_seq(res[2][0], res[2][1], w, 0, ro, rl, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)


@pytest.mark.parametrize("B", [1, 5, 8, 9])
def test_combine_shares_splits_across_warps(gpu_lib, B):
    """Up to 8 rows per combine CTA deal each row's splits to several warps (16 / rows
    of them) and merge their partials; 9 rows take one warp per row. Every row must
    match the oracle whichever way its splits were merged."""
    w = workloads.dsv3(11 + B, B=B, H=16, len_range=(3000, 5000))
    shape = gu.shape_for(w, splits=48)
    cache, _ = gu.fill_cache(w, shape)
    out, lse, _ = gu.attend(w, shape, cache, w.q)
    for b in range(w.B):
        ro, rl = attention.absorbed(w.q[b], w.latent[b], w.rope[b], w.W_UV, w.scale)
        _check_seq(out, lse, w, b, ro, rl, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)


def test_verify_causal_window(gpu_lib):
    w = workloads.verify(3, B=4, q_len=8, len_range=(8, 400), H=32)
    w.seq_lens[0] = 8          # first draft row sees exactly one token
    w.latent[0], w.rope[0] = w.latent[0][:8], w.rope[0][:8]
    shape = gu.shape_for(w)
    cache, _ = gu.fill_cache(w, shape)
    out, lse, _ = gu.attend(w, shape, cache, w.q, q_len=8)
    for b in range(w.B):
        ro, rl = attention.absorbed(w.q[b], w.latent[b], w.rope[b], w.W_UV, w.scale)
        _check_seq(out, lse, w, b, ro, rl, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)


# ------------------------------------------------------------------ INT2

def _int2_setup(B, H, len_range, n_calib=8192, seed=4):
    w = workloads.int2_rotated(seed, B=B, H=H, len_range=len_range, n_calib=n_calib)
    R, _ = oint2.fit_rotation(w.calib)
    T = oint2.clip_thresholds(w.calib, R)
    return w, R.astype(np.float32), T.astype(np.float32)


def _int2_reference_pool(w, R32, T32, seqs, with_new=True):
    """Oracle codes / scale-zero / rope for the given sequences, placed in a pool."""
    out = {}
    for b in seqs:
        C = w.latent[b]
        KR = w.rope[b]
        if with_new:
            C = np.concatenate([C, w.new_latent[b]])
            KR = np.concatenate([KR, w.new_rope[b]])
        codes, sz = oint2.quantize(C, R32, T32)
        out[b] = (codes, sz, KR)
    return out


@pytest.mark.parametrize("impl_name,H", [("simt", 32), ("tcgen05", 32), ("tcgen05", 128)])
def test_int2_append_and_decode_small(gpu_lib, impl_name, H):
    import mla_latent_kv_08_gb300 as mla
    import torch
    w, R32, T32 = _int2_setup(B=4, H=H, len_range=(40, 300))
    impl = mla.MLA_IMPL_SIMT if impl_name == "simt" else mla.MLA_IMPL_TCGEN05
    shape = gu.shape_for(w, kind=mla.MLA_KV_INT2_ROT, impl=impl)
    assert mla.mla_resolve_impl(shape) == impl
    cache = mla.Cache.allocate(shape)
    st0 = gu.append_tokens(cache, w, w.latent, w.rope, np.zeros(w.B, np.int32), R32, T32)
    st1 = gu.append_tokens(cache, w, w.new_latent, w.new_rope, w.start_pos, R32, T32)
    torch.cuda.synchronize()
    assert mla.mla_read_status_word(st0)[0] == mla.MLA_OK and mla.mla_read_status_word(st1)[0] == mla.MLA_OK
    ref = _int2_reference_pool(w, R32, T32, range(w.B))
    nb = w.num_blocks
    lens_new = w.seq_lens + 32
    ref_codes = layout.write_paged(nb, 64, 128, w.block_table, [ref[b][0] for b in range(w.B)], [0] * w.B, np.uint8)
    ref_sz = layout.write_paged(nb, 64, 32, w.block_table, [ref[b][1].reshape(-1, 32) for b in range(w.B)],
                                [0] * w.B, np.uint16)
    ref_rope = layout.write_paged(nb, 64, 64, w.block_table, [workloads.bf16_bits(ref[b][2]) for b in range(w.B)],
                                  [0] * w.B, np.uint16)
    np.testing.assert_array_equal(cache.codes.cpu().numpy(), ref_codes)
    np.testing.assert_array_equal(cache.scale_zero.cpu().view(torch.int16).numpy().view(np.uint16).reshape(nb, 64, 32), ref_sz)
    np.testing.assert_array_equal(cache.rope.cpu().view(torch.int16).numpy().view(np.uint16), ref_rope)
    # decode over the appended lengths against the oracle's own dequantised codes
    w.seq_lens = lens_new.astype(np.int32)
    out, lse, _ = gu.attend(w, shape, cache, w.q, R=R32)
    for b in range(w.B):
        Chat = oint2.decode(ref[b][0], ref[b][1])
        ro, rl = oint2.attention_rotated(w.q[b], Chat, ref[b][2], R32, w.W_UV, w.scale)
        _check_seq(out, lse, w, b, ro, rl, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)


# ------------------------------------------------------------ prefill chunks

@pytest.mark.parametrize("impl_name", ["tcgen05", "simt"])
@pytest.mark.parametrize("H,q_len,lens", [(16, 96, (200, 700)), (128, 40, (100, 400))])
def test_prefill_chunk_in_latent_form(gpu_lib, impl_name, H, q_len, lens):
    """Chunked prefill is the verify call with a long causal window: the chunk's
    q_len tokens are already appended; row i sees positions 0 .. L - q_len + i
    (many 128-row tiles, causal masks inside KV tiles)."""
    import mla_latent_kv_08_gb300 as mla
    w = workloads.verify(40 + q_len, B=2, q_len=q_len, len_range=lens, H=H)
    impl = mla.MLA_IMPL_SIMT if impl_name == "simt" else mla.MLA_IMPL_TCGEN05
    shape = gu.shape_for(w, impl=impl)
    cache, _ = gu.fill_cache(w, shape)
    out, lse, ws = gu.attend(w, shape, cache, w.q, q_len=q_len)
    assert mla.mla_get_status(ws) == (mla.MLA_OK, 0)
    for b in range(w.B):
        ro, rl = attention.absorbed(w.q[b], w.latent[b], w.rope[b], w.W_UV, w.scale)
        _check_seq(out, lse, w, b, ro, rl, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)


# ------------------------------------------------------------ many sequences

@pytest.mark.parametrize("impl_name", ["tcgen05", "simt"])
def test_more_sequences_than_one_planner_block(gpu_lib, impl_name):
    """B = 1100 short sequences (1..100 tokens): the planner's scans run over more than
    one 1024-wide chunk, streams hold many items; every row matches the oracle."""
    import mla_latent_kv_08_gb300 as mla
    w = workloads.dsv3(31, B=1100, H=16, len_range=(1, 100))
    impl = mla.MLA_IMPL_SIMT if impl_name == "simt" else mla.MLA_IMPL_TCGEN05
    shape = gu.shape_for(w, impl=impl)
    cache, _ = gu.fill_cache(w, shape)
    out, lse, ws = gu.attend(w, shape, cache, w.q)
    assert mla.mla_get_status(ws) == (mla.MLA_OK, 0)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    for b in list(range(0, w.B, 37)) + [w.B - 1]:
        ro, rl = attention.absorbed(w.q[b], w.latent[b], w.rope[b], w.W_UV, w.scale)
        _check_seq(out, lse, w, b, ro, rl, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)


# ------------------------------------------------------------ failure detection

def test_bounded_wait_gives_up_and_the_context_stays_usable(gpu_lib):
    """A wait on a barrier that nothing arrives on gives up after its limit, records
    the timeout flag, and the kernel returns; a decode afterwards is still correct."""
    import mla_latent_kv_08_gb300 as mla
    import torch
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    mla.mla_selftest_wait_timeout(2_000_000, status)          # 2 ms
    code, flags = mla.mla_read_status_word(status)
    assert code == mla.MLA_ERR_TIMEOUT and flags == 4
    w = workloads.dsv3(23, B=2, H=128, len_range=(100, 400))
    shape = gu.shape_for(w)
    cache, _ = gu.fill_cache(w, shape)
    out, lse, ws = gu.attend(w, shape, cache, w.q)
    assert mla.mla_get_status(ws) == (mla.MLA_OK, 0)
    for b in range(w.B):
        ro, rl = attention.absorbed(w.q[b], w.latent[b], w.rope[b], w.W_UV, w.scale)
        _check_seq(out, lse, w, b, ro, rl, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)


# ------------------------------------------------------------ stale pool bytes

def _pool_fill(cache, value):
    """Every pool byte set: latent/rope/scale_zero to `value`, codes to 0xFF or 0."""
    import math
    for name in ("latent", "rope", "scale_zero"):
        t = getattr(cache, name, None)
        if t is not None:
            t.fill_(value)
    if getattr(cache, "codes", None) is not None:
        cache.codes.fill_(0xFF if math.isnan(value) else 0)


@pytest.mark.parametrize("impl_name", ["tcgen05", "simt"])
def test_stale_slots_past_the_end_do_not_leak(gpu_lib, impl_name):
    """The slots of a sequence's last block past its length hold whatever the pool
    held before (here NaN): the result must equal the one over a zero-filled pool,
    bit for bit, and be finite (P = 0 must never meet the stale bytes)."""
    import mla_latent_kv_08_gb300 as mla
    import torch
    w = workloads.dsv3(21, B=4, H=128, len_range=(70, 700))
    assert np.any(w.seq_lens % 64 != 0)
    impl = mla.MLA_IMPL_SIMT if impl_name == "simt" else mla.MLA_IMPL_TCGEN05
    shape = gu.shape_for(w, impl=impl)
    res = []
    for fill in (0.0, float("nan")):
        cache = mla.Cache.allocate(shape, zero=False)
        _pool_fill(cache, fill)
        gu.append_tokens(cache, w, w.latent, w.rope, np.zeros(w.B, np.int32))
        torch.cuda.synchronize()
        res.append(gu.attend(w, shape, cache, w.q)[:2])
    (o0, l0), (o1, l1) = res
    assert np.isfinite(o1).all() and np.isfinite(l1).all()
    np.testing.assert_array_equal(o1, o0)
    np.testing.assert_array_equal(l1, l0)


def test_int2_stale_slots_past_the_end_do_not_leak(gpu_lib):
    """As above for the rotated-INT2 cache on the tensor cores (NaN scale/zero and
    rope bytes, 0xFF codes in the stale slots)."""
    import mla_latent_kv_08_gb300 as mla
    import torch
    w, R32, T32 = _int2_setup(B=3, H=32, len_range=(40, 300))
    assert np.any(w.seq_lens % 64 != 0)
    shape = gu.shape_for(w, kind=mla.MLA_KV_INT2_ROT, impl=mla.MLA_IMPL_TCGEN05)
    res = []
    for fill in (0.0, float("nan")):
        cache = mla.Cache.allocate(shape, zero=False)
        _pool_fill(cache, fill)
        gu.append_tokens(cache, w, w.latent, w.rope, np.zeros(w.B, np.int32), R32, T32)
        torch.cuda.synchronize()
        res.append(gu.attend(w, shape, cache, w.q, R=R32)[:2])
    (o0, l0), (o1, l1) = res
    assert np.isfinite(o1).all() and np.isfinite(l1).all()
    np.testing.assert_array_equal(o1, o0)
    np.testing.assert_array_equal(l1, l0)


# ------------------------------------------------------------ device checks

def test_bad_block_id_sets_flag_and_nan_rows(gpu_lib):
    import mla_latent_kv_08_gb300 as mla
    w = workloads.dsv3(13, B=3, H=16, len_range=(100, 200))
    shape = gu.shape_for(w)
    cache, _ = gu.fill_cache(w, shape)
    w.block_table = w.block_table.copy()
    w.block_table[1, 0] = w.num_blocks + 5          # out of range for decode only
    out, lse, ws = gu.attend(w, shape, cache, w.q)
    code, flags = mla.mla_get_status(ws)
    assert code == mla.MLA_ERR_BOUNDS and flags & 1
    assert np.all(np.isnan(out[1])) and np.all(np.isnan(lse[1]))
    for b in (0, 2):
        ro, rl = attention.absorbed(w.q[b], w.latent[b], w.rope[b], w.W_UV, w.scale)
        _check_seq(out, lse, w, b, ro, rl, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)


@pytest.mark.parametrize("kind_name", ["rot", "rope"])
def test_int2_bad_block_id_sets_flag_and_nan_rows(gpu_lib, kind_name):
    """The rotated-INT2 tensor-core decode with one out-of-range block id: the flag is
    raised, that sequence's rows are NaN, and the other sequences match the oracle."""
    import mla_latent_kv_08_gb300 as mla
    import torch
    w, R32, T32 = _int2_setup(B=3, H=16, len_range=(100, 200))
    TR32 = _rope_thresholds(12) if kind_name == "rope" else None
    kind = mla.MLA_KV_INT2_ROT if kind_name == "rot" else mla.MLA_KV_INT2_ROT_QR
    shape = gu.shape_for(w, kind=kind, impl=mla.MLA_IMPL_TCGEN05)
    cache, st = gu.fill_cache(w, shape, R32, T32 if kind_name == "rot" else np.concatenate([T32, TR32]))
    torch.cuda.synchronize()
    assert mla.mla_read_status_word(st)[0] == mla.MLA_OK
    w.block_table = w.block_table.copy()
    w.block_table[1, 0] = w.num_blocks + 5          # out of range for decode only
    out, lse, ws = gu.attend(w, shape, cache, w.q, R=R32)
    code, flags = mla.mla_get_status(ws)
    assert code == mla.MLA_ERR_BOUNDS and flags & 1
    assert np.all(np.isnan(out[1])) and np.all(np.isnan(lse[1]))
    for b in (0, 2):
        ro, rl, o_op, l_op = _int2_references(w, w.q[b], b, kind_name, R32, T32, TR32)
        _check_seq(out, lse, w, b, o_op, l_op, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)
        _check_seq(out, lse, w, b, ro, rl, gu.BF16_REL_TOL, 2 * gu.BF16_LSE_TOL)


def test_bad_length_sets_flag(gpu_lib):
    import mla_latent_kv_08_gb300 as mla
    w = workloads.dsv3(14, B=2, H=16, len_range=(100, 120))
    shape = gu.shape_for(w)
    cache, _ = gu.fill_cache(w, shape)
    good = w.seq_lens.copy()
    w.seq_lens = np.array([good[0], w.block_table.shape[1] * 64 + 1], np.int32)
    out, lse, ws = gu.attend(w, shape, cache, w.q)
    code, flags = mla.mla_get_status(ws)
    assert code == mla.MLA_ERR_BOUNDS and flags & 2
    assert np.all(np.isnan(out[1]))
    ro, rl = attention.absorbed(w.q[0], w.latent[0], w.rope[0], w.W_UV, w.scale)
    _check_seq(out, lse, w, 0, ro, rl, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)


def test_host_argument_errors_launch_nothing(gpu_lib):
    import mla_latent_kv_08_gb300 as mla
    import torch
    w = workloads.dsv3(15, B=2, H=16, len_range=(10, 20))
    shape = gu.shape_for(w)
    cache, _ = gu.fill_cache(w, shape)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(mla.MlaError) as e:
        gu_out = torch.empty((2, 1, 16, 128), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((2, 1, 16), dtype=torch.float32, device="cuda")
        mla.mla_decode(cache, gu.dev(w.block_table), gu.dev(w.seq_lens), gu.dev(w.q, torch.bfloat16),
                       gu.dev(w.W_UV, torch.bfloat16), w.scale, gu_out, lse, small)
    assert e.value.code == mla.MLA_ERR_WORKSPACE


# ----------------------------------------------------- tensor-core vs generic

@pytest.mark.parametrize("H,q_len,lens", [(128, 1, (1, 700)), (64, 1, (60, 200)), (128, 4, (4, 300))])
def test_tcgen05_and_simt_agree_with_oracle(gpu_lib, H, q_len, lens):
    import mla_latent_kv_08_gb300 as mla
    w = workloads.dsv3(50 + H + q_len, B=3, H=H, len_range=lens, q_len=q_len)
    res = {}
    for impl in (mla.MLA_IMPL_TCGEN05, mla.MLA_IMPL_SIMT):
        shape = gu.shape_for(w, impl=impl)
        assert mla.mla_resolve_impl(shape, q_len) == impl
        cache, _ = gu.fill_cache(w, shape)
        res[impl] = gu.attend(w, shape, cache, w.q, q_len=q_len)[:2]
    for b in range(w.B):
        ro, rl = attention.absorbed(w.q[b], w.latent[b], w.rope[b], w.W_UV, w.scale)
        for impl, (o, l) in res.items():
            _check_seq(o, l, w, b, ro, rl, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)


def _shorten(w, lens):
    """Cut each sequence of a workload to the given length (its blocks stay valid)."""
    for b, L in enumerate(lens):
        w.seq_lens[b] = L
        w.latent[b], w.rope[b] = w.latent[b][:L], w.rope[b][:L]


@pytest.mark.parametrize("kind_name,q_len", [("bf16", 1), ("bf16", 2), ("int2", 1), ("rope", 1)])
def test_lengths_at_tile_boundaries(gpu_lib, kind_name, q_len):
    """Sequence lengths on both sides of the 64-token tile (and block) boundaries, one
    token, and two tiles and a bit, on the tensor-core kernels: the decode (bf16, rotated
    INT2, rope-INT2) and the paired verify kernel (bf16, q_len 2)."""
    import mla_latent_kv_08_gb300 as mla
    import torch
    lens = [max(q_len, 1), 63, 64, 65, 127, 128, 129, 191]
    if kind_name == "bf16":
        w = workloads.dsv3(77 + q_len, B=len(lens), H=128, len_range=(200, 260), q_len=q_len)
        _shorten(w, lens)
        shape = gu.shape_for(w, impl=mla.MLA_IMPL_TCGEN05)
        cache, _ = gu.fill_cache(w, shape)
        out, lse, ws = gu.attend(w, shape, cache, w.q, q_len=q_len)
        assert mla.mla_get_status(ws)[0] == mla.MLA_OK
        for b in range(w.B):
            ro, rl = attention.absorbed(w.q[b], w.latent[b], w.rope[b], w.W_UV, w.scale)
            _check_seq(out, lse, w, b, ro, rl, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)
        return
    w, R32, T32 = _int2_setup(B=len(lens), H=128, len_range=(200, 260))
    _shorten(w, lens)
    kind = mla.MLA_KV_INT2_ROT if kind_name == "int2" else mla.MLA_KV_INT2_ROT_QR
    T = T32
    if kind_name == "rope":
        rng = np.random.default_rng(12)
        KRcal = workloads.bf16_round(rng.standard_normal((8192, 64)).astype(np.float32)).astype(np.float64)
        TR32 = oint2.rope_thresholds(KRcal).astype(np.float32)
        T = np.concatenate([T32, TR32])
    shape = gu.shape_for(w, kind=kind, impl=mla.MLA_IMPL_TCGEN05)
    cache, st = gu.fill_cache(w, shape, R32, T)
    torch.cuda.synchronize()
    assert mla.mla_read_status_word(st)[0] == mla.MLA_OK
    out, lse, ws = gu.attend(w, shape, cache, w.q, R=R32)
    assert mla.mla_get_status(ws)[0] == mla.MLA_OK
    f16 = lambda x: np.asarray(x, np.float64).astype(np.float16).astype(np.float64)   # noqa: E731
    for b in range(w.B):
        if kind_name == "int2":
            codes, sz = oint2.quantize(w.latent[b], R32, T32)
            K = oint2.decode(codes, sz).astype(np.float64)
            ro, rl = oint2.attention_rotated(w.q[b], K, w.rope[b], R32, w.W_UV, w.scale)
        else:
            codes, sz = oint2.quantize_rope_int2(w.latent[b], w.rope[b], R32, T32, TR32)
            Y = oint2.decode(codes, sz).astype(np.float64)
            ro, rl = oint2.attention_rope_int2(w.q[b], Y, R32, w.W_UV, w.scale)
        if w.seq_lens[b] > 1:
            _check_seq(out, lse, w, b, ro, rl, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)
            continue
        # One token: the LSE is that token's score itself, with no averaging of the
        # fp16 operand roundings of the rotated query and the dequantised key (the INT2
        # kernels' operand type). The kernel must match the score formed from those
        # fp16 operands to the usual bar, and the definition within twice it.
        q = np.asarray(w.q[b], np.float64)[0]                        # [H, r + d_R]
        if kind_name == "int2":
            qk = f16(q[:, :w.r] @ R32.astype(np.float64)) @ f16(K[0, :w.r]) + q[:, w.r:] @ w.rope[b][0].astype(np.float64)
        else:
            qy = np.concatenate([q[:, :w.r] @ R32.astype(np.float64), q[:, w.r:]], axis=1)
            qk = f16(qy) @ f16(Y[0])
        assert float(np.max(np.abs(lse[b, 0] - w.scale * qk))) <= gu.BF16_LSE_TOL
        _check_seq(out, lse, w, b, ro, rl, gu.BF16_REL_TOL, 2 * gu.BF16_LSE_TOL)


def test_auto_picks_tensor_cores_for_dsv3(gpu_lib):
    import mla_latent_kv_08_gb300 as mla
    w = workloads.dsv3(1, B=2, H=128, len_range=(64, 64))
    assert mla.mla_resolve_impl(gu.shape_for(w)) == mla.MLA_IMPL_TCGEN05
    assert mla.mla_resolve_impl(gu.shape_for(w, kind=mla.MLA_KV_FP32)) == mla.MLA_IMPL_SIMT


@pytest.mark.parametrize("impl_name,kind", [("tcgen05", "bf16"), ("simt", "bf16"), ("tcgen05", "int2")])
def test_decode_replays_from_a_cuda_graph(gpu_lib, impl_name, kind):
    """A decode step captured as a CUDA graph (planner, attention and combine kernels
    with their programmatic dependencies) and replayed after the query buffer was
    rewritten in place gives bit-for-bit the eager result for the new query."""
    import torch
    impl = {"tcgen05": gu.mla.MLA_IMPL_TCGEN05, "simt": gu.mla.MLA_IMPL_SIMT}[impl_name]
    R = T = None
    if kind == "int2":
        w, R, T = _int2_setup(B=4, H=128, len_range=(300, 1500))
        shape = gu.shape_for(w, kind=gu.mla.MLA_KV_INT2_ROT, impl=impl)
    else:
        w = workloads.dsv3(4, B=5, H=128, len_range=(300, 1500))
        shape = gu.shape_for(w, impl=impl)
    cache, _ = gu.fill_cache(w, shape, R=R, T=T)
    dt = gu.torch_dtype(w)
    # the second query, rounded to the cache's dtype once so that the oracle sees
    # exactly the values the kernels read
    q2 = gu.dev(np.random.default_rng(44).standard_normal(w.q.shape).astype(np.float32), dt).float().cpu().numpy()
    qd = gu.dev(w.q.astype(np.float32), dt)
    W = gu.dev(w.W_UV.astype(np.float32), dt)
    Rd = None if R is None else gu.dev(R.astype(np.float32))
    bt = gu.dev(w.block_table)
    sl = gu.dev(w.seq_lens.astype(np.int32))
    out = torch.empty((w.B, 1, w.H, w.d_v), dtype=dt, device="cuda")
    lse = torch.empty((w.B, 1, w.H), dtype=torch.float32, device="cuda")
    ws = gu.mla.alloc_workspace(shape, w.B, 1)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        gu.mla.mla_decode(cache, bt, sl, qd, W, w.scale, out, lse, ws, R=Rd, stream=side)
    side.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        gu.mla.mla_decode(cache, bt, sl, qd, W, w.scale, out, lse, ws, R=Rd, stream=side)
    torch.cuda.synchronize()
    # eager reference for the second query
    qd.copy_(gu.dev(q2, dt))
    gu.mla.mla_decode(cache, bt, sl, qd, W, w.scale, out, lse, ws, R=Rd)
    torch.cuda.synchronize()
    ref_o, ref_l = out.clone(), lse.clone()
    out.zero_()
    lse.zero_()
    graph.replay()
    torch.cuda.synchronize()
    code, flags = gu.mla.mla_get_status(ws)
    assert code == gu.mla.MLA_OK, (code, flags)
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
    if kind == "bf16":
        o = out.float().cpu().numpy()
        l = lse.cpu().numpy()
        for b in range(w.B):
            ro, rl = attention.absorbed(q2[b], w.latent[b], w.rope[b], w.W_UV, w.scale)
            _check_seq(o, l, w, b, ro, rl, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)


def test_tensor_core_decode_with_the_generic_combine(gpu_lib):
    """d_v = 64: the tensor-core decode (bf16 split partials) feeds the CUDA-core
    combine, which reads them in that format."""
    import dataclasses
    import mla_latent_kv_08_gb300 as mla
    w = workloads.dsv3(9, B=4, H=128, len_range=(200, 2500))
    w = dataclasses.replace(w, W_UV=np.ascontiguousarray(w.W_UV[:, :, :64]), d_v=64)
    shape = gu.shape_for(w, impl=mla.MLA_IMPL_TCGEN05)
    assert mla.mla_resolve_impl(shape) == mla.MLA_IMPL_TCGEN05
    cache, _ = gu.fill_cache(w, shape)
    out, lse, ws = gu.attend(w, shape, cache, w.q)
    assert mla.mla_get_status(ws)[0] == mla.MLA_OK
    for b in range(w.B):
        ro, rl = attention.absorbed(w.q[b], w.latent[b], w.rope[b], w.W_UV, w.scale)
        _check_seq(out, lse, w, b, ro, rl, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)


@pytest.mark.parametrize("kind_name,impl_name,q_len",
                         [("rot", "tcgen05", 2), ("rot", "tcgen05", 5), ("rope", "tcgen05", 3), ("rot", "simt", 3)])
def test_int2_verify_causal_window(gpu_lib, kind_name, impl_name, q_len):
    """Speculative verify on the rotated-INT2 caches: q_len draft rows a sequence, row i
    seeing positions 0 .. L - q_len + i, against the oracle's attention over the
    dequantised rows. At H = 128 a sequence's rows span several 128-row tiles, and
    sequence 0 holds exactly q_len tokens, so that its first row sees a single one."""
    import mla_latent_kv_08_gb300 as mla
    import torch
    w, R32, T32 = _int2_setup(B=3, H=128, len_range=(q_len, 700))
    w.seq_lens[0] = q_len
    w.latent[0], w.rope[0] = w.latent[0][:q_len], w.rope[0][:q_len]
    rng = np.random.default_rng(40 + q_len)
    q = workloads.bf16_round(rng.standard_normal((w.B, q_len, w.H, w.r + w.d_rope)).astype(np.float32))
    impl = mla.MLA_IMPL_SIMT if impl_name == "simt" else mla.MLA_IMPL_TCGEN05
    if kind_name == "rot":
        shape = gu.shape_for(w, kind=mla.MLA_KV_INT2_ROT, impl=impl)
        cache, st = gu.fill_cache(w, shape, R32, T32)
    else:
        KRcal = workloads.bf16_round(rng.standard_normal((8192, 64)).astype(np.float32)).astype(np.float64)
        TR32 = oint2.rope_thresholds(KRcal).astype(np.float32)
        shape = gu.shape_for(w, kind=mla.MLA_KV_INT2_ROT_QR, impl=impl)
        cache, st = gu.fill_cache(w, shape, R32, np.concatenate([T32, TR32]))
    assert mla.mla_resolve_impl(shape) == impl
    torch.cuda.synchronize()
    assert mla.mla_read_status_word(st)[0] == mla.MLA_OK
    out, lse, ws = gu.attend(w, shape, cache, q, R=R32, q_len=q_len)
    assert mla.mla_get_status(ws)[0] == mla.MLA_OK
    for b in range(w.B):
        ro, rl, o_op, l_op = _int2_references(w, q[b], b, kind_name, R32, T32, TR32 if kind_name == "rope" else None)
        if impl_name == "simt":
            _check_seq(out, lse, w, b, ro, rl, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)
            continue
        # Rows whose softmax sits on a few tokens see the fp16 roundings of the rotated
        # query and of the dequantised key (the tensor-core operand type of these kinds)
        # with little averaging, as a single token does. The kernel must match the
        # attention formed from those same operands (in fp64) to the usual bars, and the
        # definition within twice the LSE bar.
        _check_seq(out, lse, w, b, o_op, l_op, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)
        _check_seq(out, lse, w, b, ro, rl, gu.BF16_REL_TOL, 2 * gu.BF16_LSE_TOL)


def _int2_references(w, qb, b, kind_name, R32, T32, TR32=None):
    """Sequence b against the oracle: the definition over the oracle's dequantised codes
    (ro, rl), and the same attention formed in fp64 from the tensor-core kernel's operands
    (o_op, l_op): q.R and the dequantised key rounded to fp16 (INT2_ROT's rope dims bf16
    on both sides as given; INT2_ROT_QR's rope dims fp16 like the rest)."""
    f16 = lambda x: np.asarray(x, np.float64).astype(np.float16).astype(np.float64)   # noqa: E731
    R64 = R32.astype(np.float64)
    q64 = np.asarray(qb, np.float64)
    if kind_name == "rot":
        codes, sz = oint2.quantize(w.latent[b], R32, T32)
        K = oint2.decode(codes, sz).astype(np.float64)
        ro, rl = oint2.attention_rotated(qb, K, w.rope[b], R32, w.W_UV, w.scale)
        q_op = np.concatenate([f16(q64[..., :w.r] @ R64), q64[..., w.r:]], axis=-1)
        C_op, KR_op = f16(K), w.rope[b]
    else:
        codes, sz = oint2.quantize_rope_int2(w.latent[b], w.rope[b], R32, T32, TR32)
        Y = oint2.decode(codes, sz).astype(np.float64)
        ro, rl = oint2.attention_rope_int2(qb, Y, R32, w.W_UV, w.scale)
        q_op = f16(np.concatenate([q64[..., :w.r] @ R64, q64[..., w.r:]], axis=-1))
        C_op, KR_op = f16(Y[:, :w.r]), f16(Y[:, w.r:])
    _, l_op, o_rot = attention.absorbed(q_op, C_op, KR_op, np.zeros((w.H, w.r, 1)), w.scale, return_latent=True)
    o_op = np.einsum("qhr,hrv->qhv", o_rot @ R64.T, np.asarray(w.W_UV, np.float64))
    return ro, rl, o_op, l_op


def _rope_thresholds(seed):
    rng = np.random.default_rng(seed)
    KRcal = workloads.bf16_round(rng.standard_normal((8192, 64)).astype(np.float32)).astype(np.float64)
    return oint2.rope_thresholds(KRcal).astype(np.float32)


@pytest.mark.parametrize("kind_name", ["rot", "rope"])
def test_int2_split_count_does_not_change_result(gpu_lib, kind_name):
    """The rotated-INT2 tensor-core decode with the sequences cut 1, 7 and 200 ways
    (different work items over the 64-token tiles, merged by the combine): the same LSE
    to 1e-5 and the same output to the bf16 rounding of the split partials; and sequence
    0 against the oracle as in the INT2 verify test."""
    import mla_latent_kv_08_gb300 as mla
    import torch
    w, R32, T32 = _int2_setup(B=3, H=64, len_range=(2000, 3000))
    TR32 = _rope_thresholds(12) if kind_name == "rope" else None
    kind = mla.MLA_KV_INT2_ROT if kind_name == "rot" else mla.MLA_KV_INT2_ROT_QR
    T = T32 if kind_name == "rot" else np.concatenate([T32, TR32])
    res = []
    for hint in (1, 7, 200):
        shape = gu.shape_for(w, kind=kind, impl=mla.MLA_IMPL_TCGEN05, splits=hint)
        cache, st = gu.fill_cache(w, shape, R32, T)
        torch.cuda.synchronize()
        assert mla.mla_read_status_word(st)[0] == mla.MLA_OK
        res.append(gu.attend(w, shape, cache, w.q, R=R32)[:2])
    for o, l in res[1:]:
        assert np.max(np.abs(l - res[0][1])) < 1e-5
        assert gu.rel_err(o, res[0][0]) < 8e-3      # bf16 output rounding of near-equal fp32 values
    ro, rl, o_op, l_op = _int2_references(w, w.q[0], 0, kind_name, R32, T32, TR32)
    _check_seq(res[2][0], res[2][1], w, 0, o_op, l_op, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)
    _check_seq(res[2][0], res[2][1], w, 0, ro, rl, gu.BF16_REL_TOL, 2 * gu.BF16_LSE_TOL)


@pytest.mark.parametrize("impl_name,H", [("simt", 32), ("tcgen05", 32), ("tcgen05", 128)])
def test_int2_rope_codes_append_and_decode(gpu_lib, impl_name, H):
    """INT2_ROT_QR (the rope key quantised as two more INT2 groups): codes and
    scale/zero of every appended token bit-exact against the oracle's encoding, and the
    decode against the oracle's attention over the dequantised rows."""
    import mla_latent_kv_08_gb300 as mla
    import torch
    w, R32, T32 = _int2_setup(B=4, H=H, len_range=(40, 300))
    rng = np.random.default_rng(12)
    KRcal = workloads.bf16_round(rng.standard_normal((8192, 64)).astype(np.float32)).astype(np.float64)
    TR32 = oint2.rope_thresholds(KRcal).astype(np.float32)
    impl = mla.MLA_IMPL_SIMT if impl_name == "simt" else mla.MLA_IMPL_TCGEN05
    shape = gu.shape_for(w, kind=mla.MLA_KV_INT2_ROT_QR, impl=impl)
    assert mla.mla_resolve_impl(shape) == impl
    cache = mla.Cache.allocate(shape)
    assert cache.rope is None and cache.bytes_per_token() == 216
    Tall = np.concatenate([T32, TR32])
    st0 = gu.append_tokens(cache, w, w.latent, w.rope, np.zeros(w.B, np.int32), R32, Tall)
    st1 = gu.append_tokens(cache, w, w.new_latent, w.new_rope, w.start_pos, R32, Tall)
    torch.cuda.synchronize()
    assert mla.mla_read_status_word(st0)[0] == mla.MLA_OK and mla.mla_read_status_word(st1)[0] == mla.MLA_OK
    ref = []
    for b in range(w.B):
        C = np.concatenate([w.latent[b], w.new_latent[b]])
        KR = np.concatenate([w.rope[b], w.new_rope[b]])
        ref.append(oint2.quantize_rope_int2(C, KR, R32, T32, TR32))
    nb = w.num_blocks
    ref_codes = layout.write_paged(nb, 64, 144, w.block_table, [x[0] for x in ref], [0] * w.B, np.uint8)
    ref_sz = layout.write_paged(nb, 64, 36, w.block_table, [x[1].reshape(-1, 36) for x in ref], [0] * w.B, np.uint16)
    np.testing.assert_array_equal(cache.codes.cpu().numpy(), ref_codes)
    np.testing.assert_array_equal(cache.scale_zero.cpu().view(torch.int16).numpy().view(np.uint16).reshape(nb, 64, 36),
                                  ref_sz)
    w.seq_lens = (w.seq_lens + 32).astype(np.int32)
    out, lse, ws = gu.attend(w, shape, cache, w.q, R=R32)
    assert mla.mla_get_status(ws)[0] == mla.MLA_OK
    for b in range(w.B):
        Y = oint2.decode(ref[b][0], ref[b][1]).astype(np.float64)
        ro, rl = oint2.attention_rope_int2(w.q[b], Y, R32, w.W_UV, w.scale)
        _check_seq(out, lse, w, b, ro, rl, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)


# ------------------------------------------------------------ folded output rotation

def test_fold_rotation_matches_the_definition(gpu_lib):
    """W_folded[h] = R^T . W_UV[h], rounded once to bf16: every element within one bf16
    rounding (plus fp32 accumulation) of the fp64 product."""
    import mla_latent_kv_08_gb300 as mla
    import torch
    rng = np.random.default_rng(3)
    H, r, dv = 8, 512, 128
    R = workloads.haar_orthogonal(np.random.Generator(np.random.PCG64(9)), r).astype(np.float32)
    W = workloads.bf16_round(rng.standard_normal((H, r, dv)).astype(np.float32) / math.sqrt(r))
    shape = mla.Shape(num_heads=H, kv_lora_rank=r, rope_dim=64, v_head_dim=dv, block_size=64, num_blocks=1,
                      kind=mla.MLA_KV_INT2_ROT)
    Wf = torch.empty((H, r, dv), dtype=torch.bfloat16, device="cuda")
    mla.mla_fold_rotation(shape, gu.dev(R), gu.dev(W, torch.bfloat16), Wf)
    torch.cuda.synchronize()
    ref = np.einsum("ki,hkj->hij", R.astype(np.float64), W.astype(np.float64))
    got = Wf.float().cpu().numpy()
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)


@pytest.mark.parametrize("kind_name,impl_name,H", [("rot", "tcgen05", 128), ("rot", "simt", 32),
                                                   ("rope", "tcgen05", 128), ("rope", "simt", 32)])
def test_int2_decode_with_folded_up_projection(gpu_lib, kind_name, impl_name, H):
    """MLA_FLAG_WUV_FOLDED: the decode with W'_UV = R^T . W_UV (no o . R^T per call)
    matches the oracle, which rotates back and up-projects in fp64."""
    import mla_latent_kv_08_gb300 as mla
    import torch
    w, R32, T32 = _int2_setup(B=3, H=H, len_range=(60, 700))
    kind = mla.MLA_KV_INT2_ROT if kind_name == "rot" else mla.MLA_KV_INT2_ROT_QR
    impl = mla.MLA_IMPL_SIMT if impl_name == "simt" else mla.MLA_IMPL_TCGEN05
    T = T32
    if kind_name == "rope":
        rng = np.random.default_rng(12)
        KRcal = workloads.bf16_round(rng.standard_normal((8192, 64)).astype(np.float32)).astype(np.float64)
        TR32 = oint2.rope_thresholds(KRcal).astype(np.float32)
        T = np.concatenate([T32, TR32])
    shape = gu.shape_for(w, kind=kind, impl=impl)
    cache, st = gu.fill_cache(w, shape, R32, T)
    torch.cuda.synchronize()
    assert mla.mla_read_status_word(st)[0] == mla.MLA_OK
    Wf = torch.empty((w.H, w.r, w.d_v), dtype=torch.bfloat16, device="cuda")
    mla.mla_fold_rotation(shape, gu.dev(R32), gu.dev(w.W_UV, torch.bfloat16), Wf)
    fshape = gu.shape_for(w, kind=kind, impl=impl)
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
    for b in range(w.B):
        if kind_name == "rot":
            codes, sz = oint2.quantize(w.latent[b], R32, T32)
            ro, rl = oint2.attention_rotated(w.q[b], oint2.decode(codes, sz), w.rope[b], R32, w.W_UV, w.scale)
        else:
            codes, sz = oint2.quantize_rope_int2(w.latent[b], w.rope[b], R32, T32, TR32)
            Y = oint2.decode(codes, sz).astype(np.float64)
            ro, rl = oint2.attention_rope_int2(w.q[b], Y, R32, w.W_UV, w.scale)
        _check_seq(o, l, w, b, ro, rl, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)


@pytest.mark.parametrize("kind_name,impl_name,H,fold", [("rot", "tcgen05", 128, True), ("rot", "simt", 32, True),
                                                        ("rope", "tcgen05", 128, True), ("rope", "simt", 32, True),
                                                        ("rot", "tcgen05", 64, False), ("rope", "simt", 32, False)])
def test_int2_decode_with_query_given_rotated(gpu_lib, kind_name, impl_name, H, fold):
    """MLA_FLAG_Q_ROTATED: the caller passes q with its latent dims already in the
    rotated basis (bf16(q_lat . R)); with W_UV folded too, R is not passed at all. The
    oracle gets the same query expressed back in the unrotated basis (q_rot . R^T, fp64),
    so that its own q . R reproduces the caller's rotated dims."""
    import mla_latent_kv_08_gb300 as mla
    import torch
    w, R32, T32 = _int2_setup(B=3, H=H, len_range=(60, 700))
    kind = mla.MLA_KV_INT2_ROT if kind_name == "rot" else mla.MLA_KV_INT2_ROT_QR
    impl = mla.MLA_IMPL_SIMT if impl_name == "simt" else mla.MLA_IMPL_TCGEN05
    T = T32
    if kind_name == "rope":
        rng = np.random.default_rng(12)
        KRcal = workloads.bf16_round(rng.standard_normal((8192, 64)).astype(np.float32)).astype(np.float64)
        TR32 = oint2.rope_thresholds(KRcal).astype(np.float32)
        T = np.concatenate([T32, TR32])
    shape = gu.shape_for(w, kind=kind, impl=impl)
    cache, st = gu.fill_cache(w, shape, R32, T)
    torch.cuda.synchronize()
    assert mla.mla_read_status_word(st)[0] == mla.MLA_OK
    r = w.r
    q_rot = np.array(w.q, dtype=np.float64)
    q_rot[..., :r] = workloads.bf16_round((q_rot[..., :r] @ R32.astype(np.float64)).astype(np.float32))
    q_back = q_rot.copy()
    q_back[..., :r] = q_rot[..., :r] @ R32.astype(np.float64).T
    W = gu.dev(w.W_UV, torch.bfloat16)
    fshape = gu.shape_for(w, kind=kind, impl=impl)
    fshape.flags = mla.MLA_FLAG_Q_ROTATED
    if fold:
        fshape.flags |= mla.MLA_FLAG_WUV_FOLDED
        Wf = torch.empty((w.H, w.r, w.d_v), dtype=torch.bfloat16, device="cuda")
        mla.mla_fold_rotation(shape, gu.dev(R32), W, Wf)
        W = Wf
    out = torch.empty((w.B, 1, w.H, w.d_v), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, 1, w.H), dtype=torch.float32, device="cuda")
    ws = mla.alloc_workspace(fshape, w.B, 1)
    mla.mla_decode(cache, gu.dev(w.block_table), gu.dev(w.seq_lens.astype(np.int32)),
                   gu.dev(q_rot.astype(np.float32), torch.bfloat16), W, w.scale, out, lse, ws,
                   R=None if fold else gu.dev(R32), shape=fshape)
    torch.cuda.synchronize()
    assert mla.mla_get_status(ws)[0] == mla.MLA_OK
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    for b in range(w.B):
        if kind_name == "rot":
            codes, sz = oint2.quantize(w.latent[b], R32, T32)
            ro, rl = oint2.attention_rotated(q_back[b], oint2.decode(codes, sz), w.rope[b], R32, w.W_UV, w.scale)
        else:
            codes, sz = oint2.quantize_rope_int2(w.latent[b], w.rope[b], R32, T32, TR32)
            Y = oint2.decode(codes, sz).astype(np.float64)
            ro, rl = oint2.attention_rope_int2(q_back[b], Y, R32, w.W_UV, w.scale)
        _check_seq(o, l, w, b, ro, rl, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)


# ------------------------------------------------------------ joint rope/nope kind

@pytest.mark.parametrize("H", [32, 128])
def test_int2_joint_codes_append_and_decode(gpu_lib, H):
    """INT2_JOINT ([c ; k_R] rotated by one 576-dim eigenbasis, 18 INT2 groups): the
    appended codes and scale/zero of every token bit-exact against the oracle's
    encoding (the fp32 rotation chain over all 576 inputs), and the decode against the
    oracle's joint attention over the dequantised rows."""
    import mla_latent_kv_08_gb300 as mla
    import torch
    w, _, _ = _int2_setup(B=3, H=H, len_range=(40, 300))
    rng = np.random.default_rng(12)
    KRcal = workloads.bf16_round(rng.standard_normal((w.calib.shape[0], 64)).astype(np.float32)).astype(np.float64)
    Xj = np.concatenate([w.calib, KRcal], axis=1)
    Rj, _ = oint2.fit_rotation(Xj)
    Tj = oint2.clip_thresholds(Xj, Rj)
    Rj32, Tj32 = Rj.astype(np.float32), Tj.astype(np.float32)
    shape = gu.shape_for(w, kind=mla.MLA_KV_INT2_JOINT)
    assert mla.mla_resolve_impl(shape) == mla.MLA_IMPL_SIMT
    cache = mla.Cache.allocate(shape)
    assert cache.rope is None and cache.bytes_per_token() == 216
    st0 = gu.append_tokens(cache, w, w.latent, w.rope, np.zeros(w.B, np.int32), Rj32, Tj32)
    st1 = gu.append_tokens(cache, w, w.new_latent, w.new_rope, w.start_pos, Rj32, Tj32)
    torch.cuda.synchronize()
    assert mla.mla_read_status_word(st0)[0] == mla.MLA_OK and mla.mla_read_status_word(st1)[0] == mla.MLA_OK
    ref = []
    for b in range(w.B):
        K = np.concatenate([np.concatenate([w.latent[b], w.new_latent[b]]),
                            np.concatenate([w.rope[b], w.new_rope[b]])], axis=1)
        ref.append(oint2.quantize(K, Rj32, Tj32))
    nb = w.num_blocks
    ref_codes = layout.write_paged(nb, 64, 144, w.block_table, [x[0] for x in ref], [0] * w.B, np.uint8)
    ref_sz = layout.write_paged(nb, 64, 36, w.block_table, [x[1].reshape(-1, 36) for x in ref], [0] * w.B, np.uint16)
    np.testing.assert_array_equal(cache.codes.cpu().numpy(), ref_codes)
    np.testing.assert_array_equal(cache.scale_zero.cpu().view(torch.int16).numpy().view(np.uint16).reshape(nb, 64, 36),
                                  ref_sz)
    w.seq_lens = (w.seq_lens + 32).astype(np.int32)
    out, lse, ws = gu.attend(w, shape, cache, w.q, R=Rj32)
    assert mla.mla_get_status(ws)[0] == mla.MLA_OK
    for b in range(w.B):
        Y = oint2.decode(ref[b][0], ref[b][1]).astype(np.float64)
        ro, rl = oint2.attention_joint(w.q[b], Y, Rj32, w.W_UV, w.scale)
        _check_seq(out, lse, w, b, ro, rl, gu.BF16_REL_TOL, gu.BF16_LSE_TOL)
