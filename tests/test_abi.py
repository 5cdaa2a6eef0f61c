"""The C-ABI library: it builds for sm_103a, loads without a GPU, exports every
symbol include/mla.h declares, and its host-side checks reject bad arguments
before anything is launched. No compute call is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from mla_latent_kv_08_gb300 import build
    build.build()
    import mla_latent_kv_08_gb300 as mla
    return mla.load_library()


def _declared():
    src = open(os.path.join(ROOT, "include", "mla.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    import mla_latent_kv_08_gb300 as mla
    names = _declared()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(mla.EXPORTED) == names


def test_status_strings_and_version(lib):
    import mla_latent_kv_08_gb300 as mla
    assert mla.mla_version() == 104
    for code in range(-6, 1):
        assert mla.status_string(code) != "unknown status"
    assert mla.status_string(-99) == "unknown status"


def _shape(**kw):
    import mla_latent_kv_08_gb300 as mla
    base = dict(num_heads=128, kv_lora_rank=512, rope_dim=64, v_head_dim=128, block_size=64, num_blocks=10)
    base.update(kw)
    return mla.Shape(**base)


def test_shape_validation(lib):
    import mla_latent_kv_08_gb300 as mla
    assert mla.mla_resolve_impl(_shape()) in (mla.MLA_IMPL_SIMT, mla.MLA_IMPL_TCGEN05)
    assert mla.mla_resolve_impl(_shape(kv_lora_rank=500)) == mla.MLA_ERR_INVALID
    assert mla.mla_resolve_impl(_shape(rope_dim=7)) == mla.MLA_ERR_INVALID
    assert mla.mla_resolve_impl(_shape(kind=7)) == mla.MLA_ERR_INVALID
    assert mla.mla_resolve_impl(_shape(kind=mla.MLA_KV_INT2_ROT, group_size=6)) == mla.MLA_ERR_INVALID
    assert mla.mla_resolve_impl(_shape(kv_lora_rank=2048)) == mla.MLA_ERR_UNSUPPORTED
    assert mla.mla_resolve_impl(_shape(), q_len=0) == mla.MLA_ERR_INVALID
    # flags: MLA_FLAG_WUV_FOLDED and MLA_FLAG_Q_ROTATED, for the rotated INT2 kinds only
    both = mla.MLA_FLAG_WUV_FOLDED | mla.MLA_FLAG_Q_ROTATED
    assert mla.mla_resolve_impl(_shape(flags=4)) == mla.MLA_ERR_INVALID
    assert mla.mla_resolve_impl(_shape(kind=mla.MLA_KV_INT2_ROT, flags=4)) == mla.MLA_ERR_INVALID
    assert mla.mla_resolve_impl(_shape(flags=mla.MLA_FLAG_WUV_FOLDED)) == mla.MLA_ERR_INVALID
    assert mla.mla_resolve_impl(_shape(flags=mla.MLA_FLAG_Q_ROTATED)) == mla.MLA_ERR_INVALID
    assert mla.mla_resolve_impl(_shape(kind=mla.MLA_KV_INT2_ROT, flags=mla.MLA_FLAG_WUV_FOLDED)) >= 0
    assert mla.mla_resolve_impl(_shape(kind=mla.MLA_KV_INT2_ROT, flags=mla.MLA_FLAG_Q_ROTATED)) >= 0
    assert mla.mla_resolve_impl(_shape(kind=mla.MLA_KV_INT2_ROT_QR, flags=both)) >= 0
    # the joint rope/nope kind: generic kernel only, no folded up-projection, whole row in groups
    joint = mla.MLA_KV_INT2_JOINT
    assert mla.mla_resolve_impl(_shape(kind=joint)) == mla.MLA_IMPL_SIMT
    assert mla.mla_resolve_impl(_shape(kind=joint, impl=mla.MLA_IMPL_TCGEN05)) == mla.MLA_ERR_UNSUPPORTED
    assert mla.mla_resolve_impl(_shape(kind=joint, flags=mla.MLA_FLAG_WUV_FOLDED)) == mla.MLA_ERR_INVALID
    assert mla.mla_resolve_impl(_shape(kind=joint, flags=mla.MLA_FLAG_Q_ROTATED)) == mla.MLA_ERR_INVALID
    assert mla.mla_resolve_impl(_shape(kind=joint, rope_dim=48)) == mla.MLA_ERR_INVALID
    # the extra per-token key: a multiple of 8 up to 1024, BF16/FP32 kinds only
    assert mla.mla_resolve_impl(_shape(index_dim=64)) in (mla.MLA_IMPL_SIMT, mla.MLA_IMPL_TCGEN05)
    assert mla.mla_resolve_impl(_shape(index_dim=12)) == mla.MLA_ERR_INVALID
    assert mla.mla_resolve_impl(_shape(index_dim=2048)) == mla.MLA_ERR_INVALID
    assert mla.mla_resolve_impl(_shape(kind=mla.MLA_KV_INT2_ROT, index_dim=64)) == mla.MLA_ERR_INVALID
    # the rope key as INT2 groups: d_R a multiple of the group size; both kernels
    assert mla.mla_resolve_impl(_shape(kind=mla.MLA_KV_INT2_ROT_QR)) == mla.MLA_IMPL_TCGEN05
    assert mla.mla_resolve_impl(_shape(kind=mla.MLA_KV_INT2_ROT_QR, impl=mla.MLA_IMPL_SIMT)) == mla.MLA_IMPL_SIMT
    assert mla.mla_resolve_impl(_shape(kind=mla.MLA_KV_INT2_ROT_QR, rope_dim=48)) == mla.MLA_ERR_INVALID
    assert mla.mla_resolve_impl(_shape(kind=mla.MLA_KV_INT2_ROT_QR, index_dim=64)) == mla.MLA_ERR_INVALID
    # the generic kernel takes any supported shape, e.g. the tiny fp32 one
    assert mla.mla_resolve_impl(_shape(num_heads=8, kv_lora_rank=64, rope_dim=16, v_head_dim=32,
                                       block_size=256, kind=mla.MLA_KV_FP32)) == mla.MLA_IMPL_SIMT


def test_workspace_size_scales(lib):
    import mla_latent_kv_08_gb300 as mla
    a = mla.mla_workspace_bytes(_shape(), 32, 1)
    b = mla.mla_workspace_bytes(_shape(), 32, 8)
    assert 0 < a < b
    with pytest.raises(mla.MlaError):
        mla.mla_workspace_bytes(_shape(kv_lora_rank=7), 32, 1)


def test_null_arguments_rejected_before_launch(lib):
    import mla_latent_kv_08_gb300 as mla
    s = _shape().c()
    cache = mla.mla_cache(None, None, None, None)
    rc = lib.mla_decode(ctypes.byref(s), ctypes.byref(cache), None, 4, None, 2, None, None, None,
                        ctypes.c_float(0.1), None, None, None, 0, None)
    assert rc == mla.MLA_ERR_INVALID
    rc = lib.mla_verify(ctypes.byref(s), ctypes.byref(cache), None, 4, None, 2, 3, None, None, None,
                        ctypes.c_float(0.1), None, None, None, 0, None)
    assert rc == mla.MLA_ERR_INVALID
    rc = lib.mla_latent_append(ctypes.byref(s), ctypes.byref(cache), None, 4, 2, None, None, 5, None, None,
                               None, None, None, None)
    assert rc == mla.MLA_ERR_INVALID
    rc = lib.mla_decode(None, ctypes.byref(cache), None, 4, None, 2, None, None, None,
                        ctypes.c_float(0.1), None, None, None, 0, None)
    assert rc == mla.MLA_ERR_INVALID
    # append then decode: either part's missing arguments are refused before any launch
    rc = lib.mla_append_decode(ctypes.byref(s), ctypes.byref(cache), None, 4, 2, None, None, 5, None, None,
                               None, None, None, None, None, None, ctypes.c_float(0.1), None, None, None, 0, None)
    assert rc == mla.MLA_ERR_INVALID
    assert lib.mla_get_status(None, None, None) == mla.MLA_ERR_INVALID


def test_selftest_arguments_checked_before_launch(lib):
    import mla_latent_kv_08_gb300 as mla
    fake = ctypes.c_void_p(16)                     # never dereferenced: the arguments are refused first
    assert lib.mla_selftest_wait_timeout(ctypes.c_uint64(2_000_000), None, None) == mla.MLA_ERR_INVALID
    assert lib.mla_selftest_wait_timeout(ctypes.c_uint64(10), fake, None) == mla.MLA_ERR_INVALID
    assert lib.mla_selftest_wait_timeout(ctypes.c_uint64(10 ** 9), fake, None) == mla.MLA_ERR_INVALID


def test_index_append_refused_without_an_index_field(lib):
    import mla_latent_kv_08_gb300 as mla
    cache = mla.mla_cache(None, None, None, None)
    fake = ctypes.c_void_p(256)                    # never dereferenced: refused before launch
    s0 = _shape().c()                              # index_dim 0
    assert lib.mla_latent_append_index(ctypes.byref(s0), ctypes.byref(cache), fake, 4, 2, fake, fake, 3, fake,
                                       None, None) == mla.MLA_ERR_INVALID
    s1 = _shape(index_dim=64).c()                  # no cache pointer
    assert lib.mla_latent_append_index(ctypes.byref(s1), ctypes.byref(cache), fake, 4, 2, fake, fake, 3, fake,
                                       None, None) == mla.MLA_ERR_INVALID


def test_cache_layout_bytes_per_kind():
    """The binding allocates each cache kind as the header lays it out, and its per-token
    footprint is the documented one (DeepSeek-V3 shape): bf16 1152 B, fp32 2304 B,
    rotated INT2 with a bf16 rope key 320 B, and with the rope key as INT2 too 216 B."""
    import mla_latent_kv_08_gb300 as mla
    nb, bs = 3, 64
    expect = {mla.MLA_KV_BF16: 1152, mla.MLA_KV_FP32: 2304, mla.MLA_KV_INT2_ROT: 320, mla.MLA_KV_INT2_ROT_QR: 216}
    for kind, per_token in expect.items():
        cache = mla.Cache.allocate(_shape(kind=kind, num_blocks=nb, block_size=bs), device="cpu")
        assert cache.bytes_per_token() == per_token
        parts = [x for x in (cache.latent, cache.codes, cache.scale_zero, cache.rope) if x is not None]
        assert sum(x.numel() * x.element_size() for x in parts) == per_token * nb * bs
    qr = mla.Cache.allocate(_shape(kind=mla.MLA_KV_INT2_ROT_QR, num_blocks=nb, block_size=bs), device="cpu")
    assert qr.rope is None and tuple(qr.codes.shape) == (nb, bs, 144) and tuple(qr.scale_zero.shape) == (nb, bs, 18, 2)


def test_fold_rotation_argument_checks(lib):
    """mla_fold_rotation refuses non-INT2 kinds, null pointers and in-place output
    before launching anything."""
    import mla_latent_kv_08_gb300 as mla
    buf = ctypes.create_string_buffer(64)
    p = ctypes.cast(buf, ctypes.c_void_p)
    q = ctypes.cast(ctypes.create_string_buffer(64), ctypes.c_void_p)
    int2 = _shape(kind=mla.MLA_KV_INT2_ROT)
    assert lib.mla_fold_rotation(ctypes.byref(_shape().c()), p, p, q, None) == mla.MLA_ERR_INVALID
    assert lib.mla_fold_rotation(ctypes.byref(int2.c()), None, p, q, None) == mla.MLA_ERR_INVALID
    assert lib.mla_fold_rotation(ctypes.byref(int2.c()), p, p, None, None) == mla.MLA_ERR_INVALID
    assert lib.mla_fold_rotation(ctypes.byref(int2.c()), p, q, q, None) == mla.MLA_ERR_INVALID
