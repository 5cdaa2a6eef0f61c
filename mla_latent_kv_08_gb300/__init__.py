"""Python binding of the GB300 MLA latent-cache decode library (libmla_gb300.so).

Argument marshalling only: every step of append, decode and verify runs in the
library's CUDA kernels. PyTorch provides device memory and streams. The C ABI
is declared in ``include/mla.h``; the functions here carry the same names.

The library must be built (``python -m mla_latent_kv_08_gb300.build`` or
``__graft_entry__.build()``); importing this package never falls back to
anything else when it is missing.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmla_gb300.so")

MLA_OK = 0
MLA_ERR_INVALID = -1
MLA_ERR_UNSUPPORTED = -2
MLA_ERR_BOUNDS = -3
MLA_ERR_WORKSPACE = -4
MLA_ERR_CUDA = -5
MLA_ERR_TIMEOUT = -6

MLA_KV_BF16 = 0
MLA_KV_FP32 = 1
MLA_KV_INT2_ROT = 2
MLA_KV_INT2_ROT_QR = 3
MLA_KV_INT2_JOINT = 4

MLA_IMPL_AUTO = 0
MLA_IMPL_SIMT = 1
MLA_IMPL_TCGEN05 = 2
MLA_FLAG_WUV_FOLDED = 1
MLA_FLAG_Q_ROTATED = 2
MLA_DTYPE_F64, MLA_DTYPE_F32, MLA_DTYPE_BF16 = 0, 1, 2

# Every symbol include/mla.h declares.
EXPORTED = (
    "mla_workspace_bytes", "mla_latent_append", "mla_decode", "mla_verify", "mla_get_status",
    "mla_read_status_word", "mla_status_string", "mla_resolve_impl", "mla_version",
    "mla_profile_enable", "mla_profile_read", "mla_decode_noalloc", "mla_selftest_wait_timeout",
    "mla_latent_append_index", "mla_fold_rotation", "mla_append_decode",
    "mla_calib_covariance", "mla_calib_projection_energy", "mla_calib_eigh", "mla_calib_eigh_weighted",
    "mla_calib_project_abs", "mla_calib_thresholds",
)


class MlaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


class mla_shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_heads", "kv_lora_rank", "rope_dim", "v_head_dim", "block_size", "num_blocks",
        "group_size", "kind", "impl", "num_splits_hint", "index_dim", "flags")]


class mla_cache(ctypes.Structure):
    _fields_ = [("latent", ctypes.c_void_p), ("codes", ctypes.c_void_p),
                ("scale_zero", ctypes.c_void_p), ("rope", ctypes.c_void_p)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmla_gb300.so and declare its signatures. Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -m mla_latent_kv_08_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    sp = ctypes.POINTER(mla_shape)
    cp = ctypes.POINTER(mla_cache)
    i32p = ctypes.POINTER(ctypes.c_int32)
    lib.mla_workspace_bytes.argtypes = [sp, i32, i32]
    lib.mla_workspace_bytes.restype = sz
    lib.mla_latent_append.argtypes = [sp, cp, vp, i32, i32, vp, vp, i32, vp, vp, vp, vp, vp, vp]
    lib.mla_latent_append.restype = i32
    lib.mla_latent_append_index.argtypes = [sp, cp, vp, i32, i32, vp, vp, i32, vp, vp, vp]
    lib.mla_latent_append_index.restype = i32
    lib.mla_decode.argtypes = [sp, cp, vp, i32, vp, i32, vp, vp, vp, ctypes.c_float, vp, vp, vp, sz, vp]
    lib.mla_append_decode.argtypes = [sp, cp, vp, i32, i32, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                      ctypes.c_float, vp, vp, vp, sz, vp]
    lib.mla_append_decode.restype = i32
    lib.mla_decode.restype = i32
    lib.mla_verify.argtypes = [sp, cp, vp, i32, vp, i32, i32, vp, vp, vp, ctypes.c_float, vp, vp, vp, sz, vp]
    lib.mla_verify.restype = i32
    lib.mla_get_status.argtypes = [vp, i32p, vp]
    lib.mla_get_status.restype = i32
    lib.mla_read_status_word.argtypes = [vp, i32p, vp]
    lib.mla_read_status_word.restype = i32
    lib.mla_status_string.argtypes = [i32]
    lib.mla_status_string.restype = ctypes.c_char_p
    lib.mla_resolve_impl.argtypes = [sp, i32]
    lib.mla_resolve_impl.restype = i32
    lib.mla_version.argtypes = []
    lib.mla_version.restype = i32
    lib.mla_decode_noalloc.argtypes = [sp, cp, vp, i32, vp, i32, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp]
    lib.mla_decode_noalloc.restype = i32
    lib.mla_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp, vp]
    lib.mla_selftest_wait_timeout.restype = i32
    lib.mla_fold_rotation.argtypes = [sp, vp, vp, vp, vp]
    lib.mla_fold_rotation.restype = i32
    i64 = ctypes.c_int64
    lib.mla_calib_covariance.argtypes = [vp, i64, i32, i32, vp, vp]
    lib.mla_calib_projection_energy.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, vp]
    lib.mla_calib_eigh.argtypes = [vp, i32, vp, vp, vp]
    lib.mla_calib_eigh_weighted.argtypes = [vp, vp, i32, vp, vp, vp]
    lib.mla_calib_project_abs.argtypes = [vp, i64, i32, i32, vp, vp, vp]
    lib.mla_calib_thresholds.argtypes = [vp, i64, i32, i32, ctypes.c_double, vp]
    for name in ("mla_calib_covariance", "mla_calib_projection_energy", "mla_calib_eigh", "mla_calib_eigh_weighted",
                 "mla_calib_project_abs", "mla_calib_thresholds"):
        getattr(lib, name).restype = i32
    lib.mla_profile_enable.argtypes = [i32]
    lib.mla_profile_enable.restype = i32
    lib.mla_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double), i32p, i32p]
    lib.mla_profile_read.restype = i32
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load_library().mla_status_string(int(code)).decode()


def _check(code: int, where: str) -> None:
    if code != MLA_OK:
        raise MlaError(code, where)


# ---------------------------------------------------------------- shapes

@dataclasses.dataclass
class Shape:
    """Problem shape (mirrors ``mla_shape``)."""

    num_heads: int
    kv_lora_rank: int
    rope_dim: int
    v_head_dim: int
    block_size: int
    num_blocks: int
    kind: int = MLA_KV_BF16
    group_size: int = 32
    impl: int = MLA_IMPL_AUTO
    num_splits_hint: int = 0
    index_dim: int = 0
    flags: int = 0

    def c(self) -> mla_shape:
        return mla_shape(self.num_heads, self.kv_lora_rank, self.rope_dim, self.v_head_dim,
                         self.block_size, self.num_blocks, self.group_size, self.kind, self.impl,
                         self.num_splits_hint, self.index_dim, self.flags)

    @property
    def D(self) -> int:
        return self.kv_lora_rank + self.rope_dim

    @property
    def E(self) -> int:
        """Elements per cache row (BF16/FP32 kinds): latent, rope key, extra key."""
        return self.D + self.index_dim


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


@dataclasses.dataclass
class Cache:
    """Device tensors of one paged latent cache (see ``mla_cache``)."""

    shape: Shape
    latent: object = None
    codes: object = None
    scale_zero: object = None
    rope: object = None

    def c(self) -> mla_cache:
        return mla_cache(_ptr(self.latent), _ptr(self.codes), _ptr(self.scale_zero), _ptr(self.rope))

    @classmethod
    def allocate(cls, shape: Shape, device="cuda", zero: bool = True) -> "Cache":
        """Allocate the pool for ``shape`` with torch (the library never allocates)."""
        import torch
        alloc = torch.zeros if zero else torch.empty
        nb, bs, r, dR = shape.num_blocks, shape.block_size, shape.kv_lora_rank, shape.rope_dim
        if shape.kind == MLA_KV_INT2_ROT:
            return cls(shape,
                       codes=alloc((nb, bs, r // 4), dtype=torch.uint8, device=device),
                       scale_zero=alloc((nb, bs, r // shape.group_size, 2), dtype=torch.float16, device=device),
                       rope=alloc((nb, bs, dR), dtype=torch.bfloat16, device=device))
        if shape.kind in (MLA_KV_INT2_ROT_QR, MLA_KV_INT2_JOINT):   # codes over the whole row
            return cls(shape,
                       codes=alloc((nb, bs, (r + dR) // 4), dtype=torch.uint8, device=device),
                       scale_zero=alloc((nb, bs, (r + dR) // shape.group_size, 2), dtype=torch.float16,
                                        device=device))
        dt = torch.float32 if shape.kind == MLA_KV_FP32 else torch.bfloat16
        return cls(shape, latent=alloc((nb, bs, r + dR + shape.index_dim), dtype=dt, device=device))

    def bytes_per_token(self) -> int:
        s = self.shape
        if s.kind == MLA_KV_INT2_ROT:
            return s.kv_lora_rank // 4 + (s.kv_lora_rank // s.group_size) * 4 + 2 * s.rope_dim
        if s.kind in (MLA_KV_INT2_ROT_QR, MLA_KV_INT2_JOINT):
            qd = s.kv_lora_rank + s.rope_dim
            return qd // 4 + (qd // s.group_size) * 4
        return (4 if s.kind == MLA_KV_FP32 else 2) * (s.kv_lora_rank + s.rope_dim + s.index_dim)


# ---------------------------------------------------------------- entry points

def mla_workspace_bytes(shape: Shape, B: int, q_len: int = 1) -> int:
    n = load_library().mla_workspace_bytes(ctypes.byref(shape.c()), int(B), int(q_len))
    if n == 0:
        raise MlaError(MLA_ERR_INVALID, "mla_workspace_bytes")
    return int(n)


def alloc_workspace(shape: Shape, B: int, q_len: int = 1, device="cuda"):
    import torch
    return torch.empty(mla_workspace_bytes(shape, B, q_len), dtype=torch.uint8, device=device)


def mla_latent_append(cache: Cache, block_table, start_pos, cu_new, c_kv, k_rope, R=None, clip=None,
                      status=None, stream=None) -> None:
    """Write len(c_kv) new tokens into the paged cache (see include/mla.h)."""
    lib = load_library()
    B = int(start_pos.shape[0])
    code = lib.mla_latent_append(ctypes.byref(cache.shape.c()), ctypes.byref(cache.c()), _ptr(block_table),
                                 int(block_table.shape[1]), B, _ptr(start_pos), _ptr(cu_new),
                                 int(c_kv.shape[0]), _ptr(c_kv), _ptr(k_rope), _ptr(R), _ptr(clip),
                                 _ptr(status), _stream(stream))
    _check(code, "mla_latent_append")


def mla_latent_append_index(cache: Cache, block_table, start_pos, cu_new, index_key, status=None,
                            stream=None) -> None:
    """Write the extra per-token key of len(index_key) tokens (see include/mla.h)."""
    lib = load_library()
    code = lib.mla_latent_append_index(ctypes.byref(cache.shape.c()), ctypes.byref(cache.c()), _ptr(block_table),
                                       int(block_table.shape[1]), int(start_pos.shape[0]), _ptr(start_pos),
                                       _ptr(cu_new), int(index_key.shape[0]), _ptr(index_key), _ptr(status),
                                       _stream(stream))
    _check(code, "mla_latent_append_index")


def mla_decode(cache: Cache, block_table, seq_lens, q, W_UV, scale: float, out, lse, workspace,
               R=None, stream=None, shape: Optional[Shape] = None) -> None:
    """Decode attention, q [B, 1, H, r + d_R] -> out [B, 1, H, d_v], lse [B, 1, H].
    ``shape`` overrides ``cache.shape`` (e.g. to set flags for this call)."""
    lib = load_library()
    code = lib.mla_decode(ctypes.byref((shape or cache.shape).c()), ctypes.byref(cache.c()), _ptr(block_table),
                          int(block_table.shape[1]), _ptr(seq_lens), int(seq_lens.shape[0]), _ptr(q),
                          _ptr(W_UV), _ptr(R), float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
                          int(workspace.numel() * workspace.element_size()), _stream(stream))
    _check(code, "mla_decode")


def mla_append_decode(cache: Cache, block_table, start_pos, cu_new, c_kv, k_rope, seq_lens, q, W_UV,
                      scale: float, out, lse, workspace, R=None, clip=None, append_status=None, stream=None,
                      shape: Optional[Shape] = None) -> None:
    """mla_latent_append of len(c_kv) new tokens, then mla_decode over the cache that
    holds them, in one call (see include/mla.h)."""
    lib = load_library()
    code = lib.mla_append_decode(ctypes.byref((shape or cache.shape).c()), ctypes.byref(cache.c()),
                                 _ptr(block_table), int(block_table.shape[1]), int(seq_lens.shape[0]),
                                 _ptr(start_pos), _ptr(cu_new), int(c_kv.shape[0]), _ptr(c_kv), _ptr(k_rope),
                                 _ptr(clip), _ptr(append_status), _ptr(seq_lens), _ptr(q), _ptr(W_UV), _ptr(R),
                                 float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                 int(workspace.numel() * workspace.element_size()), _stream(stream))
    _check(code, "mla_append_decode")


def mla_verify(cache: Cache, block_table, seq_lens, q, W_UV, scale: float, out, lse, workspace,
               R=None, stream=None, shape: Optional[Shape] = None) -> None:
    """Speculative verify, q [B, q_len, H, r + d_R] with the causal draft window."""
    lib = load_library()
    code = lib.mla_verify(ctypes.byref((shape or cache.shape).c()), ctypes.byref(cache.c()), _ptr(block_table),
                          int(block_table.shape[1]), _ptr(seq_lens), int(seq_lens.shape[0]), int(q.shape[1]),
                          _ptr(q), _ptr(W_UV), _ptr(R), float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
                          int(workspace.numel() * workspace.element_size()), _stream(stream))
    _check(code, "mla_verify")


def mla_fold_rotation(shape: Shape, R, W_UV, W_folded, stream=None) -> None:
    """W_folded[h] = R^T . W_UV[h] (bf16), for decode with MLA_FLAG_WUV_FOLDED (see include/mla.h)."""
    lib = load_library()
    _check(lib.mla_fold_rotation(ctypes.byref(shape.c()), _ptr(R), _ptr(W_UV), _ptr(W_folded), _stream(stream)),
           "mla_fold_rotation")


def mla_decode_noalloc(cache: Cache, block_table, seq_lens, q, W_UV, scale: float, out, lse, R=None,
                       status=None, stream=None) -> None:
    """mla_decode with the library's fixed internal scratch instead of a caller
    workspace, for callers that cannot allocate device memory at call time (see
    include/mla.h for the size limit and the ordering rule)."""
    lib = load_library()
    code = lib.mla_decode_noalloc(ctypes.byref(cache.shape.c()), ctypes.byref(cache.c()), _ptr(block_table),
                                  int(block_table.shape[1]), _ptr(seq_lens), int(seq_lens.shape[0]), _ptr(q),
                                  _ptr(W_UV), _ptr(R), float(scale), _ptr(out), _ptr(lse), _ptr(status),
                                  _stream(stream))
    _check(code, "mla_decode_noalloc")


def mla_get_status(workspace, stream=None):
    """(status code, raw flag word) of the last decode/verify on this workspace."""
    flags = ctypes.c_int32(0)
    code = load_library().mla_get_status(_ptr(workspace), ctypes.byref(flags), _stream(stream))
    return int(code), int(flags.value)


def mla_read_status_word(status, stream=None):
    flags = ctypes.c_int32(0)
    code = load_library().mla_read_status_word(_ptr(status), ctypes.byref(flags), _stream(stream))
    return int(code), int(flags.value)


def mla_selftest_wait_timeout(timeout_ns: int, status, stream=None) -> None:
    """Launch the bounded-wait self-test (see mla.h); read `status` afterwards."""
    _check(load_library().mla_selftest_wait_timeout(int(timeout_ns), _ptr(status), _stream(stream)),
           "mla_selftest_wait_timeout")


def mla_resolve_impl(shape: Shape, q_len: int = 1) -> int:
    return int(load_library().mla_resolve_impl(ctypes.byref(shape.c()), int(q_len)))


def mla_version() -> int:
    return int(load_library().mla_version())


def mla_profile_enable(enable=True) -> None:
    """True / 1: event pairs around attention kernels + launch counts; 2: launch counts
    only; False / 0: off."""
    mode = int(enable) if not isinstance(enable, bool) else (1 if enable else 0)
    _check(load_library().mla_profile_enable(mode), "mla_profile_enable")


def mla_profile_read():
    """(summed attention-kernel ms, attention launches, total kernel launches)."""
    ms = ctypes.c_double(0.0)
    n_att = ctypes.c_int32(0)
    n_all = ctypes.c_int32(0)
    _check(load_library().mla_profile_read(ctypes.byref(ms), ctypes.byref(n_att), ctypes.byref(n_all)),
           "mla_profile_read")
    return float(ms.value), int(n_att.value), int(n_all.value)


# ---------------------------------------------------------------- calibration

def _np_ptr(a):
    return a.ctypes.data if a is not None else None


def _dtype_code(t) -> int:
    import torch
    return {torch.float64: MLA_DTYPE_F64, torch.float32: MLA_DTYPE_F32, torch.bfloat16: MLA_DTYPE_BF16}[t.dtype]


def calib_covariance(X, stream=None):
    """Sigma = X^T X (fp64, device) for calibration rows X [n, d] on the device."""
    import torch
    n, d = X.shape
    sigma = torch.empty((d, d), dtype=torch.float64, device=X.device)
    _check(load_library().mla_calib_covariance(_ptr(X), int(n), int(d), _dtype_code(X), _ptr(sigma), _stream(stream)),
           "mla_calib_covariance")
    return sigma


def calib_projection_energy(W_UK, W_UV, stream=None):
    """M = sum_h W_UK[h]^T W_UK[h] + W_UV[h] W_UV[h]^T (fp64, device)."""
    import torch
    H, dn, r = W_UK.shape
    dv = W_UV.shape[2]
    M = torch.empty((r, r), dtype=torch.float64, device=W_UK.device)
    _check(load_library().mla_calib_projection_energy(_ptr(W_UK), _ptr(W_UV), int(H), int(dn), int(r), int(dv),
                                                      _dtype_code(W_UK), _ptr(M), _stream(stream)),
           "mla_calib_projection_energy")
    return M


def calib_eigh(A):
    """Host eigenbasis of a symmetric fp64 matrix: (eigenvalues ascending, R fp64, R fp32)."""
    import numpy as np
    A = np.ascontiguousarray(A, dtype=np.float64)
    d = A.shape[0]
    w = np.empty(d, np.float64)
    R64 = np.empty((d, d), np.float64)
    R32 = np.empty((d, d), np.float32)
    _check(load_library().mla_calib_eigh(_np_ptr(A), d, _np_ptr(w), _np_ptr(R64), _np_ptr(R32)), "mla_calib_eigh")
    return w, R64, R32


def calib_eigh_weighted(S, M):
    """Host eigenbasis of S^1/2 M S^1/2: (eigenvalues ascending, R fp64, R fp32)."""
    import numpy as np
    S = np.ascontiguousarray(S, dtype=np.float64)
    M = np.ascontiguousarray(M, dtype=np.float64)
    d = S.shape[0]
    w = np.empty(d, np.float64)
    R64 = np.empty((d, d), np.float64)
    R32 = np.empty((d, d), np.float32)
    _check(load_library().mla_calib_eigh_weighted(_np_ptr(S), _np_ptr(M), d, _np_ptr(w), _np_ptr(R64), _np_ptr(R32)),
           "mla_calib_eigh_weighted")
    return w, R64, R32


def calib_project_abs(X, R64, stream=None):
    """|X . R| (fp64, device) for calibration rows X [n, d] and R [d, d] fp64, both on the device."""
    import torch
    n, d = X.shape
    out = torch.empty((n, d), dtype=torch.float64, device=X.device)
    _check(load_library().mla_calib_project_abs(_ptr(X), int(n), int(d), _dtype_code(X), _ptr(R64), _ptr(out),
                                                _stream(stream)), "mla_calib_project_abs")
    return out


def calib_thresholds(absY, group_size: int = 32, pct: float = 99.0):
    """Host clip thresholds (fp32 [d / group_size]) from |X . R| [n, d] (host fp64,
    reordered in place)."""
    import numpy as np
    absY = np.ascontiguousarray(absY, dtype=np.float64)
    n, d = absY.shape
    clip = np.empty(d // group_size, np.float32)
    _check(load_library().mla_calib_thresholds(_np_ptr(absY), int(n), int(d), int(group_size), float(pct),
                                               _np_ptr(clip)), "mla_calib_thresholds")
    return clip


def calibrate_rotation(X, group_size: int = 32, pct: float = 99.0, W_UK=None, W_UV=None):
    """The per-layer calibration of a rotated-INT2 cache from calibration rows X [n, d]
    on the device: Sigma on the GPU, its eigenbasis on the host (the up-projection-aware
    one when W_UK and W_UV are given), |X . R| on the GPU and the clip thresholds on the
    host. Returns (R fp32 [d, d], clip fp32 [d / group_size], eigenvalues, R fp64) as
    numpy arrays."""
    import torch
    S = calib_covariance(X).cpu().numpy()
    if W_UK is not None:
        M = calib_projection_energy(W_UK, W_UV).cpu().numpy()
        w, R64, R32 = calib_eigh_weighted(S, M)
    else:
        w, R64, R32 = calib_eigh(S)
    absY = calib_project_abs(X, torch.from_numpy(R64).to(X.device)).cpu().numpy()
    clip = calib_thresholds(absY, group_size, pct)
    return R32, clip, w, R64
