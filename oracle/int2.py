"""Rotation fit, clip thresholds and grouped INT2 codes (oracle, test
infrastructure only).

Source: "MLA model support (GLM-5.1 / DeepSeek-style)" (OSCAR issue #10),
maintainer reply, "How the rotation adapts to the latent":
  * estimate the latent covariance Sigma = c^T c over the calibration tokens;
  * eigendecompose it (eigh) and order eigenvectors by ascending eigenvalue, so
    that low-variance directions fall in the same INT2 groups;
  * the result is one [r x r] orthogonal matrix per layer;
  * the clip thresholds are fit on the rotated latent;
  * the cache holds the rotated + quantised latent and the up-projection runs on
    the dequantised latent.

Readings adopted where the page is silent:
  * Sigma is exactly c^T c (no centring, no 1/N; 1/N would not move the
    eigenvectors).
  * Eigenvector signs: each column is flipped so that its largest-magnitude
    entry is positive.
  * Rotation is applied as a row vector: y = c . R, so column j of R is the
    j-th eigenvector (ascending) and group 0 holds the lowest-variance dims.
  * Clip threshold of group g: the 99th percentile (linear interpolation) of
    |y| over all calibration tokens and the group's dims, fp64, stored fp32.
  * Encoding, packing and dequantisation: ``int2_quant.c`` (fp32 order fixed
    there).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import attention

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "int2_quant.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle_int2.so")
_lib = None


def build_native(force: bool = False) -> str:
    """Compile the plain-C encoder with gcc (no fused multiply-add contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _native():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build_native())
        f32p = ctypes.POINTER(ctypes.c_float)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        lib.oracle_rotate_chain.argtypes = [f32p, f32p, ctypes.c_int64, ctypes.c_int, f32p]
        lib.oracle_int2_encode.argtypes = [f32p, f32p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, u8p, u16p]
        lib.oracle_int2_decode.argtypes = [u8p, u16p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, f32p]
        _lib = lib
    return _lib


def _ptr(a, ty):
    return a.ctypes.data_as(ctypes.POINTER(ty))


# ---------------------------------------------------------------- calibration

def latent_covariance(X: np.ndarray) -> np.ndarray:
    """Sigma = X^T X over calibration latents X [N, r] (fp64)."""
    X = np.asarray(X, dtype=np.float64)
    return X.T @ X


def fit_rotation(X: np.ndarray):
    """Per-layer rotation: eigenvectors of Sigma, ascending eigenvalue.

    Returns (R [r, r] fp64 with columns = eigenvectors, eigenvalues ascending).
    """
    Sigma = latent_covariance(X)
    w, V = np.linalg.eigh(Sigma)               # ascending by contract of eigh
    order = np.argsort(w, kind="stable")       # explicit: ascending eigenvalue
    w, V = w[order], V[:, order]
    return _sign_fix(V), w


def _sign_fix(V: np.ndarray) -> np.ndarray:
    """Flip each column so that its largest-magnitude entry is positive."""
    idx = np.argmax(np.abs(V), axis=0)
    signs = np.sign(V[idx, np.arange(V.shape[1])])
    signs[signs == 0] = 1.0
    return V * signs[None, :]


def projection_energy(W_UK: np.ndarray, W_UV: np.ndarray) -> np.ndarray:
    """M = sum_h (W_UK^h^T W_UK^h + W_UV^h W_UV^h^T) [r, r] (fp64): how strongly a
    latent direction reaches the keys and the values after the up-projection.
    W_UK [H, d_n, r], W_UV [H, r, d_v]."""
    K = np.asarray(W_UK, dtype=np.float64)
    V = np.asarray(W_UV, dtype=np.float64)
    return np.einsum("hnr,hns->rs", K, K) + np.einsum("hrv,hsv->rs", V, V)


def fit_rotation_weighted(X: np.ndarray, W_UK: np.ndarray, W_UV: np.ndarray):
    """Up-projection-aware variant of the per-layer rotation (the page names this as
    the open refinement: shape the INT2 error in the latent directions that matter
    after reconstruction, "MLA model support (GLM-5.1 / DeepSeek-style)", maintainer
    reply). Reading taken: the eigenbasis, ascending, of G = S^1/2 M S^1/2 with S =
    c^T c and M the projection energy above; same sign rule as fit_rotation. With
    M a multiple of the identity it is fit_rotation's basis.

    Returns (R [r, r] fp64, eigenvalues of G ascending)."""
    S = latent_covariance(X)
    ws, Vs = np.linalg.eigh(S)
    S_half = (Vs * np.sqrt(np.maximum(ws, 0.0))[None, :]) @ Vs.T
    G = S_half @ projection_energy(W_UK, W_UV) @ S_half
    G = 0.5 * (G + G.T)
    w, V = np.linalg.eigh(G)
    order = np.argsort(w, kind="stable")
    return _sign_fix(V[:, order]), w[order]


def upprojected_error(C: np.ndarray, C_hat: np.ndarray, M: np.ndarray) -> float:
    """Relative error energy of a reconstructed latent after the up-projection:
    sum_t e_t M e_t^T / sum_t c_t M c_t^T with e = c_hat - c (fp64)."""
    C = np.asarray(C, dtype=np.float64)
    E = np.asarray(C_hat, dtype=np.float64) - C
    return float(np.einsum("tr,rs,ts->", E, M, E) / np.einsum("tr,rs,ts->", C, M, C))


def clip_thresholds(X: np.ndarray, R: np.ndarray, group: int = 32, pct: float = 99.0) -> np.ndarray:
    """T_g = pct-th percentile of |X R| over the calibration tokens and group g's dims."""
    Y = np.asarray(X, dtype=np.float64) @ np.asarray(R, dtype=np.float64)
    r = Y.shape[1]
    return np.array([np.percentile(np.abs(Y[:, g * group:(g + 1) * group]), pct)
                     for g in range(r // group)], dtype=np.float64)


# ---------------------------------------------------------------- encoder (C)

def rotate_fp32(c: np.ndarray, R32: np.ndarray) -> np.ndarray:
    """y = c . R as the fp32 fused chain of the encoding definition."""
    c = np.ascontiguousarray(c, dtype=np.float32)
    R32 = np.ascontiguousarray(R32, dtype=np.float32)
    n, r = c.shape
    y = np.empty((n, r), dtype=np.float32)
    _native().oracle_rotate_chain(_ptr(c, ctypes.c_float), _ptr(R32, ctypes.c_float), n, r,
                                  _ptr(y, ctypes.c_float))
    return y


def encode(y: np.ndarray, T32: np.ndarray, group: int = 32):
    """Rotated rows y [n, r] -> (codes [n, r/4] u8, sz [n, r/group, 2] fp16 bits)."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    T32 = np.ascontiguousarray(T32, dtype=np.float32)
    n, r = y.shape
    codes = np.zeros((n, r // 4), dtype=np.uint8)
    sz = np.zeros((n, r // group, 2), dtype=np.uint16)
    _native().oracle_int2_encode(_ptr(y, ctypes.c_float), _ptr(T32, ctypes.c_float), n, r, group,
                                 _ptr(codes, ctypes.c_uint8), _ptr(sz, ctypes.c_uint16))
    return codes, sz


def quantize(c: np.ndarray, R32: np.ndarray, T32: np.ndarray, group: int = 32):
    """Rotate then encode: the full append-side transform of one batch of latents."""
    return encode(rotate_fp32(c, R32), T32, group)


def decode(codes: np.ndarray, sz: np.ndarray, group: int = 32) -> np.ndarray:
    """Dequantised rotated latent c^ [n, r] fp32: fmaf(code, s, z)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    sz = np.ascontiguousarray(sz, dtype=np.uint16)
    n = codes.shape[0]
    r = codes.shape[1] * 4
    out = np.empty((n, r), dtype=np.float32)
    _native().oracle_int2_decode(_ptr(codes, ctypes.c_uint8), _ptr(sz, ctypes.c_uint16), n, r, group,
                                 _ptr(out, ctypes.c_float))
    return out


def unpack_codes(codes: np.ndarray) -> np.ndarray:
    """[n, r/4] u8 -> [n, r] integer codes, element e at bits 2*(e%4) of byte e/4."""
    codes = np.asarray(codes, dtype=np.uint8)
    shifts = np.array([0, 2, 4, 6], dtype=np.uint8)
    return ((codes[:, :, None] >> shifts[None, None, :]) & 3).reshape(codes.shape[0], -1)


# ---------------------------------------------------------------- attention

def attention_rotated(q: np.ndarray, Chat: np.ndarray, KR: np.ndarray, R: np.ndarray,
                      W_UV: np.ndarray, scale: float):
    """Absorbed attention against a rotated latent c^ (fp64 after dequantisation).

    Scores use the rotated query q~_lat . R (so that q~_lat . c = (q~_lat R) . (c R));
    the latent output is taken back with o_lat = o_rot . R^T before W_UV.
    q [q_len, H, r + d_R], Chat [L, r] (rotated basis), R [r, r].
    """
    R = np.asarray(R, dtype=np.float64)
    r = R.shape[0]
    q = q.astype(np.float64)
    q_rot = np.concatenate([q[..., :r] @ R, q[..., r:]], axis=-1)
    _, lse, o_rot = attention.absorbed(q_rot, Chat, KR, np.zeros((q.shape[1], r, 1)), scale,
                                       return_latent=True)
    o_lat = o_rot @ R.T
    out = np.einsum("qhr,hrv->qhv", o_lat, np.asarray(W_UV, dtype=np.float64))
    return out, lse


# ---------------------------------------------------------------- rope-key variants
# "MLA model support (GLM-5.1 / DeepSeek-style)" (OSCAR issue #10), a later reply
# about GLM-5.2 support: two designs "regarding ROPE+NOPE" were being benchmarked and
# neither is described. The rotated-INT2 cache above keeps the rope key in bf16.
# Readings adopted for the two alternatives built here (none of the details are on
# the pages):
#   * rope-INT2: the rope key is quantised too, unrotated (a RoPE'd key turns with
#     the position, so a fixed covariance basis has no meaning for it), as two more
#     INT2 groups of 32 with fp16 scale/zero and their own clip thresholds (the 99th
#     percentile of |k_R| over calibration rope keys). The encoded row is
#     [c . R ; k_R], 576 values in 18 groups; the latent groups are bit-identical to
#     the bf16-rope cache's.
#   * joint: [c ; k_R] is rotated as one 576-dim vector into the eigenbasis of
#     Sigma_j = [c;k_R]^T [c;k_R] (ascending, same sign rule), clipped and encoded in
#     18 groups. Scores use q . R_j; the output is o_j . R_j^T, whose first r dims are
#     the latent output.

def rope_thresholds(KR_calib: np.ndarray, group: int = 32, pct: float = 99.0) -> np.ndarray:
    """Clip thresholds of the rope groups: pct-th percentile of |k_R| per group."""
    d = np.asarray(KR_calib).shape[1]
    return clip_thresholds(KR_calib, np.eye(d), group, pct)


def quantize_rope_int2(c: np.ndarray, KR: np.ndarray, R32: np.ndarray, T32: np.ndarray,
                       TR32: np.ndarray, group: int = 32):
    """rope-INT2 encoding of tokens (c [n, r], k_R [n, d_R]): the row [c . R ; k_R]
    (fp32 rotation chain for the latent part, the rope key as given) encoded in
    groups with thresholds [T ; T_R]. Returns codes [n, (r+d_R)/4], sz [n, (r+d_R)/group, 2]."""
    y = np.concatenate([rotate_fp32(c, R32), np.asarray(KR, dtype=np.float32)], axis=1)
    T = np.concatenate([np.asarray(T32, np.float32), np.asarray(TR32, np.float32)])
    return encode(y, T, group)


def attention_rope_int2(q: np.ndarray, Y_hat: np.ndarray, R: np.ndarray, W_UV: np.ndarray,
                        scale: float):
    """Absorbed attention against a rope-INT2 cache: Y_hat [L, r + d_R] is the
    dequantised row [c^ ; k_R^] (rotated latent, then the rope key)."""
    r = np.asarray(R).shape[0]
    return attention_rotated(q, Y_hat[:, :r], Y_hat[:, r:], R, W_UV, scale)


def attention_joint(q: np.ndarray, Y_hat: np.ndarray, Rj: np.ndarray, W_UV: np.ndarray,
                    scale: float):
    """Absorbed attention against a jointly rotated cache: Y_hat [L, r + d_R] holds
    [c ; k_R] . R_j (dequantised). Scores: (q . R_j) . Y_hat (= q . [c ; k_R] before
    quantisation); output: o_j . R_j^T, of which the first r dims are o_lat."""
    Rj = np.asarray(Rj, dtype=np.float64)
    D = Rj.shape[0]
    r = np.asarray(W_UV).shape[1]
    q = q.astype(np.float64)
    qj = q @ Rj
    L = Y_hat.shape[0]
    _, lse, oj = attention.absorbed(qj, Y_hat, np.zeros((L, 0)), np.zeros((q.shape[1], D, 1)), scale,
                                    return_latent=True)
    o_lat = (oj @ Rj.T)[..., :r]
    out = np.einsum("qhr,hrv->qhv", o_lat, np.asarray(W_UV, dtype=np.float64))
    return out, lse
