"""Seeded synthetic inputs for MLA latent-cache decode, shared by the tests, the
benchmark and the oracle checks.

This module only draws random numbers and lays them out: it holds none of the
method's arithmetic (no attention, no rotation fit, no quantisation). Every
array is produced from ``numpy.random.Generator(PCG64(seed))`` so both sides of
a parity test see the same bits.

Workload recipes (shapes and value laws):

* ``tiny``      B=2, L=(100,256), q_len=1, H=8, r=64, d_R=16, d_n=32, d_v=32,
                scale 1/sqrt(48), fp32; c, k_R, q ~ N(0,1); W_UK, W_UV ~ N(0, 1/8^2);
                one 256-token block per sequence.
* ``dsv3``      B=32, q_len=1, H=128, r=512, d_R=64, d_n=128, d_v=128,
                scale 1/sqrt(192), bf16; L ~ U_int[1024, 8192]; block size 64 with
                a randomly permuted block pool; latent dim j ~ N(0, sigma_j^2) with
                sigma_j log-uniform in [0.1, 3]; k_R, q ~ N(0,1); W_UV ~ N(0, 1/512).
* ``long``      dsv3 dims with H=64, B=2, L=(32768, 131072).
* ``verify``    dsv3 dims, B=16, q_len=8, L ~ U_int[4096, 32768] (drafts included).
* ``int2``      dsv3 shapes; 65536 calibration latents N(0, diag(v)) . Q with v
                log-uniform in [0.01, 9] and Q Haar-random; cache latents drawn
                fresh from the same law; 32 new tokens appended per sequence.

Values that feed bf16 buffers are rounded to bf16 here (round-to-nearest-even on
the fp32 bit pattern) so that both sides start from identical numbers.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

__all__ = [
    "Workload",
    "bf16_round",
    "bf16_bits",
    "tiny",
    "dsv3",
    "long_context",
    "verify",
    "int2_rotated",
    "make_paging",
]


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 array -> uint16 bf16 bit patterns, round-to-nearest-even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp32 array -> fp32 array holding the nearest bf16 values (RNE)."""
    b = bf16_bits(x).astype(np.uint32) << 16
    return b.view(np.float32).reshape(np.shape(x))


@dataclasses.dataclass
class Workload:
    """One decode problem: per-sequence token data plus the paged layout.

    Token data is logical (per sequence, position order). ``block_table`` maps
    logical block j of sequence b to a physical block of the pool.
    """

    name: str
    dtype: str                      # "fp32" or "bf16": element type of q / cache / W_UV
    B: int
    q_len: int
    H: int
    r: int                          # kv_lora_rank
    d_rope: int                     # qk_rope_head_dim
    d_nope: int                     # qk_nope_head_dim
    d_v: int                        # v_head_dim
    scale: float
    block_size: int
    seq_lens: np.ndarray            # [B] int32, tokens in cache incl. drafts
    latent: list                    # per b: [L_b, r] float32 (bf16-exact if bf16)
    rope: list                      # per b: [L_b, d_rope] float32
    q: np.ndarray                   # [B, q_len, H, r + d_rope] absorbed query (fp32 values)
    W_UV: np.ndarray                # [H, r, d_v]
    block_table: np.ndarray         # [B, max_blocks] int32, -1 where unused
    num_blocks: int
    # pre-absorption query and W_UK exist only where the recipe defines them
    q_nope: Optional[np.ndarray] = None   # [B, q_len, H, d_nope]
    q_rope: Optional[np.ndarray] = None   # [B, q_len, H, d_rope]
    W_UK: Optional[np.ndarray] = None     # [H, d_nope, r]
    # rotated-INT2 recipe extras
    calib: Optional[np.ndarray] = None    # [N_cal, r] float64 calibration latents
    new_latent: Optional[list] = None     # per b: [n_new, r] appended tokens
    new_rope: Optional[list] = None       # per b: [n_new, d_rope]
    start_pos: Optional[np.ndarray] = None  # [B] position of the first appended token

    @property
    def D(self) -> int:
        return self.r + self.d_rope

    @property
    def total_tokens(self) -> int:
        return int(np.sum(self.seq_lens))


def make_paging(rng: np.random.Generator, lens_alloc: np.ndarray, block_size: int,
                permute: bool = True, spare_blocks: int = 0):
    """Block table for sequences that will hold ``lens_alloc`` tokens.

    The pool has sum(ceil(L/bs)) + spare_blocks blocks; physical ids are a
    random permutation of the pool (or identity when ``permute`` is False).
    """
    nblk = [(int(L) + block_size - 1) // block_size for L in lens_alloc]
    pool = int(sum(nblk)) + spare_blocks
    ids = rng.permutation(pool).astype(np.int32) if permute else np.arange(pool, dtype=np.int32)
    max_blocks = max(nblk) if nblk else 1
    table = np.full((len(lens_alloc), max_blocks), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(nblk):
        table[b, :n] = ids[k:k + n]
        k += n
    return table, pool


def _normal(rng, shape, std=1.0):
    return (rng.standard_normal(shape) * std).astype(np.float32)


def tiny(seed: int = 0) -> Workload:
    """Tiny fp32 decode with the pre-absorption query and W_UK."""
    rng = np.random.Generator(np.random.PCG64(seed))
    B, H, r, dR, dn, dv = 2, 8, 64, 16, 32, 32
    lens = np.array([100, 256], dtype=np.int32)
    bs = 256
    latent = [_normal(rng, (int(L), r)) for L in lens]
    rope = [_normal(rng, (int(L), dR)) for L in lens]
    q_nope = _normal(rng, (B, 1, H, dn))
    q_rope = _normal(rng, (B, 1, H, dR))
    W_UK = _normal(rng, (H, dn, r), 1.0 / math.sqrt(64))
    W_UV = _normal(rng, (H, r, dv), 1.0 / math.sqrt(64))
    table = np.array([[0], [1]], dtype=np.int32)
    # The absorbed query is formed by the caller (oracle for expected values,
    # and the same oracle-made q handed to the library as its input).
    return Workload("tiny", "fp32", B, 1, H, r, dR, dn, dv, 1.0 / math.sqrt(48.0), bs,
                    lens, latent, rope, np.zeros((B, 1, H, r + dR), np.float32), W_UV,
                    table, 2, q_nope=q_nope, q_rope=q_rope, W_UK=W_UK)


def _dsv3_like(name, seed, B, q_len, H, lens, *, bs=64, permute=True, spare=0,
               lens_alloc=None, sigma=None, rng=None, with_wuk=False) -> Workload:
    rng = rng or np.random.Generator(np.random.PCG64(seed))
    r, dR, dn, dv = 512, 64, 128, 128
    if sigma is None:
        sigma = np.exp(rng.uniform(math.log(0.1), math.log(3.0), size=r)).astype(np.float32)
    latent = [bf16_round(_normal(rng, (int(L), r)) * sigma[None, :]) for L in lens]
    rope = [bf16_round(_normal(rng, (int(L), dR))) for L in lens]
    q = bf16_round(_normal(rng, (B, q_len, H, r + dR)))
    W_UV = bf16_round(_normal(rng, (H, r, dv), 1.0 / math.sqrt(r)))
    table, pool = make_paging(rng, lens if lens_alloc is None else lens_alloc, bs,
                              permute=permute, spare_blocks=spare)
    w = Workload(name, "bf16", B, q_len, H, r, dR, dn, dv, 1.0 / math.sqrt(192.0), bs,
                 np.asarray(lens, np.int32), latent, rope, q, W_UV, table, pool)
    if with_wuk:
        w.W_UK = bf16_round(_normal(rng, (H, dn, r), 1.0 / math.sqrt(r)))
    return w


def dsv3(seed: int = 1, B: int = 32, H: int = 128, len_range=(1024, 8192),
         q_len: int = 1, permute: bool = True, with_wuk: bool = False) -> Workload:
    """DeepSeek-V3-shaped bf16 decode (paged, permuted block table)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    sigma = np.exp(rng.uniform(math.log(0.1), math.log(3.0), size=512)).astype(np.float32)
    lens = rng.integers(len_range[0], len_range[1], size=B, endpoint=True).astype(np.int32)
    return _dsv3_like("dsv3", seed, B, q_len, H, lens, sigma=sigma, rng=rng,
                      permute=permute, with_wuk=with_wuk)


def long_context(seed: int = 2, lens=(32768, 131072), H: int = 64) -> Workload:
    """Two long sequences, H=64, DS-V3 dims and value laws."""
    rng = np.random.Generator(np.random.PCG64(seed))
    sigma = np.exp(rng.uniform(math.log(0.1), math.log(3.0), size=512)).astype(np.float32)
    lens = np.asarray(lens, np.int32)
    return _dsv3_like("long", seed, len(lens), 1, H, lens, sigma=sigma, rng=rng)


def verify(seed: int = 3, B: int = 16, q_len: int = 8, len_range=(4096, 32768),
           H: int = 128) -> Workload:
    """Speculative verify: q_len draft rows per sequence, drafts already cached."""
    rng = np.random.Generator(np.random.PCG64(seed))
    sigma = np.exp(rng.uniform(math.log(0.1), math.log(3.0), size=512)).astype(np.float32)
    lens = rng.integers(len_range[0], len_range[1], size=B, endpoint=True).astype(np.int32)
    return _dsv3_like("verify", seed, B, q_len, H, lens, sigma=sigma, rng=rng)


def haar_orthogonal(rng: np.random.Generator, n: int) -> np.ndarray:
    """Haar-distributed orthogonal matrix: QR of a Gaussian matrix, with the
    column signs fixed by the sign of R's diagonal (Mezzadri 2007)."""
    Z = rng.standard_normal((n, n))
    Q, Rm = np.linalg.qr(Z)
    return Q * np.sign(np.diag(Rm))[None, :]


def int2_rotated(seed: int = 4, B: int = 32, H: int = 128, len_range=(1024, 8192),
                 n_calib: int = 65536, n_new: int = 32) -> Workload:
    """Rotated INT2 cache recipe.

    Latents follow N(0, diag(v)) . Q (v log-uniform in [0.01, 9], Q Haar), both
    for the calibration set (float64) and for the cache (bf16-rounded). Each
    sequence then receives ``n_new`` appended tokens at positions L_b..L_b+n_new-1.
    ``seq_lens`` are the lengths before the append.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    r, dR = 512, 64
    var = np.exp(rng.uniform(math.log(0.01), math.log(9.0), size=r))
    Q = haar_orthogonal(rng, r)
    mix = (np.sqrt(var)[:, None] * Q)            # row-vector law: x = z . diag(sqrt v) . Q
    calib = rng.standard_normal((n_calib, r)) @ mix
    lens = rng.integers(len_range[0], len_range[1], size=B, endpoint=True).astype(np.int32)
    latent = [bf16_round((rng.standard_normal((int(L), r)) @ mix).astype(np.float32)) for L in lens]
    rope = [bf16_round(_normal(rng, (int(L), dR))) for L in lens]
    new_latent = [bf16_round((rng.standard_normal((n_new, r)) @ mix).astype(np.float32)) for _ in lens]
    new_rope = [bf16_round(_normal(rng, (n_new, dR))) for _ in lens]
    q = bf16_round(_normal(rng, (B, 1, H, r + dR)))
    W_UV = bf16_round(_normal(rng, (H, r, 128), 1.0 / math.sqrt(r)))
    table, pool = make_paging(rng, lens + n_new, 64, permute=True)
    w = Workload("int2", "bf16", B, 1, H, r, dR, 128, 128, 1.0 / math.sqrt(192.0), 64,
                 lens, latent, rope, q, W_UV, table, pool)
    w.calib = calib
    w.new_latent = new_latent
    w.new_rope = new_rope
    w.start_pos = lens.copy()
    return w
