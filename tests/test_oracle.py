"""Pins for the CPU oracle: facts the pages print, closed forms, invariants and
brute force, each chosen so that a dropped term, a wrong index or a transposed
operand in the oracle fails at least one of them. CPU only."""
import math
import os

import numpy as np
import pytest

import workloads
from oracle import attention, layout
from oracle import int2 as oint2

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = (s.strip() for s in line.split("="))
            vals[k] = float(v)
    return vals


# ----------------------------------------------------------------- footprint

def test_footprint_matches_pages():
    g = _golden("footprint.txt")
    # DeepSeek V2/V3/V3.2: kv_lora_rank 512 + qk_rope_head_dim 64.
    assert layout.footprint_elems(512, 64) == g["deepseek_v3_latent_elems_per_layer"]
    # GLM-5.3-Flash: linear layers hold nothing, 11 latent layers x 640 x 2 B.
    types = ["linear_attention"] * int(g["glm53_linear_layers"]) + ["full_attention"] * int(g["glm53_latent_layers"])
    assert len(types) == g["glm53_layers_total"]
    per_tok = layout.kv_bytes_per_token(types, 512, 64, 64, bytes_per_elem=int(g["glm53_bytes_per_elem"]))
    assert layout.footprint_elems(512, 64, 64) == g["glm53_elems_per_latent_layer"]
    assert per_tok == g["glm53_bytes_per_token"]
    assert abs(per_tok * 2**20 / 1e9 - g["glm53_gb_at_1m_tokens"]) < 0.5
    assert abs(g["glm53_after_gb"] * 1e9 / per_tok / 1e3 - g["glm53_after_tokens_k"]) < 5


def test_footprint_ratios_match_pages():
    g = _golden("footprint.txt")
    # Old DeepSeek estimate: K and V at full hidden width (2 x 7168) per layer.
    assert abs(2 * 7168 / layout.footprint_elems(512, 64) - g["deepseek_estimate_fall_factor"]) < 0.5
    # Full-head K/V (H x (d_nope + d_rope + d_v)) over the latent, DS-V3 shapes.
    ratio = 128 * (128 + 64 + 128) / layout.footprint_elems(512, 64)
    assert abs(ratio - g["latent_kv_shrink_factor"]) / g["latent_kv_shrink_factor"] < 0.05
    assert abs(g["full_head_kv_gb_32k"] / g["latent_kv_gb_32k"] - g["latent_kv_shrink_factor"]) / 70 < 0.05


# ------------------------------------------------------- absorb == full head

def test_absorbed_equals_full_head_tiny():
    g = _golden("footprint.txt")
    w = workloads.tiny(0)
    for b in range(w.B):
        qt = attention.absorb_query(w.q_nope[b], w.q_rope[b], w.W_UK)
        o1, l1 = attention.absorbed(qt, w.latent[b], w.rope[b], w.W_UV, w.scale)
        o2, l2 = attention.full_head(w.q_nope[b], w.q_rope[b], w.latent[b], w.rope[b],
                                     w.W_UK, w.W_UV, w.scale)
        assert np.max(np.abs(o1 - o2)) <= 10 * g["absorb_equivalence_error"]
        assert np.max(np.abs(l1 - l2)) <= 10 * g["absorb_equivalence_error"]


def test_absorbed_equals_full_head_dsv3_dims_causal():
    rng = np.random.default_rng(7)
    H, r, dR, dn, dv, L, ql = 16, 512, 64, 128, 128, 300, 4
    C = rng.standard_normal((L, r)) * np.exp(rng.uniform(np.log(.1), np.log(3), r))
    KR = rng.standard_normal((L, dR))
    qn = rng.standard_normal((ql, H, dn))
    qr = rng.standard_normal((ql, H, dR))
    WUK = rng.standard_normal((H, dn, r)) / math.sqrt(r)
    WUV = rng.standard_normal((H, r, dv)) / math.sqrt(r)
    qt = attention.absorb_query(qn, qr, WUK)
    o1, l1 = attention.absorbed(qt, C, KR, WUV, 1 / math.sqrt(192))
    o2, l2 = attention.full_head(qn, qr, C, KR, WUK, WUV, 1 / math.sqrt(192))
    assert np.max(np.abs(o1 - o2)) < 1e-12
    assert np.max(np.abs(l1 - l2)) < 1e-12


# ---------------------------------------------------------- brute force

def _brute(q, C, KR, WUV, scale):
    """Definition with explicit loops, written independently of the oracle."""
    ql, H, D = q.shape
    L, r = C.shape
    dv = WUV.shape[2]
    out = np.zeros((ql, H, dv))
    lse = np.zeros((ql, H))
    for i in range(ql):
        for h in range(H):
            n_vis = L - ql + i + 1
            s = []
            for t in range(n_vis):
                acc = 0.0
                for d in range(r):
                    acc += q[i, h, d] * C[t, d]
                for d in range(KR.shape[1]):
                    acc += q[i, h, r + d] * KR[t, d]
                s.append(scale * acc)
            tot = sum(math.exp(x) for x in s)
            lse[i, h] = math.log(tot)
            for v in range(dv):
                acc = 0.0
                for t in range(n_vis):
                    p = math.exp(s[t]) / tot
                    for d in range(r):
                        acc += p * C[t, d] * WUV[h, d, v]
                out[i, h, v] = acc
    return out, lse


@pytest.mark.parametrize("L,ql", [(1, 1), (5, 1), (8, 3)])
def test_brute_force_tiny(L, ql):
    rng = np.random.default_rng(L * 10 + ql)
    H, r, dR, dv = 2, 4, 2, 3
    q = rng.standard_normal((ql, H, r + dR))
    C = rng.standard_normal((L, r))
    KR = rng.standard_normal((L, dR))
    WUV = rng.standard_normal((H, r, dv))
    o1, l1 = attention.absorbed(q, C, KR, WUV, 0.7)
    o2, l2 = _brute(q, C, KR, WUV, 0.7)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


# ----------------------------------------------------------- closed forms

def test_softmax_rows_sum_to_one():
    w = workloads.dsv3(1, B=2, H=8, len_range=(100, 300), q_len=3)
    for b in range(w.B):
        P = attention.softmax_weights(w.q[b], w.latent[b], w.rope[b], w.scale)
        assert np.max(np.abs(P.sum(-1) - 1.0)) < 1e-14
        assert np.all(P >= 0)
        # causal: row i has exactly L - q_len + i + 1 non-zero weights
        L = w.latent[b].shape[0]
        for i in range(3):
            assert np.all(P[i, :, L - 3 + i + 1:] == 0)


def test_single_token_closed_form():
    rng = np.random.default_rng(3)
    H, r, dR, dv = 4, 16, 8, 5
    q = rng.standard_normal((1, H, r + dR))
    C = rng.standard_normal((1, r))
    KR = rng.standard_normal((1, dR))
    WUV = rng.standard_normal((H, r, dv))
    out, lse = attention.absorbed(q, C, KR, WUV, 0.3)
    for h in range(H):
        # one token: p = 1, o_h = (W_UV^h)^T c_0, lse = its scaled score
        np.testing.assert_allclose(out[0, h], C[0] @ WUV[h], atol=1e-13)
        s = 0.3 * (q[0, h, :r] @ C[0] + q[0, h, r:] @ KR[0])
        assert abs(lse[0, h] - s) < 1e-13


def test_identical_keys_uniform():
    rng = np.random.default_rng(4)
    H, r, dR, dv, L = 3, 8, 4, 6, 37
    q = rng.standard_normal((1, H, r + dR))
    C = np.repeat(rng.standard_normal((1, r)), L, 0)
    KR = np.repeat(rng.standard_normal((1, dR)), L, 0)
    WUV = rng.standard_normal((H, r, dv))
    out, lse = attention.absorbed(q, C, KR, WUV, 0.5)
    for h in range(H):
        s = 0.5 * (q[0, h, :r] @ C[0] + q[0, h, r:] @ KR[0])
        assert abs(lse[0, h] - (s + math.log(L))) < 1e-12
        np.testing.assert_allclose(out[0, h], C[0] @ WUV[h], atol=1e-12)


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(5)
    H, r, dR, dv, L = 2, 8, 4, 3, 20
    C = rng.standard_normal((L, r))
    KR = rng.standard_normal((L, dR))
    WUV = rng.standard_normal((H, r, dv))
    k7 = np.concatenate([C[7], KR[7]])
    q = np.stack([k7 * 50.0, k7 * 50.0])[None]        # [1, H, D], aligned with token 7
    out, _ = attention.absorbed(q, C, KR, WUV, 1.0)
    for h in range(H):
        np.testing.assert_allclose(out[0, h], C[7] @ WUV[h], atol=1e-9)


def test_split_lse_identity():
    """LSE over all tokens = logsumexp of the LSEs of two disjoint ranges, and the
    output is the LSE-weighted mix of the two range outputs (q_len = 1)."""
    w = workloads.dsv3(1, B=1, H=4, len_range=(500, 500))
    C, KR, q = w.latent[0], w.rope[0], w.q[0]
    o, l = attention.absorbed(q, C, KR, w.W_UV, w.scale)
    o1, l1 = attention.absorbed(q, C[:123], KR[:123], w.W_UV, w.scale)
    o2, l2 = attention.absorbed(q, C[123:], KR[123:], w.W_UV, w.scale)
    lse = np.logaddexp(l1, l2)
    np.testing.assert_allclose(l, lse, atol=1e-12)
    mix = np.exp(l1 - lse)[..., None] * o1 + np.exp(l2 - lse)[..., None] * o2
    np.testing.assert_allclose(o, mix, atol=1e-12)


def test_row_subset_matches_full():
    w = workloads.verify(3, B=1, q_len=4, len_range=(200, 200), H=8)
    o, l = attention.absorbed(w.q[0], w.latent[0], w.rope[0], w.W_UV, w.scale)
    rows = [(0, 0), (3, 7), (2, 5)]
    os_, ls = attention.row_subset(w.q[0], w.latent[0], w.rope[0], w.W_UV, w.scale, rows)
    for k, (i, h) in enumerate(rows):
        np.testing.assert_allclose(os_[k], o[i, h], atol=1e-12)
        assert abs(ls[k] - l[i, h]) < 1e-12


# ----------------------------------------------------------------- paging

def test_paged_roundtrip_and_permutation_invariance():
    w = workloads.dsv3(1, B=3, H=4, len_range=(65, 300))
    rows = [np.concatenate([w.latent[b], w.rope[b]], 1) for b in range(w.B)]
    pool = layout.write_paged(w.num_blocks, 64, w.D, w.block_table, rows, [0] * w.B)
    for b in range(w.B):
        back = layout.read_paged(pool, w.block_table[b], int(w.seq_lens[b]), 64)
        np.testing.assert_array_equal(back, rows[b])
    # a different (identity) placement gives the same gathered rows
    ident, n = workloads.make_paging(np.random.default_rng(0), w.seq_lens, 64, permute=False)
    pool2 = layout.write_paged(n, 64, w.D, ident, rows, [0] * w.B)
    for b in range(w.B):
        np.testing.assert_array_equal(layout.read_paged(pool2, ident[b], int(w.seq_lens[b]), 64), rows[b])
    # block ids really are permuted (the placement test is not vacuous)
    assert not np.array_equal(w.block_table[w.block_table >= 0], np.arange(w.num_blocks))


# --------------------------------------------------------------- rotation

def test_rotation_recovers_known_eigenbasis():
    """X = diag(sqrt d) Q^T has X^T X = Q diag(d) Q^T exactly: R must be Q with its
    columns in ascending-d order, up to the sign rule."""
    rng = np.random.default_rng(11)
    n = 24
    Q = workloads.haar_orthogonal(rng, n)
    d = rng.permutation(np.linspace(1.0, 40.0, n))
    X = np.sqrt(d)[:, None] * Q.T
    R, w = oint2.fit_rotation(X)
    order = np.argsort(d)
    np.testing.assert_allclose(w, d[order], rtol=1e-12)
    for j in range(n):
        col = Q[:, order[j]]
        col = col * np.sign(col[np.argmax(np.abs(col))])
        np.testing.assert_allclose(R[:, j], col, atol=1e-10)
        assert R[np.argmax(np.abs(R[:, j])), j] > 0


def test_rotation_properties_on_calibration_set():
    w = workloads.int2_rotated(4, B=1, H=4, len_range=(64, 64), n_calib=8192)
    R, ev = oint2.fit_rotation(w.calib)
    assert np.max(np.abs(R.T @ R - np.eye(512))) < 1e-12
    Sig = oint2.latent_covariance(w.calib)
    Dm = R.T @ Sig @ R
    assert np.all(np.diff(np.diag(Dm)) >= 0)                        # ascending
    off = Dm - np.diag(np.diag(Dm))
    assert np.max(np.abs(off)) < 1e-9 * ev[-1]
    # ascending eigenvalue -> group 0 holds the lowest-variance rotated dims
    Y = w.calib @ R
    var = Y.var(0)
    assert var[:32].mean() < var[-32:].mean() / 50


def test_rotation_is_lossless_before_quantisation():
    w = workloads.int2_rotated(4, B=1, H=8, len_range=(150, 150), n_calib=4096)
    R, _ = oint2.fit_rotation(w.calib)
    C = w.latent[0].astype(np.float64)
    Y = C @ R
    o1, l1 = attention.absorbed(w.q[0], C, w.rope[0], w.W_UV, w.scale)
    o2, l2 = oint2.attention_rotated(w.q[0], Y, w.rope[0], R, w.W_UV, w.scale)
    assert np.max(np.abs(o1 - o2)) < 1e-12
    assert np.max(np.abs(l1 - l2)) < 1e-12


def test_clip_thresholds_clip_one_percent():
    w = workloads.int2_rotated(4, B=1, H=4, len_range=(64, 64), n_calib=16384)
    R, _ = oint2.fit_rotation(w.calib)
    T = oint2.clip_thresholds(w.calib, R)
    Y = np.abs(w.calib @ R)
    for g in range(16):
        frac = np.mean(Y[:, 32 * g:32 * g + 32] > T[g])
        assert 0.009 <= frac <= 0.011
    assert T[-1] > 3 * T[0]                              # thresholds grow with the group's variance


# -------------------------------------------------------------- INT2 codes

def test_int2_worked_example():
    """Hand-worked encoding of two 4-element groups (r = 8, group 4)."""
    y = np.array([[0.0, 1.0, 2.0, 3.0, -2.0, 0.5, 0.25, 2.0]], dtype=np.float32)
    T = np.array([10.0, 1.0], dtype=np.float32)
    codes, sz = oint2.encode(y, T, group=4)
    # group 0: lo 0, hi 3, s 1, z 0 -> codes 0,1,2,3 -> 0b11_10_01_00
    # group 1: clipped to [-1, .5, .25, 1]; s = fp16(2/3) = 0.66650390625, z = -1
    #          (v - z)/s = 0, 2.2506, 1.8755, 3.0007 -> codes 0,2,2,3 -> 0b11_10_10_00
    assert codes.tolist() == [[0xE4, 0xE8]]
    s = sz.view(np.float16).astype(np.float64)
    assert s[0, 0, 0] == 1.0 and s[0, 0, 1] == 0.0
    assert s[0, 1, 0] == 0.66650390625 and s[0, 1, 1] == -1.0
    deq = oint2.decode(codes, sz, group=4)
    np.testing.assert_array_equal(deq[0], np.array(
        [0, 1, 2, 3, -1, 0.3330078125, 0.3330078125, 0.99951171875], dtype=np.float32))
    np.testing.assert_array_equal(oint2.unpack_codes(codes)[0], [0, 1, 2, 3, 0, 2, 2, 3])


def test_int2_constant_group_has_zero_scale():
    y = np.full((1, 8), 0.75, dtype=np.float32)
    codes, sz = oint2.encode(y, np.array([5.0, 5.0], np.float32), group=4)
    assert codes.tolist() == [[0, 0]]
    assert np.all(sz.view(np.float16)[..., 0] == 0)
    np.testing.assert_array_equal(oint2.decode(codes, sz, group=4), y)


def test_int2_invariants_and_rotation_chain():
    w = workloads.int2_rotated(4, B=2, H=4, len_range=(64, 64), n_calib=8192)
    R, _ = oint2.fit_rotation(w.calib)
    T = oint2.clip_thresholds(w.calib, R).astype(np.float32)
    c = np.concatenate(w.new_latent)                         # [64, 512]
    R32 = R.astype(np.float32)
    y = oint2.rotate_fp32(c, R32)
    # the fp32 chain is c . R (not c . R^T) to fp32 accuracy
    y64 = c.astype(np.float64) @ R32.astype(np.float64)
    assert np.max(np.abs(y - y64)) < 1e-4 * np.max(np.abs(y64))
    assert np.max(np.abs(c.astype(np.float64) @ R32.T.astype(np.float64) - y64)) > 1e-2
    codes, sz = oint2.encode(y, T)
    u = oint2.unpack_codes(codes)
    assert u.min() >= 0 and u.max() <= 3
    s = sz.view(np.float16)[..., 0].astype(np.float32).repeat(32, 1)
    z = sz.view(np.float16)[..., 1].astype(np.float32).repeat(32, 1)
    deq = oint2.decode(codes, sz)
    assert np.all(deq >= z - 1e-6) and np.all(deq <= z + 3 * s + 1e-5 * np.abs(z + 3 * s))
    yc = np.clip(y, -T.repeat(32)[None], T.repeat(32)[None])
    err = np.abs(deq - yc)
    # rounding to the nearest level, plus the fp16 rounding of z and s
    assert np.all(err <= s / 2 + 2e-3 * (np.abs(yc) + s) + 1e-6)
    # python re-decoding agrees with the C decoder (codes * s + z is exact-then-rounded once)
    np.testing.assert_array_equal(deq, (u.astype(np.float32) * s + z).astype(np.float32))


# ------------------------------------------------- up-projection-aware rotation

def test_projection_energy_closed_form():
    rng = np.random.default_rng(3)
    K = rng.standard_normal((3, 5, 8))
    V = rng.standard_normal((3, 8, 4))
    M = oint2.projection_energy(K, V)
    # direct sum over heads, written out
    ref = sum(K[h].T @ K[h] + V[h] @ V[h].T for h in range(3))
    np.testing.assert_allclose(M, ref, rtol=1e-12)
    # c M c^T is the energy c reaches the keys and values with
    c = rng.standard_normal(8)
    energy = sum(np.sum((K[h] @ c) ** 2) + np.sum((c @ V[h]) ** 2) for h in range(3))
    assert abs(c @ M @ c - energy) < 1e-10 * energy


def test_weighted_rotation_reduces_to_plain_for_isotropic_weights():
    """M = I (W_UK the identity, no W_UV): G = S, so the basis is fit_rotation's."""
    rng = np.random.default_rng(4)
    r = 16
    X = rng.standard_normal((4000, r)) * np.exp(rng.uniform(-1.5, 1.5, size=r))[None, :]
    R0, w0 = oint2.fit_rotation(X)
    R1, w1 = oint2.fit_rotation_weighted(X, np.eye(r)[None], np.zeros((1, r, 1)))
    np.testing.assert_allclose(R1, R0, atol=1e-8)
    np.testing.assert_allclose(w1, w0, rtol=1e-10)
    assert np.max(np.abs(R1.T @ R1 - np.eye(r))) < 1e-12


def test_weighted_rotation_follows_the_weights_for_white_latents():
    """S = I (orthonormal calibration columns): G = M, the basis is M's eigenbasis."""
    rng = np.random.default_rng(5)
    r = 12
    X, _ = np.linalg.qr(rng.standard_normal((500, r)))            # X^T X = I
    K = rng.standard_normal((2, 6, r))
    V = rng.standard_normal((2, r, 3))
    R, w = oint2.fit_rotation_weighted(X, K, V)
    M = oint2.projection_energy(K, V)
    np.testing.assert_allclose(R.T @ M @ R, np.diag(w), atol=1e-9 * np.max(w))
    assert np.all(np.diff(w) >= 0)


def test_upprojected_error_closed_form():
    rng = np.random.default_rng(6)
    r = 10
    A = rng.standard_normal((r, r))
    M = A @ A.T
    lam, U = np.linalg.eigh(M)
    C = rng.standard_normal((50, r))
    assert oint2.upprojected_error(C, C, M) == 0.0
    # a perturbation of size d along eigenvector k of M on every token
    d, k = 0.01, 3
    err = oint2.upprojected_error(C, C + d * U[:, k][None, :], M)
    assert abs(err - 50 * d * d * lam[k] / np.einsum("tr,rs,ts->", C, M, C)) < 1e-12


def test_weighted_rotation_study():
    """The up-projection-aware reading measured against the plain rotation on the INT2
    workload's law (the comparison reported in the design notes): no gain with
    isotropic synthetic weights, and a clear loss with anisotropic ones, because it
    puts latent directions of very different variance into the same INT2 group."""
    w = workloads.int2_rotated(4, B=4, H=32, len_range=(512, 768), n_calib=32768)
    rng = np.random.default_rng(7)
    r = w.r
    K = rng.standard_normal((w.H, 128, r)) / np.sqrt(r)
    V = np.asarray(w.W_UV, np.float64)
    C = np.concatenate(w.latent).astype(np.float64)
    scale = np.exp(rng.uniform(np.log(0.2), np.log(5.0), size=r))
    res = {}
    for label, (KK, VV) in (("isotropic", (K, V)),
                            ("anisotropic", (K * scale[None, None, :], V * scale[None, :, None]))):
        M = oint2.projection_energy(KK, VV)
        for name, R in (("plain", oint2.fit_rotation(w.calib)[0]),
                        ("weighted", oint2.fit_rotation_weighted(w.calib, KK, VV)[0])):
            T = oint2.clip_thresholds(w.calib, R)
            codes, sz = oint2.quantize(C.astype(np.float32), R.astype(np.float32), T.astype(np.float32))
            Chat = oint2.decode(codes, sz).astype(np.float64) @ R.T
            res[label, name] = oint2.upprojected_error(C, Chat, M)
    print({k: round(v, 4) for k, v in res.items()})
    assert res["isotropic", "weighted"] > 0.97 * res["isotropic", "plain"]
    assert res["anisotropic", "weighted"] > 1.3 * res["anisotropic", "plain"]


# ------------------------------------------------------- rope-key variants (next-2)

def _rope_setup(n=96, seed=21):
    w = workloads.int2_rotated(seed, B=1, H=4, len_range=(n, n), n_calib=4096)
    R, _ = oint2.fit_rotation(w.calib)
    T = oint2.clip_thresholds(w.calib, R)
    return w, R, T


def test_rope_int2_latent_groups_match_the_bf16_rope_cache():
    """Quantising the rope key as two more groups leaves the latent's 16 groups (codes
    and scale/zero) bit-identical to the cache that keeps the rope key in bf16."""
    w, R, T = _rope_setup()
    C, KR = w.latent[0], w.rope[0]
    TR = oint2.rope_thresholds(KR.astype(np.float64))
    codes, sz = oint2.quantize(C, R.astype(np.float32), T.astype(np.float32))
    c2, s2 = oint2.quantize_rope_int2(C, KR, R.astype(np.float32), T.astype(np.float32), TR.astype(np.float32))
    assert c2.shape == (C.shape[0], 144) and s2.shape == (C.shape[0], 18, 2)
    np.testing.assert_array_equal(c2[:, :128], codes)
    np.testing.assert_array_equal(s2[:, :16], sz)


def test_rope_int2_is_lossless_on_four_level_keys():
    """Rope groups whose values are the four levels -1.5, -0.5, 0.5, 1.5 (clip 1.5)
    encode with scale 1 and zero -1.5 exactly, decode exactly, and the attention over
    the rope-INT2 row equals the attention over the bf16-rope cache."""
    w, R, T = _rope_setup()
    rng = np.random.default_rng(3)
    n = w.latent[0].shape[0]
    levels = np.array([-1.5, -0.5, 0.5, 1.5], np.float32)
    KR = levels[rng.integers(0, 4, size=(n, 64))]
    KR[:, [0, 32]] = -1.5
    KR[:, [1, 33]] = 1.5                 # every token's two groups span the full range
    TR = np.array([1.5, 1.5], np.float32)
    c2, s2 = oint2.quantize_rope_int2(w.latent[0], KR, R.astype(np.float32), T.astype(np.float32), TR)
    Y = oint2.decode(c2, s2)
    np.testing.assert_array_equal(Y[:, 512:], KR)
    np.testing.assert_array_equal(oint2.unpack_codes(c2)[:, 512:], (KR + 1.5).astype(np.int64))
    o1, l1 = oint2.attention_rope_int2(w.q[0], Y.astype(np.float64), R, w.W_UV, w.scale)
    o2, l2 = oint2.attention_rotated(w.q[0], Y[:, :512], KR, R, w.W_UV, w.scale)
    assert np.max(np.abs(o1 - o2)) < 1e-12 and np.max(np.abs(l1 - l2)) < 1e-12


def test_joint_rotation_attention_is_exact_without_quantisation():
    """With the rotated row kept exact, the jointly rotated attention is the plain
    absorbed attention: scores through q . R_j, output through o_j . R_j^T (a Haar
    rotation, not symmetric, so an R_j / R_j^T swap anywhere fails)."""
    rng = np.random.default_rng(5)
    L, H, r, dR = 40, 4, 512, 64
    C = rng.standard_normal((L, r))
    KR = rng.standard_normal((L, dR))
    q = rng.standard_normal((2, H, r + dR))
    W = rng.standard_normal((H, r, 16)) / np.sqrt(r)
    Rj = workloads.haar_orthogonal(rng, r + dR)
    Y = np.concatenate([C, KR], 1) @ Rj
    o1, l1 = oint2.attention_joint(q, Y, Rj, W, 0.05)
    o2, l2 = attention.absorbed(q, C, KR, W, 0.05)
    assert np.max(np.abs(o1 - o2)) < 1e-10 and np.max(np.abs(l1 - l2)) < 1e-10


def test_rope_variants_study():
    """Bytes and error of the three rope-key layouts on the INT2 workload's law (the
    comparison reported in the design notes). Per token: bf16 rope key 128 B codes +
    64 B scale/zero + 128 B rope = 320 B; rope-INT2 and joint 144 B + 72 B = 216 B.
    INT2 costs each covered dim about the same relative error (~0.38 on this law), so
    both variants add about 4 % to the score error of the bf16-rope cache."""
    w = workloads.int2_rotated(4, B=4, H=32, len_range=(512, 768), n_calib=32768)
    rng = np.random.default_rng(11)
    KRcal = workloads.bf16_round(rng.standard_normal((32768, 64)).astype(np.float32)).astype(np.float64)
    R, _ = oint2.fit_rotation(w.calib)
    T = oint2.clip_thresholds(w.calib, R)
    TR = oint2.rope_thresholds(KRcal)
    Xj = np.concatenate([w.calib, KRcal], axis=1)
    Rj, _ = oint2.fit_rotation(Xj)
    Tj = oint2.clip_thresholds(Xj, Rj)
    R32, T32, TR32, Rj32, Tj32 = (a.astype(np.float32) for a in (R, T, TR, Rj, Tj))
    res = {}
    for b in range(w.B):
        C, KR, q = (a.astype(np.float64) for a in (w.latent[b], w.rope[b], w.q[b]))
        K = np.concatenate([C, KR], 1)
        S = q[0] @ K.T
        ref, rl = attention.absorbed(q, C, KR, w.W_UV, w.scale)
        codes, sz = oint2.quantize(C, R32, T32)
        Ch = oint2.decode(codes, sz).astype(np.float64)
        c2, s2 = oint2.quantize_rope_int2(C, KR, R32, T32, TR32)
        Y2 = oint2.decode(c2, s2).astype(np.float64)
        c3, s3 = oint2.quantize(K, Rj32, Tj32)
        Y3 = oint2.decode(c3, s3).astype(np.float64)
        layouts = (
            ("bf16 rope", codes.nbytes + sz.nbytes + KR.shape[0] * 64 * 2, np.concatenate([Ch @ R.T, KR], 1),
             oint2.attention_rotated(q, Ch, KR, R, w.W_UV, w.scale)),
            ("rope-INT2", c2.nbytes + s2.nbytes, np.concatenate([Y2[:, :512] @ R.T, Y2[:, 512:]], 1),
             oint2.attention_rope_int2(q, Y2, R, w.W_UV, w.scale)),
            ("joint", c3.nbytes + s3.nbytes, Y3 @ Rj.T, oint2.attention_joint(q, Y3, Rj, w.W_UV, w.scale)),
        )
        for name, nbytes, Kh, (o, l) in layouts:
            row = (nbytes / C.shape[0], np.linalg.norm(q[0] @ Kh.T - S) / np.linalg.norm(S),
                   np.linalg.norm(Kh[:, 512:] - KR) / np.linalg.norm(KR),
                   np.linalg.norm(o - ref) / np.linalg.norm(ref), float(np.max(np.abs(l - rl))))
            res.setdefault(name, []).append(row)
    m = {k: np.mean(np.array(v), axis=0) for k, v in res.items()}
    print({k: [round(float(x), 4) for x in v] for k, v in m.items()})
    assert m["bf16 rope"][0] == 320 and m["rope-INT2"][0] == 216 and m["joint"][0] == 216
    assert m["bf16 rope"][2] == 0.0                      # rope key kept exactly
    for name in ("rope-INT2", "joint"):
        assert 0.3 < m[name][2] < 0.5                    # INT2 error on the rope dims
        assert 1.0 < m[name][1] / m["bf16 rope"][1] < 1.1
