"""The library's calibration on the GPU: Sigma, the projection energy and |X . R|
against their fp64 definitions, and the whole calibration (GPU Sigma, host eigh, GPU
projection, host percentiles) against the oracle's fit, down to identical INT2 codes
for the cache it calibrates."""
import numpy as np
import pytest

import workloads
from oracle import int2 as oint2
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["f64", "f32", "bf16"])
def test_covariance_matches_the_definition(gpu_lib, dtype):
    import mla_latent_kv_08_gb300 as mla
    import torch
    rng = np.random.default_rng(2)
    X = rng.standard_normal((3000, 200)) * np.exp(rng.uniform(-2, 1, 200))
    tdt = {"f64": torch.float64, "f32": torch.float32, "bf16": torch.bfloat16}[dtype]
    Xd = torch.from_numpy(X).to(tdt).cuda()
    Xr = Xd.double().cpu().numpy()                    # the values the kernel sees
    S = mla.calib_covariance(Xd).cpu().numpy()
    ref = Xr.T @ Xr
    assert np.abs(S - ref).max() <= 1e-13 * np.abs(ref).max()


def test_projection_energy_matches_the_oracle(gpu_lib):
    import mla_latent_kv_08_gb300 as mla
    import torch
    rng = np.random.default_rng(3)
    H, dn, r, dv = 6, 48, 136, 40
    W_UK = rng.standard_normal((H, dn, r))
    W_UV = rng.standard_normal((H, r, dv))
    M = mla.calib_projection_energy(torch.from_numpy(W_UK).cuda(), torch.from_numpy(W_UV).cuda()).cpu().numpy()
    ref = oint2.projection_energy(W_UK, W_UV)
    assert np.abs(M - ref).max() <= 1e-13 * np.abs(ref).max()


def test_project_abs_matches_the_definition(gpu_lib):
    import mla_latent_kv_08_gb300 as mla
    import torch
    rng = np.random.default_rng(4)
    X = rng.standard_normal((1000, 96))
    R = np.linalg.qr(rng.standard_normal((96, 96)))[0]
    got = mla.calib_project_abs(torch.from_numpy(X).cuda(), torch.from_numpy(R).cuda()).cpu().numpy()
    ref = np.abs(X @ R)
    assert np.abs(got - ref).max() <= 1e-13 * ref.max()


def test_calibration_reproduces_the_oracle_fit_and_codes(gpu_lib):
    """65536 calibration latents of the INT2 workload's law: the library's eigenvalues,
    R and clip thresholds equal the oracle's fit within fp64 / fp32 rounding; the cache
    it calibrates holds, bit for bit, the oracle encoder's codes for that R and those
    thresholds, and differs from the oracle-calibrated cache in a tiny fraction of
    codes (the fp32 roundings of R that land on the other side)."""
    import mla_latent_kv_08_gb300 as mla
    import torch
    from oracle import layout
    w = workloads.int2_rotated(4, B=3, H=32, len_range=(40, 200), n_calib=65536)
    R32, clip, wv, R64 = mla.calibrate_rotation(torch.from_numpy(np.asarray(w.calib)).cuda())
    Rref, wref = oint2.fit_rotation(w.calib)
    Tref = oint2.clip_thresholds(w.calib, Rref)
    assert np.abs(wv - wref).max() <= 1e-10 * wref.max()
    assert np.abs(R64 - Rref).max() < 1e-8
    assert np.abs(R32.astype(np.float64) - Rref.astype(np.float32)).max() < 1e-8
    np.testing.assert_allclose(clip, Tref.astype(np.float32), rtol=2e-7)
    shape = gu.shape_for(w, kind=mla.MLA_KV_INT2_ROT)
    cache, st = gu.fill_cache(w, shape, R32, clip)
    torch.cuda.synchronize()
    assert mla.mla_read_status_word(st)[0] == mla.MLA_OK
    mine = [oint2.quantize(w.latent[b], R32, clip) for b in range(w.B)]
    ref_codes = layout.write_paged(w.num_blocks, 64, 128, w.block_table, [x[0] for x in mine], [0] * w.B, np.uint8)
    np.testing.assert_array_equal(cache.codes.cpu().numpy(), ref_codes)
    theirs = [oint2.quantize(w.latent[b], Rref.astype(np.float32), Tref.astype(np.float32)) for b in range(w.B)]
    a = np.concatenate([oint2.unpack_codes(x[0]).ravel() for x in mine])
    b = np.concatenate([oint2.unpack_codes(x[0]).ravel() for x in theirs])
    assert np.mean(a != b) < 1e-4


def test_weighted_calibration_matches_the_oracle(gpu_lib):
    import mla_latent_kv_08_gb300 as mla
    import torch
    w = workloads.int2_rotated(4, B=1, H=16, len_range=(10, 20), n_calib=16384)
    rng = np.random.default_rng(7)
    W_UK = workloads.bf16_round(rng.standard_normal((16, 128, 512)).astype(np.float32) / np.sqrt(512))
    R32, clip, wv, R64 = mla.calibrate_rotation(torch.from_numpy(np.asarray(w.calib)).cuda(),
                                                W_UK=torch.from_numpy(W_UK).to(torch.bfloat16).cuda(),
                                                W_UV=torch.from_numpy(w.W_UV).to(torch.bfloat16).cuda())
    Rref, wref = oint2.fit_rotation_weighted(w.calib, W_UK.astype(np.float64), w.W_UV.astype(np.float64))
    assert np.abs(wv - wref).max() <= 1e-10 * np.abs(wref).max()
    assert np.abs(R64 - Rref).max() < 1e-7
