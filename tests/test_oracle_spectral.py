"""Pins of the SQU-KV oracle (oracle/spectral.py) against facts that do not depend on it:
- eigen-decomposition identities;
- the rank of data built with a known rank;
- the second moments its scales produce;
- that the storage order is a permutation with the modeled coordinates where the decoder wants
  them;
- hand-checked codes and record bytes;
- nearest-centroid brute force;
- the direction of [ABL]'s finding: SpectralQuant ahead of TurboQuant on low-rank data at the
  same budget."""

import numpy as np
import pytest

from oracle import codebook, codec, layout, rotation, spectral, tables


def _low_rank(n, d, r, noise_var, rng, Q=None):
    if Q is None:
        Q, _ = np.linalg.qr(rng.standard_normal((d, r)))
    return rng.standard_normal((n, r)) @ Q.T + np.sqrt(noise_var) * rng.standard_normal((n, d)), Q


def test_calibration_eigen_identities():
    rng = np.random.default_rng(1)
    X, _ = _low_rank(3000, 64, 8, 0.01, rng)
    E, lam, _ = spectral.calibrate(X)
    U = X / np.linalg.norm(X, axis=1, keepdims=True)
    M = U.T @ U / U.shape[0]
    assert np.allclose(E.T @ E, np.eye(64), atol=1e-12)
    assert np.allclose(M @ E, E * lam[None, :], atol=1e-12)
    assert np.all(np.diff(lam) <= 1e-15)
    assert abs(np.sum(lam) - 1.0) < 1e-12  # trace of the second moment of unit vectors


@pytest.mark.parametrize("r", [4, 16, 24])
def test_effective_dim_recovers_the_rank(r):
    rng = np.random.default_rng(2 + r)
    X, Q = _low_rank(4000, 128, r, 0.01, rng)
    E, lam, d_eff = spectral.calibrate(X)
    assert d_eff == r
    sv = np.linalg.svd(Q.T @ E[:, :r], compute_uv=False)  # principal-angle cosines
    assert np.min(sv) > 0.999


def test_effective_dim_gap_rule_on_fixed_spectra():
    # one dominant eigenvalue does not prune the modeled subspace: the largest ratio wins
    assert spectral.effective_dim(np.array([10.0, 1.0, 1.0, 1.0, 1e-3, 1e-3, 1e-3, 1e-3])) == 4
    assert spectral.effective_dim(np.array([3.0, 3.0, 3.0, 1e-4, 1e-4])) == 3
    assert spectral.effective_dim(np.array([1.0, 0.5, 0.0, 0.0])) == 2  # zeros are floored


def test_storage_order():
    for side, chunk, first in (("k", 32, 8), ("v", 16, 4)):
        r = spectral.rank_of_coord(side)
        assert sorted(r) == list(range(128))
        top = spectral.top_mask(side)
        # the modeled coordinates are the first `first` of every `chunk`-coordinate piece
        assert np.array_equal(np.flatnonzero(top), [c for c in range(128) if c % chunk < first])
        assert np.all(np.diff(r[~top]) > 0)  # tail ranks in increasing coordinate order
    assert spectral.rank_of_coord("k")[[0, 32, 64, 96, 1]].tolist() == [0, 1, 2, 3, 4]
    assert spectral.rank_of_coord("v")[[0, 16, 112, 1]].tolist() == [0, 1, 7, 8]


def test_scales_give_sphere_coordinate_second_moments():
    rng = np.random.default_rng(3)
    d = 128
    X, _ = _low_rank(5000, d, 16, 0.01, rng)
    E, lam, _ = spectral.calibrate(X)
    E32, s32 = spectral.storage_tables(E, lam, "k")
    Z = (spectral.unit_rows(X) @ E32.astype(np.float64)) / s32.astype(np.float64)
    assert np.allclose(np.mean(Z * Z, axis=0), 1.0 / d, rtol=2e-6)  # fp32 rounding of the tables


def test_codes_are_nearest_centroids_and_pack_round_trips():
    rng = np.random.default_rng(4)
    d = 128
    X, _ = _low_rank(400, d, 16, 0.02, rng)
    E, lam, _ = spectral.calibrate(X)
    C4, T4 = codebook.fp32_tables(d, 4)
    C1, T1 = codebook.fp32_tables(d, 1)
    for side in ("k", "v"):
        E32, s32 = spectral.storage_tables(E, lam, side)
        f = spectral.encode(X, side, E32, s32, C4, T4, C1, T1)
        top = spectral.top_mask(side)
        z32 = f["z"].astype(np.float32).astype(np.float64)
        near4 = np.argmin(np.abs(z32[:, top][..., None] - C4.astype(np.float64)), axis=-1)
        clear = f["code_margin"][:, top] > 1e-6
        assert np.array_equal(f["codes"][:, top][clear], near4[clear])
        assert np.array_equal(f["codes"][:, ~top], (f["z"][:, ~top] > 0).astype(np.int64))
        rec = spectral.pack(f["codes"], side)
        assert rec.shape == (400, 32)
        assert np.array_equal(spectral.unpack(rec, side), f["codes"])


def test_record_bytes_by_hand():
    # key side: coordinate 0 modeled with code 13 (s=1, k=5), coordinate 1 modeled with code 2
    # (s=0, k=5), coordinate 8 a floor coordinate with code 1 (positive)
    codes = np.zeros((1, 128), dtype=np.int64)
    codes[0, 0], codes[0, 1], codes[0, 8] = 13, 2, 1
    top = spectral.top_mask("k")
    codes[0, top & (np.arange(128) > 1)] = 7  # s=0, k=0 elsewhere among the modeled ones
    rec = spectral.pack(codes, "k")
    assert rec[0, 0] == 0x55  # magnitudes 5, 5 in the first byte
    assert np.all(rec[0, 1:16] == 0)
    assert rec[0, 16] == 0x01 and rec[0, 17] == 0x01  # signs: coordinate 0 and coordinate 8
    assert np.all(rec[0, 18:] == 0)


def test_reconstruction_uses_each_coordinates_codebook():
    # a vector along one basis direction: every coordinate but that one is ~0
    d = 128
    E = rotation.rotation_matrix(tables.rotation_signs(9, 1, d)).T  # any orthonormal basis
    lam = np.full(d, 1.0 / d)
    C4, T4 = codebook.fp32_tables(d, 4)
    C1, T1 = codebook.fp32_tables(d, 1)
    E32, s32 = spectral.storage_tables(E, lam, "v")
    assert np.allclose(s32, 1.0)
    x = 3.0 * E32[:, 0].astype(np.float64)[None, :]  # coordinate 0 (modeled), z_0 = 1
    f = spectral.encode(x, "v", E32, s32, C4, T4, C1, T1)
    xh = spectral.reconstruct(f["codes"], f["norm"], "v", E32, s32, C4, C1)
    zhat = np.where(spectral.top_mask("v"), C4.astype(np.float64)[np.minimum(f["codes"][0], 15)],
                    C1.astype(np.float64)[np.minimum(f["codes"][0], 1)])
    assert np.allclose(xh[0], 3.0 * (E32.astype(np.float64) @ zhat), atol=1e-6)
    assert f["codes"][0, 0] == 15  # z = 1 is far above the top threshold


def test_low_rank_data_favours_the_calibrated_basis_at_equal_budget():
    # [ABL] "Contribuições Principais" 3 / "Resultados": on structured data calibrated on a
    # separate set, SpectralQuant beats the data-oblivious rotation at the same storage
    rng = np.random.default_rng(6)
    d = 128
    Xc, Q = _low_rank(4000, d, 16, 0.01, rng)
    X, _ = _low_rank(2000, d, 16, 0.01, rng, Q)
    E, lam, d_eff = spectral.calibrate(Xc)
    assert d_eff == 16
    C4, T4 = codebook.fp32_tables(d, 4)
    C1, T1 = codebook.fp32_tables(d, 1)
    E32, s32 = spectral.storage_tables(E, lam, "k")
    f = spectral.encode(X, "k", E32, s32, C4, T4, C1, T1)
    xs = spectral.reconstruct(f["codes"], f["norm"], "k", E32, s32, C4, C1)
    R = rotation.rotation_matrix(tables.rotation_signs(7, tables.STREAM_D_K, d))
    C2, T2 = codebook.fp32_tables(d, 2)
    tqc = codec.SideCodec(2, True, False)
    g = codec.encode(X, tqc, C2, T2, R)
    xt = codec.reconstruct(tqc, g["codes"], g["norm"], C2, R)
    err = lambda a: np.sum((X - a) ** 2) / np.sum(X * X)
    assert err(xs) < 0.5 * err(xt), (err(xs), err(xt))  # measured 0.030 vs 0.116
    assert spectral.pack(f["codes"], "k").shape[1] == layout.pack_codes(g["codes"], 2).shape[1]


def test_scheme_name():
    k, v = codec.scheme_codecs("squ", 2)
    assert k.spectral and v.spectral and not k.qjl and not k.rotate
    with pytest.raises(ValueError):
        codec.scheme_codecs("squ", 3)


def test_pipeline_store_and_read_back():
    # OracleContext with SQU-KV sides: the cache bytes written by append parse back to the
    # encoder's codes and norms, and reconstruct through each head's own tables
    from oracle.pipeline import OracleContext
    rng = np.random.default_rng(8)
    d, B, H, T = 128, 2, 2, 40
    tabs = {}
    for side in ("k", "v"):
        per = []
        for h in range(H):
            Xc, _ = _low_rank(800, d, 8, 0.05, rng)
            E, lam, _ = spectral.calibrate(Xc)
            per.append(spectral.storage_tables(E, lam, side))
        tabs[side] = per
    kc, vc = codec.scheme_codecs("squ", 2)
    orc = OracleContext(d, 4, H, B, 64, kc, vc, 0, spectral_k=tabs["k"], spectral_v=tabs["v"])
    K = rng.standard_normal((B, H, T, d))
    V = rng.standard_normal((B, H, T, d))
    buf = orc.new_cache()
    fields = orc.append(buf, K, V, [0, 0])
    C4, T4 = codebook.fp32_tables(d, 4)
    C1, T1 = codebook.fp32_tables(d, 1)
    for b in range(B):
        for h in range(H):
            for side, X in (("k", K[b, h]), ("v", V[b, h])):
                got = orc.stored_fields(buf, side, b, h, T)
                want = fields[(b, h)][0 if side == "k" else 1]
                assert np.array_equal(got["codes"], want["codes"])
                assert np.array_equal(got["norm"], want["norm"])
            Kh, Vh = orc.reconstruct(buf, b, h, T)
            want_k = spectral.reconstruct(fields[(b, h)][0]["codes"], fields[(b, h)][0]["norm"], "k",
                                          *tabs["k"][h], C4, C1)
            assert np.allclose(Kh, want_k, atol=1e-12)


def test_package_calibration_agrees_with_the_oracle():
    # the package's host calibration (its own numpy code) gives the oracle's eigenvalues, scales
    # and subspace; eigenvectors agree up to sign
    from turboquant_quantized_kv_tq_gb300.calibration import spectral_basis
    rng = np.random.default_rng(9)
    X, _ = _low_rank(3000, 128, 12, 0.02, rng)
    E, lam, d_eff = spectral.calibrate(X)
    E32o, s32o = spectral.rank_tables(E, lam)
    Ep, sp, dp = spectral_basis(X)
    assert dp == d_eff == 12
    assert np.allclose(sp, s32o, rtol=1e-5)
    G = np.abs(Ep[:, :12].astype(np.float64).T @ E32o[:, :12].astype(np.float64))
    assert np.allclose(G, np.eye(12), atol=1e-4)
