"""Pins for the oracle encoder, layout, reconstruction, attention and HeadQ (no GPU)."""

import numpy as np
import pytest

from oracle import attention, codebook, codec, headq, layout, rotation, tables
from oracle.pipeline import OracleContext


def test_codes_are_nearest_centroid_brute_force():
    rng = np.random.default_rng(0)
    for d in (8, 128):
        for bits in (1, 2, 3, 4):
            c32, t32 = codebook.fp32_tables(d, bits)
            y = rng.standard_normal((200, d)) / np.sqrt(d)
            codes = codec.quantize_codes(y, t32)
            for i in range(200):
                for j in range(d):
                    if codec.boundary_distance(y[i, j], t32) < 1e-6:
                        continue
                    dist = [abs(np.float32(y[i, j]) - v) for v in c32]
                    assert codes[i, j] == int(np.argmin(dist))


def test_tie_goes_to_lower_cell():
    c32, t32 = codebook.fp32_tables(128, 2)
    assert codec.quantize_codes(np.array([t32[1]], dtype=np.float64), t32)[0] == 1
    assert codec.quantize_codes(np.array([np.nextafter(t32[1], np.float32(1))], dtype=np.float64), t32)[0] == 2


def test_sign_magnitude_table_by_hand():
    # b = 2: c = 0,1,2,3 -> (s, k) = (0,1), (0,0), (1,0), (1,1); b = 3: c = 5 -> s=1, k=1
    s, k = layout.to_sign_magnitude(np.array([0, 1, 2, 3]), 2)
    assert list(s) == [0, 0, 1, 1] and list(k) == [1, 0, 0, 1]
    s, k = layout.to_sign_magnitude(np.array([5, 2]), 3)
    assert list(s) == [1, 0] and list(k) == [1, 1]
    for bits in (1, 2, 3, 4):
        c = np.arange(1 << bits)
        assert np.array_equal(layout.from_sign_magnitude(*layout.to_sign_magnitude(c, bits), bits), c)


def test_packed_bytes_by_hand():
    # d = 8, 4-bit codes 0..7 -> symbols (s<<3)|k: c<8 -> s=0, k=7-c -> 7,6,5,4,3,2,1,0
    b = layout.pack_codes(np.arange(8)[None, :], 4)
    assert list(b[0]) == [0x67, 0x45, 0x23, 0x01]
    # 2-bit codes [3, 0, 2, 1, ...]: symbols 3, 1, 2, 0 -> byte 0b00_10_01_11
    b = layout.pack_codes(np.array([[3, 0, 2, 1, 0, 0, 0, 0]]), 2)
    assert b[0, 0] == 0b00100111 and b[0, 1] == 0b01010101
    # 3-bit: k stream (2-bit) then s stream (1-bit); codes [7, 0, 4, 3, 0, 0, 0, 0]
    b = layout.pack_codes(np.array([[7, 0, 4, 3, 0, 0, 0, 0]]), 3)
    # k = [3, 3, 0, 0, 3, 3, 3, 3] -> bytes 0x0F, 0xFF ; s = [1,0,1,0,0,0,0,0] -> 0x05
    assert list(b[0]) == [0x0F, 0xFF, 0x05]
    # side code nibbles, two's complement, low nibble first
    assert list(layout.pack_side(np.array([[-1, 7, -7, 0]]))[0]) == [0x7F, 0x09]


def test_pack_roundtrip():
    rng = np.random.default_rng(3)
    for bits in (1, 2, 3, 4):
        c = rng.integers(0, 1 << bits, size=(17, 128))
        assert np.array_equal(layout.unpack_codes(layout.pack_codes(c, bits), bits, 128), c)
    z = rng.integers(-7, 8, size=(5, 16))
    assert np.array_equal(layout.unpack_side(layout.pack_side(z), 16), z)


def test_blocks_aligned_and_disjoint():
    shape = layout.CacheShape(3, 2, 64, 128, 3, True, 2, True, 128, 16, 4)
    lay = layout.layout(shape)
    k, v = lay["k"], lay["v"]
    # K block: codes 48 B, norm 4, signs 16, rho 2, side 8, scale 2 per token, 16 tokens each
    assert k["fields"] == {"k_codes": (0, 48), "k_norm": (768, 4), "k_signs": (832, 16), "k_rho": (1088, 2),
                           "k_side": (1120, 8), "k_side_scale": (1248, 2)}
    assert k["block"] == 1280 and v["block"] == 16 * (32 + 4 + 16 + 2)
    assert k["offset"] == 0 and v["offset"] % 256 == 0 and v["offset"] >= 3 * 2 * 4 * k["block"]
    assert lay["total"] == v["offset"] + 3 * 2 * 4 * v["block"]
    owner = np.full(lay["total"], -1, dtype=np.int64)
    for name, _ in layout.side_fields(shape, "k") + layout.side_fields(shape, "v"):
        for b in range(3):
            for h in range(2):
                idx = layout.field_positions(shape, name, b, h, np.arange(64)).ravel()
                assert np.all(owner[idx] == -1), name
                owner[idx] = 1
    assert np.all(owner[:3 * 2 * 4 * k["block"]] == 1)
    assert np.all(owner[v["offset"]:] == 1)


def test_value_streams_grouped_by_16_coordinates():
    # d = 32, 3-bit values with QJL (m = 32): the 2-bit stream (8 B per token) in groups of
    # 16 coordinates = 4 B, then the 1-bit stream (4 B per token) in groups of 2 B; the QJL
    # signs likewise; key fields stay whole records
    shape = layout.CacheShape(1, 1, 16, 32, 4, False, 3, True, 32)
    p = np.array([0, 5])
    got = layout.record_byte_positions(shape, "v_codes", p)
    two = [(j // 4) * 64 + p * 4 + j % 4 for j in range(8)]
    one = [128 + (j // 2) * 32 + p * 2 + j % 2 for j in range(4)]
    assert np.array_equal(got, np.stack(two + one, axis=1))
    sg = layout.record_byte_positions(shape, "v_signs", p)
    assert np.array_equal(sg, np.stack([(j // 2) * 32 + p * 2 + j % 2 for j in range(4)], axis=1))
    kc = layout.record_byte_positions(shape, "k_codes", p)
    assert np.array_equal(kc, p[:, None] * 16 + np.arange(16)[None, :])


def test_zero_vector():
    d = 128
    c32, t32 = codebook.fp32_tables(d, 3)
    R = rotation.rotation_matrix(tables.rotation_signs(0, 1, d))
    S = tables.sketch_matrix(0, 3, d, d)
    f = codec.encode(np.zeros((1, d)), codec.SideCodec(3, True, True), c32, t32, R, S)
    assert f["norm"][0] == 0
    assert np.all(f["codes"] == 3)  # y = 0 sits on the middle threshold t = 0: lower cell
    c_mid = np.float64(c32[3])
    assert abs(float(f["rho"][0]) - abs(c_mid) * np.sqrt(d)) < 1e-3  # r = -C[3] in every coordinate
    xh = codec.reconstruct(codec.SideCodec(3, True, True), f["codes"], f["norm"], c32, R, f["rho"], f["signs"], S)
    assert np.all(xh == 0)


def test_reconstruction_error_matches_codebook_mse():
    # QJL off: E||u - u_hat||^2 = d * MSE(codebook) for uniform unit vectors (rotation keeps them uniform)
    rng = np.random.default_rng(4)
    d = 128
    R = rotation.rotation_matrix(tables.rotation_signs(2, 1, d))
    for bits in (2, 4):
        c, t = codebook.lloyd_max(d, bits)
        c32, t32 = c.astype(np.float32), t.astype(np.float32)
        x = rng.standard_normal((20000, d))
        f = codec.encode(x, codec.SideCodec(bits, True, False), c32, t32, R)
        xh = codec.reconstruct(codec.SideCodec(bits, True, False), f["codes"], f["norm"], c32, R)
        rel = np.sum((x - xh) ** 2, axis=1) / np.sum(x * x, axis=1)
        assert abs(rel.mean() / (d * codebook.mse(c, t, d)) - 1) < 0.02


def test_qjl_reconstruction_unbiased_inner_products():
    rng = np.random.default_rng(6)
    d = 64
    R = np.eye(d)
    c32, t32 = codebook.fp32_tables(d, 2)
    x = rng.standard_normal((1, d))
    a = rng.standard_normal(d)
    base = codec.encode(x, codec.SideCodec(2, False, False), c32, t32, R)
    ests = []
    for _ in range(4000):
        S = rng.standard_normal((d, d)).astype(np.float32)
        f = codec.encode(x, codec.SideCodec(2, False, True), c32, t32, R, S)
        xh = codec.reconstruct(codec.SideCodec(2, False, True), f["codes"], f["norm"], c32, R, f["rho"], f["signs"], S)
        ests.append(a @ xh[0])
    ests = np.array(ests)
    truth = a @ x[0]
    # the stored fp16 rho and fp32 norm bias the mean by < 1e-3 relative
    assert abs(ests.mean() - truth) < 4 * ests.std() / np.sqrt(len(ests)) + 1e-3 * abs(truth)
    xb = codec.reconstruct(codec.SideCodec(2, False, False), base["codes"], base["norm"], c32, R)
    assert abs(ests.mean() - truth) < abs(a @ xb[0] - truth) + 4 * ests.std() / np.sqrt(len(ests))


def test_softmax_shift_invariance():
    # [HEADQ] "Espaço de Pontuação da Chave": a shared key translation shifts all scores equally
    rng = np.random.default_rng(7)
    d, T = 64, 300
    q = rng.standard_normal(d)
    K = rng.standard_normal((T, d))
    V = rng.standard_normal((T, d))
    mu = 3 * rng.standard_normal(d)
    o1 = attention.decode_attention(q, K, V)
    o2 = attention.decode_attention(q, K + mu, V)
    assert np.allclose(o1, o2, atol=1e-12, rtol=0)
    assert np.allclose(attention.softmax(np.arange(5.0)), attention.softmax(np.arange(5.0) + 123.0), atol=1e-15)


def test_attention_brute_force_loops_d8():
    rng = np.random.default_rng(8)
    d, T = 8, 13
    q, K, V = rng.standard_normal(d), rng.standard_normal((T, d)), rng.standard_normal((T, d))
    s = [sum(q[i] * K[j, i] for i in range(d)) / d ** 0.5 for j in range(T)]
    mx = max(s)
    e = [np.exp(v - mx) for v in s]
    tot = sum(e)
    o = [sum(e[j] / tot * V[j, i] for j in range(T)) for i in range(d)]
    assert np.allclose(attention.decode_attention(q, K, V), o, atol=1e-14)


def test_gqa_mapping_and_empty_sequence():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((2, 4, 8))
    K = rng.standard_normal((2, 2, 5, 8))
    V = rng.standard_normal((2, 2, 5, 8))
    out = attention.decode_attention_gqa(q, K, V, [5, 0])
    assert np.allclose(out[0, 3], attention.decode_attention(q[0, 3], K[0, 1], V[0, 1]))
    assert np.all(out[1] == 0)


def test_headq_full_rank_fine_side_code_recovers_scores():
    # special case: r = d and a very fine side quantizer restore the unquantized logits
    rng = np.random.default_rng(10)
    d, T = 16, 50
    K = rng.standard_normal((T, d))
    q = rng.standard_normal(d)
    R = rotation.rotation_matrix(tables.rotation_signs(0, 1, d))
    c32, t32 = codebook.fp32_tables(d, 2)
    f = codec.encode(K, codec.SideCodec(2, True, False), c32, t32, R)
    U = np.eye(d)
    side = codec.headq_encode(K, f["codes"], f["norm"], c32, R, U, side_bits=16)
    kbase = codec.reconstruct(codec.SideCodec(2, True, False), f["codes"], f["norm"], c32, R)
    s_hat = headq.corrected_logits(q, kbase, U, side["side"], side["side_scale"])
    exact = K @ q / np.sqrt(d)
    base_err = np.max(np.abs(kbase @ q / np.sqrt(d) - exact))
    assert np.max(np.abs(s_hat - exact)) < 2e-3 * base_err


def test_headq_wrong_sign_hurts():
    # [HEADQ] "Contribuições Principais" (wrong-sign control): flipping the correction increases error
    rng = np.random.default_rng(12)
    d, T, r = 128, 400, 16
    A = np.linalg.qr(rng.standard_normal((d, 24)))[0]
    calib = rng.standard_normal((4096, 24)) @ A.T + 0.1 * rng.standard_normal((4096, d))
    U = headq.calibration_basis(calib, r)
    K = rng.standard_normal((T, d))
    q = A @ rng.standard_normal(24) + 0.1 * rng.standard_normal(d)
    R = rotation.rotation_matrix(tables.rotation_signs(0, 1, d))
    c32, t32 = codebook.fp32_tables(d, 2)
    f = codec.encode(K, codec.SideCodec(2, True, False), c32, t32, R)
    side = codec.headq_encode(K, f["codes"], f["norm"], c32, R, U)
    kbase = codec.reconstruct(codec.SideCodec(2, True, False), f["codes"], f["norm"], c32, R)
    exact = K @ q / np.sqrt(d)
    good = headq.corrected_logits(q, kbase, U, side["side"], side["side_scale"])
    wrong = headq.corrected_logits(q, kbase, U, -side["side"], side["side_scale"])
    base = kbase @ q / np.sqrt(d)
    e_good, e_base, e_wrong = (np.mean((v - exact) ** 2) for v in (good, base, wrong))
    assert e_good < 0.5 * e_base < e_wrong


def test_pipeline_roundtrip_through_bytes():
    # the stored-and-parsed fields reconstruct exactly what the encoder's fields reconstruct
    rng = np.random.default_rng(13)
    for scheme, n in (("tq", 4), ("kqv", 3), ("qkqv", 4), ("plain", 2)):
        kc, vc = codec.scheme_codecs(scheme, n)
        ctx = OracleContext(128, 4, 2, 2, 64, kc, vc, seed=5)
        buf = ctx.new_cache()
        K = rng.standard_normal((2, 2, 40, 128))
        V = rng.standard_normal((2, 2, 40, 128))
        fields = ctx.append(buf, K, V, [0, 7])
        Kh, Vh = ctx.reconstruct(buf, 1, 1, 47)
        fk, fv = fields[(1, 1)]
        Kd = codec.reconstruct(kc, fk["codes"], fk["norm"], ctx.C_K, ctx.R_K, fk.get("rho"), fk.get("signs"), ctx.S_K)
        assert np.array_equal(Kh[7:], Kd)
        assert np.all(Kh[:7] == 0)
