"""Quality report of the quantized KV cache on the synthetic regimes (GPU).

For each regime and scheme the keys and values of a scaled-down workload go through the
library's write path; the stored cache is read back with ``tq_dequantize`` (K_hat, V_hat) and
decoded with ``tq_decode_attention`` (o_hat).  Everything is compared with exact float64
attention on the unquantized bf16 inputs:

* scale and direction errors of keys, values and outputs ([TQ-KV] "Métricas de Evaluación":
  error split into scale / SNR and direction): relMSE = sum ||x - x_hat||^2 / sum ||x||^2 and
  the mean of 1 - cos(x, x_hat) over vectors;
* KL(p_ref || p_hat) of the attention distributions and top-5 routing recall (the same
  section's mechanistic proxies), averaged over (batch, query head);
* for HeadQ ([HEADQ] "Cadeia de Evidências Falsificáveis"): the calibrated basis against an
  equal-rank random basis and against the correction applied with the wrong sign.

Scores of the quantized cache are q . K_hat / sqrt(d) in float64, which is what the decode
kernel computes in the rotated domain.  The HeadQ basis is the top-16 eigenvectors of the
centred covariance of the calibration queries, computed here with numpy.

    python quality.py            # prints a markdown table and one JSON line per row
"""

import argparse
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

REGIMES = [
    # (config, label, sizes, schemes)
    ("cfg2", "heavy-tailed (Student-t 3), d=128", dict(B=2, Hkv=2, T=2048),
     [("plain", 4), ("tq", 2), ("tq", 3), ("tq", 4), ("kqv", 2), ("kqv", 3), ("kqv", 4),
      ("qkqv", 2), ("qkqv", 3), ("qkqv", 4), ("squ", 2)]),
    ("sq", "low-rank K and V (rank 16), d=128", dict(B=2, Hkv=2, T=2048),
     [("tq", 2), ("squ", 2), ("kqv", 2), ("tq", 4)]),
    ("cfg4", "outlier channels (log-uniform std), d=128", dict(B=1, Hkv=2, T=4096),
     [("tq", 4), ("kqv", 2), ("kqv", 3), ("kqv", 4), ("qkqv", 4)]),
    ("cfg3", "low-rank keys (rank 16), d=1024", dict(B=2, Hkv=2, T=1024),
     [("tq", 2), ("tq", 4), ("kqv", 2), ("kqv", 4)]),
    # peaked attention on low-rank keys ([TQ-KV] "Contribuciones Clave" 3 reports its KL
    # blow-up at d = 1024): the same recipes with the queries scaled so the exact scores have
    # standard deviation 3 over each regime's tokens, at d = 1024 and at d = 128
    ("cfg3", "low-rank keys, peaked attention (score std 3), d=1024", dict(B=2, Hkv=2, T=1024, score_std=3.0),
     [("tq", 2), ("tq", 4), ("kqv", 2), ("kqv", 4)]),
    ("sq", "low-rank K and V, peaked attention (score std 3), d=128", dict(B=2, Hkv=2, T=1024, score_std=3.0),
     [("tq", 2), ("tq", 4), ("kqv", 2), ("kqv", 4)]),
]


def _torch_bf16(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def _softmax(s):
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=-1, keepdims=True)


def _vec_errors(x, xh):
    """relMSE = sum ||x - x_hat||^2 / sum ||x||^2 over the last axis's vectors (a ratio of sums:
    attention outputs over long contexts have small, widely varying norms), and the mean of
    1 - cos(x, x_hat)"""
    x = x.reshape(-1, x.shape[-1])
    xh = xh.reshape(-1, xh.shape[-1])
    n2 = np.sum(x * x, axis=1)
    ok = n2 > 0
    rel = np.sum((x - xh) ** 2) / np.sum(n2)
    cos = np.sum(x * xh, axis=1)[ok] / np.sqrt(n2[ok] * np.sum(xh * xh, axis=1)[ok] + 1e-300)
    return float(rel), float(np.mean(1.0 - cos))


def _attention_metrics(q, K, Kh, d, G):
    """KL(p_ref || p_hat) and top-5 recall, averaged over (batch, query head)."""
    B, Hq, _ = q.shape
    kls, rec = [], []
    for b in range(B):
        for hq in range(Hq):
            kv = hq // G
            s = K[b, kv] @ q[b, hq] / np.sqrt(d)
            sh = Kh[b, kv] @ q[b, hq] / np.sqrt(d)
            p, ph = _softmax(s), _softmax(sh)
            kls.append(float(np.sum(p * (np.log(p + 1e-300) - np.log(ph + 1e-300)))))
            t1, t2 = set(np.argsort(-s)[:5]), set(np.argsort(-sh)[:5])
            rec.append(len(t1 & t2) / 5.0)
    return float(np.mean(kls)), float(np.mean(rec))


def _reference_output(q, K, V, d, G):
    B, Hq, _ = q.shape
    o = np.zeros((B, Hq, d))
    for b in range(B):
        for hq in range(Hq):
            kv = hq // G
            p = _softmax(K[b, kv] @ q[b, hq] / np.sqrt(d))
            o[b, hq] = p @ V[b, kv]
    return o


def _dequantize_all(kv, B, Hkv, T, d):
    Kh = np.zeros((B, Hkv, T, d))
    Vh = np.zeros((B, Hkv, T, d))
    for b in range(B):
        for h in range(Hkv):
            k, v = kv.dequantize(b, h, 0, T)
            Kh[b, h] = k.cpu().numpy()
            Vh[b, h] = v.cpu().numpy()
    return Kh, Vh


def _row(regime, label, scheme, n, K, V, Kh, Vh, q, o_ref, o_hat, d, G):
    kr, kd = _vec_errors(K, Kh)
    vr, vd = _vec_errors(V, Vh)
    orr, od = _vec_errors(o_ref, o_hat)
    kl, r5 = _attention_metrics(q, K, Kh, d, G)
    return {"regime": regime, "label": label, "scheme": scheme, "n": n,
            "K_relmse": kr, "K_dir": kd, "V_relmse": vr, "V_dir": vd,
            "out_relmse": orr, "out_dir": od, "kl": kl, "top5": r5}


def _calibration_sets(name, inp, sizes):
    """Per-side calibration vectors [H_kv][n][d] for SQU-KV: the regime's own calibration sets
    when it has them, else a separate draw of the same recipe (another seed)."""
    from workloads import make_inputs
    if "calib_k" in inp.extra:
        return inp.extra["calib_k"], inp.extra["calib_v"]
    cal = make_inputs(name, B=1, T=4096, Hkv=sizes["Hkv"], Hq=inp.Hq, seed=inp.seed + 100)
    return cal.k_f32()[0].astype(np.float64), cal.v_f32()[0].astype(np.float64)


def score_scale(q, K, d, G, target_std):
    """Factor that gives the exact scores q . k / sqrt(d) standard deviation ``target_std`` over
    all (batch, query head, token)."""
    s = np.concatenate([(K[b, hq // G] @ q[b, hq] / np.sqrt(d)).ravel()
                        for b in range(q.shape[0]) for hq in range(q.shape[1])])
    return float(target_std / np.std(s))


def run_regime(name, label, sizes, schemes, device, keep=None):
    """Rows of one regime.  ``keep``: a list that receives (scheme, n, cache, inputs, q) for each
    scheme (the tests recompute a row from the oracle's reading of the same cache)."""
    import torch
    from turboquant_quantized_kv_tq_gb300 import QuantizedKVCache
    from turboquant_quantized_kv_tq_gb300.calibration import spectral_tables
    from workloads import CONFIGS, make_inputs
    c = CONFIGS[name]
    G = c["Hq"] // c["Hkv"]
    inp = make_inputs(name, B=sizes["B"], T=sizes["T"], Hkv=sizes["Hkv"], Hq=G * sizes["Hkv"])
    B, Hq, Hkv, d, T = inp.B, inp.Hq, inp.Hkv, inp.d, inp.T
    K = inp.k_f32().astype(np.float64)
    V = inp.v_f32().astype(np.float64)
    q32 = inp.q
    if "score_std" in sizes:
        q32 = (inp.q * score_scale(inp.q.astype(np.float64), K, d, G, sizes["score_std"])).astype(np.float32)
    q = q32.astype(np.float64)
    o_ref = _reference_output(q, K, V, d, G)
    Kt, Vt = _torch_bf16(inp.K).to(device), _torch_bf16(inp.V).to(device)
    rows = []
    for scheme, n in schemes:
        kv = QuantizedKVCache(d, Hq, Hkv, B, (T + 63) // 64 * 64, scheme=scheme, n=n, seed=inp.seed,
                              device=device)
        if scheme == "squ":
            for side, X in enumerate(_calibration_sets(name, inp, sizes)):
                E, sc, _ = spectral_tables(X)
                kv.set_spectral_basis(side, torch.from_numpy(E).to(device), torch.from_numpy(sc).to(device))
        kv.append(Kt, Vt, [0] * B)
        o_hat = kv.decode(torch.from_numpy(q32).to(device), [T] * B).cpu().numpy().astype(np.float64)
        Kh, Vh = _dequantize_all(kv, B, Hkv, T, d)
        rows.append(_row(name, label, scheme, n, K, V, Kh, Vh, q, o_ref, o_hat, d, G))
        if keep is not None:
            keep.append((scheme, n, kv, inp, q32))
    return rows


def run_headq(device):
    """cfg5: HeadQ (TQ-KV n=2 keys + rank-16 side code, 4-bit values) with the calibrated basis,
    an equal-rank random basis, and the calibrated correction applied with the wrong sign; TQ-KV
    n=2 keys without a side code for reference."""
    import torch
    from turboquant_quantized_kv_tq_gb300 import QuantizedKVCache
    from workloads import make_inputs
    inp = make_inputs("cfg5", B=2, T=2048, Hkv=2, Hq=8)
    B, Hq, Hkv, d, T = inp.B, inp.Hq, inp.Hkv, inp.d, inp.T
    G = Hq // Hkv
    K = inp.k_f32().astype(np.float64)
    V = inp.v_f32().astype(np.float64)
    q = inp.q.astype(np.float64)
    o_ref = _reference_output(q, K, V, d, G)
    Kt, Vt = _torch_bf16(inp.K).to(device), _torch_bf16(inp.V).to(device)
    calib = inp.extra["calib"]  # [Hkv][n_calib][d]
    U_cal = np.zeros((Hkv, d, 16), dtype=np.float32)
    for h in range(Hkv):
        x = calib[h].astype(np.float64)
        x = x - x.mean(axis=0, keepdims=True)
        w, vecs = np.linalg.eigh(x.T @ x)
        U_cal[h] = vecs[:, np.argsort(-w)[:16]].astype(np.float32)
    rng = np.random.default_rng(1234)
    U_rand = np.stack([np.linalg.qr(rng.standard_normal((d, 16)))[0] for _ in range(Hkv)]).astype(np.float32)
    cap = (T + 63) // 64 * 64
    qd = torch.from_numpy(inp.q).to(device)

    def cache(U):
        kv = QuantizedKVCache(d, Hq, Hkv, B, cap, scheme=None, seed=inp.seed, k_codec=(2, 1, 0),
                              v_codec=(4, 1, 0), headq_rank=16 if U is not None else 0, device=device)
        if U is not None:
            kv.set_headq_basis(torch.from_numpy(U).to(device))
        kv.append(Kt, Vt, [0] * B)
        return kv

    rows = []
    base = cache(None)
    Kb, Vb = _dequantize_all(base, B, Hkv, T, d)
    # (2-bit keys with 4-bit values and no side code is not a built decode: the output is the
    # exact attention over the dequantized cache, which is what the decode computes)
    o_b = _reference_output(q, Kb, Vb, d, G)
    rows.append(_row("cfg5", "HeadQ regime, d=128", "tq-k2 (no side code)", 2, K, V, Kb, Vb, q, o_ref, o_b, d, G))
    for label, U in (("headq calibrated", U_cal), ("headq random basis", U_rand)):
        kv = cache(U)
        Kh, Vh = _dequantize_all(kv, B, Hkv, T, d)
        o_h = kv.decode(qd, [T] * B).cpu().numpy().astype(np.float64)
        rows.append(_row("cfg5", "HeadQ regime, d=128", label, 2, K, V, Kh, Vh, q, o_ref, o_h, d, G))
        if label == "headq calibrated":
            Kw = 2.0 * Kb - Kh  # base minus the calibrated correction
            r = _row("cfg5", "HeadQ regime, d=128", "headq wrong sign", 2, K, V, Kw, Vh, q, o_ref, o_h, d, G)
            r["out_relmse"] = r["out_dir"] = None  # the decode has no wrong-sign mode
            rows.append(r)
    return rows


def _fmt(x):
    return "—" if x is None else f"{x:.3g}"


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--device", default="cuda:0")
    args = ap.parse_args()
    rows = []
    for name, label, sizes, schemes in REGIMES:
        rows += run_regime(name, label, sizes, schemes, args.device)
    rows += run_headq(args.device)
    print("| regime | scheme | n | K relMSE | K 1-cos | V relMSE | V 1-cos | out relMSE | out 1-cos | KL | top-5 |")
    print("|---|---|---|---|---|---|---|---|---|---|---|")
    for r in rows:
        print(f"| {r['label']} | {r['scheme']} | {r['n']} | {_fmt(r['K_relmse'])} | {_fmt(r['K_dir'])} | "
              f"{_fmt(r['V_relmse'])} | {_fmt(r['V_dir'])} | {_fmt(r['out_relmse'])} | {_fmt(r['out_dir'])} | "
              f"{_fmt(r['kl'])} | {r['top5']:.3f} |")
    for r in rows:
        print(json.dumps(r))


if __name__ == "__main__":
    main()
