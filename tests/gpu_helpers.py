"""Shared helpers of the GPU parity tests: build the same cache on the GPU (through the C ABI)
and in the oracle, and compare fields under the parity rule.

Parity rule (codes and sign bits bit-exact except coordinates within 1e-6 of a decision
boundary, at most 1e-4 of all coordinates; norms within 2 fp32 ulp; rho within 1 fp16 ulp;
attention outputs within 2e-3 relative error, row-normalized max norm).
"""

import numpy as np

from oracle import codec as ocodec
from oracle import headq as oheadq
from oracle.pipeline import OracleContext
from turboquant_quantized_kv_tq_gb300 import QuantizedKVCache
from workloads import make_inputs

BOUNDARY = 1e-6
EXEMPT_FRACTION = 1e-4
ATTN_TOL = 2e-3


def to_torch(arr, dtype):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr))


def scheme_codecs(scheme, n):
    if scheme == "headq":
        # K: TQ-KV n-bit base + HeadQ side code; V: TQ-KV 4-bit
        return ocodec.SideCodec(n, True, False), ocodec.SideCodec(4, True, False)
    return ocodec.scheme_codecs(scheme, n)


def headq_basis(inp, rank=16):
    """Per-KV-head calibration basis (d x rank), fp32, from the calibration queries."""
    return np.stack([oheadq.calibration_basis(inp.extra["calib"][h], rank)
                     for h in range(inp.Hkv)]).astype(np.float32)


class Pair:
    """A GPU cache and an oracle context for the same configuration."""

    def __init__(self, inp, scheme, n, capacity=None, seed=None):
        import torch
        self.inp = inp
        kc, vc = scheme_codecs(scheme, n)
        self.kc, self.vc = kc, vc
        cap = capacity or ((inp.T + 63) // 64 * 64)
        seed = inp.seed if seed is None else seed
        hq = 16 if scheme == "headq" else 0
        self.U = headq_basis(inp) if hq else None
        self.gpu = QuantizedKVCache(inp.d, inp.Hq, inp.Hkv, inp.B, cap, scheme=None, seed=seed,
                                    k_codec=(kc.bits, int(kc.rotate), int(kc.qjl)),
                                    v_codec=(vc.bits, int(vc.rotate), int(vc.qjl)), headq_rank=hq)
        if hq:
            self.gpu.set_headq_basis(torch.from_numpy(self.U).cuda())
        self.orc = OracleContext(inp.d, inp.Hq, inp.Hkv, inp.B, cap, kc, vc, seed,
                                 headq_rank=hq, headq_basis=self.U)

    def append_gpu(self, t0=0, t1=None, start=None, chunk=None):
        """Append tokens [t0, t1) of every slab, in chunks of ``chunk`` tokens."""
        import torch
        t1 = self.inp.T if t1 is None else t1
        chunk = chunk or (t1 - t0)
        for s in range(t0, t1, chunk):
            e = min(t1, s + chunk)
            k = to_torch(self.inp.K[:, :, s:e], self.inp.dtype).cuda()
            v = to_torch(self.inp.V[:, :, s:e], self.inp.dtype).cuda()
            self.gpu.append(k, v, [s] * self.inp.B if start is None else [x + s - t0 for x in start])
        torch.cuda.synchronize()

    def gpu_bytes(self):
        return self.gpu.cache.cpu().numpy()

    def decode_gpu(self, seq_len):
        import torch
        q = torch.from_numpy(self.inp.q).cuda()
        out = self.gpu.decode(q, seq_len)
        torch.cuda.synchronize()
        return out.cpu().numpy().astype(np.float64)


def compare_slab(pair, buf, b, h, T, tokens=None):
    """Compare the GPU-written fields of slab (b, h), tokens [0, T), with the oracle's encoding.

    Returns (n_exempt_mismatches, n_coordinates).  Raises AssertionError on a rule violation.
    """
    inp, orc = pair.inp, pair.orc
    K = inp.k_f32()[b, h, :T].astype(np.float64)
    V = inp.v_f32()[b, h, :T].astype(np.float64)
    exempt_total, coords = 0, 0
    for side, X in (("k", K), ("v", V)):
        o = orc.encode_side(X, side, h)
        g = orc.stored_fields(buf, side, b, h, T)
        nu_o = o["norm"]
        ulp = np.spacing(np.abs(nu_o)).astype(np.float64)
        assert np.all(np.abs(g["norm"].astype(np.float64) - nu_o) <= 2 * ulp + 1e-38), (side, "norm")
        mism = g["codes"] != o["codes"]
        exempt = o["code_margin"] < BOUNDARY
        bad = mism & ~exempt
        assert not bad.any(), (side, "codes", np.argwhere(bad)[:5], o["code_margin"][bad][:5])
        exempt_total += int(mism.sum())
        coords += mism.size
        vec_ok = ~mism.any(axis=1)
        if "signs" in o:
            ulp16 = np.spacing(np.abs(o["rho"])).astype(np.float64)
            drho = np.abs(g["rho"].astype(np.float64) - o["rho"].astype(np.float64))
            assert np.all((drho <= ulp16 + 1e-12) | ~vec_ok), (side, "rho")
            smis = g["signs"] != o["signs"]
            sex = (np.abs(o["Sr"]) < BOUNDARY) | ~vec_ok[:, None]
            assert not (smis & ~sex).any(), (side, "signs", np.argwhere(smis & ~sex)[:5])
            exempt_total += int(smis.sum())
            coords += smis.size
        if side == "k" and "side" in o:
            sc_o, sc_g = o["side_scale"], g["side_scale"]
            same_scale = sc_o == sc_g
            # the scale's fp16 rounding is a decision: max|z|/7 may round the other way only
            # within 1e-6 (relative) of an fp16 midpoint, or where the key's base code differs
            # (exempt, at a cell boundary: its residual, and so z, differs)
            sex_scale = (o["scale_margin"] < BOUNDARY) | ~vec_ok
            assert not (~same_scale & ~sex_scale).any(), \
                ("side scale", np.argwhere(~same_scale & ~sex_scale)[:5])
            exempt_total += int((~same_scale).sum())
            coords += same_scale.size
            # a key whose scale differs has every side code decided against another scale
            zmis = g["side"] != o["side"]
            zex = (o["side_margin"] < BOUNDARY) | ~same_scale[:, None] | ~vec_ok[:, None]
            assert not (zmis & ~zex).any(), ("side code", np.argwhere(zmis & ~zex)[:5])
            exempt_total += int(zmis.sum())
            coords += zmis.size
    return exempt_total, coords


def check_exempt(ex, n):
    """The exempt mismatches of one test: at most 1e-4 of every coordinate it compared."""
    assert ex <= EXEMPT_FRACTION * n, (ex, n, EXEMPT_FRACTION * n)


def rel_err(out, ref):
    """max over (b, h) of ||out - ref||_inf / ||ref||_inf (rows with ref == 0 compare absolutely)."""
    num = np.max(np.abs(out - ref), axis=-1)
    den = np.max(np.abs(ref), axis=-1)
    r = np.where(den > 0, num / np.where(den > 0, den, 1), num)
    return float(np.max(r))


def small_inputs(name, B=2, T=300, Hkv=2, Hq=None, seed=None, d=None):
    from workloads import CONFIGS
    c = CONFIGS[name]
    G = c["Hq"] // c["Hkv"]
    Hq = Hq if Hq is not None else G * Hkv
    return make_inputs(name, B=B, T=T, Hkv=Hkv, Hq=Hq, seed=seed, d=d)
