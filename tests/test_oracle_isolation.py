"""The oracle's side of every comparison runs without the product library: importing the oracle
and the seeded input generators, and running the bench's reference arm setup, must not map
``libtq.so`` into the process (the input generators live outside the package for this reason)."""

import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_PROBE = r"""
import sys
sys.path.insert(0, {root!r})
import numpy as np
import workloads
import oracle
from oracle import codec, codebook, layout, pipeline, spectral, tables, headq, attention, rotation
inp = workloads.make_inputs("cfg2", B=1, T=32, Hkv=1, Hq=4)
kc, vc = codec.scheme_codecs("kqv", 4)
orc = pipeline.OracleContext(128, 4, 1, 1, 64, kc, vc, inp.seed)
buf = orc.new_cache()
orc.append(buf, inp.k_f32()[:, :, :32].astype(np.float64), inp.v_f32()[:, :, :32].astype(np.float64), [0])
orc.decode(buf, inp.q, [32])
loaded = [m for m in sys.modules if m.startswith("turboquant_quantized_kv_tq_gb300")]
maps = open("/proc/self/maps").read() if sys.platform.startswith("linux") else ""
print("MODULES", loaded)
print("MAPPED", "libtq.so" in maps)
"""


def test_oracle_and_inputs_do_not_load_the_library():
    out = subprocess.run([sys.executable, "-c", _PROBE.format(root=ROOT)], capture_output=True, text=True,
                         timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    assert "MODULES []" in out.stdout, out.stdout
    assert "MAPPED False" in out.stdout, out.stdout
