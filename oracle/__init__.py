"""Plain float64 CPU oracle for the rotated-codebook quantized KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports, calls or
links anything here; only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code, tables or constants with the CUDA library: every table it needs
(codebooks, rotation signs, sketch matrices, cache layout) it builds itself
from the definitions written in its own modules.

Sources.  The method is described by three technical summaries of papers,
cited below by short tags:

* [TQ-KV]  "Resumen Técnico: Inferencia Estadística y Medidas de Calidad de
  Cuantizaciones de Cache KV Inspiradas en TurboQuant"
  (gist.science/es/paper/2605.08114).
* [ABL]    "Resumo Técnico: Ablação, Inferência Estatística e Validação para
  Compressão de KV-Cache" (gist.science/pt/paper/2607.09683).
* [HEADQ]  "Resumo Técnico: HeadQ: Distorção Visível ao Modelo e Correção no
  Espaço de Pontuação para Quantização de KV-Cache"
  (gist.science/pt/paper/2605.03562).

Modules:

* ``codebook``  Beta sphere-marginal density and its Lloyd-Max codebook.
* ``tables``    counter-based SplitMix64 draws: rotation signs D, sketch S.
* ``rotation``  explicit Sylvester Hadamard matrix and R = H D / sqrt(d).
* ``codec``     per-vector encoder (norm split, rotation, scalar code, QJL
  residual sketch, HeadQ side code) and the matching reconstruction.
* ``layout``    the packed cache layout (byte streams, 16-token blocks) and its parser.
* ``attention`` textbook softmax decode attention with grouped query heads.
* ``headq``     calibration basis by PCA and the corrected logits.

Parity status: every function is pinned by ``tests/test_oracle_*.py`` against
closed forms, published values, invariants or brute force.  The HeadQ PCA basis
(``headq.calibration_basis``) is pinned through what is unique about it (an
eigenvector's sign and a degenerate subspace are not): its projector against
a planted subspace, orthonormality, maximal captured variance against other
frames, invariance to a common offset and to scale, and the leading direction
by brute force at d = 2.  It is calibration data handed identically to both
sides, so it never enters a parity comparison.
"""

from . import codebook, tables, rotation, codec, layout, attention, headq, pipeline  # noqa: F401
