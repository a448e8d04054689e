"""Plain fp64 CPU oracle for OptR-style rotated INT2 KV-cache attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product path (``int2_kv_cache_gb300``) never imports, calls or executes it, and
this package imports nothing from the product path (callers hand it the seeded
arrays of ``int2_kv_cache_gb300.workloads``, which hold no arithmetic).

Everything here is written from the method's published description, in float64
numpy, with no blocking, fusion or reordering beyond what the definitions state:

* ``rotations``  -- Sylvester Hadamard, signed Hadamard, skew-symmetric matrix
  exponential ("Output-Aware Rotation for INT2 KV-Cache Quantization", §4.2,
  Eq. 11).
* ``quant``      -- group-wise asymmetric INT2 quantize / dequantize Q_2(.; c, G)
  and the rotated map D_{R,c} (§3.1, Eq. 4; Implementation Details of §5 and
  Table A: group 128, clip ratio c, fp16 scale and zero), 2-bit packing.
* ``cache``      -- the paged cache record layout and the write path
  (key centring §4.1 and Eqs. 19-21, rotation, quantize, pack, append).
* ``attention``  -- decode attention by definition (Eqs. 1-2, 5, rotated query
  Eqs. 22/26), an explicit split-K variant with its log-sum-exp combine.
* ``output``     -- W_O folding (Eqs. 29-31), the post-W_O output (Eqs. 3, 7),
  NMSE, the exact key/value error decomposition (Eq. 8), summary statistics.
* ``calib``      -- the candidate-rotation x clip-ratio sweep scored by post-W_O
  NMSE with argmin selection ("Output-aware INT2 KV-cache rotation evaluation").
* ``optr``       -- Algorithm 1 on one KV head: the key and value losses (Eqs.
  12-16), straight-through gradients (Eq. 18) through R = R^0 exp(A - A^T)
  (Eq. 11), Adam, selection every 20 steps.
* ``report``     -- the per-head output-error report (Figure 5: RMS error as a
  percentage of plain INT2; the Eq. 8 key/value split).
* ``window``     -- BF16 sink and recent windows beside the INT2 cache (§5
  implementation details, Table A; appendix "OptR Algorithm"): membership, the
  window record layout, bf16 rounding, the windowed decode readout.

Every function here is pinned by ``tests/test_oracle_*.py`` against closed
forms, library routines, brute force on tiny inputs or constants printed on the
pages; the page-1 NMSE values (52.35 / 1.96) are the one quantity left
"parity unpinned" (their generator and data recipe are not published).
"""
from . import rotations, quant, cache, attention, output, calib, window, report, optr  # noqa: F401
