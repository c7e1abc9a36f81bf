"""CPU oracle for ragged (head-wise non-uniform) paged decode attention and
Quest-style page top-K.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference arm of ``bench.py`` may import this package.  The library under
``non_uniform_paged_gb300`` never imports it, and this package imports
nothing from there: the two share no code.  Both sides receive their inputs
from the ``synth`` generator module.

Everything here is plain numpy / Python, single-threaded, float64 where the
pages leave the precision open, written for a reader checking it against the
pages by eye rather than for speed:

* ``oracle.tangram``    -- budget scaling, retained-token top-k, ragged page
  tables with budget-aware clustering, the proportional workload split map,
  the per-CTA work list, exact softmax decode attention and the log-sum-exp
  merge (Tangram review page, sections 3.1-3.3);
* ``oracle.flexicache`` -- per-page min/max key vectors, the Quest page bound
  and per-KV-head top-K page selection (FlexiCache review page, "Core method /
  Sparse decode" and "Assumption 2").

Pins (tests marked ``not gpu``) tie each function to something other than
itself; see ``tests/test_oracle_pins.py``.  Every function has at least one
pin; none is "parity unpinned".
"""
from . import tangram, flexicache  # noqa: F401
