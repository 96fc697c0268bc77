"""fp64 CPU oracle of MLA decode: test infrastructure, not the product.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs import this package.  The CUDA library
(``mla_latent_kv_82_b300``) never imports it, and the two share no code.

* ``oracle.mla``   -- vectorised float64 explicit and absorbed decode,
                      paged addressing, cache-size closed forms;
* ``oracle.brute`` -- pure-Python scalar decode for tiny inputs;
* ``oracle.fp8``   -- the E4M3 codec and the row quantiser of the FP8
                      cache (the decode over its dequantised rows is
                      ``oracle.mla`` unchanged);
* ``oracle.case``  -- assembles a workload's inputs (from ``synth``) and
                      runs the oracle on whole sequences or samples.

Parity pins live in ``tests/test_oracle.py`` and ``tests/test_oracle_fp8.py``.  Nothing here is "parity
unpinned": every function above is checked there against closed forms,
brute force, special cases or invariants.
"""
from . import mla, brute, fp8  # noqa: F401
