"""CPU float64 oracle for the LoLA hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import, call or build anything in this package.  The CUDA library does not depend on
it and shares no code, header, table or helper with it.

* ``lola_ref``: numpy statements of the method (running-state and set-based forms)
  and the closed forms it reduces to;
* ``inc``: the plain-C incremental form, threaded over heads, for full-size workloads,
  with a replay mode that validates another implementation's decisions.
"""
