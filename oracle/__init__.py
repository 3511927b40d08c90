"""CPU oracle for MLA chunked prefill over a paged packed-latent KV cache.

TEST INFRASTRUCTURE ONLY.  This package is the slow, obviously-correct CPU
definition that the CUDA path is checked against.  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs
of ``bench.py`` may import it.  The product path (``mla_prefix_cache_gb300`` and
its C-ABI library) never imports, links or calls anything here, and nothing here
imports the product package: the two share no code.

Modules
-------
``mla_oracle``  vectorised numpy oracle (fp32 by default, any float dtype):
                gather + FP8 decode, up-projection, RoPE rotation, unchunked
                full-softmax attention with (out, lse), merge_attn_states, and a
                literal chunk-loop variant.
``brute``       scalar fp64 loops with exactly-rounded sums (math.fsum) for tiny
                inputs, used to pin the vectorised oracle.

Parity status: every function is pinned by ``tests/test_oracle_pins.py`` (closed
forms, invariants, brute force, library cross-checks); none is "parity unpinned".
"""
from . import mla_oracle, brute  # noqa: F401
