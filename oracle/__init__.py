"""CPU oracle for DCP causal multi-token MLA verification attention.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or
execute this package: only the test suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it. It shares
no code with the CUDA library (``decode_context_mla_causal_gb300``) and does
not import it; the only module both sides use is the seeded input generator in
``workloads``, which holds none of the method's arithmetic.

Everything is plain NumPy in float64 and follows the plain definitions:

* ``fp8``        -- decode of FP8 E4M3 codes and of BF16 bit patterns.
* ``metadata``   -- per-row causal boundary, rank-local lengths (by counting),
                    subpage expansion, split bounds, at a static bound.
* ``attention``  -- gather of a global sequence from the interleaved rank
                    pools, global causal attention, per-shard attention and the
                    LSE merge of shard results.
* ``kv_write``   -- the step before the path: the new tokens' slot mapping
                    (-1 where a rank does not own a token), the E4M3 encoding of
                    x / scale (round to nearest even, saturating) and the write
                    into the rank pools.
* ``exchange``   -- the step after the path: each rank's output in the
                    all-to-all wire format (BF16 output, the float32 LSE as two
                    16-bit halves), the all-to-all itself, the combine at the
                    destination, and project-before-merge (a per-head W_V
                    applied to each rank's output before the exchange).

Sources (cited by page title and section throughout):

* "Context Parallel Guide (PCP & DCP)" (ATOM docs), section "Decode Context
  Parallel (DCP) Guide": token->rank interleave, ``--dcp-config``
  ``interleave_size``, "How it works", "DCP + Speculative Decode".
* "Support Kimi-K3 DCP with DSpark" (vLLM PR #52188), review thread: the
  per-row rank-local length formula.
* "[ROCm][MLA][DCP] Support causal multi-token verification" (vLLM PR #51705),
  sections "Implementation" and "Validation": the verify path itself.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``,
``tests/test_kv_write_pins.py`` or ``tests/test_exchange_pins.py`` except the split/partial intermediates, which are implementation-defined and
therefore never compared (only merged outputs and per-rank LSE are).
"""

from . import fp8, metadata, attention, kv_write, exchange  # noqa: F401
