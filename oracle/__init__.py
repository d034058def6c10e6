"""Float64 CPU oracle for paged KV attention over a flattened varlen batch.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports this
package; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import or run it.  It shares no code with the CUDA path:
the two meet only in the seeded input generator (``workloads.py``), which holds
none of the method's arithmetic.

Modules, each citing the passage it follows:

* ``flatten`` - the runner's flat-batch tensors (``query_start_loc``,
  ``seq_lens``, ``block_table``, ``slot_mapping``, ``positions``) from a
  schedule, and the slot-mapped KV write ("Model execution", section
  "Flattening a step" and its ``flatten_batch.py`` example).
* ``ref`` - exact attention of every new row over its request's context,
  gathered through the block table, as a plain two-pass softmax in float64
  ("Inside the engine ...", section "Never materialise the TxT matrix": the
  textbook S = QK^T, row softmax, times V; section "Attention over a block
  table, not a contiguous tensor").
* ``brute`` - the same attention by materialising each request's full masked
  score matrix (the textbook form the first page describes).
* ``merge`` - the online softmax (running m and l, accumulator rescaled by
  e^(m_old - m_new)) over key tiles, split-KV partials and their
  log-sum-exp merge (sections "Never materialise the TxT matrix" and
  "Prefill has a full grid; decode at batch 1 has almost none").

* ``cascade`` - attention of requests sharing a block-aligned prefix: the
  plain result over shared ++ own blocks, and its two-level form (prefix
  partial over all rows + per-request suffix partial, merged by log-sum-exp)
  that a cascade kernel computes.
* ``fp8`` - E4M3 codes of an 8-bit KV cache with per-tensor scales (the
  reading taken for the FP8 KV cache the "Model execution" page names; pinned
  in ``tests/test_oracle_fp8.py``).

Pins (``tests/test_oracle.py``) tie these to what the pages and mathematics fix:
the printed flatten example, torch's float64 scaled-dot-product attention on the
contiguous equivalent, closed forms (uniform weights -> prefix mean, one key ->
v, head-constant V -> GQA mapping) and paging/split invariance.
"""

from . import brute, cascade, flatten, merge, ref  # noqa: F401
