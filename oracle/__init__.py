"""CPU fp64 oracle for mask-aware softmax attention (test infrastructure only).

This package defines, plainly and slowly, what the CUDA library computes:

* ``masks``     - which (query i, key j) pairs each mask allows;
* ``attention`` - exact masked softmax attention forward and its analytic
                  backward, in fp64 on the host;
* ``plan``      - the tile classification (skip / full / partial), the per
                  query-tile and per key-tile lists, and the longest-first
                  work orders, by brute force over the materialised mask;
* ``counts``    - valid-pair counts, by popcount and by closed forms;
* ``blockmap``  - block-sparse maps from block scores: mean-pooled query/key block
                  scores and top-k selection per query block.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import it.  It shares no code
with the CUDA path; the only common module is the seeded input generator
``long_context_masked_gb300.inputs``, which holds no attention arithmetic.

Sources: "Long-Context Attention Benchmark: From Kernel Efficiency to
Distributed Context Parallelism" (LongCA-bench): the summary page (sections 2.1.1
"Input Mask Patterns", 2.1.2 "Input Data Sampling", A.2 "Details of Sparse Data
Sampling", A.3 "Details of Sparse Attention Kernels", A.4.1 "Performance Metric: FLOPS") and the reading note page ("Key
design" items 1 and 2).  The pages name the masks and the computation
("standard attention", softmax(QK^T/sqrt(d) + mask)V) but print no formula
beyond that; every reading taken where they are silent is listed in the
docstring of the function that takes it.

Parity pins: every function here is pinned by ``tests/test_oracle_*.py`` against
hand-drawn masks (``tests/golden/``), closed-form pair counts, brute-force
loops, finite differences, a library attention routine and reductions between
masks.  No function is left unpinned.
"""
from . import masks, attention, plan, counts, blockmap  # noqa: F401
from .masks import allowed, mask_rows, materialize_mask, map_head_of  # noqa: F401
from .attention import (attn_fwd_ref, attn_bwd_ref, attn_fwd_rows_ref,  # noqa: F401
                        attn_dq_rows_ref, attn_dkdv_cols_ref)
from .plan import col_list_byte, row_list_byte, tile_plan_ref, tile_rows_ref  # noqa: F401
from .counts import n_valid_popcount, n_valid_closed_form  # noqa: F401
from .blockmap import topk_count, topk_block_map, pooled_block_scores  # noqa: F401
