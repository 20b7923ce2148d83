"""Plain fp64 CPU oracle for query-aware sparse KV selection.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only the test suite, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may use it.  It shares no code with
the CUDA library (no headers, helpers, tables or constant generators); the two
meet only through the seeded input generators in ``synth``.

Every function restates a definition from one of the source pages in the
plainest form that a reader can check by eye:

* "TokenSelect" = the explainer page "論文解説: TokenSelect — 動的トークン
  レベルKVキャッシュ選択による長文推論の高速化" (arXiv 2411.05159).
* "SnapKV" = the explainer page "NeurIPS 2024論文解説: SnapKV — 生成前に
  KVキャッシュの重要トークンを選択する手法" (arXiv 2402.02938).
* "TokenButler" = the summary page "Technische Zusammenfassung: TokenButler"
  (arXiv 2503.07518).

Floating point is fp64 throughout; the only other rounding is the explicit
round-to-nearest-even to bf16 of the stored compressed key index.

Pins (what fixes this oracle other than itself) live in
``tests/test_oracle_pins.py``.  Parity status per function:

* ``bf16.round_bf16``            pinned (hand values, torch cast)
* ``tokenselect.index_rows``     pinned (selector projections, exact cases)
* ``tokenselect.query_index``    pinned (selector projection, GQA mapping)
* ``tokenselect.scores``         pinned (hand example, GQA mapping)
* ``tokenselect.thresholds``     pinned (order-statistic definition)
* ``tokenselect.select``         pinned (subset enumeration, H=1 top-K,
                                   hand example, V_min property)
* ``tokenselect.sparse_attention`` pinned (dense SDPA at 100 % budget,
                                   closed-form uniform cases)
* ``snapkv.*``                   pinned (identity at c>=n, library pooling,
                                   closed-form uniform case, softmax sums)
* ``tokenselect.select_per_kv_head``, ``sparse_attention_per_head``
                                 pinned (tests/test_oracle_pins_per_head.py)
* ``tokenselect.expand_neighbors`` pinned (tests/test_oracle_pins_expand.py)
* ``paged.*``                    pinned (hand-worked pages and ring, pool cut
                                   from a contiguous cache by reshapes, page
                                   permutation, flush round trip;
                                   tests/test_oracle_pins_paged.py)
"""

from . import bf16, tokenselect, snapkv, paged  # noqa: F401
