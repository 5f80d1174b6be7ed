"""Oracle: a plain, slow CPU restatement of the CSA2 sparse-attention path.

TEST INFRASTRUCTURE ONLY. Nothing in the product imports this package: only the tests, the smoke
check in ``__graft_entry__.py`` and the CPU-baseline leg of ``bench.py`` use it. It shares no code,
table or constant with the CUDA library; both sides receive the same seeded inputs and nothing else.

Modules
  fp4        pair-merge, E2M1/E4M3 values, the FP4 quantiser and the block-major cache layout.
  indexer    entry scores, block maxima, Top-K with lower-id tie-break, hierarchical selection.
  attention  sparse attention over selected entries plus the sliding window (fp64), and the dense
             attention used by the "Top-K covering everything" invariant.
  chain      the Full / Reindex / Reuse layer pattern.
  projection the cache write path: latent projection of hidden rows, then pair-merge and pack.

Sources the definitions follow (web pages about the DeepSeek-V4.1-Flash technical report):
  [digest]   "DeepSeek-v4.1 Flash: Pushing the Limits of KV Cache Compression" (paper-digest.app),
             Core Mechanics and Terminology.
  [abstract] "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" (thelatestinai.com),
             Abstract.
  [card]     "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" (observer.broadside
             card), Key ideas.
The pages describe structure only; numeric formats and tie rules are this project's readings and are
spelled out in each function's docstring.

Parity status: every function here is pinned by ``tests/test_oracle_*.py`` against values or
properties that do not come from this package (hand-worked golden bytes, torch's float8 codec,
integer brute force, closed forms of softmax). The absolute attention outputs have no printed value on
the pages to pin against; they are pinned by closed forms and invariants only.
"""

from . import fp4, indexer, attention, chain  # noqa: F401
