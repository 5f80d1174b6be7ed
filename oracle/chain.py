"""Full / Reindex / Reuse layer pattern over one shared cache.

Test infrastructure only (see the package docstring).

Follows [card] Key ideas, "CSA2 with three static layer modes": Full makes the global KV and the index,
Reindex reuses an earlier layer's KV but rescores with its own indexer query, Reuse reuses both KV and
Top-K indices; every layer keeps its own query and sliding-window KV. The pages give no order of the
modes; the reading taken for a 20-layer chain with 1 Full, 4 Reindex and 15 Reuse layers is
[F U U U][X U U U] x 4 (every fourth layer makes indices, the first of them Full).
"""

FULL, REINDEX, REUSE = "full", "reindex", "reuse"


def modes(n_layers=20, period=4):
    """Layer modes: layer 0 Full, every `period`-th layer after it Reindex, the rest Reuse."""
    out = []
    for layer in range(n_layers):
        if layer == 0:
            out.append(FULL)
        elif layer % period == 0:
            out.append(REINDEX)
        else:
            out.append(REUSE)
    return out


def index_sources(mode_list):
    """For each layer, the layer whose Top-K indices it attends with: itself for Full/Reindex, the
    nearest earlier Full/Reindex layer for Reuse."""
    src, last = [], None
    for layer, m in enumerate(mode_list):
        if m in (FULL, REINDEX):
            last = layer
        elif last is None:
            raise ValueError("a Reuse layer needs an earlier Full or Reindex layer")
        src.append(last)
    return src
