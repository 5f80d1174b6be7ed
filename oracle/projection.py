"""The cache write path, restated plainly: latent projection of hidden states, then pair-merge and FP4 pack.

Test infrastructure only (see the package docstring).

What the pages fix: the upper layers' global KV is projected from the hidden state of a middle layer
([card] Key ideas, "Causal Encoder-Decoder (CED)"), and the cache holds one 512-d latent per two merged
positions in FP4 ([digest] Core Mechanics, "Sequence" and "Channel"). The projection is a linear map with
this project's random weights (no trained weights exist here). Its precision is this project's reading:

  * x_t = fl32(sum_k h[t, k] * w[j, k]) for each latent column j: the dot product of the bf16 hidden row
    and the bf16 weight row, accumulated in float64 and rounded once to fp32. The weight is stored
    output-major, [512][hidden], like a linear layer's weight.
  * The fp32 rows x then go through the pack of `fp4.pack` with merge 2: an odd trailing token is not
    packed.
"""

import numpy as np

from . import fp4


def project(h, w):
    """Latent rows (float32 [T, 512]) of hidden rows h [T, hidden] under the weight w [512, hidden]."""
    h = np.asarray(h, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    return (h @ w.T).astype(np.float32)


def project_pack(h, w, rule, first_entry=0, n_blocks=None, base=None):
    """csa_project_pack for one sequence: project the hidden rows, merge adjacent pairs and pack them as
    entries first_entry, first_entry + 1, ... (block-major bytes, as `fp4.pack`)."""
    x = project(h, w)
    return fp4.pack(x, 2, rule, first_entry, n_blocks, base)
