"""CPU oracle for the MHLA forward pass: test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.  The library never does.
"""

from .mhla_oracle import *  # noqa: F401,F403
from .mhla_oracle import (  # noqa: F401
    PHI_RELU,
    PHI_RELU_EPS,
    TRANSFORMS,
    apply_transform,
    block_centres,
    block_distances,
    block_of_token,
    blocks_per_axis,
    forward,
    forward_dense,
    forward_listing_normaliser,
    linear_attention,
    mix,
    mixing_matrix,
    num_blocks,
    phi,
    readout,
    summaries,
)
from .mhla_backward import backward, phi_derivative  # noqa: F401,E402
from .mhla_causal import blocks_are_contiguous, forward_causal, forward_causal_dense  # noqa: F401,E402
from .mhla_causal_backward import backward_causal, backward_causal_dense  # noqa: F401,E402
from .mhla_module import LEPE_K, LN_EPS, layer_norm, lepe, linear, module_forward  # noqa: F401,E402
