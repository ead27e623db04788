"""fp64 CPU oracle (test infrastructure only; see ``bsa_oracle`` and ``bsa_oracle_ext``)."""

from .bsa_oracle import (  # noqa: F401
    ORDER_GLOBAL,
    ORDER_GROUPED,
    active_keys,
    backward,
    backward_blocks,
    backward_sampled,
    block_flops,
    check_layout,
    expand_mask,
    forward,
    forward_dense,
    masked_attention,
    oracle_csc,
    oracle_lut,
    query_block,
)
from .bsa_oracle_ext import element_mask, forward_ext, n_blocks  # noqa: F401,E402
from .bsa_oracle_topk import topk_attention, topk_flops  # noqa: F401,E402
