"""fp64 CPU oracle (test infrastructure only; see lce_oracle's header)."""
from .lce_oracle import (  # noqa: F401
    forward, forward_backward, out_of_range_targets, sampled_reference, valid_rows,
)
from .optim_oracle import optimizer_step  # noqa: F401
from .embed_oracle import embedding_backward, embedding_forward  # noqa: F401
