"""CPU oracle for the differential-attention forward (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (the CUDA library and its Python binding) never imports it and
shares no code with it.
"""

from .diffattn_oracle import (  # noqa: F401
    attention_map,
    diff_attn_head,
    diff_attn_v1,
    diff_attn_v1_decode,
    diff_attn_v2,
    diff_attn_v2_decode,
    difference_map,
    dequant_e4m3,
    e4m3_decode,
    head_rmsnorm,
    lambda_init,
    lambda_reparam,
    sigmoid,
    softmax_rows,
)
from .brute import brute_v1, brute_v2  # noqa: F401
from .backward import diff_attn_v1_backward, diff_attn_v2_backward, lambda_reparam_backward  # noqa: F401
from .projections import diff_v1_layer, diff_v2_layer  # noqa: F401
