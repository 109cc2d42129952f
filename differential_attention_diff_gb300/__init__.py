"""Differential attention (V1 and V2) for NVIDIA GB300, sm_103a.

The operator lives in the C-ABI library ``libdiffattn.so`` (``include/diffattn.h``);
``binding`` is its thin Python binding.  Build with
``python -m differential_attention_diff_gb300.build``.
"""

from .binding import (  # noqa: F401
    DiffAttnError,
    diffattn_get_device_status,
    diffattn_lambda_init,
    diffattn_v1_bwd,
    diffattn_v1_fwd,
    diffattn_v2_decode,
    diffattn_v2_decode_num_splits,
    diffattn_v2_decode_workspace_size,
    diffattn_v2_fwd,
    diffattn_v2_gate,
    load,
)
