"""GB300-native (sm_103a) Mixture-of-Experts FFN hot path.

Python binding over the C ABI of include/moe.h.  The library is loaded on
first use; nothing here computes on the CPU.
"""
from ._binding import (  # noqa: F401
    LIB_PATH, MoeError, Permutation, Workspace, load_library, moe_grouped_fc1_swiglu, moe_grouped_fc2,
    moe_grouped_ffn_fwd, moe_permute,
    moe_route_topk, moe_unpermute_combine, rows_capacity,
)
from ._binding import (  # noqa: F401
    moe_combine_bwd, moe_grouped_dgrad_fc1, moe_grouped_dgrad_fc2_dswiglu, moe_grouped_ffn_bwd,
    moe_grouped_wgrad, moe_unpermute_sum,
)
from ._binding import (  # noqa: F401
    PermutationMX, moe_grouped_fc1_swiglu_mxfp8, moe_grouped_fc2_mxfp8, moe_grouped_quantize_mxfp8,
    moe_permute_mxfp8, moe_quantize_weights_mxfp8, mx_tile_scale_bytes,
    moe_dequantize_rows_mxfp8, moe_dequantize_weights_mxfp8, moe_unpermute_combine_mxfp8,
    moe_unpermute_combine_nvfp4,
)
from ._binding import (  # noqa: F401
    SCORE_SIGMOID, SCORE_SOFTMAX, moe_route_topk_bwd, moe_route_topk_sigmoid,
)
from .layer import (HostPipeline, MoeBackward, MoeBackwardMX, MoeForward, MoeForwardMX, MxWeights,  # noqa: F401
                    moe_forward)
