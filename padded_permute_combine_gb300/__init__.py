"""GB300-native MoE token routing: route build, binned / padded gather
(permute), scatter (combine), router-weight gradient and the dense
routing-map compaction, as hand-written sm_103a CUDA kernels behind the C ABI
in include/moe_route.h, with a thin Python binding of the same names."""
from . import autograd  # noqa: F401
from ._lib import MoeError, load  # noqa: F401
from .ops import (  # noqa: F401
    Route,
    moe_binned_gather,
    moe_binned_gather_weighted,
    moe_binned_scatter,
    moe_binned_wgrad,
    moe_check_routing,
    moe_padded_gather,
    moe_padded_gather_weighted,
    moe_padded_scatter,
    moe_padded_wgrad,
    moe_route_build,
    moe_route_build_binned_gather,
    moe_route_build_padded_gather,
    moe_routing_map_to_indices_bwd,
    moe_routing_map_to_indices_fwd,
    moe_topk_gating,
)
