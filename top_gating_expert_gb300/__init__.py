"""GB300-native (sm_103a) MoE layer forward: routing, dispatch, grouped expert FFN and
combine as hand-written CUDA kernels behind a C ABI (``include/moe.h``).

The compute entry points live in :mod:`top_gating_expert_gb300.moe`; importing that
module loads the in-tree CUDA library and fails loudly if it has not been built.
"""
