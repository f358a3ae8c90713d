"""GB300-native MoE expert-parallel dispatch/combine (layout, notify, dispatch, combine).

The compute path is the C-ABI library ``libep_gb300.so`` built from ``csrc/``
for sm_103a; :mod:`combine_get_dispatch_notify_gb300.ep` is its thin Python
binding.  :mod:`combine_get_dispatch_notify_gb300.workloads` generates seeded
synthetic inputs.
"""
__all__ = ["ep", "workloads"]
