"""GB300-native fused Mixture-of-Experts router.

The router's top-K forward/backward and aux-loss score forward/backward run
as hand-written sm_103a CUDA kernels behind a C ABI (include/moe_router.h);
``score_top_expert_gb300.router`` is its Python binding.  The router entry
points are loaded lazily so that ``score_top_expert_gb300.workloads`` (the
seeded input generators) imports without the compiled library.
"""
_ROUTER_NAMES = ("router_topk_fwd", "router_topk_fwd_compact", "router_topk_fwd_maps",
                 "router_expert_maps", "router_topk_bwd",
                 "router_aux_scores_fwd", "router_aux_scores_bwd", "router_aux_loss_fwd", "router_aux_loss_fwd_noalloc",
                 "router_aux_loss_bwd",
                 "force_path", "force_fwd_lanes", "device_status", "selftest_bounded_wait",
                 "RouterError", "lib", "library_path")

__all__ = list(_ROUTER_NAMES)


def __getattr__(name):
    if name in _ROUTER_NAMES:
        from . import router
        return getattr(router, name)
    raise AttributeError(f"module {__name__!r} has no attribute {name!r}")
