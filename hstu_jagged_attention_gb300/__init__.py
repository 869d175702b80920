"""GB300 (sm_103a) HSTU jagged causal attention forward.

``binding`` exposes the C ABI of ``libhstu.so`` under its own names
(``hstu_attn_fwd``, ``hstu_plan_create``, ...); ``workloads`` draws the
seeded synthetic inputs; ``build`` compiles the library with nvcc.
Importing the package does not load the library; the first call does, and
fails loudly if the library has not been built.
"""
from .binding import (  # noqa: F401
    HstuError,
    Plan,
    hstu_attn_fwd,
    hstu_attn_fwd_noalloc,
    hstu_attn_fwd_plan,
    hstu_last_status,
    hstu_launch_shape,
    hstu_plan_create,
    hstu_plan_destroy,
    hstu_plan_num_items,
    hstu_plan_worklist,
    hstu_set_debug_flags,
    hstu_set_wait_timeout_ns,
    hstu_status_string,
    hstu_trace_read,
    hstu_worklist_build,
)
