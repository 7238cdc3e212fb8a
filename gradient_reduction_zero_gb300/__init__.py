"""GB300-native data-parallel / ZeRO-1 step: ring reduce-scatter + average,
global-norm clip, sharded AdamW, bf16 cast and all-gather for N simulated
ranks resident in one GPU's HBM, as hand-written sm_103a CUDA behind a C-ABI
(include/dpz.h).

``dpz`` is the ctypes binding; importing it (or any of its names from this
package) loads libdpz.so and raises ImportError if it is not built: there is
no fallback.  ``memory`` is pure host-side accounting.
"""
import importlib

_BINDING = {"AdamWCfg", "DpzError", "dp_allgather", "dp_allreduce_avg", "dp_grad_global_norm",
            "dp_grad_global_norm_static", "dp_reduce_scatter_avg", "dp_reduce_scatter_avg_range",
            "dp_reduce_scatter_avg_bucket", "dp_grad_norm_finalize", "dp_zero1_step",
            "dp_zero1_update", "dp_zero2_update", "make_cfg", "workspace", "zero1_adamw_step"}


def __getattr__(name):
    if name in ("dpz", "memory"):
        return importlib.import_module(f"{__name__}.{name}")
    if name in _BINDING:
        return getattr(importlib.import_module(f"{__name__}.dpz"), name)
    raise AttributeError(name)
