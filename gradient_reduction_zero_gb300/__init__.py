"""GB300-native data-parallel / ZeRO-1 step: ring reduce-scatter + average,
global-norm clip, sharded AdamW, bf16 cast and all-gather for N simulated
ranks resident in one GPU's HBM, as hand-written sm_103a CUDA behind a C-ABI
(include/dpz.h).  ``dpz`` is the ctypes binding."""
from . import dpz  # noqa: F401  (raises if libdpz.so is not built)
from .dpz import (  # noqa: F401
    AdamWCfg, DpzError, dp_allgather, dp_allreduce_avg, dp_grad_global_norm,
    dp_reduce_scatter_avg, dp_zero1_step, make_cfg, workspace, zero1_adamw_step,
)
