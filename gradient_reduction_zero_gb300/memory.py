"""Memory accounting of the arena layouts, per simulated rank.

The ZeRO model-state bytes per GPU for mixed-precision Adam
("Lab 09 — Parallelism, simulated", §4): 2 bytes of bf16 weights, 2 of bf16
gradients and k = 12 bytes of fp32 optimizer state per parameter, with one
more term divided by N at each stage.  rank_buffers() gives the bytes one
simulated rank holds under this library's layouts, so that a caller can
size its buffers and check them against the model.
"""
from __future__ import annotations


def zero_model_state_bytes(params: float, N: int, stage: int, k: int = 12) -> float:
    """Model-state bytes per GPU at ZeRO stage 0..3 (weights 2, grads 2, state k)."""
    w, g, s = 2.0 * params, 2.0 * params, float(k) * params
    if stage == 0:
        return w + g + s
    if stage == 1:
        return w + g + s / N
    if stage == 2:
        return w + (g + s) / N
    if stage == 3:
        return (w + g + s) / N
    raise ValueError("stage must be 0..3")


def rank_buffers(P: int, N: int, layout: str, grad_bytes: int = 2, weight_bytes: int = 2,
                 bucket: int = 0) -> dict:
    """Bytes of each buffer one simulated rank holds.

    layout "zero1": its weight slab, its full gradient slab, and its shard of
    the fp32 master/m/v (dp_zero1_step, or the bucketed dp_*_range calls).
    layout "zero2": its weight slab, its gradient shard in the compact
    shards buffer, its master/m/v shard, and its row of the staging bucket
    (dp_reduce_scatter_avg_bucket, transient: a temporary buffer on top of the
    model state)."""
    C = P // N
    out = {"weights": P * weight_bytes, "master_m_v": 12 * C}
    if layout == "zero1":
        out["grads"] = P * grad_bytes
    elif layout == "zero2":
        out["grad_shard"] = C * grad_bytes
        out["staging_bucket"] = bucket * grad_bytes
    else:
        raise ValueError("layout must be zero1 or zero2")
    return out


def model_state_bytes(buffers: dict) -> int:
    """Model-state bytes of a rank (everything but transient buffers)."""
    return sum(v for k, v in buffers.items() if k != "staging_bucket")
