"""Closed forms the pages state for streamed, tiled operators.

TEST INFRASTRUCTURE (like the rest of ``oracle/``): the library never imports
it.  The tests pin these functions to the worked numbers the pages print
(``tests/golden/pages_worked_numbers.json``), and then use them to check the
library's own sizing arithmetic and the benchmark's FLOP / byte accounting.

Page keys used below:
  tm_zero_infinity   aicassindra.com/blogs/transformer_math/tm_zero_infinity.html
  pwwt 5430303       pwwt.cn/news/5430303 (ZeRO-Infinity's three key techniques)
  gpu_zero_sharding  aicassindra.com/blogs/gpu/gpu_zero_sharding.html
"""
from __future__ import annotations

import math

BF16_BYTES = 2


# --- arithmetic intensity --------------------------------------------------
# tm_zero_infinity, "The FLOPs-per-byte test every tier must pass".

def ait(flops: float, nbytes: float) -> float:
    """Arithmetic intensity: FLOPs done per byte moved."""
    return flops / nbytes


def machine_balance(R: float, BW: float) -> float:
    """R / BW: the intensity at which a tier of bandwidth BW stops stalling a
    GPU that sustains R FLOP/s."""
    return R / BW


def tier_hidden(ait_value: float, R: float, BW: float) -> bool:
    """A tier is hidden exactly when ait >= R / BW."""
    return ait_value >= machine_balance(R, BW)


def step_flops_per_token_checkpointed(P: float) -> float:
    """Forward 2P + recomputed forward 2P + backward 4P = 8P per token."""
    return 2 * P + 2 * P + 4 * P


def param_bytes_per_step_checkpointed(P: float) -> float:
    """fp16 parameters climb twice per step: 2 x 2P bytes."""
    return 2 * BF16_BYTES * P


def ait_params_checkpointed(T: float) -> float:
    """8PT / 4P = 2T: parameter-streaming intensity with checkpointing."""
    P = 1.0
    return step_flops_per_token_checkpointed(P) * T / param_bytes_per_step_checkpointed(P)


def tokens_needed_per_link(R: float, BW: float) -> float:
    """Smallest T with 2T >= R/BW (tier table, last column)."""
    return machine_balance(R, BW) / 2


def efficiency(ait_value: float, R: float, BW: float) -> float:
    """tm_zero_infinity, "The honest cost": per-step efficiency against an
    all-HBM run is about min(1, ait / (R/BW)) for the binding tier."""
    return min(1.0, ait_value / machine_balance(R, BW))


def adam_ait(flops: float = 12.0, nbytes: float = 24.0) -> float:
    """Applying the test: the Adam update does ~12 FLOPs per 24 bytes."""
    return ait(flops, nbytes)


def decode_ait(P: float = 1.0) -> float:
    """Pitfalls: autoregressive decode does ~2P FLOPs against 2P bytes."""
    return ait(2 * P, BF16_BYTES * P)


# --- fetch time and prefetch depth -----------------------------------------
# tm_zero_infinity, "Bandwidth-centric partitioning: allgather, not broadcast"
# and "Prefetch depth: how far ahead the pipeline must run".

def t_fetch_owner_broadcast(layer_bytes: float, bw_one: float) -> float:
    return layer_bytes / bw_one


def t_fetch_bandwidth_centric(layer_bytes: float, bw_one: float, dp: int) -> float:
    return layer_bytes / (dp * bw_one)


def prefetch_depth(t_fetch: float, t_layer: float) -> int:
    """Smallest integer d with d >= t_fetch / t_layer (at least 1)."""
    return max(1, math.ceil(t_fetch / t_layer))


def prefetch_buffer_bytes(d: int, layer_bytes: float) -> float:
    """buffer_bytes = d * layer_bytes."""
    return d * layer_bytes


def step_compute_seconds(P: float, tokens: float, R: float) -> float:
    """Checkpointed step compute: 8 * P * tokens / R."""
    return step_flops_per_token_checkpointed(P) * tokens / R


# --- memory-centric tiling --------------------------------------------------
# tm_zero_infinity, "Memory-centric tiling: operators bigger than the device";
# pwwt 5430303, 关键技术一 (具体例子).

def tile_working_bytes(layer_bytes: float, k: int, double_buffered: bool = False) -> float:
    """Working memory layer_bytes / k, doubled when double-buffered."""
    return layer_bytes / k * (2 if double_buffered else 1)


def linear_weight_bytes(K: int, M: int) -> int:
    return K * M * BF16_BYTES


def tile_bytes(K: int, M: int, N: int) -> int:
    """Bytes of one output-dimension tile W_i: K rows of M/N bf16 columns."""
    return K * (M // N) * BF16_BYTES


def ring_bytes(K: int, M: int, N: int, d: int) -> int:
    """Resident weight tiles when d tiles are fetched ahead of the one being
    computed: (d + 1) tiles (d = 1 is the "doubled" double-buffered case)."""
    return (min(d, N - 1) + 1) * tile_bytes(K, M, N)


# --- the streamed linear operator's FLOPs and bytes ------------------------
# tm_zero_infinity, "The FLOPs-per-byte test": forward 2P and backward 4P
# FLOPs per token; with P = K*M weights of one linear map and T tokens.

def linear_flops_forward(T: int, K: int, M: int) -> int:
    return 2 * T * K * M


def linear_flops_backward(T: int, K: int, M: int) -> int:
    return 4 * T * K * M


def linear_h2d_bytes_fwd_bwd(K: int, M: int) -> int:
    """W is fetched once for forward and again for backward (it was freed):
    gpu_zero_sharding, "End-to-end flow" (the backward pays the parameter
    cost again)."""
    return 2 * linear_weight_bytes(K, M)


def linear_d2h_bytes_fwd_bwd(K: int, M: int) -> int:
    """dW (2 bytes per weight) is written back once per step."""
    return linear_weight_bytes(K, M)


def roofline_seconds(T: int, K: int, M: int, R: float, B_h2d: float, B_d2h: float) -> float:
    """Tightest time for one forward + backward: compute, or either link
    direction, whichever binds."""
    flops = linear_flops_forward(T, K, M) + linear_flops_backward(T, K, M)
    return max(flops / R, linear_h2d_bytes_fwd_bwd(K, M) / B_h2d,
               linear_d2h_bytes_fwd_bwd(K, M) / B_d2h)


# --- capacity ceilings ------------------------------------------------------
# tm_zero_infinity, "The ceiling that is advertised, and the one that binds".

def p_max(c_nvme_total_bytes: float, bytes_per_param: float = 16.0) -> float:
    return c_nvme_total_bytes / bytes_per_param
