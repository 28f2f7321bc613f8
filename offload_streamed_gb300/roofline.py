"""Work, traffic and time bounds of one streamed forward + backward step.

The benchmark's accounting: FLOPs, host-link bytes and the roofline times it
reports.  Page keys:
  tm_zero_infinity   aicassindra.com/blogs/transformer_math/tm_zero_infinity.html
  gpu_zero_sharding  aicassindra.com/blogs/gpu/gpu_zero_sharding.html

One step over Y [T, M] = X [T, K] . W [K, M]:
  * FLOPs: forward 2 per weight and token, backward 4 (tm_zero_infinity,
    "The FLOPs-per-byte test every tier must pass": 2P forward and 4P backward
    per token), so 6 T K M;
  * host -> device: W once for the forward and once more for the backward,
    which fetches every tile again after the forward freed it (same section:
    parameters climb the hierarchy twice per step; gpu_zero_sharding,
    "End-to-end flow"), 2 bytes per weight each time: 4 K M bytes;
  * device -> host: dW once, 2 bytes per weight: 2 K M bytes.
The time bounds follow tm_zero_infinity, "The honest cost": a step runs at the
pace of whichever of compute and the links binds.
"""
from __future__ import annotations

BF16 = 2


def step_flops(T: int, K: int, M: int) -> float:
    """Forward (2 T K M) plus backward (dX and dW, 2 T K M each)."""
    return 2.0 * T * K * M + 4.0 * T * K * M


def step_h2d_bytes(K: int, M: int) -> float:
    """W over the host link twice per step (forward, then the backward's refetch)."""
    return 2.0 * BF16 * K * M


def step_d2h_bytes(K: int, M: int) -> float:
    """dW back over the host link once per step, bf16."""
    return 1.0 * BF16 * K * M


def ait_h2d(T: int) -> float:
    """Step FLOPs per host->device byte: 6 T K M / 4 K M = 1.5 T."""
    return 1.5 * T


def crossover_tokens(R: float, B_h2d: float) -> float:
    """Smallest T at which compute, not the host->device link, binds a step:
    1.5 T >= R / B_h2d."""
    return R / (1.5 * B_h2d)


def step_bound(T: int, K: int, M: int, R: float, B_h2d: float, B_d2h: float) -> tuple[float, str]:
    """Tightest step time when forward and backward may overlap across the call
    boundary: max(6TKM/R, 4KM/B_h2d, 2KM/B_d2h), and which term binds
    ("tensor", "h2d" or "d2h")."""
    terms = {"tensor": step_flops(T, K, M) / R,
             "h2d": step_h2d_bytes(K, M) / B_h2d,
             "d2h": step_d2h_bytes(K, M) / B_d2h}
    bound = max(terms, key=terms.get)
    return terms[bound], bound


def phase_bound(T: int, K: int, M: int, R: float, B_h2d: float, B_h2d_bidir: float,
                B_d2h_bidir: float) -> tuple[float, float]:
    """Per-phase step time, forward and backward summed separately: the
    forward moves W in (2KM bytes) under 2TKM FLOPs; the backward moves W in
    again and dW out (2KM bytes each way, both directions at once, so at the
    links' concurrent rates) under 4TKM FLOPs.  Returns (t_forward,
    t_backward)."""
    w = BF16 * K * M
    t_f = max(2.0 * T * K * M / R, w / B_h2d)
    t_b = max(4.0 * T * K * M / R, w / B_h2d_bidir, w / B_d2h_bidir)
    return t_f, t_b


def link_seconds(h2d_bytes: float, d2h_bytes: float, B_h2d: float, B_d2h: float, B_bidir: float) -> float:
    """Shortest time the host link needs to move h2d_bytes in and d2h_bytes
    out, with each direction at its solo rate (B_h2d, B_d2h) while it runs
    alone and both at B_bidir each while both run: the two directions run
    together for the smaller amount and the larger one's remainder runs
    alone (when 2 B_bidir is at least either solo rate, as it is on this
    link, overlapping them is never slower)."""
    both = min(h2d_bytes, d2h_bytes)
    return both / B_bidir + (h2d_bytes - both) / B_h2d + (d2h_bytes - both) / B_d2h


def e2e_bound(T: int, K: int, M: int, R: float, act_in: float, act_out: float, B_h2d: float, B_d2h: float,
              B_bidir: float) -> float:
    """A step whose activations also cross the host link (act_in bytes in,
    act_out bytes out, besides the weights' 4 K M in and 2 K M out): no
    faster than its FLOPs at R or its link traffic (link_seconds), whichever
    takes longer.  With no activations and a link-bound step this is the
    per-phase bound's link time, since the weights' bytes already fill the
    backward's two directions equally."""
    return max(step_flops(T, K, M) / R,
               link_seconds(step_h2d_bytes(K, M) + act_in, step_d2h_bytes(K, M) + act_out, B_h2d, B_d2h, B_bidir))


def gemm_flops(T: int, K: int, n: int) -> float:
    """One tile GEMM: forward, dW and dX each do 2 T K n FLOPs over a tile (or
    tile group) of n weight columns."""
    return 2.0 * T * K * n


def gemm_bytes(kind: str, T: int, K: int, n: int, accumulate: bool = True) -> float:
    """Algorithmic HBM bytes of one tile GEMM: each operand read once and each
    output written once; dX (fp32) is read and written once per launch that
    adds to it (the first launch of a pass only writes it).
      fwd: X [T,K], W_i [K,n] in, Y_i [T,n] out (bf16)
      dw:  X [T,K], dY_i [T,n] in, dW_i [K,n] out (bf16)
      dx:  dY_i [T,n], W_i [K,n] in (bf16), dX [T,K] fp32 (read +) write."""
    if kind == "fwd":
        return BF16 * (T * K + K * n + T * n)
    if kind == "dw":
        return BF16 * (T * K + T * n + K * n)
    if kind == "dx":
        return BF16 * (T * n + K * n) + (8.0 if accumulate else 4.0) * T * K
    raise ValueError(f"unknown GEMM kind {kind!r}")
