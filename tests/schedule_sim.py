"""A discrete model of the streamed operator's schedule, for pinning the
closed forms of its work, traffic and time (test infrastructure).

The model follows the method's steps and their order, not any formula for
their totals.  The pages' sections: tm_zero_infinity, "Prefetch depth" (a
ring d tiles deep) and "Memory-centric tiling" (output-dimension tiles);
gpu_zero_sharding, "End-to-end flow" (backward walks the tiles in reverse and
fetches each again; gradients leave as they are produced).

Three serial resources: the host->device link (B_h2d bytes/s), the
device->host link (B_d2h) and the GPU (R FLOP/s).  Per step:
  forward:  for i = 0..N-1: fetch W_i into a ring slot, then Y_i = X W_i;
  backward: for i = N-1..0: fetch W_i again, dW_i = X^T dY_i into a staging
            slot, write dW_i back, dX += dY_i W_i^T.
A fetch waits for its link and for the ring slot's last reader; a GEMM
waits for the GPU and for its operands; a write-back waits for its link and
its dW_i.  Every transfer and GEMM is issued in program order on its
resource, as streams do.  With ``phase_barrier`` every phase starts when
everything before it has finished.
"""
from __future__ import annotations


def simulate(T: int, K: int, M: int, N: int, d: int, R: float, B_h2d: float, B_d2h: float,
             steps: int, staging: int = 2, phase_barrier: bool = False) -> dict:
    Mi = M // N
    tile = K * Mi * 2                 # bytes of W_i (and of dW_i), bf16
    t_gemm = 2 * T * K * Mi / R       # one tile GEMM: T x Mi outputs, K deep (or K x Mi, T deep)
    link_in = link_out = gpu = 0.0    # when each resource is next free
    slot_free = [0.0] * (d + 1)       # ring slots, used in turn
    stage_free = [0.0] * staging
    fetches = stages = 0
    moved_in = moved_out = 0
    flops = 0.0

    def barrier():
        nonlocal link_in, link_out, gpu
        t = max(link_in, link_out, gpu)
        link_in = link_out = gpu = t

    for _ in range(steps):
        if phase_barrier:
            barrier()
        for i in range(N):            # forward
            s = fetches % (d + 1)
            fetches += 1
            start = max(link_in, slot_free[s])
            landed = start + tile / B_h2d
            link_in = landed
            moved_in += tile
            gpu = max(gpu, landed) + t_gemm
            flops += 2 * T * K * Mi
            slot_free[s] = gpu
        if phase_barrier:
            barrier()
        for i in reversed(range(N)):  # backward
            s = fetches % (d + 1)
            fetches += 1
            start = max(link_in, slot_free[s])
            landed = start + tile / B_h2d
            link_in = landed
            moved_in += tile
            g = stages % staging
            stages += 1
            dw_done = max(gpu, stage_free[g]) + t_gemm
            flops += 2 * T * K * Mi
            out_start = max(link_out, dw_done)
            link_out = out_start + tile / B_d2h
            stage_free[g] = link_out
            moved_out += tile
            gpu = max(dw_done, landed) + t_gemm
            flops += 2 * T * K * Mi
            slot_free[s] = gpu
    return {"seconds": max(gpu, link_in, link_out), "h2d_bytes": moved_in, "d2h_bytes": moved_out,
            "flops": flops}
