"""Planted mistakes in the oracle must be caught by its pins.

Each case copies ``oracle/oracle.c``, applies one textual change that a
plausible bug would make (a dropped term, a flipped sign, a wrong index, a
transposed operand, a wrong tile stride), compiles the copy into a temporary
directory and runs every pin against it: at least one pin has to fail.  The
real oracle source is never modified.  All mutants keep every memory access
in bounds.
"""
import os

import pytest

from oracle import oracle as O
import oracle_pins as P

SRC = os.path.join(os.path.dirname(O.__file__), "oracle.c")

MUTANTS = {
    "forward_drops_last_k": (
        "        for (int64_t k = 0; k < K; ++k) {\n            float x = bf16_to_f32(X[t * K + k]);",
        "        for (int64_t k = 0; k < K - 1; ++k) {\n            float x = bf16_to_f32(X[t * K + k]);"),
    "forward_sign": (
        "yrow[m] = yrow[m] + x * bf16_to_f32(wrow[m]);",
        "yrow[m] = yrow[m] - x * bf16_to_f32(wrow[m]);"),
    "dx_wrong_w_row": (
        "            const uint16_t *wrow = W + k * M;\n            float acc = 0.0f;",
        "            const uint16_t *wrow = W + (K - 1 - k) * M;\n            float acc = 0.0f;"),
    "dw_drops_first_t": (
        "        for (int64_t t = 0; t < T; ++t) {\n            float x = bf16_to_f32(X[t * K + k]);\n            const uint16_t *dyrow",
        "        for (int64_t t = 1; t < T; ++t) {\n            float x = bf16_to_f32(X[t * K + k]);\n            const uint16_t *dyrow"),
    "dw_reversed_column": (
        "dwrow[m] = dwrow[m] + x * bf16_to_f32(dyrow[m]);",
        "dwrow[m] = dwrow[m] + x * bf16_to_f32(dyrow[M - 1 - m]);"),
    "tile_storage_missing_k_stride": (
        "return W[blk * K * C + k * C + col];",
        "return W[blk * C + k * C + col];"),
    "sample_dx_sign": (
        "acc = acc + bf16_to_f32(dY[t * M + m]) * bf16_to_f32(w_at(W, K, wcols, k, m));",
        "acc = acc - bf16_to_f32(dY[t * M + m]) * bf16_to_f32(w_at(W, K, wcols, k, m));"),
    "sample_dw_drops_last_t": (
        "        for (int64_t t = 0; t < T; ++t)\n            acc = acc + bf16_to_f32(X[t * K + k]) * bf16_to_f32(dY[t * M + m]);",
        "        for (int64_t t = 0; t < T - 1; ++t)\n            acc = acc + bf16_to_f32(X[t * K + k]) * bf16_to_f32(dY[t * M + m]);"),
    "sample_y_transposed_x": (
        "acc = acc + bf16_to_f32(X[t * K + k]) * bf16_to_f32(w_at(W, K, wcols, k, m));",
        "acc = acc + bf16_to_f32(X[(k % T) * K + (t % K)]) * bf16_to_f32(w_at(W, K, wcols, k, m));"),
    "round_half_up": (
        "u += 0x7FFFu + ((u >> 16) & 1u);",
        "u += 0x8000u;"),
    "round_truncates": (
        "u += 0x7FFFu + ((u >> 16) & 1u);",
        "u += 0u;"),
    "bf16_widening_shift": (
        "uint32_t u = ((uint32_t)h) << 16;",
        "uint32_t u = ((uint32_t)h) << 15;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mpath = tmp_path / "oracle_mutant.c"
    mpath.write_text(src.replace(old, new))
    lib = O.load(O.build(str(mpath), str(tmp_path / "liboracle_mutant.so"), force=True))
    failures = []
    for pin in P.ALL_PINS:
        try:
            pin(lib)
        except AssertionError as e:
            failures.append(f"{pin.__name__}: {str(e)[:80]}")
    assert failures, f"no pin caught mutant {name}"
