"""Planted mistakes: each plausible slip in the oracle must trip a pin.

Every case patches one oracle function with a wrong variant (on the CPU
only), runs the pin tests that should notice, and checks at least one fails.
"""

import numpy as np
import pytest

import oracle.e4m3 as e4m3
import oracle.gemm as gemm
import oracle.quant as quant

from tests import test_oracle_e4m3 as T_e4m3
from tests import test_oracle_gemm as T_gemm
from tests import test_oracle_quant as T_quant


def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def _encode_ties_away(x):
    """Mutant: ties round away from zero instead of to even."""
    x = np.asarray(x, dtype=np.float32)
    out = e4m3._orig_encode(x)
    grid = e4m3._POS_GRID
    mag = np.abs(x).astype(np.float64)
    hi = np.minimum(np.searchsorted(grid, mag), 0x7E)
    lo = np.maximum(hi - 1, 0)
    tie = mag == (grid[lo] + grid[hi]) / 2
    bumped = np.where(tie & (mag <= 448), hi, out & 0x7F).astype(np.uint8)
    return np.where(np.signbit(x), bumped | 0x80, bumped).astype(np.uint8)


def _encode_truncate(x):
    """Mutant: round toward zero."""
    x = np.asarray(x, dtype=np.float32)
    mag = np.abs(x).astype(np.float64)
    code = np.searchsorted(e4m3._POS_GRID, mag, side="right") - 1
    code = np.clip(code, 0, 0x7E).astype(np.uint8)
    return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)


def test_encoder_mutants_are_caught(monkeypatch):
    e4m3._orig_encode = e4m3.encode_rne_sat
    for mutant in (_encode_ties_away, _encode_truncate):
        monkeypatch.setattr(e4m3, "encode_rne_sat", mutant)
        caught = (_fails(T_e4m3.test_encode_matches_library_cast)
                  or _fails(T_e4m3.test_encode_ties_to_even_and_tiny))
        assert caught, mutant.__name__
    monkeypatch.undo()


def test_quant_mutants_are_caught(monkeypatch):
    # reciprocal-multiply instead of division; scale = 448 / amax direction slip
    def recip_block(x, fmt="e4m3"):
        x = np.asarray(x, dtype=np.float32)
        amax = np.float32(np.max(np.abs(x)))
        s = np.float32(amax / np.float32(448))
        if amax == 0:
            return np.zeros(x.shape, np.uint8), s
        return e4m3.encode_rne_sat(x * np.float32(np.float32(1) / s)), s

    def inverted_block(x, fmt="e4m3"):
        x = np.asarray(x, dtype=np.float32)
        amax = np.float32(np.max(np.abs(x)))
        s = np.float32(np.float32(448) / amax) if amax else np.float32(0)
        if amax == 0:
            return np.zeros(x.shape, np.uint8), s
        return e4m3.encode_rne_sat(x * s), s

    for mutant in (recip_block, inverted_block):
        monkeypatch.setattr(quant, "_quant_block", mutant)
        caught = (_fails(T_quant.test_quant_1x128_matches_library, "prefill")
                  or any(_fails(T_quant.test_golden_worked_blocks, *b)
                         for b in T_quant._golden_blocks()))
        assert caught, mutant.__name__
        monkeypatch.undo()


def test_gemm_mutants_are_caught(monkeypatch):
    orig = gemm._block_scaled

    def wrong_scale_row(Ad, sA, Bd, sB_rows):
        # B scale taken from the wrong 128-row tile (off by one tile)
        return orig(Ad, sA, Bd, np.roll(sB_rows, 128, axis=0))

    def scale_at_end(Ad, sA, Bd, sB_rows):
        # scales applied once after the K loop (mean scale): the slip the
        # per-block formula warns against
        return (sA.mean(1)[:, None] * sB_rows.mean(1)[None, :]) * (Ad @ Bd.T)

    def dropped_last_block(Ad, sA, Bd, sB_rows):
        return orig(Ad[:, :-128], sA[:, :-1], Bd[:, :-128], sB_rows[:, :-1])

    def transposed_b(Ad, sA, Bd, sB_rows):
        return orig(Ad, sA, Bd[::-1], sB_rows)

    for mutant in (wrong_scale_row, scale_at_end, dropped_last_block, transposed_b):
        monkeypatch.setattr(gemm, "_block_scaled", mutant)
        caught = (_fails(T_gemm.test_bruteforce, 3, 260, 256)
                  or _fails(T_gemm.test_dequantise_then_matmul))
        assert caught, mutant.__name__
        monkeypatch.undo()


def test_saturation_count_mutants_are_caught(monkeypatch):
    from tests import test_oracle_saturation as T_sat
    limit = np.float32(448)

    def counts_equal(x, fmt="e4m3"):
        # quotients equal to the limit counted too
        x = np.asarray(x, dtype=np.float32)
        amax = np.float32(np.max(np.abs(x)))
        if amax == 0:
            return 0
        s = np.float32(amax / limit)
        with np.errstate(divide="ignore", invalid="ignore"):
            y = (x / s).astype(np.float32)
        return int(np.count_nonzero(~(np.abs(y) < limit)))

    def recip(x, fmt="e4m3"):
        # reciprocal-multiply instead of the division
        x = np.asarray(x, dtype=np.float32)
        amax = np.float32(np.max(np.abs(x)))
        if amax == 0:
            return 0
        s = np.float32(amax / limit)
        with np.errstate(divide="ignore", invalid="ignore"):
            y = (x * np.float32(np.float32(1) / s)).astype(np.float32)
        return int(np.count_nonzero(~(np.abs(y) <= limit)))

    def wide_scale(x, fmt="e4m3"):
        # the scale kept in double: no FP32 rounding of amax / 448
        x = np.asarray(x, dtype=np.float32)
        amax = float(np.max(np.abs(x)))
        if amax == 0:
            return 0
        with np.errstate(divide="ignore", invalid="ignore"):
            y = (x.astype(np.float64) / (amax / 448.0))
        return int(np.count_nonzero(~(np.abs(y) <= 448.0)))

    def nan_not_counted(x, fmt="e4m3"):
        x = np.asarray(x, dtype=np.float32)
        amax = np.float32(np.max(np.abs(x)))
        if amax == 0:
            return 0
        s = np.float32(amax / limit)
        with np.errstate(divide="ignore", invalid="ignore"):
            y = (x / s).astype(np.float32)
        return int(np.count_nonzero(np.abs(y) > limit))

    pins = (T_sat.test_amax_element_against_exact_rounding,
            T_sat.test_quotient_equal_to_limit_is_not_counted,
            T_sat.test_zero_block_and_underflowing_scale,
            T_sat.test_power_of_two_scales_never_saturate)
    for mutant in (counts_equal, recip, wide_scale, nan_not_counted):
        monkeypatch.setattr(quant, "_block_saturations", mutant)
        assert any(_fails(p) for p in pins), mutant.__name__
        monkeypatch.undo()
