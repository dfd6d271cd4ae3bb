"""The reciprocal shortcut of the 128x128 weight quantiser (quant4_recip),
modelled in NumPy float32 -- the same IEEE operations the kernel performs:
q' = RN(x * RN(1 / s)) is used only when it is finite and either an exact zero
or has its low 19 fraction bits at least 8 away from zero (mod 2^19); then its
FP8 byte, and whether it is beyond the format's limit, must equal those of the
correctly rounded quotient RN(x / s).  Checked on blocks built to put x / s
within 8 ulps of every FP8 value and midpoint (so the shortcut must give way
there), and on wide-range random data (where it must be the common case).
The GPU tests compare the kernel's bytes with the oracle on the same kind of
data."""

import numpy as np
import pytest

from oracle import e4m3, e5m2

FORMATS = {"e4m3": (e4m3, 448.0), "e5m2": (e5m2, 57344.0)}


def boundary_blocks(nb, seed, lut, limit):
    """nb blocks of 128 values whose quotients x / s sit within 8 ulps of the
    FP8 values and midpoints (both signs); element 0 holds the block's amax."""
    g = np.random.default_rng(seed)
    vals = np.unique(np.abs(lut[np.isfinite(lut)]))
    vals = vals[vals <= limit]
    points = np.concatenate([vals, (vals[1:] + vals[:-1]) / 2.0])
    amax = g.uniform(0.25, 4.0, nb).astype(np.float32)
    s = (amax / np.float32(limit)).astype(np.float32)
    m = g.choice(points[points < limit], (nb, 128)) * g.choice([-1.0, 1.0], (nb, 128))
    q = m * (1.0 + g.integers(-8, 9, (nb, 128)) * 2.0 ** -23)
    x = np.clip((q * s[:, None].astype(np.float64)).astype(np.float32), -amax[:, None],
                amax[:, None])
    x[:, 0] = amax
    return x


def _shortcut(blk, limit):
    amax = np.abs(blk).max(1).astype(np.float32)
    s = (amax / np.float32(limit)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        r = (np.float32(1.0) / s).astype(np.float32)
        q_fast = (blk * r[:, None]).astype(np.float32)
        q_div = (blk / s[:, None]).astype(np.float32)
    bits = q_fast.view(np.uint32)
    f = bits & np.uint32(0x7FFFF)
    finite = (bits & np.uint32(0x7F800000)) != np.uint32(0x7F800000)
    zero = (bits & np.uint32(0x7FFFFFFF)) == 0
    trusted = finite & (zero | ((f >= 8) & (f <= 0x7FFF8)))
    return trusted, q_fast, q_div


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_trusted_quotients_give_the_same_byte_and_count(fmt):
    mod, limit = FORMATS[fmt]
    for seed in range(3):
        blk = boundary_blocks(2048, seed, mod.decode_table(), limit)
        trusted, q_fast, q_div = _shortcut(blk, limit)
        differ = mod.encode_rne_sat(q_fast) != mod.encode_rne_sat(q_div)
        assert not (differ & trusted).any()
        clamp_differ = (np.abs(q_fast) > limit) != ~(np.abs(q_div) <= limit)
        assert not (clamp_differ & trusted).any()
        assert (differ & ~trusted).any()  # the data does reach the divisions
    g = np.random.default_rng(7)
    wide = (g.standard_normal((4096, 128)) *
            np.exp(g.uniform(-30, 30, (4096, 1)))).astype(np.float32)
    wide[:8, 1::2] = 0.0
    wide[8:16] *= np.float32(1e-30)  # tiny scales: reciprocals near the top of the range
    trusted, q_fast, q_div = _shortcut(wide, limit)
    assert not ((mod.encode_rne_sat(q_fast) != mod.encode_rne_sat(q_div)) & trusted).any()
    # the shortcut is the common case; each block's amax gives way (its
    # quotient is the limit itself, a rounding point), almost nothing else
    others = np.ones(wide.shape, bool)
    others[np.arange(wide.shape[0]), np.abs(wide).argmax(1)] = False
    assert trusted[others].mean() > 0.999


def test_planted_slip_is_caught():
    """Trusting every product but those exactly on a rounding point (a window
    of 1 instead of 8) lets wrong bytes through on the boundary data: the
    window is what makes the shortcut exact, and this data is able to show
    it."""
    mod, limit = FORMATS["e4m3"]
    blk = boundary_blocks(4096, 11, mod.decode_table(), limit)
    amax = np.abs(blk).max(1).astype(np.float32)
    s = (amax / np.float32(limit)).astype(np.float32)
    r = (np.float32(1.0) / s).astype(np.float32)
    q_fast = (blk * r[:, None]).astype(np.float32)
    q_div = (blk / s[:, None]).astype(np.float32)
    f = q_fast.view(np.uint32) & np.uint32(0x7FFFF)
    loose = (f >= 1) & (f <= 0x7FFFF - 1)
    differ = mod.encode_rne_sat(q_fast) != mod.encode_rne_sat(q_div)
    assert (differ & loose).any()
