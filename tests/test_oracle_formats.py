"""Pins for the oracle's format tables (CPU only).

The e4m3 table and encoder are checked against torch's own float8_e4m3fn
cast (an independent library routine, round-to-nearest-even, which agrees
with the saturating conversion for |v| <= 464) and against the saturation
rule above that.  The e2m1 table and encoder are checked against the
closed-form value list of the format and an independent per-binade
``numpy.rint`` (round-half-even) rounding.  The ``check_*`` functions take
an oracle handle so tests/test_oracle_mutants.py can run them on planted
mistakes.
"""
import numpy as np
import pytest
import torch

E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _f32(x):
    return np.float32(x)


def torch_e4m3_values():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).float().numpy().astype(np.float64)


def torch_e4m3_encode(vals):
    t = torch.tensor(np.asarray(vals, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def e4m3_sweep(rng):
    """Every code value, every midpoint, one fp32 ulp either side of each
    midpoint, and random values -- positive and negative, |v| <= 464."""
    v = torch_e4m3_values()[:127]
    mids = 0.5 * (v[:-1] + v[1:])
    mids32 = mids.astype(np.float32)
    assert (mids32.astype(np.float64) == mids).all()  # midpoints exact
    up = np.nextafter(mids32, np.float32(np.inf))
    dn = np.nextafter(mids32, np.float32(-np.inf))
    rnd = rng.uniform(0, 464, 2000).astype(np.float32)
    lg = (2.0 ** rng.uniform(-12, 8.8, 2000)).astype(np.float32)
    pts = np.concatenate([v.astype(np.float32), mids32, up, dn, rnd, lg,
                          np.float32([464.0, 2.0 ** -10, 0.0])])
    return np.concatenate([pts, -pts])


def check_e4m3_decode(o):
    ref = torch_e4m3_values()
    got = np.array([o.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()
    assert (np.signbit(got[~nan]) == np.signbit(ref[~nan])).all()


def check_e4m3_encode(o):
    rng = np.random.default_rng(11)
    pts = e4m3_sweep(rng)
    ref = torch_e4m3_encode(pts)
    got = np.array([o.e4m3_encode(p) for p in pts], dtype=np.uint8)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(pts[i]), hex(got[i]), hex(ref[i]))
                           for i in bad[:8]]
    # satfinite above the largest finite value (torch gives NaN there)
    for v in [448.5, 464.0001, 470.0, 480.0, 512.0, 1e6, 3.0e38]:
        assert o.e4m3_encode(v) == 0x7E
        assert o.e4m3_encode(-v) == 0xFE
    assert o.e4m3_encode(-0.0) == 0x80
    # satfinite covers infinities; NaN stays NaN
    assert o.e4m3_encode(float("inf")) == 0x7E
    assert o.e4m3_encode(float("-inf")) == 0xFE
    assert o.e4m3_encode(float("nan")) & 0x7F == 0x7F
    # every finite code round-trips
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        assert o.e4m3_encode(o.e4m3_decode(c)) == c


def e2m1_closed_form(v: float) -> int:
    """Independent e2m1 rounding: the format's step is 0.5 on [0, 2), 1 on
    [2, 4), 2 on [4, 6]; numpy.rint rounds half to even, and an even
    multiple of the step is an even code."""
    a = abs(float(v))
    if a < 2.0:
        code = int(np.rint(a * 2.0))            # 0..4  (value m/2)
    elif a < 4.0:
        code = int(np.rint(a)) + 2               # 2..4 -> 4..6
    elif a <= 6.0:
        code = int(np.rint(a / 2.0)) + 4         # 2..3 -> 6..7
    else:
        code = 7
    return code | (8 if np.signbit(v) else 0)


def e2m1_sweep(rng):
    v = np.array(E2M1_VALUES)
    mids = (0.5 * (v[:-1] + v[1:])).astype(np.float32)
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(-np.inf))
    rnd = rng.uniform(0, 8, 4000).astype(np.float32)
    tiny = np.float32([1e-30, 1e-40, 2.0 ** -126, 0.0, 6.0001, 7.0, 1e9])
    pts = np.concatenate([v.astype(np.float32), mids, up, dn, rnd, tiny])
    return np.concatenate([pts, -pts])


def check_e2m1_decode(o):
    for c in range(8):
        assert o.e2m1_decode(c) == E2M1_VALUES[c]
        assert o.e2m1_decode(c | 8) == -E2M1_VALUES[c]
    assert np.signbit(o.e2m1_decode(8))


def check_e2m1_encode(o):
    rng = np.random.default_rng(12)
    for p in e2m1_sweep(rng):
        assert o.e2m1_encode(p) == e2m1_closed_form(p), float(p)
    assert o.e2m1_encode(float("inf")) == 0x7
    assert o.e2m1_encode(float("-inf")) == 0xF


def check_f16_decode(o):
    """IEEE binary16 decode against numpy's float16 (an independent
    library) on all 65536 bit patterns."""
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    got = np.array([o.f16_decode(c) for c in range(65536)])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()
    assert (np.signbit(got[~nan]) == np.signbit(ref[~nan])).all()


def check_swizzle_golden(o):
    from tests.golden_io import swizzle_points
    for t, s, S, off in swizzle_points():
        assert o.swizzle(t, s, S) == off, (t, s, S)


def check_swizzle_permute(o):
    """The page states the swizzle twice: as an index formula and as the
    reshape [T/4, 4, 4, S/4] -> permute(0, 2, 3, 1) -> [T, S].  Check the
    oracle's offsets against the reshape statement, and that the map is a
    bijection on the tile that keeps each 4-row band closed."""
    for S in (4, 8, 16, 32):
        for T in (4, 16, 32, 64):
            lin = np.arange(T * S).reshape(T, S)
            phys = (lin.reshape(T // 4, 4, 4, S // 4)
                    .transpose(0, 2, 3, 1).reshape(T * S))
            # phys[k] = linear index (t*S + s) stored at physical slot k
            where = np.empty(T * S, dtype=np.int64)
            where[phys] = np.arange(T * S)
            for t in range(T):
                for s in range(S):
                    off = o.swizzle(t, s, S)
                    assert off == where[t * S + s], (t, s, S)
                    assert (t // 4) * 4 * S <= off < (t // 4 + 1) * 4 * S
            offs = sorted(o.swizzle(t, s, S)
                          for t in range(T) for s in range(S))
            assert offs == list(range(T * S))


CHECKS = [check_e4m3_decode, check_e4m3_encode, check_e2m1_decode,
          check_e2m1_encode, check_f16_decode, check_swizzle_golden,
          check_swizzle_permute]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__)
def test_format_pins(orc, check):
    check(orc)
