"""Readers for the hand-worked fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.strip()
            if line and not line.startswith("#"):
                yield line


def nvfp4_groups():
    """[(name, g, inputs[16] (float), sf, data bytes[8], dtype)] with dtype
    0 = bf16, 1 = fp16."""
    out = []
    for line in _lines("nvfp4_groups.txt"):
        fields = [p.strip() for p in line.split(";")]
        name, g, xs, sf, data = fields[:5]
        dtype = 1 if len(fields) > 5 and fields[5] == "f16" else 0
        xs = [float(v) for v in xs.split()]
        assert len(xs) == 16, name
        data = bytes.fromhex(data)
        assert len(data) == 8, name
        out.append((name, float(g), xs, int(sf, 16), data, dtype))
    return out


def swizzle_points():
    """[(t, s, S, offset)]"""
    return [tuple(int(v) for v in line.split())
            for line in _lines("swizzle_points.txt")]


def as_bf16_bits(values):
    """Exact bf16 bit patterns of values that bf16 represents exactly."""
    f = np.asarray(values, dtype=np.float32)
    bits = f.view(np.uint32)
    assert ((bits & 0xFFFF) == 0).all(), "value not exact in bf16"
    return (bits >> 16).astype(np.uint16)


def as_f16_bits(values):
    """Exact fp16 bit patterns of values that fp16 represents exactly."""
    f = np.asarray(values, dtype=np.float64)
    h = f.astype(np.float16)
    assert (h.astype(np.float64) == f).all(), "value not exact in fp16"
    return h.view(np.uint16)


def as_bits(values, dtype):
    return as_f16_bits(values) if dtype == 1 else as_bf16_bits(values)
