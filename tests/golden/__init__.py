"""Readers for the hand-worked fixtures in this folder (no arithmetic of the method)."""
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def _lines(name):
    with open(os.path.join(HERE, name)) as f:
        for ln in f:
            ln = ln.strip()
            if ln and not ln.startswith("#"):
                yield ln


def _hex(s):
    return [int(t, 16) for t in s.split()]


def q8_0_blocks():
    """[(x float list of 32, expected 34 bytes)]"""
    out, x = [], None
    for ln in _lines("q8_0_blocks.txt"):
        key, val = ln.split(":", 1)
        if key == "x":
            x = [float(t) for t in val.split()]
            x += [0.0] * (32 - len(x))
        else:
            b = _hex(val)
            b += [0] * (34 - len(b))
            out.append((x, b))
    return out


def int4_blocks():
    """[(x, scale bytes, nibble bytes, dequantised values)]"""
    out, cur = [], {}
    for ln in _lines("int4_blocks.txt"):
        key, val = ln.split(":", 1)
        cur[key] = val
        if key == "back":
            out.append(([float(t) for t in cur["x"].split()], _hex(cur["scale"]),
                        _hex(cur["nibbles"]), [float(t) for t in val.split()]))
            cur = {}
    return out


def f16_values():
    """[(value, binary16 bits)]"""
    return [(float(a), int(b, 16)) for a, b in (ln.split() for ln in _lines("f16_values.txt"))]
