"""Readers for the text fixtures under tests/golden/ (parsing only)."""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _float(tok: str) -> float:
    try:
        return float(tok)
    except ValueError:
        return float.fromhex(tok)


def read_blocks(name: str = "q4_0_blocks.txt"):
    """List of (name, 18 raw bytes, 32 expected fp32 values)."""
    out, cur = [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "block":
                cur = {"name": rest}
            elif key == "bytes":
                cur["bytes"] = np.frombuffer(bytes.fromhex(rest), dtype=np.uint8)
            elif key == "values":
                cur["values"] = np.array([_float(t) for t in rest.split()], dtype=np.float32)
                out.append((cur["name"], cur["bytes"], cur["values"]))
    return out


def _values(rest: str) -> np.ndarray:
    """Whitespace-separated values; "v*n" stands for n copies of v."""
    vals = []
    for tok in rest.split():
        v, star, n = tok.partition("*")
        vals.extend([_float(v)] * (int(n) if star else 1))
    return np.array(vals, dtype=np.float32)


def read_typed_blocks(name: str = "legacy_blocks.txt"):
    """List of (type name, block name, raw bytes, expected fp32 values: 32 per
    legacy block, 256 per Q4_K super-block)."""
    out, cur, typ = [], {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "type":
                typ = rest
            elif key == "block":
                cur = {"name": rest}
            elif key == "bytes":
                cur["bytes"] = np.frombuffer(bytes.fromhex(rest), dtype=np.uint8)
            elif key == "values":
                cur["values"] = _values(rest)
                out.append((typ, cur["name"], cur["bytes"], cur["values"]))
    return out


def read_mul_mat(name: str = "q4_0_mul_mat_small.txt"):
    rec = {"W": [], "X": [], "Y": [], "S": []}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key in ("M", "K", "N"):
                rec[key] = int(rest)
            elif key == "W":
                rec["W"].append(np.frombuffer(bytes.fromhex(rest), dtype=np.uint8))
            else:
                rec[key].append([_float(t) for t in rest.split()])
    rec["W"] = np.stack(rec["W"])
    rec["X"] = np.array(rec["X"], dtype=np.float32)
    rec["Y"] = np.array(rec["Y"], dtype=np.float64)
    rec["S"] = np.array(rec["S"], dtype=np.float64)
    return rec


def same_f32_bits(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Element-wise: identical fp32 bit patterns, or both NaN (payloads may differ)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    same = a.view(np.uint32) == b.view(np.uint32)
    return same | (np.isnan(a) & np.isnan(b))
