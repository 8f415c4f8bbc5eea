"""Helpers shared by the tests (comparison only; no arithmetic of the method)."""
import re
import os

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def ulp_distance(a, b) -> int:
    """max |ord(a) - ord(b)| with ord the sign-magnitude order of the FP64 bit patterns."""
    ia = np.ascontiguousarray(a, dtype=np.float64).view(np.int64).ravel()
    ib = np.ascontiguousarray(b, dtype=np.float64).view(np.int64).ravel()
    lo = np.int64(-0x8000000000000000)
    oa = np.where(ia < 0, lo - ia, ia)
    ob = np.where(ib < 0, lo - ib, ib)
    same = (oa >= 0) == (ob >= 0)
    with np.errstate(over="ignore"):
        d = np.where(same, np.abs(np.where(same, oa - ob, 0)), np.iinfo(np.int64).max)
    small = (~same) & (np.abs(oa) < 2**40) & (np.abs(ob) < 2**40)
    d = np.where(small, np.abs(oa) + np.abs(ob), d)
    return int(d.max()) if d.size else 0


def decode_x(limbs) -> int:
    """192-bit two's complement little-endian limbs (int64 bit patterns) -> Python int."""
    u = [int(v) & (2**64 - 1) for v in limbs]
    x = u[0] | (u[1] << 64) | (u[2] << 128)
    return x - (1 << 192) if x >> 191 else x


def header_functions():
    """Names of the functions include/ozaki2.h declares."""
    text = open(os.path.join(ROOT, "include", "ozaki2.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ozaki2_\w+)\s*\(", text)))
