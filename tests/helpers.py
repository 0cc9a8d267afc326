"""Test helpers: golden-file parsing and the per-element acceptance check."""

from __future__ import annotations

import os

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden_cases(name: str = "textbook_gemm.txt"):
    """Parse a golden file into a list of (case name, {"A","B","C"} arrays)."""
    cases = []
    cur = None
    mat = None
    rows_left = 0
    with open(os.path.join(GOLDEN_DIR, name), encoding="utf-8") as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            if rows_left:
                cur[1][mat].append([float(t) for t in tok])
                rows_left -= 1
                continue
            if tok[0] == "case":
                cur = (tok[1], {})
                cases.append(cur)
            elif tok[0] in ("A", "B", "C"):
                mat = tok[0]
                rows_left = int(tok[1])
                cur[1][mat] = []
            else:
                raise ValueError(f"bad golden line: {raw!r}")
    out = []
    for cname, mats in cases:
        out.append((cname, {k: np.array(v, dtype=np.float32 if k != "C"
                                         else np.float64)
                            for k, v in mats.items()}))
    return out


def within_tolerance(c_test, c_ref, bound, K):
    """Boolean mask of |C - C_ref| <= 1e-5·sqrt(K)·(|A|·|B|) + 1e-30."""
    tol = 1e-5 * np.sqrt(max(K, 0)) * bound + 1e-30
    err = np.abs(np.asarray(c_test, dtype=np.float64) - c_ref)
    return err <= tol


def assert_within_tolerance(c_test, c_ref, bound, K, what=""):
    ok = within_tolerance(c_test, c_ref, bound, K)
    if not ok.all():
        bad = np.argwhere(~ok)
        i = tuple(bad[0])
        err = abs(float(np.asarray(c_test)[i]) - float(c_ref[i]))
        raise AssertionError(
            f"{what}: {bad.shape[0]} of {ok.size} elements outside tolerance; "
            f"first at {i}: got {float(np.asarray(c_test)[i])!r}, "
            f"oracle {float(c_ref[i])!r}, |err| {err:.3e}, "
            f"tol {1e-5 * np.sqrt(K) * bound[i] + 1e-30:.3e}")


def assert_bitexact(c_test, c_ref64, what=""):
    """c_test (float32) must equal float32(c_ref64) bit for bit."""
    a = np.ascontiguousarray(c_test, dtype=np.float32).view(np.uint32)
    b = np.ascontiguousarray(np.asarray(c_ref64).astype(np.float32)).view(
        np.uint32)
    if not np.array_equal(a, b):
        bad = np.argwhere(a != b)
        i = tuple(bad[0])
        raise AssertionError(
            f"{what}: {bad.shape[0]} elements differ bitwise; first at {i}: "
            f"{np.asarray(c_test)[i]!r} vs {np.asarray(c_ref64)[i]!r}")
