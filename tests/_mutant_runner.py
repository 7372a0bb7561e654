"""Runs every attention pin against one compiled (possibly broken) copy of the
oracle's C source.  Exit status 1 when at least one pin fails, 0 when all pass.
Used by tests/test_oracle_mutants.py in a child process."""
import ctypes
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
from tests import pins  # noqa: E402


def main_rotary(lib_path):
    lib = ctypes.CDLL(lib_path)
    dp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.oracle_rotary.argtypes = [dp, dp, dp, dp, i64, i64, i64, i32]
    lib.oracle_rotary.restype = i32

    def rot(x, c, s, interleaved):
        x = np.ascontiguousarray(x, dtype=np.float64)
        c, s = (np.ascontiguousarray(t, dtype=np.float32) for t in (c, s))
        B, H, N, d = x.shape
        out = np.empty_like(x)
        p = lambda a: ctypes.c_void_p(a.ctypes.data)
        assert lib.oracle_rotary(p(x), p(c), p(s), p(out), B * H, N, d, int(interleaved)) == 0
        return out

    try:
        pins.check_rotary_complex(rot)
    except AssertionError:
        print("failed: check_rotary_complex")
        return 1
    return 0


def _attn_and_bwd(lib):
    i64, dp, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    fn = lib.oracle_attention_qk
    fn.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64, i64, i32, ctypes.c_double, dp, i64, i32, dp]
    fn.restype = i32
    bw = lib.oracle_attention_bwd
    bw.argtypes = [dp, dp, dp, dp, dp, dp, dp, i64, i64, i64, i64, i32, ctypes.c_double, i32]
    bw.restype = i32
    p = lambda a: ctypes.c_void_p(a.ctypes.data)

    def attn(q, k, v, causal, scale):
        q, k, v = (np.ascontiguousarray(a, dtype=np.float64) for a in (q, k, v))
        B, H, N, d = q.shape
        o, lse = np.empty((B, H, N, d)), np.empty((B, H, N))
        assert fn(p(q), p(k), p(v), p(o), p(lse), B * H, N, k.shape[2], d, int(causal), float(scale),
                  None, N, 1, None) == 0
        return o, lse

    def bwd(q, k, v, g, causal, scale):
        q, k, v, g = (np.ascontiguousarray(a, dtype=np.float64) for a in (q, k, v, g))
        B, H, N, d = q.shape
        dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
        assert bw(p(q), p(k), p(v), p(g), p(dq), p(dk), p(dv), B * H, N, k.shape[2], d, int(causal),
                  float(scale), 1) == 0
        return dq, dk, dv

    return attn, bwd


def main_bwd(lib_path):
    attn, bwd = _attn_and_bwd(ctypes.CDLL(lib_path))
    failed = []
    for check in pins.BWD_CHECKS:
        try:
            with np.errstate(all="ignore"):
                check(attn, bwd)
        except AssertionError:
            failed.append(check.__name__)
    print("failed:", ",".join(failed))
    return 1 if failed else 0


def main(lib_path):
    lib = ctypes.CDLL(lib_path)
    i64, dp, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    fn = lib.oracle_attention_qk
    fn.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64, i64, i32, ctypes.c_double, dp, i64, i32, dp]
    fn.restype = i32

    def attn(q, k, v, causal, scale, rows=None):
        q, k, v = (np.ascontiguousarray(a, dtype=np.float64) for a in (q, k, v))
        B, H, N, d = q.shape
        Nk = k.shape[2]
        r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        R = N if r is None else len(r)
        o = np.empty((B, H, R, d))
        lse = np.empty((B, H, R))
        p = lambda a: ctypes.c_void_p(a.ctypes.data)
        st = fn(p(q), p(k), p(v), p(o), p(lse), B * H, N, Nk, d, int(causal), float(scale),
                None if r is None else p(r), R, 2, None)
        assert st == 0
        return o, lse

    failed = []
    for check in pins.ALL_CHECKS:
        try:
            with np.errstate(all="ignore"):
                check(attn)
        except AssertionError:
            failed.append(check.__name__)
    print("failed:", ",".join(failed))
    return 1 if failed else 0


if __name__ == "__main__":
    mode = sys.argv[2] if len(sys.argv) > 2 else ""
    sys.exit({"rotary": main_rotary, "bwd": main_bwd}.get(mode, main)(sys.argv[1]))
