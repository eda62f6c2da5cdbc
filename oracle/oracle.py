"""Python face of the CPU oracle (``fathom_oracle.c``).

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers; the CUDA library never
imports, links or runs anything here, and nothing here imports the CUDA
library.  Every function is argument marshalling over the plain C loops in
``fathom_oracle.c``, which cite the passages of the Fathom review page
("Fathom: 쿼리마다 깊이를 바꾸는 스캔으로 1M 토큰 디코딩을 1.67배 빠르게 하다")
they follow.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fathom_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libfathom_oracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, no fast-math)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _P(t):
    return ctypes.POINTER(t)


_i, _d, _u8, _u16, _u32, _u64, _f, _i32 = (
    ctypes.c_int, ctypes.c_double, ctypes.c_uint8, ctypes.c_uint16,
    ctypes.c_uint32, ctypes.c_uint64, ctypes.c_float, ctypes.c_int32)

_SIGS = {
    "oracle_round_fp16": (_d, [_d]),
    "oracle_fp16_bits": (_u16, [_d]),
    "oracle_fp16_value": (_d, [_u16]),
    "oracle_code": (_i, [_f, _d]),
    "oracle_quantize_pack": (_i, [_i, _i, _i, _P(_f), _P(_u64), _P(_u16), _P(_u8)]),
    "oracle_dequant": (_d, [_i, _i, _d]),
    "oracle_importance": (None, [_i, _i, _P(_f), _P(_f), _P(_d)]),
    "oracle_depth_of": (_i, [_d, _d]),
    "oracle_plan": (_i, [_i, _i, _P(_f), _P(_f), _i, _P(_d), _P(_u8), _P(_d), _P(_d), _P(_i)]),
    "oracle_plan_fixed": (None, [_i, _i, _P(_f), _P(_f), _i, _i, _P(_u8)]),
    "oracle_runs": (None, [_i, _i, _P(_u8), _P(_u32)]),
    "oracle_gather": (None, [_i, _P(_u32), _P(_u64), _P(_u16), _P(_u64), _P(_u16)]),
    "oracle_scores": (None, [_i, _i, _i, _i, _P(_u64), _P(_u16), _P(_u8), _P(_f), _P(_d)]),
    "oracle_scores_staged": (None, [_i, _i, _i, _P(_u32), _P(_u64), _P(_u16), _P(_u8), _P(_f), _P(_d)]),
    "oracle_select": (_i, [_i, _i, _P(_d), _i, _i, _i, _P(_i32), _P(_d)]),
    "oracle_attention": (None, [_i, _i, _i, _P(_u16), _P(_u16), _P(_f), _P(_i32), _i, _P(_d)]),
    "oracle_reconstruct": (None, [_i, _i, _i, _P(_u64), _P(_u16), _P(_d)]),
    "oracle_attention_keys": (None, [_i, _i, _i, _P(_d), _P(_u16), _P(_f), _P(_i32), _i, _P(_d)]),
    "oracle_exact_scores": (None, [_i, _i, _i, _P(_f), _P(_f), _P(_d)]),
    "oracle_greedy_budgets": (None, [_i, _i, _P(_d), _i, _i, _i, _P(_i32)]),
    "oracle_calibrate": (None, [_i, _i, _P(_f), _P(_d), _P(_d), _P(_d)]),
    "oracle_eigh": (_i, [_i, _P(_d), _P(_d), _P(_d)]),
    "oracle_rotate": (None, [_i, _i, _P(_f), _P(_d), _P(_d), _P(_f)]),
    "oracle_rotate_query": (None, [_i, _i, _P(_f), _P(_d), _P(_d)]),
}


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


_CT = {np.float32: _f, np.float64: _d, np.uint8: _u8, np.uint16: _u16,
       np.uint32: _u32, np.uint64: _u64, np.int32: _i32, np.intc: _i}


def _ptr(a, dtype):
    if a is None:
        return None
    assert a.dtype == dtype and a.flags.c_contiguous, (a.dtype, dtype)
    return a.ctypes.data_as(_P(_CT[np.dtype(dtype).type]))


def _arr(x, dtype):
    return np.ascontiguousarray(np.asarray(x), dtype=dtype)


# ---------------------------------------------------------------- scalars
def round_fp16(a: float) -> float:
    return lib().oracle_round_fp16(float(a))


def fp16_bits(v: float) -> int:
    return lib().oracle_fp16_bits(float(v))


def fp16_value(bits: int) -> float:
    return lib().oracle_fp16_value(int(bits))


def code(k: float, a16: float) -> int:
    return lib().oracle_code(float(np.float32(k)), float(a16))


def dequant(c_t: int, t: int, a16: float) -> float:
    return lib().oracle_dequant(int(c_t), int(t), float(a16))


def depth_of(g: float, theta: float) -> int:
    return lib().oracle_depth_of(float(g), float(theta))


# ---------------------------------------------------------------- store
def quantize_pack(keys):
    """keys [U][n][D] (or [n][D]) fp32 -> (planes [U][D][4][nb] u64,
    scales [U][D][nb] u16 fp16 bits, codes [U][n][D] u8)."""
    k = _arr(keys, np.float32)
    squeeze = k.ndim == 2
    if squeeze:
        k = k[None]
    U, n, D = k.shape
    nb = (n + 63) // 64
    planes = np.zeros((U, D, 4, nb), np.uint64)
    scales = np.zeros((U, D, nb), np.uint16)
    codes = np.zeros((U, n, D), np.uint8)
    lib().oracle_quantize_pack(U, n, D, _ptr(k, np.float32), _ptr(planes, np.uint64),
                               _ptr(scales, np.uint16), _ptr(codes, np.uint8))
    if squeeze:
        return planes[0], scales[0], codes[0]
    return planes, scales, codes


# ---------------------------------------------------------------- plan
def importance(q, var):
    q = _arr(q, np.float32)
    var = _arr(var, np.float32)
    G, D = q.shape
    g = np.zeros(D, np.float64)
    lib().oracle_importance(D, G, _ptr(q, np.float32), _ptr(var, np.float32), _ptr(g, np.float64))
    return g


def plan(q, var, B, bracket=None, trace=False):
    """q [G][D] fp32, var [D] fp32 -> (depth [D] u8, theta, steps[, probes, sums])."""
    q = _arr(q, np.float32)
    var = _arr(var, np.float32)
    G, D = q.shape
    depth = np.zeros(D, np.uint8)
    theta = np.zeros(1, np.float64)
    br = None if bracket is None else _arr(bracket, np.float64)
    probes = np.full(30, np.nan) if trace else None
    sums = np.full(30, -1, np.intc) if trace else None
    steps = lib().oracle_plan(D, G, _ptr(q, np.float32), _ptr(var, np.float32), int(B),
                              _ptr(br, np.float64), _ptr(depth, np.uint8), _ptr(theta, np.float64),
                              _ptr(probes, np.float64), _ptr(sums, np.intc))
    if trace:
        return depth, float(theta[0]), steps, probes, sums
    return depth, float(theta[0]), steps


def plan_fixed(q, var, n_sel, t_fixed):
    q = _arr(q, np.float32)
    var = _arr(var, np.float32)
    G, D = q.shape
    depth = np.zeros(D, np.uint8)
    lib().oracle_plan_fixed(D, G, _ptr(q, np.float32), _ptr(var, np.float32), int(n_sel),
                            int(t_fixed), _ptr(depth, np.uint8))
    return depth


def runs(depth, n):
    """depth [D] -> run list [D][6] u32
    {src_word, n_words, dst_word, src_scale, n_scales, dst_scale}."""
    depth = _arr(depth, np.uint8)
    D = depth.shape[0]
    r = np.zeros((D, 6), np.uint32)
    lib().oracle_runs(D, int(n), _ptr(depth, np.uint8), _ptr(r, np.uint32))
    return r


def gather(run_list, planes_unit, scales_unit, stage_words, stage_scales):
    """One unit: store [D][4][nb] / [D][nb] -> staging (stage_words u64, stage_scales u16)."""
    r = _arr(run_list, np.uint32)
    D = r.shape[0]
    P = _arr(planes_unit, np.uint64)
    S = _arr(scales_unit, np.uint16)
    sp = np.zeros(stage_words, np.uint64)
    ss = np.zeros(stage_scales, np.uint16)
    lib().oracle_gather(D, _ptr(r, np.uint32), _ptr(P, np.uint64), _ptr(S, np.uint16),
                        _ptr(sp, np.uint64), _ptr(ss, np.uint16))
    return sp, ss


# ---------------------------------------------------------------- scan
def scores(planes, scales, depth, q, n):
    """planes [U][D][4][nb], scales [U][D][nb], depth [U][D], q [U][G][D] -> [U][G][n] fp64."""
    P = _arr(planes, np.uint64)
    S = _arr(scales, np.uint16)
    dep = _arr(depth, np.uint8)
    qq = _arr(q, np.float32)
    U, G, D = qq.shape
    out = np.zeros((U, G, n), np.float64)
    lib().oracle_scores(U, int(n), D, G, _ptr(P, np.uint64), _ptr(S, np.uint16),
                        _ptr(dep, np.uint8), _ptr(qq, np.float32), _ptr(out, np.float64))
    return out


def scores_staged(run_list, stage_planes, stage_scales, depth, q, n):
    r = _arr(run_list, np.uint32)
    sp = _arr(stage_planes, np.uint64)
    ss = _arr(stage_scales, np.uint16)
    dep = _arr(depth, np.uint8)
    qq = _arr(q, np.float32)
    G, D = qq.shape
    out = np.zeros((G, n), np.float64)
    lib().oracle_scores_staged(int(n), D, G, _ptr(r, np.uint32), _ptr(sp, np.uint64),
                               _ptr(ss, np.uint16), _ptr(dep, np.uint8), _ptr(qq, np.float32),
                               _ptr(out, np.float64))
    return out


def select(scores_gn, k, n_sink, n_recent):
    """scores [G][n] (fp64 or fp32 values) -> (idx [G][k] i32 ascending, their scores)."""
    s = _arr(scores_gn, np.float64)
    G, n = s.shape
    idx = np.zeros((G, k), np.int32)
    sel = np.zeros((G, k), np.float64)
    rc = lib().oracle_select(n, G, _ptr(s, np.float64), int(k), int(n_sink), int(n_recent),
                             _ptr(idx, np.int32), _ptr(sel, np.float64))
    if rc != 0:
        raise ValueError("oracle_select: need |forced| <= k <= n")
    return idx, sel


def attention(krows, vrows, q, idx):
    """krows/vrows [n][D] bf16 bits (u16), q [G][D] fp32, idx [G][k] -> out [G][D] fp64."""
    K = _arr(krows, np.uint16)
    V = _arr(vrows, np.uint16)
    qq = _arr(q, np.float32)
    ii = _arr(idx, np.int32)
    n, D = K.shape
    G, k = ii.shape
    out = np.zeros((G, D), np.float64)
    lib().oracle_attention(n, D, G, _ptr(K, np.uint16), _ptr(V, np.uint16), _ptr(qq, np.float32),
                           _ptr(ii, np.int32), int(k), _ptr(out, np.float64))
    return out


# ---------------------------------------------------------------- fidelity / budgets
def reconstruct(planes_unit, scales_unit, n):
    """One unit's store planes [D][4][cb], scales [D][cb] -> keys [n][D] fp64 at all four planes."""
    P = _arr(planes_unit, np.uint64)
    S = _arr(scales_unit, np.uint16)
    D, _, cb = P.shape
    out = np.zeros((n, D), np.float64)
    lib().oracle_reconstruct(int(n), D, cb, _ptr(P, np.uint64), _ptr(S, np.uint16), _ptr(out, np.float64))
    return out


def attention_keys(keys, vrows, q, idx):
    """Attention with fp64 keys [n][D] and bf16 value rows (u16 bits) -> [G][D] fp64."""
    K = _arr(keys, np.float64)
    V = _arr(vrows, np.uint16)
    qq = _arr(q, np.float32)
    ii = _arr(idx, np.int32)
    n, D = K.shape
    G, k = ii.shape
    out = np.zeros((G, D), np.float64)
    lib().oracle_attention_keys(n, D, G, _ptr(K, np.float64), _ptr(V, np.uint16), _ptr(qq, np.float32),
                                _ptr(ii, np.int32), int(k), _ptr(out, np.float64))
    return out


def exact_scores(keys, q):
    """keys [n][D] fp32 (bf16 rows widened exactly), q [G][D] fp32 -> [G][n] fp64: q . k."""
    k = _arr(keys, np.float32)
    qq = _arr(q, np.float32)
    n, D = k.shape
    G = qq.shape[0]
    out = np.zeros((G, n), np.float64)
    lib().oracle_exact_scores(n, D, G, _ptr(k, np.float32), _ptr(qq, np.float32), _ptr(out, np.float64))
    return out


def dense_attention(krows, vrows, q):
    """Attention of every head over all n rows (bf16 bits) -> [G][D] fp64."""
    n = np.asarray(krows).shape[0]
    G = np.asarray(q).shape[0]
    idx = np.tile(np.arange(n, dtype=np.int32), (G, 1))
    return attention(krows, vrows, q, idx)


def rel_l2(a, ref):
    """Relative L2 error per row, ||a - ref|| / ||ref|| (||a|| where ref is zero)."""
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    num = np.sqrt(np.sum((a - ref) ** 2, axis=-1))
    den = np.sqrt(np.sum(ref ** 2, axis=-1))
    return np.where(den > 0, num / np.where(den > 0, den, 1.0), num)


def greedy_budgets(err, b_min, step, b_mean):
    """err [layers][levels] -> budgets [layers] int32 (levels b_min + step*i)."""
    e = _arr(err, np.float64)
    L, levels = e.shape
    out = np.zeros(L, np.int32)
    lib().oracle_greedy_budgets(L, levels, _ptr(e, np.float64), int(b_min), int(step), int(b_mean),
                                _ptr(out, np.int32))
    return out


# ---------------------------------------------------------------- calibration / KLT
def calibrate(keys, with_cov=False):
    k = _arr(keys, np.float32)
    m, D = k.shape
    mean = np.zeros(D, np.float64)
    var = np.zeros(D, np.float64)
    cov = np.zeros((D, D), np.float64) if with_cov else None
    lib().oracle_calibrate(m, D, _ptr(k, np.float32), _ptr(mean, np.float64),
                           _ptr(var, np.float64), _ptr(cov, np.float64))
    return (mean, var, cov) if with_cov else (mean, var)


def eigh(A):
    A = _arr(A, np.float64)
    D = A.shape[0]
    lam = np.zeros(D, np.float64)
    V = np.zeros((D, D), np.float64)
    lib().oracle_eigh(D, _ptr(A, np.float64), _ptr(lam, np.float64), _ptr(V, np.float64))
    return lam, V


def rotate(keys, mu, V):
    k = _arr(keys, np.float32)
    n, D = k.shape
    out = np.zeros((n, D), np.float32)
    lib().oracle_rotate(n, D, _ptr(k, np.float32), _ptr(_arr(mu, np.float64), np.float64),
                        _ptr(_arr(V, np.float64), np.float64), _ptr(out, np.float32))
    return out


def rotate_query(q, V):
    qq = _arr(q, np.float32)
    G, D = qq.shape
    out = np.zeros((G, D), np.float64)
    lib().oracle_rotate_query(G, D, _ptr(qq, np.float32), _ptr(_arr(V, np.float64), np.float64),
                              _ptr(out, np.float64))
    return out
