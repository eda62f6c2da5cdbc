"""Thin Python binding of libfathom (include/fathom.h).

Argument marshalling only: every function takes torch tensors, checks dtype,
device and contiguity, passes raw pointers and the current CUDA stream to the
C ABI of the same name, and raises ``FathomError`` on a non-zero status.  All
computation runs in the CUDA kernels of libfathom; there is no fallback: if
the library is missing or CUDA is unavailable the call fails.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# FATHOM_LIB names another build of the same library (e.g. the debug build with
# bounds checks, libfathom_debug.so) to load instead of the default one.
LIB_PATH = os.environ.get("FATHOM_LIB") or os.path.join(_PKG, "_build", "libfathom.so")

F32, BF16 = 0, 1
WS_SCAN_TOPK, WS_SPARSE_ATTN, WS_DENSE_ATTN, WS_KLT_ONLINE = 0, 1, 2, 3
SRC_STORE, SRC_STAGING = 0, 1
MAX_D, MAX_G, MAX_K = 128, 8, 2048

# (name, restype, argtypes) of every symbol include/fathom.h declares
_vp, _i32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t


class Shape(ctypes.Structure):
    _fields_ = [("units", ctypes.c_int32), ("n", ctypes.c_int32), ("D", ctypes.c_int32),
                ("G", ctypes.c_int32), ("k", ctypes.c_int32), ("n_sink", ctypes.c_int32),
                ("n_recent", ctypes.c_int32), ("n_cap", ctypes.c_int32), ("scan_ctas_per_sm", ctypes.c_int32)]

    def __repr__(self):
        return (f"Shape(units={self.units}, n={self.n}, D={self.D}, G={self.G}, k={self.k}, "
                f"n_sink={self.n_sink}, n_recent={self.n_recent}, n_cap={self.n_cap}, "
                f"scan_ctas_per_sm={self.scan_ctas_per_sm})")

    @property
    def cap(self) -> int:
        """Tokens the per-unit arrays are laid out for."""
        return self.n_cap if self.n_cap > 0 else self.n


RUN_FIELDS = ("src_word", "n_words", "dst_word", "src_scale", "n_scales", "dst_scale")
RUN_BYTES = 24

SIGNATURES = {
    "fathom_calibrate": (ctypes.c_int, [_i32, _i32, _i32, _vp, _vp, _vp, _vp]),
    "fathom_calibrate_klt": (ctypes.c_int, [_i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp]),
    "fathom_rotate_keys": (ctypes.c_int, [ctypes.POINTER(Shape), _vp, ctypes.c_int, _i32, _vp, _vp, _vp, _vp]),
    "fathom_rotate_query": (ctypes.c_int, [ctypes.POINTER(Shape), _vp, _i32, _vp, _vp, _vp]),
    "fathom_quantize_pack": (ctypes.c_int, [ctypes.POINTER(Shape), _vp, ctypes.c_int, _vp, _vp, _vp]),
    "fathom_append_block": (ctypes.c_int, [ctypes.POINTER(Shape), _vp, ctypes.c_int, _i32, _i32, _vp, _vp, _vp]),
    "fathom_plan": (ctypes.c_int, [ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "fathom_plan_fixed": (ctypes.c_int, [ctypes.POINTER(Shape), _vp, _vp, _i32, _i32, _vp, _vp, _vp]),
    "fathom_gather": (ctypes.c_int, [ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _sz, _sz, _vp]),
    "fathom_scan_topk": (ctypes.c_int, [ctypes.POINTER(Shape), _vp, _vp, ctypes.c_int, _sz, _sz, _vp,
                                        _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "fathom_scan": (ctypes.c_int, [ctypes.POINTER(Shape), _vp, _vp, ctypes.c_int, _sz, _sz, _vp, _vp, _vp, _vp,
                                   _sz, _vp]),
    "fathom_select": (ctypes.c_int, [ctypes.POINTER(Shape), _vp, _vp, ctypes.c_int, _sz, _sz, _vp, _vp, _vp, _vp,
                                     _vp, _sz, _vp]),
    "fathom_exact_topk": (ctypes.c_int, [ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "fathom_sparse_attn": (ctypes.c_int, [ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "fathom_dense_attn": (ctypes.c_int, [ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "fathom_sparse_attn_planes": (ctypes.c_int, [ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz,
                                                 _vp]),
    "fathom_sparse_attn_noalloc": (ctypes.c_int, [ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp]),
    "fathom_klt_online": (ctypes.c_int, [ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "fathom_rel_err": (ctypes.c_int, [_i32, _i32, _vp, _vp, _vp, _vp]),
    "fathom_set_overlap": (ctypes.c_int, [_i32, _i32, _vp, _vp, _vp, _vp]),
    "fathom_greedy_budgets": (ctypes.c_int, [_i32, _i32, _vp, _i32, _i32, _i32, _vp]),
    "fathom_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(Shape), ctypes.c_int]),
    "fathom_last_error": (ctypes.c_char_p, []),
    "fathom_version": (ctypes.c_char_p, []),
    "fathom_debug_status": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p]),
}


class FathomError(RuntimeError):
    def __init__(self, name, status, msg):
        super().__init__(f"{name} failed with status {status}: {msg}")
        self.status = status


_lib = None


def lib():
    """Load libfathom.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libfathom is not built ({LIB_PATH} missing): run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _call(name, *args):
    rc = getattr(lib(), name)(*args)
    if rc != 0:
        raise FathomError(name, rc, lib().fathom_last_error().decode())
    return rc


def _p(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, dtypes, shape=None, dev=True, min_numel=None):
    """Dtype, shape (exact), size (at least min_numel elements: the library sees only
    a pointer, so a shorter tensor would be read or written past its end),
    contiguity, and memory the GPU can reach, in that order."""
    if t is None:
        raise ValueError(f"{name} is required")
    if dtypes and t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(shape)}")
    if min_numel is not None and t.numel() < min_numel:
        raise ValueError(f"{name}: {t.numel()} elements, the call needs at least {min_numel}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dev and not _reachable(t):
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    return t


def _reachable(t) -> bool:
    """Memory the GPU can load from and store to: device memory or pinned host memory."""
    return t.is_cuda or t.is_pinned()


def _check_out(t, name, dtypes, min_numel):
    """A caller-provided output (None: the binding allocates it)."""
    if t is not None:
        _check(t, name, dtypes, min_numel=min_numel)
    return t


def _store_words(shape: Shape) -> int:
    """Elements of a bit-plane store [units][D][4][cap blocks]."""
    return shape.units * shape.D * 4 * nblocks(shape.cap)


def _store_scales(shape: Shape) -> int:
    """Elements of the store's scales [units][D][cap blocks]."""
    return shape.units * shape.D * nblocks(shape.cap)


def _rows(shape: Shape) -> int:
    """Elements of per-unit rows [units][cap][D]."""
    return shape.units * shape.cap * shape.D


def make_shape(units, n, D=128, G=4, k=1, n_sink=4, n_recent=32, n_cap=0, scan_ctas_per_sm=0) -> Shape:
    return Shape(units, n, D, G, k, n_sink, n_recent, n_cap, scan_ctas_per_sm)


def nblocks(n: int) -> int:
    return (n + 63) // 64


def version() -> str:
    return lib().fathom_version().decode()


def workspace_size(shape: Shape, which: int) -> int:
    return int(lib().fathom_workspace_size(ctypes.byref(shape), which))


def alloc_workspace(shape: Shape, which: int, device="cuda") -> torch.Tensor:
    nbytes = workspace_size(shape, which)
    if nbytes == 0:
        raise FathomError("fathom_workspace_size", 1, lib().fathom_last_error().decode())
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ calls
def fathom_calibrate(calib, mean=None, var=None, stream=None):
    """calib [U][m][D] fp32 -> (mean [U][D], var [U][D]) fp32 (ddof = 1)."""
    _check(calib, "calib", (torch.float32,))
    if calib.dim() != 3:
        raise ValueError(f"calib: shape {tuple(calib.shape)} is not [units][m][D]")
    U, m, D = calib.shape
    _check_out(mean, "mean", (torch.float32,), U * D)
    _check_out(var, "var", (torch.float32,), U * D)
    if var is None:
        var = torch.empty(U, D, dtype=torch.float32, device=calib.device)
    if mean is None:
        mean = torch.empty(U, D, dtype=torch.float32, device=calib.device)
    _call("fathom_calibrate", U, m, D, _p(calib), _p(mean), _p(var), _stream(stream))
    return mean, var


def fathom_calibrate_klt(calib, mean=None, V=None, lam=None, stream=None):
    """calib [groups][m][D] fp32 -> (mean [groups][D] fp64, V [groups][D][D] fp64 (eigenvectors
    as columns, eigenvalues descending), lambda [groups][D] fp32)."""
    _check(calib, "calib", (torch.float32,))
    if calib.dim() != 3:
        raise ValueError(f"calib: shape {tuple(calib.shape)} is not [groups][m][D]")
    Gr, m, D = calib.shape
    dev = calib.device
    _check_out(mean, "mean", (torch.float64,), Gr * D)
    _check_out(V, "V", (torch.float64,), Gr * D * D)
    _check_out(lam, "lam", (torch.float32,), Gr * D)
    if mean is None:
        mean = torch.empty(Gr, D, dtype=torch.float64, device=dev)
    if V is None:
        V = torch.empty(Gr, D, D, dtype=torch.float64, device=dev)
    if lam is None:
        lam = torch.empty(Gr, D, dtype=torch.float32, device=dev)
    _call("fathom_calibrate_klt", Gr, m, D, _p(calib), _p(mean), _p(V), _p(lam), _stream(stream))
    return mean, V, lam


def fathom_rotate_keys(shape: Shape, keys, groups, mean, V, out=None, stream=None):
    """keys [U][n][D] fp32 or bf16 -> (k - mu_g) V_g [U][n][D] fp32, g = u % groups."""
    _check(keys, "keys", (torch.float32, torch.bfloat16, torch.int16), min_numel=_rows(shape))
    _check(mean, "mean", (torch.float64,), (groups, shape.D))
    _check(V, "V", (torch.float64,), (groups, shape.D, shape.D))
    _check_out(out, "out", (torch.float32,), _rows(shape))
    dt = F32 if keys.dtype == torch.float32 else BF16
    if out is None:
        out = torch.empty(shape.units, shape.cap, shape.D, dtype=torch.float32, device=keys.device)
    _call("fathom_rotate_keys", ctypes.byref(shape), _p(keys), dt, int(groups), _p(mean), _p(V), _p(out),
          _stream(stream))
    return out


def fathom_rotate_query(shape: Shape, q, groups, V, out=None, stream=None):
    """q [U][G][D] fp32 -> q V_g [U][G][D] fp32, g = u % groups."""
    _check(q, "q", (torch.float32,), (shape.units, shape.G, shape.D))
    _check(V, "V", (torch.float64,), (groups, shape.D, shape.D))
    _check_out(out, "out", (torch.float32,), shape.units * shape.G * shape.D)
    if out is None:
        out = torch.empty_like(q)
    _call("fathom_rotate_query", ctypes.byref(shape), _p(q), int(groups), _p(V), _p(out), _stream(stream))
    return out


def fathom_quantize_pack(shape: Shape, keys, planes=None, scales=None, stream=None):
    """keys [U][n][D] fp32 or bf16 -> planes [U][D][4][nb] (int64 storage of u64),
    scales [U][D][nb] (int16 storage of fp16 bits)."""
    _check(keys, "keys", (torch.float32, torch.bfloat16, torch.int16), min_numel=_rows(shape))
    _check_out(planes, "planes", (torch.int64,), _store_words(shape))
    _check_out(scales, "scales", (torch.int16,), _store_scales(shape))
    dt = F32 if keys.dtype == torch.float32 else BF16
    nb = nblocks(shape.cap)
    dev = keys.device
    if planes is None:
        planes = torch.empty(shape.units, shape.D, 4, nb, dtype=torch.int64, device=dev)
    if scales is None:
        scales = torch.empty(shape.units, shape.D, nb, dtype=torch.int16, device=dev)
    _call("fathom_quantize_pack", ctypes.byref(shape), _p(keys), dt, _p(planes), _p(scales),
          _stream(stream))
    return planes, scales


def fathom_append_block(shape: Shape, keys, block, count, planes, scales, stream=None):
    """Quantise block `block` (its first `count` tokens) of every unit of the key rows
    keys [U][cap][D] (fp32 or bf16) into the store planes [U][D][4][cap blocks],
    scales [U][D][cap blocks], in place."""
    _check(keys, "keys", (torch.float32, torch.bfloat16, torch.int16), (shape.units, shape.cap, shape.D))
    _check(planes, "planes", (torch.int64,), (shape.units, shape.D, 4, nblocks(shape.cap)))
    _check(scales, "scales", (torch.int16,), (shape.units, shape.D, nblocks(shape.cap)))
    dt = F32 if keys.dtype == torch.float32 else BF16
    _call("fathom_append_block", ctypes.byref(shape), _p(keys), dt, int(block), int(count), _p(planes), _p(scales),
          _stream(stream))
    return planes, scales


def fathom_plan(shape: Shape, q, var, budget, bracket=None, depth=None, theta=None, runs=None,
                stream=None, want_theta=True):
    """-> depth [U][D] u8, theta [U] f64 (None when want_theta is False: the call
    then passes no theta buffer and the depths and runs are the same), runs
    [U][D][6] (int32 storage of u32)."""
    _check(q, "q", (torch.float32,), (shape.units, shape.G, shape.D))
    _check(var, "var", (torch.float32,), (shape.units, shape.D))
    _check(budget, "budget", (torch.int32,), (shape.units,))
    if bracket is not None:
        _check(bracket, "bracket", (torch.float64,), (shape.units, 2))
    _check_out(depth, "depth", (torch.uint8,), shape.units * shape.D)
    _check_out(theta, "theta", (torch.float64,), shape.units)
    _check_out(runs, "runs", (torch.int32,), shape.units * shape.D * 6)
    dev = q.device
    if depth is None:
        depth = torch.empty(shape.units, shape.D, dtype=torch.uint8, device=dev)
    if not want_theta:
        theta = None
    elif theta is None:
        theta = torch.empty(shape.units, dtype=torch.float64, device=dev)
    if runs is None:
        runs = torch.empty(shape.units, shape.D, 6, dtype=torch.int32, device=dev)
    _call("fathom_plan", ctypes.byref(shape), _p(q), _p(var), _p(budget), _p(bracket), _p(depth),
          _p(theta), _p(runs), _stream(stream))
    return depth, theta, runs


def fathom_plan_fixed(shape: Shape, q, var, n_channels, depth_each, depth=None, runs=None,
                      stream=None):
    _check(q, "q", (torch.float32,), (shape.units, shape.G, shape.D))
    _check(var, "var", (torch.float32,), (shape.units, shape.D))
    _check_out(depth, "depth", (torch.uint8,), shape.units * shape.D)
    _check_out(runs, "runs", (torch.int32,), shape.units * shape.D * 6)
    dev = q.device
    if depth is None:
        depth = torch.empty(shape.units, shape.D, dtype=torch.uint8, device=dev)
    if runs is None:
        runs = torch.empty(shape.units, shape.D, 6, dtype=torch.int32, device=dev)
    _call("fathom_plan_fixed", ctypes.byref(shape), _p(q), _p(var), int(n_channels), int(depth_each),
          _p(depth), _p(runs), _stream(stream))
    return depth, runs


def fathom_gather(shape: Shape, store_planes, store_scales, runs, stage_planes, stage_scales,
                  stream=None):
    """stage_planes [U][W] int64, stage_scales [U][S] int16 (per-unit strides W, S)."""
    _check(store_planes, "store_planes", (torch.int64,), min_numel=_store_words(shape))
    _check(store_scales, "store_scales", (torch.int16,), min_numel=_store_scales(shape))
    _check(runs, "runs", (torch.int32,), (shape.units, shape.D, 6))
    W = stage_planes.shape[-1] if stage_planes is not None and stage_planes.dim() else 0
    S = stage_scales.shape[-1] if stage_scales is not None and stage_scales.dim() else 0
    _check(stage_planes, "stage_planes", (torch.int64,), min_numel=shape.units * W)
    _check(stage_scales, "stage_scales", (torch.int16,), min_numel=shape.units * S)
    _call("fathom_gather", ctypes.byref(shape), _p(store_planes), _p(store_scales), _p(runs),
          _p(stage_planes), _p(stage_scales), W, S, _stream(stream))
    return stage_planes, stage_scales


def fathom_scan_topk(shape: Shape, planes, scales, runs, q, workspace, source=SRC_STORE,
                     topk_idx=None, topk_score=None, scores=None, stream=None):
    """-> topk_idx [U][G][k] int32 ascending, topk_score [U][G][k] fp32 (scores, if given,
    receives every token's score [U][G][n])."""
    if source == SRC_STAGING:      # [units][W] and [units][S]: the last dimension is the per-unit stride
        W = planes.shape[-1] if planes is not None and planes.dim() else 0
        S = scales.shape[-1] if scales is not None and scales.dim() else 0
        need_p, need_s = shape.units * W, shape.units * S
    else:
        W = S = 0
        need_p, need_s = _store_words(shape), _store_scales(shape)
    _check(planes, "planes", (torch.int64,), min_numel=need_p)
    _check(scales, "scales", (torch.int16,), min_numel=need_s)
    _check(runs, "runs", (torch.int32,), (shape.units, shape.D, 6))
    _check(q, "q", (torch.float32,), (shape.units, shape.G, shape.D))
    _check(workspace, "workspace", (torch.uint8,))
    _check_out(topk_idx, "topk_idx", (torch.int32,), shape.units * shape.G * shape.k)
    _check_out(topk_score, "topk_score", (torch.float32,), shape.units * shape.G * shape.k)
    dev = q.device
    if topk_idx is None:
        topk_idx = torch.empty(shape.units, shape.G, shape.k, dtype=torch.int32, device=dev)
    if topk_score is None:
        topk_score = torch.empty(shape.units, shape.G, shape.k, dtype=torch.float32, device=dev)
    if scores is not None:
        _check(scores, "scores", (torch.float32,), (shape.units, shape.G, shape.n))
    _call("fathom_scan_topk", ctypes.byref(shape), _p(planes), _p(scales), int(source), W, S,
          _p(runs), _p(q), _p(topk_idx), _p(topk_score), _p(scores), _p(workspace),
          workspace.numel(), _stream(stream))
    return topk_idx, topk_score


def _scan_inputs(shape, planes, scales, runs, q, workspace, source):
    if source == SRC_STAGING:
        W = planes.shape[-1] if planes is not None and planes.dim() else 0
        S = scales.shape[-1] if scales is not None and scales.dim() else 0
        need_p, need_s = shape.units * W, shape.units * S
    else:
        W = S = 0
        need_p, need_s = _store_words(shape), _store_scales(shape)
    _check(planes, "planes", (torch.int64,), min_numel=need_p)
    _check(scales, "scales", (torch.int16,), min_numel=need_s)
    _check(runs, "runs", (torch.int32,), (shape.units, shape.D, 6))
    _check(q, "q", (torch.float32,), (shape.units, shape.G, shape.D))
    _check(workspace, "workspace", (torch.uint8,))
    return W, S


def fathom_scan(shape: Shape, planes, scales, runs, q, workspace, source=SRC_STORE, scores=None, stream=None):
    """The scan half of fathom_scan_topk: candidate lists in the workspace (scores, if
    given, receives every token's score [U][G][n])."""
    W, S = _scan_inputs(shape, planes, scales, runs, q, workspace, source)
    if scores is not None:
        _check(scores, "scores", (torch.float32,), (shape.units, shape.G, shape.n))
    _call("fathom_scan", ctypes.byref(shape), _p(planes), _p(scales), int(source), W, S, _p(runs), _p(q),
          _p(scores), _p(workspace), workspace.numel(), _stream(stream))


def fathom_select(shape: Shape, planes, scales, runs, q, workspace, source=SRC_STORE, topk_idx=None,
                  topk_score=None, stream=None):
    """The selection half: -> topk_idx [U][G][k] int32 ascending, topk_score [U][G][k] fp32."""
    W, S = _scan_inputs(shape, planes, scales, runs, q, workspace, source)
    _check_out(topk_idx, "topk_idx", (torch.int32,), shape.units * shape.G * shape.k)
    _check_out(topk_score, "topk_score", (torch.float32,), shape.units * shape.G * shape.k)
    if topk_idx is None:
        topk_idx = torch.empty(shape.units, shape.G, shape.k, dtype=torch.int32, device=q.device)
    if topk_score is None:
        topk_score = torch.empty(shape.units, shape.G, shape.k, dtype=torch.float32, device=q.device)
    _call("fathom_select", ctypes.byref(shape), _p(planes), _p(scales), int(source), W, S, _p(runs), _p(q),
          _p(topk_idx), _p(topk_score), _p(workspace), workspace.numel(), _stream(stream))
    return topk_idx, topk_score


def fathom_exact_topk(shape: Shape, k_rows, q, workspace, topk_idx=None, topk_score=None, scores=None,
                      stream=None):
    """Fidelity reference: the kept set with every token scored exactly, q . k
    over all D channels of its bf16 row.  k_rows [U][cap][D] bf16 -> topk_idx
    [U][G][k] int32 ascending, topk_score [U][G][k] fp32 (workspace of kind
    WS_SCAN_TOPK)."""
    _check(k_rows, "k_rows", (torch.bfloat16, torch.int16), (shape.units, shape.cap, shape.D))
    _check(q, "q", (torch.float32,), (shape.units, shape.G, shape.D))
    _check(workspace, "workspace", (torch.uint8,))
    _check_out(topk_idx, "topk_idx", (torch.int32,), shape.units * shape.G * shape.k)
    _check_out(topk_score, "topk_score", (torch.float32,), shape.units * shape.G * shape.k)
    dev = q.device
    if topk_idx is None:
        topk_idx = torch.empty(shape.units, shape.G, shape.k, dtype=torch.int32, device=dev)
    if topk_score is None:
        topk_score = torch.empty(shape.units, shape.G, shape.k, dtype=torch.float32, device=dev)
    if scores is not None:
        _check(scores, "scores", (torch.float32,), (shape.units, shape.G, shape.n))
    _call("fathom_exact_topk", ctypes.byref(shape), _p(k_rows), _p(q), _p(topk_idx), _p(topk_score),
          _p(scores), _p(workspace), workspace.numel(), _stream(stream))
    return topk_idx, topk_score


def fathom_dense_attn(shape: Shape, k_rows, v_rows, q, workspace, out=None, stream=None):
    """Fidelity reference: attention of every head over all n tokens.
    k_rows, v_rows [U][cap][D] bf16 -> out [U][G][D] fp32 (workspace of kind
    WS_DENSE_ATTN)."""
    _check(k_rows, "k_rows", (torch.bfloat16, torch.int16), (shape.units, shape.cap, shape.D))
    _check(v_rows, "v_rows", (torch.bfloat16, torch.int16), (shape.units, shape.cap, shape.D))
    _check(q, "q", (torch.float32,), (shape.units, shape.G, shape.D))
    _check(workspace, "workspace", (torch.uint8,))
    _check_out(out, "out", (torch.float32,), shape.units * shape.G * shape.D)
    if out is None:
        out = torch.empty(shape.units, shape.G, shape.D, dtype=torch.float32, device=q.device)
    _call("fathom_dense_attn", ctypes.byref(shape), _p(k_rows), _p(v_rows), _p(q), _p(out),
          _p(workspace), workspace.numel(), _stream(stream))
    return out


def fathom_klt_online(shape: Shape, k_rows, workspace=None, mean=None, V=None, lam=None, stream=None):
    """Per-unit rotated basis from the unit's own key rows [U][cap][D] bf16 ->
    (mean [U][D] f64, V [U][D][D] f64, lambda [U][D] f32)."""
    _check(k_rows, "k_rows", (torch.bfloat16, torch.int16), (shape.units, shape.cap, shape.D))
    _check_out(mean, "mean", (torch.float64,), shape.units * shape.D)
    _check_out(V, "V", (torch.float64,), shape.units * shape.D * shape.D)
    _check_out(lam, "lam", (torch.float32,), shape.units * shape.D)
    dev = "cuda"
    if workspace is None:
        workspace = alloc_workspace(shape, WS_KLT_ONLINE, device=dev)
    _check(workspace, "workspace", (torch.uint8,))
    U, D = shape.units, shape.D
    if mean is None:
        mean = torch.empty(U, D, dtype=torch.float64, device=dev)
    if V is None:
        V = torch.empty(U, D, D, dtype=torch.float64, device=dev)
    if lam is None:
        lam = torch.empty(U, D, dtype=torch.float32, device=dev)
    _call("fathom_klt_online", ctypes.byref(shape), _p(k_rows), _p(mean), _p(V), _p(lam), _p(workspace),
          workspace.numel(), _stream(stream))
    return mean, V, lam


def fathom_rel_err(a, ref, err=None, stream=None):
    """a, ref [..., D] fp32 (device) -> err [...] fp64: ||a - ref|| / ||ref|| per row."""
    _check(a, "a", (torch.float32,))
    _check(ref, "ref", (torch.float32,), tuple(a.shape))
    D = a.shape[-1]
    rows = a.numel() // D if D else 0
    if err is None:
        err = torch.empty(a.shape[:-1], dtype=torch.float64, device=a.device)
    _check(err, "err", (torch.float64,), tuple(a.shape[:-1]))
    _call("fathom_rel_err", rows, D, _p(a), _p(ref), _p(err), _stream(stream))
    return err


def fathom_set_overlap(a, b, count=None, stream=None):
    """a, b [..., k] int32 ascending (device) -> count [...] int32: shared indices per row."""
    _check(a, "a", (torch.int32,))
    _check(b, "b", (torch.int32,), tuple(a.shape))
    k = a.shape[-1]
    rows = a.numel() // k if k else 0
    if count is None:
        count = torch.empty(a.shape[:-1], dtype=torch.int32, device=a.device)
    _check(count, "count", (torch.int32,), tuple(a.shape[:-1]))
    _call("fathom_set_overlap", rows, k, _p(a), _p(b), _p(count), _stream(stream))
    return count


def fathom_greedy_budgets(err, b_min, step, b_mean):
    """err [layers][levels] (host array-like, fp64) -> budgets [layers] (numpy int32)."""
    import numpy as np
    e = np.ascontiguousarray(np.asarray(err, dtype=np.float64))
    if e.ndim != 2:
        raise ValueError("err must be [layers][levels]")
    out = np.zeros(e.shape[0], dtype=np.int32)
    _call("fathom_greedy_budgets", e.shape[0], e.shape[1], e.ctypes.data, int(b_min), int(step), int(b_mean),
          out.ctypes.data)
    return out


def fathom_sparse_attn_planes(shape: Shape, planes, scales, v_rows, q, topk_idx, workspace, out=None,
                              stream=None):
    """Sparse attention with the winners' keys rebuilt from the store's four planes.
    planes [U][D][4][cb], scales [U][D][cb], v_rows [U][cap][D] bf16 -> out [U][G][D] fp32."""
    cb = nblocks(shape.cap)
    _check(planes, "planes", (torch.int64,), (shape.units, shape.D, 4, cb))
    _check(scales, "scales", (torch.int16,), (shape.units, shape.D, cb))
    _check(v_rows, "v_rows", (torch.bfloat16, torch.int16), (shape.units, shape.cap, shape.D))
    _check(q, "q", (torch.float32,), (shape.units, shape.G, shape.D))
    _check(topk_idx, "topk_idx", (torch.int32,), (shape.units, shape.G, shape.k))
    _check(workspace, "workspace", (torch.uint8,))
    _check_out(out, "out", (torch.float32,), shape.units * shape.G * shape.D)
    if out is None:
        out = torch.empty(shape.units, shape.G, shape.D, dtype=torch.float32, device=q.device)
    _call("fathom_sparse_attn_planes", ctypes.byref(shape), _p(planes), _p(scales), _p(v_rows), _p(q),
          _p(topk_idx), _p(out), _p(workspace), workspace.numel(), _stream(stream))
    return out


def fathom_sparse_attn_noalloc(shape: Shape, k_rows, v_rows, q, topk_idx, out, stream=None):
    """fathom_sparse_attn with the library's own fixed scratch (no workspace, no
    allocation inside the call): for callers that may not allocate device memory.
    `out` [U][G][D] fp32 must be provided by the caller."""
    _check(k_rows, "k_rows", (torch.bfloat16, torch.int16), (shape.units, shape.cap, shape.D))
    _check(v_rows, "v_rows", (torch.bfloat16, torch.int16), (shape.units, shape.cap, shape.D))
    _check(q, "q", (torch.float32,), (shape.units, shape.G, shape.D))
    _check(topk_idx, "topk_idx", (torch.int32,), (shape.units, shape.G, shape.k))
    _check(out, "out", (torch.float32,), (shape.units, shape.G, shape.D))
    _call("fathom_sparse_attn_noalloc", ctypes.byref(shape), _p(k_rows), _p(v_rows), _p(q),
          _p(topk_idx), _p(out), _stream(stream))
    return out


def fathom_sparse_attn(shape: Shape, k_rows, v_rows, q, topk_idx, workspace, out=None, stream=None):
    """k_rows, v_rows [U][n][D] bf16 (device or pinned host) -> out [U][G][D] fp32."""
    _check(k_rows, "k_rows", (torch.bfloat16, torch.int16), (shape.units, shape.cap, shape.D))
    _check(v_rows, "v_rows", (torch.bfloat16, torch.int16), (shape.units, shape.cap, shape.D))
    _check(q, "q", (torch.float32,), (shape.units, shape.G, shape.D))
    _check(topk_idx, "topk_idx", (torch.int32,), (shape.units, shape.G, shape.k))
    _check(workspace, "workspace", (torch.uint8,))
    _check_out(out, "out", (torch.float32,), shape.units * shape.G * shape.D)
    if out is None:
        out = torch.empty(shape.units, shape.G, shape.D, dtype=torch.float32, device=q.device)
    _call("fathom_sparse_attn", ctypes.byref(shape), _p(k_rows), _p(v_rows), _p(q), _p(topk_idx),
          _p(out), _p(workspace), workspace.numel(), _stream(stream))
    return out


def fathom_debug_status(mode=0):
    """Debug build only: the first failed bounds check of the scan, gather and
    attention kernels, as three integers (site << 48 | index; 0: none).  mode 1
    also clears them; mode 2 plants a self-test record first."""
    out = (ctypes.c_uint64 * 3)()
    _call("fathom_debug_status", int(mode), ctypes.cast(out, ctypes.c_void_p))
    return [int(x) for x in out]
