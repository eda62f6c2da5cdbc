"""The Python binding's argument checks, on CPU.

The C ABI receives only pointers, so the binding checks every tensor the
library will read or write (dtype, shape or size, contiguity, memory the GPU
can reach) before the call: a tensor one element short would otherwise be
read or written past its end on the GPU.  The library is never called here:
the call itself, the stream lookup and the device check are replaced, so a
correctly sized call reaches the (recorded) library call, and a short tensor
raises first, naming the argument."""
import pytest
import torch

from bit_plane_kv_gb300 import binding as B

U, N, D, G, K = 2, 200, 128, 4, 64
CB = B.nblocks(N)                     # 4 blocks
W, S = 100, 40                        # staging strides (words, scales) per unit


class Reached(Exception):
    pass


@pytest.fixture(autouse=True)
def no_library(monkeypatch):
    def fake_call(name, *args):
        raise Reached(name)
    monkeypatch.setattr(B, "_call", fake_call)
    monkeypatch.setattr(B, "_stream", lambda stream=None: None)
    monkeypatch.setattr(B, "_reachable", lambda t: True)


def z(*shape, dtype=torch.float32):
    return torch.zeros(*shape, dtype=dtype)


def shape_(n_cap=0):
    return B.make_shape(U, N, D, G, K, 4, 32, n_cap)


def short(t):
    """Same dtype, one element fewer (and flat)."""
    return torch.zeros(t.numel() - 1, dtype=t.dtype)


I64, I32, I16, U8, F64, BF = torch.int64, torch.int32, torch.int16, torch.uint8, torch.float64, torch.bfloat16

# (binding function, positional names, builder of valid arguments)
CASES = {
    "fathom_quantize_pack": (["shape", "keys"], lambda: dict(
        shape=shape_(), keys=z(U, N, D), planes=z(U, D, 4, CB, dtype=I64), scales=z(U, D, CB, dtype=I16))),
    "fathom_append_block": (["shape", "keys", "block", "count", "planes", "scales"], lambda: dict(
        shape=shape_(), keys=z(U, N, D, dtype=BF), block=3, count=8, planes=z(U, D, 4, CB, dtype=I64),
        scales=z(U, D, CB, dtype=I16))),
    "fathom_calibrate": (["calib"], lambda: dict(calib=z(U, 16, D), mean=z(U, D), var=z(U, D))),
    "fathom_calibrate_klt": (["calib"], lambda: dict(
        calib=z(2, 16, D), mean=z(2, D, dtype=F64), V=z(2, D, D, dtype=F64), lam=z(2, D))),
    "fathom_rotate_keys": (["shape", "keys", "groups", "mean", "V"], lambda: dict(
        shape=shape_(), keys=z(U, N, D, dtype=BF), groups=2, mean=z(2, D, dtype=F64), V=z(2, D, D, dtype=F64),
        out=z(U, N, D))),
    "fathom_rotate_query": (["shape", "q", "groups", "V"], lambda: dict(
        shape=shape_(), q=z(U, G, D), groups=2, V=z(2, D, D, dtype=F64), out=z(U, G, D))),
    "fathom_plan": (["shape", "q", "var", "budget"], lambda: dict(
        shape=shape_(), q=z(U, G, D), var=z(U, D), budget=z(U, dtype=I32), bracket=z(U, 2, dtype=F64),
        depth=z(U, D, dtype=U8), theta=z(U, dtype=F64), runs=z(U, D, 6, dtype=I32))),
    "fathom_plan_fixed": (["shape", "q", "var", "n_channels", "depth_each"], lambda: dict(
        shape=shape_(), q=z(U, G, D), var=z(U, D), n_channels=32, depth_each=4, depth=z(U, D, dtype=U8),
        runs=z(U, D, 6, dtype=I32))),
    "fathom_gather": (["shape", "store_planes", "store_scales", "runs", "stage_planes", "stage_scales"], lambda: dict(
        shape=shape_(), store_planes=z(U, D, 4, CB, dtype=I64), store_scales=z(U, D, CB, dtype=I16),
        runs=z(U, D, 6, dtype=I32), stage_planes=z(U, W, dtype=I64), stage_scales=z(U, S, dtype=I16))),
    "fathom_scan_topk": (["shape", "planes", "scales", "runs", "q", "workspace"], lambda: dict(
        shape=shape_(), planes=z(U, D, 4, CB, dtype=I64), scales=z(U, D, CB, dtype=I16), runs=z(U, D, 6, dtype=I32),
        q=z(U, G, D), workspace=z(4096, dtype=U8), topk_idx=z(U, G, K, dtype=I32), topk_score=z(U, G, K),
        scores=z(U, G, N))),
    "fathom_exact_topk": (["shape", "k_rows", "q", "workspace"], lambda: dict(
        shape=shape_(), k_rows=z(U, N, D, dtype=BF), q=z(U, G, D), workspace=z(4096, dtype=U8),
        topk_idx=z(U, G, K, dtype=I32), topk_score=z(U, G, K), scores=z(U, G, N))),
    "fathom_dense_attn": (["shape", "k_rows", "v_rows", "q", "workspace"], lambda: dict(
        shape=shape_(), k_rows=z(U, N, D, dtype=BF), v_rows=z(U, N, D, dtype=BF), q=z(U, G, D),
        workspace=z(4096, dtype=U8), out=z(U, G, D))),
    "fathom_klt_online": (["shape", "k_rows"], lambda: dict(
        shape=shape_(), k_rows=z(U, N, D, dtype=BF), workspace=z(4096, dtype=U8), mean=z(U, D, dtype=F64),
        V=z(U, D, D, dtype=F64), lam=z(U, D))),
    "fathom_sparse_attn": (["shape", "k_rows", "v_rows", "q", "topk_idx", "workspace"], lambda: dict(
        shape=shape_(), k_rows=z(U, N, D, dtype=BF), v_rows=z(U, N, D, dtype=BF), q=z(U, G, D),
        topk_idx=z(U, G, K, dtype=I32), workspace=z(4096, dtype=U8), out=z(U, G, D))),
    "fathom_sparse_attn_planes": (["shape", "planes", "scales", "v_rows", "q", "topk_idx", "workspace"], lambda: dict(
        shape=shape_(), planes=z(U, D, 4, CB, dtype=I64), scales=z(U, D, CB, dtype=I16),
        v_rows=z(U, N, D, dtype=BF), q=z(U, G, D), topk_idx=z(U, G, K, dtype=I32), workspace=z(4096, dtype=U8),
        out=z(U, G, D))),
    "fathom_sparse_attn_noalloc": (["shape", "k_rows", "v_rows", "q", "topk_idx", "out"], lambda: dict(
        shape=shape_(), k_rows=z(U, N, D, dtype=BF), v_rows=z(U, N, D, dtype=BF), q=z(U, G, D),
        topk_idx=z(U, G, K, dtype=I32), out=z(U, G, D))),
}


def invoke(name, kw):
    pos, _ = CASES[name]
    args = [kw.pop(p) for p in pos]
    return getattr(B, name)(*args, **kw)


@pytest.mark.parametrize("name", sorted(CASES))
def test_valid_arguments_reach_the_library_call(name):
    with pytest.raises(Reached):
        invoke(name, CASES[name][1]())


# every tensor argument except the workspaces, whose size the library itself checks
@pytest.mark.parametrize("name,arg", [(nm, a) for nm in sorted(CASES) for a, v in CASES[nm][1]().items()
                                      if isinstance(v, torch.Tensor) and a != "workspace"])
def test_every_tensor_one_element_short_is_rejected(name, arg):
    kw = CASES[name][1]()
    kw[arg] = short(kw[arg])
    with pytest.raises(ValueError, match=rf"^{arg}\b"):
        invoke(name, kw)


def test_wrong_dtype_is_rejected():
    kw = CASES["fathom_scan_topk"][1]()
    kw["planes"] = kw["planes"].to(torch.int32)
    with pytest.raises(TypeError, match=r"^planes\b"):
        invoke("fathom_scan_topk", kw)


def test_staging_strides_come_from_the_last_dimension():
    kw = CASES["fathom_scan_topk"][1]()
    kw.update(planes=z(U, W, dtype=I64), scales=z(U, S, dtype=I16), source=B.SRC_STAGING)
    with pytest.raises(Reached):
        invoke("fathom_scan_topk", dict(kw))
    # a flat staging area of U * W words reads as one unit of U * W words: too short for U units
    kw["planes"] = z(U * W, dtype=I64)
    with pytest.raises(ValueError, match=r"^planes\b"):
        invoke("fathom_scan_topk", kw)


def test_store_sized_for_n_is_too_short_for_a_capacity_layout():
    # the shape says the store is laid out for 320 tokens (5 blocks); a store of 4 blocks is short
    for name in ("fathom_scan_topk", "fathom_gather", "fathom_quantize_pack"):
        kw = CASES[name][1]()
        kw["shape"] = shape_(n_cap=320)
        with pytest.raises(ValueError):
            invoke(name, kw)


def test_non_contiguous_and_unreachable_memory_are_rejected(monkeypatch):
    kw = CASES["fathom_sparse_attn"][1]()
    kw["q"] = z(U, D, G).transpose(1, 2)
    with pytest.raises(ValueError, match=r"^q must be contiguous"):
        invoke("fathom_sparse_attn", kw)
    monkeypatch.setattr(B, "_reachable", lambda t: False)
    with pytest.raises(ValueError, match="CUDA tensor or pinned"):
        invoke("fathom_sparse_attn", CASES["fathom_sparse_attn"][1]())
