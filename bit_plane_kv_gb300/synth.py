"""Seeded synthetic inputs shaped like the Fathom workloads.

This module only draws random numbers.  It holds none of the method's
arithmetic (no quantisation, importance, planning, scoring, selection or
attention); both the CUDA path and the CPU oracle receive the tensors drawn
here.  Every tensor comes from its own torch generator seeded from
(workload seed, unit, tensor kind), so a unit's inputs do not depend on how
many other units are drawn or on the order of the draws.

Distributions (one "unit" = one sequence x layer x KV head), after the
Fathom review page's experimental setup (Qwen3-8B shape: 36 layers, 8 KV
heads, 4 query heads per KV head, 128 channels; §1) with synthetic content:

* sigma_j = exp(z_j), z_j ~ N(0, 1): log-normal channel scales, so a few
  channels dominate;  "outliers" channels (chosen by a seeded permutation)
  are scaled by 8.
* keys k_ij ~ N(0, sigma_j^2); calibration keys (1024 rows) likewise.
* queries q_hj ~ N(0, 1) * sigma_j^0.5.
* value rows ~ N(0, 1).
* rotated-basis workloads: keys R diag(sigma) z with a seeded random
  orthogonal R per unit (QR of a Gaussian matrix); queries R (N(0,1) sigma^0.5).
* sigma, R and the calibration keys belong to a unit's (layer, KV head): in a
  multi-session batch every sequence shares them (one calibration per layer
  and head); keys, queries and values are the unit's own.
* bf16 rows are the round-to-nearest-even of the fp32 draws.
"""
from __future__ import annotations

import dataclasses
import hashlib

import torch

CALIB_ROWS = 1024

_KIND = {"sigma": 1, "keys": 2, "q": 3, "calib": 4, "v": 5, "rot": 6, "qstep": 7}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    n: int
    seqs: int = 1
    layers: int = 1
    kv_heads: int = 1
    G: int = 4
    D: int = 128
    k: int = 512
    n_sink: int = 4
    n_recent: int = 32
    budgets: tuple = (48,)          # flat budget(s), or one per layer when per_layer
    per_layer: bool = False
    outliers: int = 0
    keys_dtype: str = "bf16"        # the store is quantised from these values
    regime: str = "hbm"             # "hbm" (store and rows in HBM) or "host"
    rotated: bool = False

    @property
    def units(self) -> int:
        return self.seqs * self.layers * self.kv_heads

    def units_per_layer(self) -> int:
        return self.seqs * self.kv_heads

    def unit_index(self, seq: int, layer: int, head: int) -> int:
        """Units are packed (sequence, layer, KV head) row-major."""
        return (seq * self.layers + layer) * self.kv_heads + head

    def layer_units(self, layer: int) -> list:
        return [self.unit_index(s, layer, h) for s in range(self.seqs) for h in range(self.kv_heads)]

    def dist_unit(self, unit: int) -> int:
        """The (layer, KV head) a unit belongs to: the index of its key distribution
        and calibration set, shared by every sequence of a multi-session batch."""
        return unit % (self.layers * self.kv_heads)


# The five workloads: shapes, budgets and regimes as the Fathom measurements
# describe them (single layer n=4096; Qwen3-8B decode at 32k; host-resident
# 256k and 1M; 32-session rotated-basis batch), seeded 20260000 + index.
WORKLOADS = {
    "single_4k": Workload("single_4k", 20260000, n=4096, k=64, budgets=(48,), keys_dtype="f32"),
    "qwen3_32k": Workload("qwen3_32k", 20260001, n=32768, layers=36, kv_heads=8, budgets=(48,),
                          outliers=3),
    "host_256k": Workload("host_256k", 20260002, n=262144, layers=4, kv_heads=8,
                          budgets=(32, 48, 64), outliers=3, regime="host"),
    "host_1m": Workload("host_1m", 20260003, n=1048576, layers=4, kv_heads=8, budgets=(48, 64),
                        outliers=3, regime="host"),
    "klt_32x64k": Workload("klt_32x64k", 20260004, n=65536, seqs=32, layers=8, kv_heads=8,
                           budgets=(24, 128, 32, 40, 48, 56, 32, 24), per_layer=True, outliers=3,
                           rotated=True),
}


def shrink(w: Workload, **kw) -> Workload:
    """Same distributions, smaller sizes (parity cases the oracle finishes quickly)."""
    return dataclasses.replace(w, **kw)


def _seed(w: Workload, unit: int, kind: str, extra: int = 0) -> int:
    h = hashlib.sha256(f"{w.seed}:{unit}:{_KIND[kind]}:{extra}".encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(w, unit, kind, device, extra=0):
    g = torch.Generator(device=device)
    g.manual_seed(_seed(w, unit, kind, extra))
    return g


def unit_sigma(w: Workload, unit: int, device="cpu") -> torch.Tensor:
    g = _gen(w, w.dist_unit(unit), "sigma", device)
    sigma = torch.exp(torch.randn(w.D, generator=g, device=device))
    if w.outliers:
        pick = torch.randperm(w.D, generator=g, device=device)[: w.outliers]
        sigma[pick] *= 8.0
    return sigma


def unit_rotation(w: Workload, unit: int, device="cpu") -> torch.Tensor:
    g = _gen(w, w.dist_unit(unit), "rot", "cpu")
    a = torch.randn(w.D, w.D, generator=g, dtype=torch.float64)
    qm, r = torch.linalg.qr(a)
    qm = qm * torch.sign(torch.diagonal(r))[None, :]
    return qm.to(device=device, dtype=torch.float32)


def _correlate(w, unit, x, sigma, device):
    x = x * sigma
    if w.rotated:
        x = x @ unit_rotation(w, unit, device).T
    return x


def unit_keys(w: Workload, unit: int, device="cpu", n: int | None = None) -> torch.Tensor:
    """[n][D] fp32 keys (draw in fp32; round with .to(torch.bfloat16) for bf16 rows)."""
    n = w.n if n is None else n
    sigma = unit_sigma(w, unit, device)
    g = _gen(w, unit, "keys", device)
    return _correlate(w, unit, torch.randn(n, w.D, generator=g, device=device), sigma, device)


def unit_calib(w: Workload, unit: int, device="cpu") -> torch.Tensor:
    """[1024][D] calibration keys of the unit's (layer, KV head)."""
    sigma = unit_sigma(w, unit, device)
    g = _gen(w, w.dist_unit(unit), "calib", device)
    return _correlate(w, unit, torch.randn(CALIB_ROWS, w.D, generator=g, device=device), sigma, device)


def unit_query(w: Workload, unit: int, device="cpu", step: int = 0) -> torch.Tensor:
    """[G][D] fp32 queries of one decode step."""
    sigma = unit_sigma(w, unit, device)
    g = _gen(w, unit, "q" if step == 0 else "qstep", device, extra=step)
    return _correlate(w, unit, torch.randn(w.G, w.D, generator=g, device=device), sigma.sqrt(), device)


def unit_values(w: Workload, unit: int, device="cpu", n: int | None = None) -> torch.Tensor:
    n = w.n if n is None else n
    g = _gen(w, unit, "v", device)
    return torch.randn(n, w.D, generator=g, device=device)


def bf16_bits(x: torch.Tensor) -> torch.Tensor:
    """Round-to-nearest-even bf16, returned as its raw 16-bit patterns (int16 view)."""
    return x.to(torch.bfloat16).view(torch.int16)
