"""Byte accounting against the figures the Fathom review page prints (CPU).

The store, the run lists and the scanned bytes follow from the oracle's own
layout and plans; these tests check them against the page's numbers:
68 bytes per token and KV head for the 4-plane store with fp16 block scales
(§3.2); 136 bits per token for the 32-channel, 4-plane comparison scan
(128 code bits + 8 scale bits, §4); "56 bits" for B = 48 with about 32 active
channels (§4); and the Qwen3-8B sizes of §1 (bf16 K/V of one 32k step about
4.8 GB; the 136-bit scan about 160 MB at 32k and 5.1 GB at 1M tokens)."""
import numpy as np
import pytest

from oracle import oracle as O

QWEN3_LAYERS, QWEN3_KV_HEADS, D, G = 36, 8, 128, 4


def scanned_bytes(depth, n):
    """Bytes a plan reads per unit: its runs' plane words and scales."""
    r = O.runs(depth, n)
    return int(r[:, 1].sum()) * 8 + int(r[:, 4].sum()) * 2


def test_store_is_68_bytes_per_token_and_head():
    n = 4096
    keys = np.random.default_rng(3).standard_normal((n, D)).astype(np.float32)
    planes, scales, _ = O.quantize_pack(keys)
    assert (planes.nbytes + scales.nbytes) / n == 68.0


def test_fixed_plan_scans_136_bits_per_token():
    rng = np.random.default_rng(4)
    n = 64 * 1000
    q = rng.standard_normal((G, D)).astype(np.float32)
    var = rng.lognormal(size=D).astype(np.float32)
    depth = O.plan_fixed(q, var, 32, 4)
    assert int((depth == 4).sum()) == 32 and int(depth.sum()) == 128
    assert scanned_bytes(depth, n) * 8 / n == 136.0


@pytest.mark.parametrize("active", [30, 32, 34])
def test_budget_48_scans_48_bits_plus_active_scales(active):
    # any plan with 48 planes over `active` channels reads 48 + 16 * active / 64 bits per token:
    # 56 bits at the page's ~32 active channels
    depth = np.zeros(D, np.uint8)
    depth[:active] = 1
    extra = 48 - active                   # deepen some channels up to 48 planes in all
    i = 0
    while extra:
        add = min(3, extra)
        depth[i] += add
        extra -= add
        i += 1
    assert int(depth.sum()) == 48 and int((depth > 0).sum()) == active
    n = 64 * 512
    assert scanned_bytes(depth, n) * 8 / n == 48 + 16 * active / 64
    if active == 32:
        assert scanned_bytes(depth, n) * 8 / n == 56.0


def test_plans_at_budget_48_use_about_32_channels():
    # on log-normal channel scales the plan at B = 48 spreads its planes over roughly the
    # 30-34 active channels the page reports, and never exceeds the budget
    rng = np.random.default_rng(5)
    actives = []
    for _ in range(50):
        sigma = np.exp(rng.standard_normal(D))
        q = (rng.standard_normal((G, D)) * np.sqrt(sigma)).astype(np.float32)
        var = (sigma ** 2).astype(np.float32)
        depth, _, _ = O.plan(q, var, 48)
        assert int(depth.sum()) <= 48
        actives.append(int((depth > 0).sum()))
    assert 24 <= np.median(actives) <= 40


def test_qwen3_8b_sizes():
    units = QWEN3_LAYERS * QWEN3_KV_HEADS
    kv_bf16_32k = units * 32768 * D * 2 * 2
    assert 4.7e9 < kv_bf16_32k < 4.9e9                      # "4.8 GB" per step at 32k
    scan136_32k = units * 32768 * 136 / 8
    scan136_1m = units * (1 << 20) * 136 / 8
    assert 155e6 < scan136_32k < 165e6                      # "160 MB" at 32k
    assert 5.0e9 < scan136_1m < 5.2e9                       # "5.1 GB" at 1M
