"""The seeded synthetic inputs (CPU): the workload table, reproducibility of
every draw, and the input recipe (log-normal channel scales, 3 outlier
channels at 8 sigma, queries at sigma^0.5, shared bases of a multi-session
batch, bf16 rows as the round-to-nearest-even of the fp32 draws)."""
import numpy as np
import pytest
import torch

from bit_plane_kv_gb300 import synth

W = synth.WORKLOADS


def test_workload_table():
    assert [W[k].seed for k in ("single_4k", "qwen3_32k", "host_256k", "host_1m", "klt_32x64k")] == \
        [20260000 + i for i in range(5)]
    s = W["single_4k"]
    assert (s.units, s.n, s.G, s.D, s.k, s.budgets, s.keys_dtype, s.regime) == (1, 4096, 4, 128, 64, (48,), "f32", "hbm")
    q = W["qwen3_32k"]
    assert (q.layers, q.kv_heads, q.n, q.k, q.budgets, q.outliers, q.regime) == (36, 8, 32768, 512, (48,), 3, "hbm")
    h = W["host_256k"]
    assert (h.layers, h.kv_heads, h.n, h.budgets, h.regime) == (4, 8, 262144, (32, 48, 64), "host")
    m = W["host_1m"]
    assert (m.layers, m.kv_heads, m.n, m.budgets, m.regime) == (4, 8, 1 << 20, (48, 64), "host")
    r = W["klt_32x64k"]
    assert (r.seqs, r.layers, r.kv_heads, r.n, r.rotated, r.per_layer) == (32, 8, 8, 65536, True, True)
    assert np.mean(r.budgets) == 48 and min(r.budgets) >= 24 and max(r.budgets) <= 128
    for w in W.values():
        assert (w.n_sink, w.n_recent, w.G, w.D) == (4, 32, 4, 128)


def test_draws_are_reproducible_and_independent_of_order():
    w = synth.shrink(W["qwen3_32k"], n=256)
    a = synth.unit_keys(w, 5)
    synth.unit_keys(w, 6), synth.unit_values(w, 5), synth.unit_query(w, 5, step=3)
    assert torch.equal(a, synth.unit_keys(w, 5))
    assert not torch.equal(a, synth.unit_keys(w, 6))
    assert not torch.equal(synth.unit_query(w, 5, step=1), synth.unit_query(w, 5, step=2))
    assert torch.equal(synth.unit_query(w, 5, step=2), synth.unit_query(w, 5, step=2))
    # a shorter draw is the prefix of a longer one
    assert torch.equal(synth.unit_keys(w, 5, n=100), a[:100])


def test_outlier_channels_are_three_at_eight_sigma():
    w = W["qwen3_32k"]
    plain = synth.shrink(w, outliers=0)
    for u in (0, 7, 100):
        ratio = (synth.unit_sigma(w, u) / synth.unit_sigma(plain, u)).numpy()
        assert np.sum(np.isclose(ratio, 8.0)) == 3 and np.sum(np.isclose(ratio, 1.0)) == w.D - 3


def test_key_and_query_scales_follow_sigma():
    w = synth.shrink(W["single_4k"], n=20000)
    sigma = synth.unit_sigma(w, 0).double().numpy()
    # sigma_j = exp(z_j), z_j ~ N(0, 1): the log-scales look standard normal
    assert abs(np.log(sigma).mean()) < 0.35 and 0.7 < np.log(sigma).std() < 1.3
    k = synth.unit_keys(w, 0).double().numpy()
    np.testing.assert_allclose(k.std(axis=0), sigma, rtol=0.05)
    qs = torch.stack([synth.unit_query(w, 0, step=s) for s in range(1, 2001)]).double().numpy()   # [steps][G][D]
    np.testing.assert_allclose(qs.reshape(-1, w.D).std(axis=0), np.sqrt(sigma), rtol=0.05)
    c = synth.unit_calib(w, 0).double().numpy()
    assert c.shape == (synth.CALIB_ROWS, w.D)
    np.testing.assert_allclose(c.std(axis=0), sigma, rtol=0.15)


def test_sessions_share_the_basis_of_their_layer_and_head():
    w = synth.shrink(W["klt_32x64k"], n=128)
    u = w.unit_index(0, 3, 5)
    v = w.unit_index(7, 3, 5)              # another session, same layer and KV head
    x = w.unit_index(0, 4, 5)              # another layer
    assert w.dist_unit(u) == w.dist_unit(v) != w.dist_unit(x)
    assert torch.equal(synth.unit_sigma(w, u), synth.unit_sigma(w, v))
    assert torch.equal(synth.unit_rotation(w, u), synth.unit_rotation(w, v))
    assert torch.equal(synth.unit_calib(w, u), synth.unit_calib(w, v))
    assert not torch.equal(synth.unit_keys(w, u), synth.unit_keys(w, v))
    assert not torch.equal(synth.unit_rotation(w, u), synth.unit_rotation(w, x))
    R = synth.unit_rotation(w, u).double()
    np.testing.assert_allclose((R.T @ R).numpy(), np.eye(w.D), atol=1e-6)


def test_units_are_packed_sequence_layer_head():
    w = W["klt_32x64k"]
    assert w.unit_index(0, 0, 1) == 1 and w.unit_index(0, 1, 0) == w.kv_heads
    assert w.unit_index(1, 0, 0) == w.layers * w.kv_heads
    lu = w.layer_units(2)
    assert len(lu) == w.seqs * w.kv_heads == w.units_per_layer()
    assert all((u // w.kv_heads) % w.layers == 2 for u in lu)


def test_bf16_rows_are_round_to_nearest_even():
    x = synth.unit_keys(W["single_4k"], 0, n=4096).reshape(-1)
    x = torch.cat([x, torch.tensor([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -1.0 - 2.0 ** -8])])   # exact ties
    b = x.view(torch.int32).numpy().astype(np.int64) & 0xFFFFFFFF
    lsb = (b >> 16) & 1
    rne = ((b + 0x7FFF + lsb) >> 16) & 0xFFFF          # round half to even on the dropped 16 bits
    got = synth.bf16_bits(x).numpy().astype(np.int64) & 0xFFFF
    np.testing.assert_array_equal(got, rne)
    # the ties went to the even neighbour
    assert list(got[-3:]) == [0x3F80, 0x3F82, 0xBF80]


@pytest.mark.parametrize("name", sorted(W))
def test_layer_units_cover_every_unit_once(name):
    w = W[name]
    seen = sorted(u for l in range(w.layers) for u in w.layer_units(l))
    assert seen == list(range(w.units))
