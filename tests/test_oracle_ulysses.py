"""Pins for the oracle's Ulysses re-layout (CPU only).

"Ulysses Context Parallelism 的工程取舍全记录" §1.2: sequence shards of all heads
become, through an all-to-all, the whole sequence of H/C heads per device
(device r: heads r*H/C ..), attention runs unsharded per device, and a second
all-to-all restores the sequence shards.
"""

import numpy as np
import pytest

import oracle
import workloads


def _rand(shape, seed):
    return np.random.RandomState(seed).standard_normal(shape)


@pytest.mark.parametrize("layout", ["contiguous", "zigzag"])
def test_scatter_worked_example(layout):
    # 4 tokens, 4 heads, C = 2; x[t, h] = 10 t + h in global order.  Written
    # out by hand: device 0 gets heads 0-1 of every token, device 1 heads 2-3.
    xg = np.array([[10 * t + h for h in range(4)] for t in range(4)], dtype=np.float64)
    perm = oracle.shard_order([0, 4], 2, layout)
    xs = xg[perm]
    want = np.array([[[0, 1], [10, 11], [20, 21], [30, 31]],
                     [[2, 3], [12, 13], [22, 23], [32, 33]]], dtype=np.float64)
    assert np.array_equal(oracle.ulysses_scatter(xs, perm, 2), want)
    assert np.array_equal(oracle.ulysses_gather(want, perm), xs)


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
def test_round_trips(layout):
    cu = workloads.make_cu_seqlens([37, 1, 90]).tolist()
    T = cu[-1]
    perm = oracle.shard_order(cu, 4, layout)
    x = _rand((T, 8, 3), 1)
    y = oracle.ulysses_scatter(x, perm, 4)
    assert y.shape == (4, T, 2, 3)
    assert np.array_equal(oracle.ulysses_gather(y, perm), x)
    l = _rand((8, T), 2)
    lu = oracle.ulysses_scatter_lse(l, perm, 4)
    assert lu.shape == (4, 2, T)
    assert np.array_equal(oracle.ulysses_gather_lse(lu, perm), l)
    # head slice r of device r, in global order, is head block r of the input
    xg = oracle.to_global(x, perm)
    for r in range(4):
        assert np.array_equal(y[r], xg[:, 2 * r:2 * r + 2])


@pytest.mark.parametrize("layout", ["zigzag", "striped"])
def test_per_device_attention_equals_full_attention(layout):
    # Ulysses composition: scatter q, k, v; unsharded attention on every
    # device's heads (GQA 2:1 kept inside each device); gather o and lse.
    # Heads are independent, so the result is the full attention.
    cu = workloads.make_cu_seqlens([40, 3, 57]).tolist()
    T, C, hq, hkv = cu[-1], 2, 4, 2
    q, k, v = _rand((T, hq, 8), 3), _rand((T, hkv, 8), 4), _rand((T, hkv, 6), 5)
    o_ref, l_ref = oracle.attn_forward(q, k, v, cu, 0.4)
    perm = oracle.shard_order(cu, C, layout)
    qs, ks, vs = q[perm], k[perm], v[perm]
    qu, ku, vu = (oracle.ulysses_scatter(t, perm, C) for t in (qs, ks, vs))
    ou, lu = [], []
    for r in range(C):
        o_r, l_r = oracle.attn_forward(qu[r], ku[r], vu[r], cu, 0.4)
        ou.append(o_r)
        lu.append(l_r)
    o_s = oracle.ulysses_gather(np.stack(ou), perm)
    l_s = oracle.ulysses_gather_lse(np.stack(lu), perm)
    np.testing.assert_allclose(o_s, o_ref[perm], atol=1e-13)
    np.testing.assert_allclose(l_s, l_ref[:, perm], atol=1e-13)


def test_head_count_must_divide():
    with pytest.raises(ValueError):
        oracle.ulysses_scatter(np.zeros((4, 3, 2)), np.arange(4), 2)
