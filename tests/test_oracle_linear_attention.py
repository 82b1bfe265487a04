"""Pins for the oracle's decayed linear attention and its AllGather CP
state recovery (CPU only).  "超长上下文训练速度翻倍秘籍": h_t = alpha h_{t-1} +
K_t^T V_t, O_t = Q_t h_t; AllGather CP gathers the rank-local states,
recovers each rank's initial state by a decayed prefix and corrects the
local outputs by (q * decay) @ init_state."""

import numpy as np
import pytest

import oracle
import workloads


def _rand(shape, seed):
    return np.random.RandomState(seed).standard_normal(shape)


def test_worked_example_scalar_heads():
    # one head, Dk = Dv = 1, alpha = 0.5, scale 1: h = 1, 0.5*1 + 2, 0.5*2.5 + 3
    q = np.ones((3, 1, 1))
    k = np.array([1.0, 2.0, 3.0]).reshape(3, 1, 1)
    v = np.ones((3, 1, 1))
    g = [np.log(0.5)]
    want = [1.0, 2.5, 4.25]
    for f in (oracle.linear_attn_forward, oracle.linear_attn_recurrent):
        np.testing.assert_allclose(f(q, k, v, [0, 3], g, 1.0).ravel(), want, rtol=1e-14)


def test_recurrence_equals_definition():
    cu = workloads.make_cu_seqlens([17, 1, 40]).tolist()
    T = cu[-1]
    q, k, v = _rand((T, 3, 4), 1), _rand((T, 3, 4), 2), _rand((T, 3, 5), 3)
    g = [-0.05, -0.5, -2.0]
    a = oracle.linear_attn_forward(q, k, v, cu, g, 0.5)
    b = oracle.linear_attn_recurrent(q, k, v, cu, g, 0.5)
    np.testing.assert_allclose(a, b, atol=1e-12)


def test_no_decay_is_a_cumulative_sum():
    q, k, v = _rand((9, 2, 3), 4), _rand((9, 2, 3), 5), _rand((9, 2, 2), 6)
    kv = np.cumsum(k[:, :, :, None] * v[:, :, None, :], axis=0)  # [T, H, Dk, Dv]
    want = 0.7 * np.einsum("thd,thde->the", q, kv)
    np.testing.assert_allclose(oracle.linear_attn_forward(q, k, v, [0, 9], [0.0, 0.0], 0.7), want, atol=1e-12)


def test_full_decay_keeps_only_the_diagonal():
    q, k, v = _rand((6, 1, 3), 7), _rand((6, 1, 3), 8), _rand((6, 1, 4), 9)
    want = 0.3 * np.einsum("thd,thd->th", q, k)[:, :, None] * v
    np.testing.assert_allclose(oracle.linear_attn_forward(q, k, v, [0, 6], [-60.0], 0.3), want, atol=1e-12)


def test_local_state_is_the_final_hidden_state():
    k, v = _rand((11, 2, 3), 10), _rand((11, 2, 4), 11)
    g = np.array([-0.1, -1.0])
    h = np.zeros((2, 3, 4))
    for t in range(11):
        h = np.exp(g)[:, None, None] * h + k[t][:, :, None] * v[t][:, None, :]
    np.testing.assert_allclose(oracle.local_state(k, v, g), h, atol=1e-12)


@pytest.mark.parametrize("C", [1, 2, 3, 8])
def test_allgather_cp_equals_unsharded(C):
    cu = workloads.make_cu_seqlens([50, 2, 31, 7]).tolist()
    T = cu[-1]
    q, k, v = _rand((T, 2, 4), 12), _rand((T, 2, 4), 13), _rand((T, 2, 3), 14)
    g = [-0.02, -0.3]
    want = oracle.linear_attn_forward(q, k, v, cu, g, 0.5)
    np.testing.assert_allclose(oracle.linear_attn_cp(q, k, v, cu, g, 0.5, C), want, atol=1e-12)
