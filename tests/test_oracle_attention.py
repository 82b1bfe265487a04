"""Pins for the float64 attention oracle (CPU only).

Each test checks the oracle against something other than itself: scalar
brute force on tiny inputs, closed forms, invariants of softmax attention,
torch's float64 CPU attention (a library routine), central finite differences
and exact gradient identities.
"""

import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand(shape, seed):
    return np.random.RandomState(seed).standard_normal(shape)


def _brute_forward(q, k, v, cu, scale, causal, gqa):
    """Scalar loops, math.exp: the definition with nothing vectorised."""
    T, hq, dk = q.shape
    hkv, dv = k.shape[1], v.shape[2]
    o = [[[0.0] * dv for _ in range(hq)] for _ in range(T)]
    lse = [[-math.inf] * T for _ in range(hq)]
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        for h in range(hq):
            kvh = h // (hq // hkv) if gqa == "blocked" else h % hkv
            for i in range(a, b):
                js = [j for j in range(a, b) if (not causal or j <= i)]
                sc = []
                for j in js:
                    acc = 0.0
                    for c in range(dk):
                        acc += q[i, h, c] * k[j, kvh, c]
                    sc.append(scale * acc)
                z = sum(math.exp(x) for x in sc)
                lse[h][i] = math.log(z)
                for c in range(dv):
                    o[i][h][c] = sum(math.exp(x) / z * v[j, kvh, c] for x, j in zip(sc, js))
    return np.array(o), np.array(lse)


@pytest.mark.parametrize("hq,hkv,gqa", [(2, 2, "blocked"), (4, 2, "blocked"), (4, 2, "interleaved"), (3, 1, "blocked")])
@pytest.mark.parametrize("causal", [True, False])
def test_forward_matches_brute_force(hq, hkv, gqa, causal):
    cu = [0, 5, 6, 13]
    T, dk, dv = 13, 4, 3
    q, k, v = _rand((T, hq, dk), 1), _rand((T, hkv, dk), 2), _rand((T, hkv, dv), 3)
    o, lse = oracle.attn_forward(q, k, v, cu, 0.7, causal=causal, gqa=gqa, row_block=3)
    ob, lb = _brute_forward(q, k, v, cu, 0.7, causal, gqa)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-12)


def test_zero_query_closed_form():
    # q = 0: every visible score is 0, so o_i is the mean of the visible v_j
    # and lse_i = log(#visible keys).
    cu = [0, 7, 20]
    T, hq, hkv = 20, 4, 2
    q = np.zeros((T, hq, 8))
    k, v = _rand((T, hkv, 8), 5), _rand((T, hkv, 6), 6)
    o, lse = oracle.attn_forward(q, k, v, cu, 0.3, causal=True)
    for s in range(2):
        a, b = cu[s], cu[s + 1]
        for i in range(a, b):
            n = i - a + 1
            for h in range(hq):
                kvh = h // 2
                np.testing.assert_allclose(o[i, h], v[a:i + 1, kvh].mean(axis=0), atol=1e-13)
                assert abs(lse[h, i] - math.log(n)) < 1e-13


def test_single_token():
    q, k, v = _rand((1, 2, 5), 7), _rand((1, 1, 5), 8), _rand((1, 1, 3), 9)
    o, lse = oracle.attn_forward(q, k, v, [0, 1], 0.5)
    for h in range(2):
        np.testing.assert_allclose(o[0, h], v[0, 0], atol=0)
        assert abs(lse[h, 0] - 0.5 * q[0, h] @ k[0, 0]) < 1e-14


def test_key_shift_invariance():
    # adding the same vector c to every key leaves o unchanged and shifts
    # lse_i by scale * q_i . c
    cu = [0, 33]
    q, k, v = _rand((33, 2, 8), 10), _rand((33, 2, 8), 11), _rand((33, 2, 8), 12)
    c = _rand((8,), 13)
    o1, l1 = oracle.attn_forward(q, k, v, cu, 0.4)
    o2, l2 = oracle.attn_forward(q, k + c, v, cu, 0.4)
    np.testing.assert_allclose(o2, o1, atol=1e-11)
    np.testing.assert_allclose(l2, l1 + 0.4 * np.einsum("thd,d->ht", q, c), atol=1e-11)


def test_causality_and_sequence_isolation():
    cu = [0, 40, 64]
    T = 64
    q, k, v = _rand((T, 2, 8), 14), _rand((T, 1, 8), 15), _rand((T, 1, 4), 16)
    o1, l1 = oracle.attn_forward(q, k, v, cu, 0.3)
    i = 25
    k2, v2 = k.copy(), v.copy()
    k2[i + 1:] += 3.0  # later keys of the same sequence and the next sequence
    v2[i + 1:] -= 2.0
    o2, l2 = oracle.attn_forward(q, k2, v2, cu, 0.3)
    assert np.array_equal(o1[: i + 1], o2[: i + 1])
    assert np.array_equal(l1[:, : i + 1], l2[:, : i + 1])
    # keys of the first sequence never reach the second one
    k3, v3 = k.copy(), v.copy()
    k3[:40] *= -1.5
    v3[:40] += 1.0
    o3, l3 = oracle.attn_forward(q, k3, v3, cu, 0.3)
    assert np.array_equal(o1[40:], o3[40:])
    assert np.array_equal(l1[:, 40:], l3[:, 40:])


def test_varlen_equals_separate_sequences():
    cu = [0, 3, 50, 51, 90]
    T = 90
    q, k, v = _rand((T, 4, 8), 17), _rand((T, 2, 8), 18), _rand((T, 2, 5), 19)
    o, lse = oracle.attn_forward(q, k, v, cu, 0.3, row_block=16)
    for s in range(4):
        a, b = cu[s], cu[s + 1]
        os_, ls = oracle.attn_forward(q[a:b], k[a:b], v[a:b], [0, b - a], 0.3)
        np.testing.assert_allclose(o[a:b], os_, atol=1e-13)
        np.testing.assert_allclose(lse[:, a:b], ls, atol=1e-13)


def _torch_ref(q, k, v, cu, scale, causal, gqa):
    """torch float64 CPU scaled_dot_product_attention per sequence; lse via
    torch.logsumexp over the masked scores."""
    q, k, v = (torch.tensor(x) for x in (q, k, v))
    hq, hkv = q.shape[1], k.shape[1]
    G = hq // hkv
    if gqa == "blocked":
        kx, vx = k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1)
    else:
        kx, vx = k.repeat(1, G, 1), v.repeat(1, G, 1)
    outs, lses = [], []
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        Q, K, V = (x[a:b].transpose(0, 1) for x in (q, kx, vx))
        outs.append(torch.nn.functional.scaled_dot_product_attention(
            Q, K, V, is_causal=causal, scale=scale).transpose(0, 1))
        S = scale * Q @ K.transpose(-1, -2)
        if causal:
            S = S.masked_fill(torch.ones(b - a, b - a, dtype=torch.bool).triu(1), -math.inf)
        lses.append(torch.logsumexp(S, dim=-1))
    return torch.cat(outs).numpy(), torch.cat(lses, dim=1).numpy()


@pytest.mark.parametrize("gqa", ["blocked", "interleaved"])
@pytest.mark.parametrize("causal", [True, False])
def test_forward_matches_torch_sdpa(gqa, causal):
    cu = [0, 100, 101, 300]
    T = 300
    q, k, v = _rand((T, 8, 16), 20), _rand((T, 2, 16), 21), _rand((T, 2, 12), 22)
    o, lse = oracle.attn_forward(q, k, v, cu, 0.25, causal=causal, gqa=gqa, row_block=64)
    ot, lt = _torch_ref(q, k, v, cu, 0.25, causal, gqa)
    np.testing.assert_allclose(o, ot, atol=1e-12)
    np.testing.assert_allclose(lse, lt, atol=1e-12)


def test_backward_matches_finite_differences():
    cu = [0, 6, 11]
    T, hq, hkv, dk, dv = 11, 4, 2, 3, 2
    q, k, v = _rand((T, hq, dk), 23), _rand((T, hkv, dk), 24), _rand((T, hkv, dv), 25)
    dout = _rand((T, hq, dv), 26)
    scale = 0.8
    g = oracle.attn_backward(q, k, v, dout, cu, scale, row_block=4)

    def loss(q_, k_, v_):
        o, _ = oracle.attn_forward(q_, k_, v_, cu, scale)
        return float((o * dout).sum())

    eps = 1e-6
    for name, x, grad in (("q", q, g["dq"]), ("k", k, g["dk"]), ("v", v, g["dv"])):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            lp = loss(args["q"], args["k"], args["v"])
            args[name] = xm
            lm = loss(args["q"], args["k"], args["v"])
            num[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(grad, num, atol=2e-8, rtol=1e-6, err_msg=name)


@pytest.mark.parametrize("gqa", ["blocked", "interleaved"])
def test_backward_matches_torch_autograd(gqa):
    cu = [0, 70, 200]
    T = 200
    q, k, v = _rand((T, 6, 16), 27), _rand((T, 2, 16), 28), _rand((T, 2, 8), 29)
    dout = _rand((T, 6, 8), 30)
    g = oracle.attn_backward(q, k, v, dout, cu, 0.3, gqa=gqa, row_block=48)
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    G = 3
    outs = []
    for s in range(2):
        a, b = cu[s], cu[s + 1]
        if gqa == "blocked":
            K, V = kt[a:b].repeat_interleave(G, 1), vt[a:b].repeat_interleave(G, 1)
        else:
            K, V = kt[a:b].repeat(1, G, 1), vt[a:b].repeat(1, G, 1)
        outs.append(torch.nn.functional.scaled_dot_product_attention(
            qt[a:b].transpose(0, 1), K.transpose(0, 1), V.transpose(0, 1),
            is_causal=True, scale=0.3).transpose(0, 1))
    torch.cat(outs).backward(torch.tensor(dout))
    np.testing.assert_allclose(g["dq"], qt.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(g["dk"], kt.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(g["dv"], vt.grad.numpy(), atol=1e-11)


def test_backward_identities():
    # sum_j dS_ij = 0 for every row, so sum_j dk_j = 0 per sequence and kv head;
    # sum_j P_ij = 1, so sum_j dv_j = sum over the group's heads of sum_i dO_i.
    cu = [0, 50, 129]
    T = 129
    q, k, v = _rand((T, 4, 8), 31), _rand((T, 2, 8), 32), _rand((T, 2, 8), 33)
    dout = _rand((T, 4, 8), 34)
    g = oracle.attn_backward(q, k, v, dout, cu, 0.35, row_block=32)
    for s in range(2):
        a, b = cu[s], cu[s + 1]
        np.testing.assert_allclose(g["dk"][a:b].sum(axis=0), 0.0, atol=1e-12)
        for kvh in range(2):
            want = dout[a:b, 2 * kvh:2 * kvh + 2].sum(axis=(0, 1))
            np.testing.assert_allclose(g["dv"][a:b, kvh].sum(axis=0), want, atol=1e-12)
    # D_i = dO_i . o_i = sum_j P_ij dP_ij
    np.testing.assert_allclose(g["D"], np.einsum("thd,thd->ht", dout, g["o"]), atol=1e-13)


@pytest.mark.parametrize("causal,gqa", [(True, "blocked"), (False, "blocked"), (True, "interleaved")])
def test_sampled_rows_agree_with_full(causal, gqa):
    """The long-sequence samplers equal the full functions on the selected
    rows, with row blocks and chunks small enough that every sequence spans
    several of them (so the blocking itself is exercised)."""
    cu = [0, 90, 91, 200]
    T = 200
    q, k, v = _rand((T, 4, 8), 35), _rand((T, 2, 8), 36), _rand((T, 2, 6), 37)
    dout = _rand((T, 4, 6), 38)
    g = oracle.attn_backward(q, k, v, dout, cu, 0.4, causal=causal, gqa=gqa, row_block=32)
    rows = [0, 17, 18, 40, 89, 90, 91, 150, 151, 152, 199]
    heads = [0, 3]
    for chunk in (128, 3):
        o, lse = oracle.attn_forward_rows(q, k, v, cu, 0.4, rows, heads, causal=causal, gqa=gqa, chunk=chunk)
        np.testing.assert_allclose(o, g["o"][rows][:, heads], atol=1e-13)
        np.testing.assert_allclose(lse, g["lse"][heads][:, rows], atol=1e-13)
        dq = oracle.attn_backward_dq_rows(q, k, v, dout, cu, 0.4, rows, heads, causal=causal, gqa=gqa, chunk=chunk)
        np.testing.assert_allclose(dq, g["dq"][rows][:, heads], atol=1e-12)
    keys = [0, 5, 80, 89, 90, 91, 120, 121, 199]
    for row_block in (1024, 7):
        dk, dv = oracle.attn_backward_dkdv_rows(q, k, v, dout, cu, 0.4, keys, [0, 1], causal=causal, gqa=gqa,
                                                row_block=row_block)
        np.testing.assert_allclose(dk, g["dk"][keys], atol=1e-12)
        np.testing.assert_allclose(dv, g["dv"][keys], atol=1e-12)
    # a torch bf16 input (how the GPU tests pass it) gives the same rows as its float64 copy
    qt = torch.from_numpy(q).to(torch.bfloat16)
    q64 = qt.to(torch.float64).numpy()
    o_t, _ = oracle.attn_forward_rows(qt, k, v, cu, 0.4, rows, heads, causal=causal, gqa=gqa)
    o_n, _ = oracle.attn_forward_rows(q64, k, v, cu, 0.4, rows, heads, causal=causal, gqa=gqa)
    np.testing.assert_array_equal(o_t, o_n)
