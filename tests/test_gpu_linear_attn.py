"""GPU parity of decayed linear attention with AllGather CP.

"超长上下文训练速度翻倍秘籍": h_t = alpha h_{t-1} + K_t^T V_t, O_t = Q_t h_t; every
rank computes its piece's local state, the gathered states give each rank its
initial state by a decayed prefix, and the output is corrected by
(q * decay) @ init_state.  The GPU result is compared with the oracle's
definition (o_t = scale sum_{s<=t} alpha^(t-s) (q_t.k_s) v_s) and with its
step-by-step AllGather CP.  Outputs are not bounded like softmax attention,
so the comparison is relative (Frobenius): 1e-5 for fp32 runs, 2e-2 for
bf16 (the bf16-gradient bar of the other tests).
"""

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

cpa = pytest.importorskip("context_long_sequence_zigzag_gb300")


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _case(lengths, H, Dk, Dv, C, dtype, seed):
    cu = workloads.make_cu_seqlens(lengths).tolist()
    T = cu[-1]
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(T, H, Dk, generator=gen) * 0.5
    k = torch.randn(T, H, Dk, generator=gen) * 0.5
    v = torch.randn(T, H, Dv, generator=gen)
    g = -torch.rand(H, generator=gen) * 0.9 - 0.05  # decay alpha in (0.39, 0.95)
    if dtype == torch.bfloat16:
        q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    scale = Dk ** -0.5
    prob = cpa.Problem(T, H, H, Dk, Dv, C, "contiguous", cu, True, scale, "blocked", dtype)
    perm = torch.from_numpy(oracle.shard_order(cu, C, "contiguous"))
    qs, ks, vs = (t.index_select(0, perm).contiguous().cuda() for t in (q, k, v))
    o_s = cpa.cp_lin_attn_fwd(prob, qs, ks, vs, g.cuda())
    torch.cuda.synchronize()
    o = torch.empty_like(o_s.cpu())
    o[perm] = o_s.cpu()
    qd, kd, vd = (t.double().numpy() for t in (q, k, v))
    ref = oracle.linear_attn_forward(qd, kd, vd, cu, g.double().numpy(), scale)
    return o.double().numpy(), ref, (qd, kd, vd, cu, g.double().numpy(), scale)


@pytest.mark.parametrize("lengths,C", [([300], 1), ([150, 2, 148], 4), ([700, 1, 99], 8), ([5, 3], 8)])
def test_fp32_matches_definition(lengths, C):
    o, ref, _ = _case(lengths, H=2, Dk=32, Dv=48, C=C, dtype=torch.float32, seed=41)
    assert _rel(o, ref) < 1e-5


def test_fp32_matches_the_pages_cp_steps():
    o, ref, (q, k, v, cu, g, scale) = _case([400, 17, 250], H=3, Dk=40, Dv=24, C=4, dtype=torch.float32, seed=42)
    steps = oracle.linear_attn_cp(q, k, v, cu, g, scale, 4)
    assert _rel(o, steps) < 1e-5


@pytest.mark.parametrize("C", [2, 8])
def test_bf16_heads_128(C):
    o, ref, _ = _case([2500, 33, 1563], H=4, Dk=128, Dv=128, C=C, dtype=torch.bfloat16, seed=43)
    assert _rel(o, ref) < 2e-2


def test_cp_size_does_not_change_the_result():
    a, _, _ = _case([1000, 24], H=2, Dk=64, Dv=64, C=1, dtype=torch.float32, seed=44)
    b, _, _ = _case([1000, 24], H=2, Dk=64, Dv=64, C=8, dtype=torch.float32, seed=44)
    assert _rel(b, a) < 1e-5


def test_bf16_full_size_sampled_heads():
    """The configuration the benchmark times: one 64K-token sequence, 16 heads
    of 128, C = 8 contiguous pieces, bf16.  The float64 recurrence runs over
    the whole sequence for two sampled heads (the first and the last)."""
    T, H, D, C = 65536, 16, 128, 8
    cu = [0, T]
    gen = torch.Generator().manual_seed(45)
    q = (torch.randn(T, H, D, generator=gen) * 0.5).to(torch.bfloat16)
    k = (torch.randn(T, H, D, generator=gen) * 0.5).to(torch.bfloat16)
    v = torch.randn(T, H, D, generator=gen).to(torch.bfloat16)
    g = -torch.rand(H, generator=gen) * 0.9 - 0.05
    scale = D ** -0.5
    prob = cpa.Problem(T, H, H, D, D, C, "contiguous", cu, True, scale, "blocked", torch.bfloat16)
    # contiguous pieces of one sequence: sharded order is global order
    o = cpa.cp_lin_attn_fwd(prob, q.cuda(), k.cuda(), v.cuda(), g.cuda()).cpu()
    heads = [0, H - 1]
    sel = lambda t: t[:, heads].double().numpy()
    ref = oracle.linear_attn_recurrent(sel(q), sel(k), sel(v), cu, g[heads].double().numpy(), scale)
    assert _rel(sel(o), ref) < 2e-2
