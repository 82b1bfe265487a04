"""GPU parity of Ulysses (all-to-all) context parallelism on one GPU.

"Ulysses Context Parallelism 的工程取舍全记录" §1.2: an all-to-all turns sequence
shards of every head into the whole sequence of H/C heads per rank, each rank
runs unsharded attention, and a second all-to-all restores the shards.  The
re-layout is checked bit-exact against the oracle's scatter / gather; the
attention against the float64 oracle (tolerances of the ring path) and
against the ring path's own result.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import (BF16_GRAD_RFRO, BF16_LSE_ATOL, BF16_O_ATOL, F32_ATOL, f64, max_abs, perm_of, rel_fro,
                      to_dev_sharded, to_host_global)

pytestmark = pytest.mark.gpu

cpa = pytest.importorskip("context_long_sequence_zigzag_gb300")


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
@pytest.mark.parametrize("C,heads,dtype", [(4, 8, torch.bfloat16), (2, 2, torch.float32), (8, 8, torch.bfloat16)])
def test_a2a_bit_exact(layout, C, heads, dtype):
    lengths = [1, 130, 7, 700, 65]
    cu = workloads.make_cu_seqlens(lengths).tolist()
    T = cu[-1]
    prob = cpa.Problem(T, heads, heads, 64, 64, C, layout, cu, dtype=dtype)
    g = torch.Generator().manual_seed(5)
    x = torch.randn(T, heads, 64, generator=g).to(dtype)
    perm = oracle.shard_order(cu, C, layout)
    xs = x[torch.from_numpy(perm)].contiguous()
    want = oracle.ulysses_scatter(xs.float().numpy(), perm, C)
    y = cpa.cp_ulysses_a2a(prob, xs.cuda())
    assert tuple(y.shape) == (C, T, heads // C, 64)
    assert torch.equal(y.cpu().float(), torch.from_numpy(want).float())
    back = cpa.cp_ulysses_a2a(prob, y, inverse=True)
    torch.cuda.synchronize()
    assert torch.equal(back.cpu(), xs)


def _run(w, gqa="blocked"):
    inp = workloads.make_inputs(w, with_dout=True)
    cu = inp["cu_seqlens"].tolist()
    perm = perm_of(cu, w.cp_size, w.layout)
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    prob = cpa.Problem(w.total_tokens, w.hq, w.hkv, w.d_qk, w.d_v, w.cp_size, w.layout, cu, w.causal, w.scale, gqa, dt)
    q, k, v, do = (to_dev_sharded(inp[n], perm) for n in ("q", "k", "v", "dout"))
    o_u, l_u = cpa.cp_ulysses_attn_fwd(prob, q, k, v)
    o_r, l_r = cpa.cp_attn_fwd(prob, q, k, v)
    g_u = cpa.cp_ulysses_attn_bwd(prob, q, k, v, o_u, l_u, do)
    g_r = cpa.cp_attn_bwd(prob, q, k, v, o_r, l_r, do)
    torch.cuda.synchronize()
    assert cpa.cp_device_status() == 0
    return inp, cu, perm, (o_u, l_u, g_u), (o_r, l_r, g_r)


CASES = [
    dict(total_tokens=600, hq=4, hkv=2, d_qk=64, d_v=64, cp_size=2, layout="zigzag", dtype="f32",
         seqlens=(300, 5, 295)),
    dict(total_tokens=3000, hq=8, hkv=4, d_qk=128, d_v=128, cp_size=4, layout="zigzag", dtype="bf16",
         seqlens=(1700, 3, 1297)),
    dict(total_tokens=2048, hq=4, hkv=4, d_qk=128, d_v=128, cp_size=4, layout="striped", dtype="bf16"),
    dict(total_tokens=1500, hq=4, hkv=2, d_qk=192, d_v=128, cp_size=2, layout="contiguous", dtype="bf16",
         sigma=0.5),
]


@pytest.mark.parametrize("kw", CASES)
def test_ulysses_attention_matches_oracle_and_ring(kw):
    w = workloads.Workload(name="t", seed=31, **kw)
    inp, cu, perm, (o_u, l_u, g_u), (o_r, l_r, g_r) = _run(w)
    o_ref, l_ref = oracle.attn_forward(inp["q"], inp["k"], inp["v"], cu, w.scale)
    ref = oracle.attn_backward(inp["q"], inp["k"], inp["v"], inp["dout"], cu, w.scale, True)
    o = f64(to_host_global(o_u, perm))
    lse = np.empty_like(f64(l_u))
    lse[:, perm.numpy()] = f64(l_u)
    grads = {n: f64(to_host_global(t, perm)) for n, t in zip(("dq", "dk", "dv"), g_u)}
    if w.dtype == "f32":
        assert max_abs(o, o_ref) < F32_ATOL and max_abs(lse, l_ref) < F32_ATOL
        for n in grads:
            assert max_abs(grads[n], ref[n]) < F32_ATOL, n
    else:
        assert max_abs(o, o_ref) < BF16_O_ATOL and max_abs(lse, l_ref) < BF16_LSE_ATOL
        for n in grads:
            assert rel_fro(grads[n], ref[n]) < BF16_GRAD_RFRO, n
    # and against the ring path on the same inputs
    assert max_abs(f64(o_u), f64(o_r)) < 2 * BF16_O_ATOL
    assert max_abs(f64(l_u), f64(l_r)) < 2 * BF16_LSE_ATOL
    for a, b in zip(g_u, g_r):
        assert rel_fro(f64(a), f64(b)) < 2 * BF16_GRAD_RFRO


def test_ulysses_needs_whole_kv_heads_per_rank():
    # "Ulysses Context Parallelism 的工程取舍全记录" §2: C may not exceed the KV head count
    prob = cpa.Problem(1024, 8, 2, 128, 128, 4, "zigzag")
    with pytest.raises(cpa.CpError) as e:
        cpa.cp_workspace_size(prob, cpa.CP_OP_ULYSSES_FWD)
    assert e.value.status == cpa.CP_ERR_UNSUPPORTED


def test_full_size_ulysses_matches_ring():
    # the S=64K bench workload: Ulysses and ring results agree element-wise
    w = workloads.get("bf16_gqa_s64k_h32kv8_d128_c8_zigzag")
    inp = workloads.make_inputs(w, device="cuda", with_dout=True)
    cu = inp["cu_seqlens"].tolist()
    prob = cpa.Problem(w.total_tokens, w.hq, w.hkv, w.d_qk, w.d_v, w.cp_size, w.layout, cu, w.causal, w.scale)
    sh = {n: cpa.cp_shard_permute(prob, inp[n]) for n in ("q", "k", "v", "dout")}
    del inp
    o_u, l_u = cpa.cp_ulysses_attn_fwd(prob, sh["q"], sh["k"], sh["v"])
    o_r, l_r = cpa.cp_attn_fwd(prob, sh["q"], sh["k"], sh["v"])
    assert float((o_u.float() - o_r.float()).abs().max()) < 2 * BF16_O_ATOL
    assert float((l_u - l_r).abs().max()) < 2 * BF16_LSE_ATOL
    del o_u, l_u
    g_u = cpa.cp_ulysses_attn_bwd(prob, sh["q"], sh["k"], sh["v"], o_r, l_r, sh["dout"])
    g_r = cpa.cp_attn_bwd(prob, sh["q"], sh["k"], sh["v"], o_r, l_r, sh["dout"])
    torch.cuda.synchronize()
    assert cpa.cp_device_status() == 0
    for a, b in zip(g_u, g_r):
        a, b = a.float(), b.float()
        assert float((a - b).norm() / b.norm()) < 2 * BF16_GRAD_RFRO
