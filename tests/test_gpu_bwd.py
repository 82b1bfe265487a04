"""GPU backward parity against the float64 oracle.

dq/dk/dv are compared by relative Frobenius error: 2e-2 for bf16 runs; fp32
runs use max-abs 1e-5.  The GPU backward consumes the GPU forward's o and lse
(as training does); the oracle recomputes everything from q, k, v, dout.
"""

import pytest
import torch

import oracle
import workloads
from gpu_util import (BF16_GRAD_RFRO, F32_ATOL, f64, max_abs, perm_of, rel_fro, to_dev_sharded,
                      to_host_global)

pytestmark = pytest.mark.gpu

cpa = pytest.importorskip("context_long_sequence_zigzag_gb300")


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _run(w: workloads.Workload, gqa="blocked"):
    inp = workloads.make_inputs(w, with_dout=True)
    cu = inp["cu_seqlens"].tolist()
    perm = perm_of(cu, w.cp_size, w.layout)
    prob = cpa.Problem(w.total_tokens, w.hq, w.hkv, w.d_qk, w.d_v, w.cp_size, w.layout, cu, w.causal,
                       w.scale, gqa, torch.float32 if w.dtype == "f32" else torch.bfloat16)
    q, k, v, do = (to_dev_sharded(inp[n], perm) for n in ("q", "k", "v", "dout"))
    o, lse = cpa.cp_attn_fwd(prob, q, k, v)
    dq, dk, dv = cpa.cp_attn_bwd(prob, q, k, v, o, lse, do)
    torch.cuda.synchronize()
    assert cpa.cp_device_status() == 0
    ref = oracle.attn_backward(inp["q"], inp["k"], inp["v"], inp["dout"], cu, w.scale, w.causal, gqa)
    got = {n: f64(to_host_global(t, perm)) for n, t in (("dq", dq), ("dk", dk), ("dv", dv))}
    return got, ref


F32_CASES = [
    dict(total_tokens=256, hq=2, hkv=2, d_qk=64, d_v=64, cp_size=2, layout="contiguous"),
    dict(total_tokens=300, hq=4, hkv=2, d_qk=64, d_v=64, cp_size=4, layout="zigzag", seqlens=(100, 1, 199)),
    dict(total_tokens=300, hq=2, hkv=1, d_qk=64, d_v=64, cp_size=4, layout="striped", seqlens=(150, 2, 148)),
]


@pytest.mark.parametrize("kw", F32_CASES)
def test_fp32_backward(kw):
    w = workloads.Workload(name="t", dtype="f32", seed=20, **kw)
    got, ref = _run(w)
    for n in ("dq", "dk", "dv"):
        assert max_abs(got[n], ref[n]) < F32_ATOL, n


BF16_CASES = [
    dict(total_tokens=2048, hq=4, hkv=1, d_qk=128, d_v=128, cp_size=2, layout="zigzag"),
    dict(total_tokens=3000, hq=2, hkv=2, d_qk=128, d_v=128, cp_size=4, layout="zigzag"),
    dict(total_tokens=2500, hq=4, hkv=2, d_qk=128, d_v=128, cp_size=3, layout="contiguous",
         seqlens=(1200, 9, 1291)),
    dict(total_tokens=1024, hq=2, hkv=2, d_qk=192, d_v=128, cp_size=4, layout="zigzag", sigma=0.5),
    # MLA-shaped heads with GQA and a ragged varlen pack (64-row query steps)
    dict(total_tokens=2000, hq=4, hkv=2, d_qk=192, d_v=128, cp_size=4, layout="zigzag", sigma=0.5,
         seqlens=(1300, 5, 695)),
    # striped shards (shifted-diagonal blocks), varlen, both head widths
    dict(total_tokens=3000, hq=4, hkv=2, d_qk=128, d_v=128, cp_size=4, layout="striped", seqlens=(1700, 3, 1297)),
    dict(total_tokens=1500, hq=2, hkv=1, d_qk=192, d_v=128, cp_size=8, layout="striped", sigma=0.5),
]


@pytest.mark.parametrize("kw", BF16_CASES)
def test_bf16_backward(kw):
    w = workloads.Workload(name="t", dtype="bf16", seed=21, **kw)
    got, ref = _run(w)
    for n in ("dq", "dk", "dv"):
        assert rel_fro(got[n], ref[n]) < BF16_GRAD_RFRO, n


def test_bf16_backward_interleaved_gqa_noncausal():
    w = workloads.Workload(name="t", total_tokens=1500, hq=4, hkv=2, d_qk=128, d_v=128, cp_size=2,
                           layout="zigzag", dtype="bf16", seed=22, causal=False)
    got, ref = _run(w, gqa="interleaved")
    for n in ("dq", "dk", "dv"):
        assert rel_fro(got[n], ref[n]) < BF16_GRAD_RFRO, n


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_split_backward_matches_combined(dtype):
    # cp_attn_bwd_prep + cp_attn_bwd_dkdv + cp_attn_bwd_dq run the same
    # kernels as cp_attn_bwd: results are bit-identical.
    d = 128 if dtype == "bf16" else 64
    w = workloads.Workload(name="t", total_tokens=1500, hq=4, hkv=2, d_qk=d, d_v=d, cp_size=4, layout="zigzag",
                           dtype=dtype, seed=23, seqlens=(1000, 500))
    inp = workloads.make_inputs(w, device="cuda", with_dout=True)
    prob = cpa.Problem(w.total_tokens, w.hq, w.hkv, d, d, 4, "zigzag", inp["cu_seqlens"].tolist(), True, w.scale,
                       "blocked", torch.float32 if dtype == "f32" else torch.bfloat16)
    q, k, v, do = (inp[n] for n in ("q", "k", "v", "dout"))
    o, lse = cpa.cp_attn_fwd(prob, q, k, v)
    dq, dk, dv = cpa.cp_attn_bwd(prob, q, k, v, o, lse, do)
    dps = cpa.cp_attn_bwd_prep(prob, o, do)
    dk2, dv2 = cpa.cp_attn_bwd_dkdv(prob, q, k, v, lse, dps, do)
    dq2 = cpa.cp_attn_bwd_dq(prob, q, k, v, lse, dps, do)
    torch.cuda.synchronize()
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)
    # D itself: rowsum(dout * o) in float64 from the same bf16/f32 tensors
    want = (do.double() * o.double()).sum(-1).transpose(0, 1)
    assert float((dps.double() - want).abs().max()) < 1e-3
