"""GPU: run-to-run determinism.

No kernel of the forward, the backward or the ring accumulates through
atomics: every output element is written by one thread after a fixed
sequence of tensor-core and FP32 operations, and every CTA's work list comes
from the same host plan.  Two runs on the same inputs must therefore give
bit-identical o, lse, dq, dk and dv, whatever order the CTAs ran in.  A race
between a block write and a later read ("超长上下文训练速度翻倍秘籍" §2 warns of
one that unit tests missed) would typically show up here as run-to-run
differences before it shows up as a tolerance failure.
"""

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

cpa = pytest.importorskip("context_long_sequence_zigzag_gb300")


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


CASES = [
    "bf16_gqa_s16k_h32kv8_d128_c2_zigzag",
    dict(total_tokens=6000, hq=4, hkv=1, d_qk=128, d_v=128, cp_size=4, layout="zigzag",
         seqlens=(1500, 7, 129, 4364)),
    dict(total_tokens=4096, hq=2, hkv=2, d_qk=192, d_v=128, cp_size=4, layout="zigzag", sigma=0.5),
    dict(total_tokens=700, hq=4, hkv=2, d_qk=64, d_v=64, cp_size=4, layout="striped", dtype="f32",
         seqlens=(300, 3, 397)),
]


def _workload(c):
    if isinstance(c, str):
        return workloads.get(c)
    c = dict(c)
    dtype = c.pop("dtype", "bf16")
    return workloads.Workload(name="det", dtype=dtype, seed=61, **c)


@pytest.mark.parametrize("case", CASES, ids=lambda c: c if isinstance(c, str) else f"{c['layout']}{c['total_tokens']}")
def test_forward_backward_bit_identical_across_runs(case):
    w = _workload(case)
    inp = workloads.make_inputs(w, device="cuda", with_dout=True)
    cu = inp["cu_seqlens"].tolist()
    prob = cpa.Problem(w.total_tokens, w.hq, w.hkv, w.d_qk, w.d_v, w.cp_size, w.layout, cu, w.causal, w.scale,
                       "blocked", torch.float32 if w.dtype == "f32" else torch.bfloat16)
    sh = {n: cpa.cp_shard_permute(prob, inp[n]) for n in ("q", "k", "v", "dout")}
    runs = []
    for _ in range(2):
        o, lse = cpa.cp_attn_fwd(prob, sh["q"], sh["k"], sh["v"])
        dq, dk, dv = cpa.cp_attn_bwd(prob, sh["q"], sh["k"], sh["v"], o, lse, sh["dout"])
        o_r, lse_r = cpa.cp_ring_attn_fwd(prob, sh["q"], sh["k"], sh["v"])
        runs.append((o, lse, dq, dk, dv, o_r, lse_r))
    torch.cuda.synchronize()
    assert cpa.cp_device_status() == 0
    names = ("o", "lse", "dq", "dk", "dv", "ring o", "ring lse")
    for name, a, b in zip(names, runs[0], runs[1]):
        assert torch.equal(a, b), name


def test_ulysses_and_linear_attention_bit_identical_across_runs():
    """The all-to-all path (re-layout kernels around the same attention
    kernels) and the decayed linear attention (chunk states, a fixed-order
    prefix over chunks, then the chunk outputs) are deterministic as well."""
    w = workloads.Workload(name="det", dtype="bf16", seed=67, total_tokens=5000, hq=8, hkv=4, d_qk=128, d_v=128,
                           cp_size=4, layout="zigzag", seqlens=(2100, 9, 2891))
    inp = workloads.make_inputs(w, device="cuda", with_dout=True)
    cu = inp["cu_seqlens"].tolist()
    prob = cpa.Problem(w.total_tokens, w.hq, w.hkv, w.d_qk, w.d_v, w.cp_size, w.layout, cu)
    sh = {n: cpa.cp_shard_permute(prob, inp[n]) for n in ("q", "k", "v", "dout")}
    lin = cpa.Problem(w.total_tokens, w.hq, w.hq, 128, 128, w.cp_size, "contiguous", cu, True, 128 ** -0.5,
                      "blocked", torch.bfloat16)
    gen = torch.Generator().manual_seed(67)
    kl = (torch.randn(w.total_tokens, w.hq, 128, generator=gen) * 0.5).to(torch.bfloat16).cuda()
    g = (-torch.rand(w.hq, generator=gen) * 0.9 - 0.05).cuda()
    ql = inp["q"]
    runs = []
    for _ in range(2):
        o, lse = cpa.cp_ulysses_attn_fwd(prob, sh["q"], sh["k"], sh["v"])
        dq, dk, dv = cpa.cp_ulysses_attn_bwd(prob, sh["q"], sh["k"], sh["v"], o, lse, sh["dout"])
        o_lin = cpa.cp_lin_attn_fwd(lin, ql, kl, ql, g)
        runs.append((o, lse, dq, dk, dv, o_lin))
    torch.cuda.synchronize()
    assert cpa.cp_device_status() == 0
    for name, a, b in zip(("o", "lse", "dq", "dk", "dv", "linear o"), runs[0], runs[1]):
        assert torch.equal(a, b), name
