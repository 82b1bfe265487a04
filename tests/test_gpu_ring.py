"""GPU: ring attention with explicit KV transport (cp_ring_attn_fwd).

Every virtual rank computes its block against the KV shard it holds while
the shards move one rank on through device-to-device copies on a second
stream ("Ulysses Context Parallelism 的工程取舍全记录" §2 and "LLM context
parallel production guide", Ring Attention: the KV transfer overlaps the
block computation; "Ulysses与Ring-Attention详解" §4.1-§4.2: each step's
(out, lse) is merged into the running result).  Checked against:
  * the float64 oracle in global order (fp32 max-abs 1e-5; bf16 max-abs 2e-2
    on o, 1e-3 on lse), over layouts, GQA, varlen packs, non-causal, the
    192-wide MLA heads and the CUDA-core fp32 path;
  * the same call with the copies serialised on the compute stream: the
    kernels and their order are the same, so the results are bit-identical;
  * the fused forward cp_attn_fwd at the S=64K, C=8 zigzag bench size (every
    row) and the oracle on sampled rows there.
"""

import pytest
import torch

import oracle
import workloads
from gpu_util import (BF16_GRAD_RFRO, BF16_LSE_ATOL, BF16_O_ATOL, F32_ATOL, f64, lse_to_global, max_abs, perm_of,
                      rel_fro, to_dev_sharded, to_host_global)

pytestmark = pytest.mark.gpu

cpa = pytest.importorskip("context_long_sequence_zigzag_gb300")


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


CASES = [
    dict(total_tokens=3000, hq=4, hkv=2, d_qk=128, d_v=128, cp_size=4, layout="zigzag", seqlens=(1700, 13, 1287)),
    dict(total_tokens=4096, hq=2, hkv=2, d_qk=128, d_v=128, cp_size=2, layout="contiguous"),
    dict(total_tokens=4096, hq=4, hkv=1, d_qk=128, d_v=128, cp_size=8, layout="zigzag"),
    dict(total_tokens=2500, hq=4, hkv=2, d_qk=128, d_v=128, cp_size=3, layout="striped", seqlens=(1200, 1300)),
    dict(total_tokens=1500, hq=2, hkv=1, d_qk=128, d_v=128, cp_size=4, layout="zigzag", causal=False),
    dict(total_tokens=2048, hq=2, hkv=2, d_qk=192, d_v=128, cp_size=4, layout="zigzag", sigma=0.5),
    dict(total_tokens=1000, hq=2, hkv=1, d_qk=128, d_v=128, cp_size=1, layout="contiguous"),
]


def _run(w, overlap=True, gqa="blocked"):
    inp = workloads.make_inputs(w, with_dout=False)
    cu = inp["cu_seqlens"].tolist()
    perm = perm_of(cu, w.cp_size, w.layout)
    prob = cpa.Problem(w.total_tokens, w.hq, w.hkv, w.d_qk, w.d_v, w.cp_size, w.layout, cu, w.causal, w.scale, gqa,
                       torch.float32 if w.dtype == "f32" else torch.bfloat16)
    q, k, v = (to_dev_sharded(inp[n], perm) for n in ("q", "k", "v"))
    o, lse = cpa.cp_ring_attn_fwd(prob, q, k, v, overlap=overlap)
    torch.cuda.synchronize()
    assert cpa.cp_device_status() == 0
    return inp, cu, perm, prob, (q, k, v), o, lse


@pytest.mark.parametrize("kw", CASES)
def test_ring_matches_oracle(kw):
    w = workloads.Workload(name="t", dtype="bf16", seed=41, backward=False, **kw)
    inp, cu, perm, prob, qkv, o, lse = _run(w)
    o_ref, lse_ref = oracle.attn_forward(inp["q"], inp["k"], inp["v"], cu, w.scale, w.causal)
    assert max_abs(f64(to_host_global(o, perm)), o_ref) < BF16_O_ATOL
    assert max_abs(f64(lse_to_global(lse, perm)), lse_ref) < BF16_LSE_ATOL
    # the copies serialised on the compute stream: same kernels, same order
    o2, lse2 = cpa.cp_ring_attn_fwd(prob, *qkv, overlap=False)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_ring_interleaved_gqa():
    w = workloads.Workload(name="t", total_tokens=2048, hq=4, hkv=2, d_qk=128, d_v=128, cp_size=4,
                           layout="zigzag", dtype="bf16", seed=42, backward=False)
    inp, cu, perm, _, _, o, lse = _run(w, gqa="interleaved")
    o_ref, lse_ref = oracle.attn_forward(inp["q"], inp["k"], inp["v"], cu, w.scale, True, "interleaved")
    assert max_abs(f64(to_host_global(o, perm)), o_ref) < BF16_O_ATOL
    assert max_abs(f64(lse_to_global(lse, perm)), lse_ref) < BF16_LSE_ATOL


@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
def test_ring_fp32_cuda_core_path(layout):
    w = workloads.Workload(name="t", total_tokens=600, hq=2, hkv=2, d_qk=64, d_v=64, cp_size=3, layout=layout,
                           dtype="f32", seed=43, backward=False, seqlens=(301, 299))
    inp, cu, perm, _, _, o, lse = _run(w)
    o_ref, lse_ref = oracle.attn_forward(inp["q"], inp["k"], inp["v"], cu, w.scale, True)
    assert max_abs(f64(to_host_global(o, perm)), o_ref) < F32_ATOL
    assert max_abs(f64(lse_to_global(lse, perm)), lse_ref) < F32_ATOL


def test_ring_full_size_bench_configuration():
    w = workloads.get("bf16_gqa_s64k_h32kv8_d128_c8_zigzag")
    inp = workloads.make_inputs(w, device="cuda", with_dout=False)
    cu = inp["cu_seqlens"].tolist()
    prob = cpa.Problem(w.total_tokens, w.hq, w.hkv, w.d_qk, w.d_v, w.cp_size, w.layout, cu)
    sh = {n: cpa.cp_shard_permute(prob, inp[n]) for n in ("q", "k", "v")}
    o_r, lse_r = cpa.cp_ring_attn_fwd(prob, sh["q"], sh["k"], sh["v"])
    o_f, lse_f = cpa.cp_attn_fwd(prob, sh["q"], sh["k"], sh["v"])
    torch.cuda.synchronize()
    assert cpa.cp_device_status() == 0
    # every row against the fused forward (both bf16 results of the same math)
    assert float((o_r.float() - o_f.float()).abs().max()) < BF16_O_ATOL
    assert float((lse_r - lse_f).abs().max()) < BF16_LSE_ATOL
    # sampled rows of the first and last head group against the oracle
    o = cpa.cp_shard_permute(prob, o_r, inverse=True)
    perm = torch.from_numpy(oracle.shard_order(cu, w.cp_size, w.layout)).cuda()
    lse = torch.empty_like(lse_r)
    lse[:, perm] = lse_r
    G = w.hq // w.hkv
    for kv in (0, w.hkv - 1):
        heads = [kv * G + g for g in range(G)]
        rows = workloads.sample_rows(w.total_tokens, 256, w.seed + 77 + kv)
        o_ref, lse_ref = oracle.attn_forward_rows(inp["q"], inp["k"], inp["v"], cu, w.scale, rows, heads)
        rows_t = torch.from_numpy(rows).cuda()
        o_gpu = f64(o.index_select(0, rows_t)[:, heads])
        assert max_abs(o_gpu, o_ref) < BF16_O_ATOL
        assert rel_fro(o_gpu, o_ref) < BF16_GRAD_RFRO
        assert max_abs(f64(lse[heads][:, rows_t]), lse_ref) < BF16_LSE_ATOL
