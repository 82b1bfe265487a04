"""GPU forward parity against the float64 oracle.

The CUDA path runs in sharded order; results are brought back to global
order with the oracle's shard map and compared element by element.
Tolerances: fp32 max-abs 1e-5; bf16 max-abs 2e-2 on o and 1e-3 on lse.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import (BF16_LSE_ATOL, BF16_O_ATOL, F32_ATOL, f64, lse_to_global, max_abs, perm_of,
                      to_dev_sharded, to_host_global)

pytestmark = pytest.mark.gpu

cpa = pytest.importorskip("context_long_sequence_zigzag_gb300")


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _run_fwd(w: workloads.Workload, gqa="blocked"):
    inp = workloads.make_inputs(w, with_dout=False)
    cu = inp["cu_seqlens"].tolist()
    perm = perm_of(cu, w.cp_size, w.layout)
    prob = cpa.Problem(w.total_tokens, w.hq, w.hkv, w.d_qk, w.d_v, w.cp_size, w.layout, cu, w.causal,
                       w.scale, gqa, torch.float32 if w.dtype == "f32" else torch.bfloat16)
    q, k, v = (to_dev_sharded(inp[n], perm) for n in ("q", "k", "v"))
    o, lse = cpa.cp_attn_fwd(prob, q, k, v)
    torch.cuda.synchronize()
    assert cpa.cp_device_status() == 0
    o_ref, lse_ref = oracle.attn_forward(inp["q"], inp["k"], inp["v"], cu, w.scale, w.causal, gqa)
    return f64(to_host_global(o, perm)), f64(lse_to_global(lse, perm)), o_ref, lse_ref


def test_fp32_reference_workload():
    # fp32, B=1, 2 heads (MHA), S=256, d=64, 2 contiguous shards, forward only
    w = workloads.get("f32_mha_s256_d64_c2_contiguous")
    o, lse, o_ref, lse_ref = _run_fwd(w)
    assert max_abs(o, o_ref) < F32_ATOL
    assert max_abs(lse, lse_ref) < F32_ATOL


F32_CASES = [
    dict(total_tokens=300, hq=4, hkv=2, d_qk=64, d_v=64, cp_size=4, layout="zigzag"),
    dict(total_tokens=500, hq=3, hkv=1, d_qk=32, d_v=64, cp_size=2, layout="contiguous", seqlens=(120, 1, 379)),
    dict(total_tokens=257, hq=2, hkv=2, d_qk=128, d_v=128, cp_size=8, layout="zigzag", causal=False),
    dict(total_tokens=700, hq=4, hkv=2, d_qk=64, d_v=64, cp_size=4, layout="striped", seqlens=(300, 3, 397)),
]


@pytest.mark.parametrize("kw", F32_CASES)
def test_fp32_variants(kw):
    w = workloads.Workload(name="t", dtype="f32", seed=5, backward=False, **kw)
    o, lse, o_ref, lse_ref = _run_fwd(w)
    assert max_abs(o, o_ref) < F32_ATOL
    assert max_abs(lse, lse_ref) < F32_ATOL


BF16_CASES = [
    # several tiles per chunk, GQA 4:1, both layouts
    dict(total_tokens=4096, hq=4, hkv=1, d_qk=128, d_v=128, cp_size=2, layout="zigzag"),
    dict(total_tokens=4096, hq=4, hkv=2, d_qk=128, d_v=128, cp_size=4, layout="contiguous"),
    # chunk sizes not multiples of 128 (ragged tails) and a short sequence
    dict(total_tokens=3000, hq=2, hkv=2, d_qk=128, d_v=128, cp_size=4, layout="zigzag"),
    dict(total_tokens=5000, hq=4, hkv=2, d_qk=128, d_v=128, cp_size=3, layout="zigzag",
         seqlens=(1500, 7, 129, 3364)),
    # non-causal, one shard
    dict(total_tokens=1000, hq=2, hkv=1, d_qk=128, d_v=128, cp_size=1, layout="contiguous", causal=False),
    # MLA-shaped heads: 192-wide q/k, 128-wide v
    dict(total_tokens=2048, hq=2, hkv=2, d_qk=192, d_v=128, cp_size=4, layout="zigzag", sigma=0.5),
    # striped shards: every (q rank, kv rank) block is a shifted causal diagonal
    dict(total_tokens=4096, hq=4, hkv=1, d_qk=128, d_v=128, cp_size=4, layout="striped"),
    dict(total_tokens=5000, hq=4, hkv=2, d_qk=128, d_v=128, cp_size=8, layout="striped",
         seqlens=(2500, 7, 1200, 1293)),
]


@pytest.mark.parametrize("kw", BF16_CASES)
def test_bf16_tensor_core_forward(kw):
    w = workloads.Workload(name="t", dtype="bf16", seed=7, backward=False, **kw)
    o, lse, o_ref, lse_ref = _run_fwd(w)
    assert max_abs(o, o_ref) < BF16_O_ATOL
    assert max_abs(lse, lse_ref) < BF16_LSE_ATOL


def test_bf16_interleaved_gqa():
    w = workloads.Workload(name="t", total_tokens=2048, hq=4, hkv=2, d_qk=128, d_v=128, cp_size=2,
                           layout="zigzag", dtype="bf16", seed=8, backward=False)
    o, lse, o_ref, lse_ref = _run_fwd(w, gqa="interleaved")
    assert max_abs(o, o_ref) < BF16_O_ATOL
    assert max_abs(lse, lse_ref) < BF16_LSE_ATOL


def test_bf16_varlen_pack():
    lengths = workloads.varlen_lengths(6000, 64, 2000, 3)
    w = workloads.Workload(name="t", total_tokens=6000, hq=4, hkv=1, d_qk=128, d_v=128, cp_size=4,
                           layout="zigzag", dtype="bf16", seed=9, backward=False, seqlens=tuple(lengths))
    o, lse, o_ref, lse_ref = _run_fwd(w)
    assert max_abs(o, o_ref) < BF16_O_ATOL
    assert max_abs(lse, lse_ref) < BF16_LSE_ATOL


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", ["zigzag", "contiguous", "striped"])
def test_stepwise_ring_equals_oracle(dtype, layout):
    # Each virtual rank: block (r, r), then (r, r-1), ... merged in ring
    # order with cp_lse_merge ("Ulysses与Ring-Attention详解" §4.1-§4.2).
    lengths = (700, 1, 300) if dtype == "f32" else (1100, 33, 900)
    T = sum(lengths)
    C = 4
    d = 64 if dtype == "f32" else 128
    w = workloads.Workload(name="t", total_tokens=T, hq=2, hkv=1, d_qk=d, d_v=d, cp_size=C, layout=layout,
                           dtype=dtype, seed=10, backward=False, seqlens=lengths)
    inp = workloads.make_inputs(w, with_dout=False)
    cu = inp["cu_seqlens"].tolist()
    perm = perm_of(cu, C, layout)
    prob = cpa.Problem(T, 2, 1, d, d, C, layout, cu, True, w.scale, "blocked",
                       torch.float32 if dtype == "f32" else torch.bfloat16)
    q, k, v = (to_dev_sharded(inp[n], perm) for n in ("q", "k", "v"))
    off = cpa.cp_shard_offsets(prob)
    o_ref, lse_ref = oracle.attn_forward(inp["q"], inp["k"], inp["v"], cu, w.scale)
    perm_np = perm.numpy()
    tol_o = F32_ATOL if dtype == "f32" else BF16_O_ATOL
    tol_l = F32_ATOL if dtype == "f32" else BF16_LSE_ATOL
    for r in range(C):
        o_acc, lse_acc = cpa.cp_attn_block_fwd(prob, r, r, q, k, v)
        for step in range(1, C):
            o_p, l_p = cpa.cp_attn_block_fwd(prob, r, (r - step) % C, q, k, v)
            cpa.cp_lse_merge(prob, o_acc, lse_acc, o_p, l_p)
        torch.cuda.synchronize()
        rows = perm_np[off[r]:off[r + 1]]
        assert max_abs(f64(o_acc), o_ref[rows]) < tol_o
        assert max_abs(f64(lse_acc), lse_ref[:, rows]) < tol_l


def test_block_classes():
    # future blocks are empty (lse = -inf, o = 0); the diagonal block of a
    # one-token-per-row problem reduces to the row's own value.
    T, C = 1024, 4
    w = workloads.Workload(name="t", total_tokens=T, hq=2, hkv=2, d_qk=128, d_v=128, cp_size=C,
                           layout="contiguous", dtype="bf16", seed=12, backward=False)
    inp = workloads.make_inputs(w, with_dout=False)
    prob = cpa.Problem(T, 2, 2, 128, 128, C, "contiguous", [0, T])
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = cpa.cp_attn_block_fwd(prob, 0, 3, q, k, v)  # rank 3 holds the future
    torch.cuda.synchronize()
    assert torch.isneginf(lse).all() and (o == 0).all()
    o, lse = cpa.cp_attn_block_fwd(prob, 3, 0, q, k, v)  # fully visible history
    ref_o, ref_l = oracle.attn_forward_keyset(inp["q"], inp["k"], inp["v"], [0, T], w.scale,
                                              np.arange(T) < T // 4)
    assert max_abs(f64(o), ref_o[3 * T // 4:]) < BF16_O_ATOL
    assert max_abs(f64(lse), ref_l[:, 3 * T // 4:]) < BF16_LSE_ATOL


def test_layouts_agree_after_unpermute():
    # "Ulysses与Ring-Attention详解" §4.2: zigzag only moves tokens between ranks;
    # the un-permuted result equals the contiguous run's.
    base = dict(total_tokens=4096, hq=2, hkv=1, d_qk=128, d_v=128, dtype="bf16", seed=13, backward=False)
    oz, lz, _, _ = _run_fwd(workloads.Workload(name="z", cp_size=4, layout="zigzag", **base))
    oc, lc, _, _ = _run_fwd(workloads.Workload(name="c", cp_size=4, layout="contiguous", **base))
    o1, l1, _, _ = _run_fwd(workloads.Workload(name="one", cp_size=1, layout="contiguous", **base))
    os_, ls, _, _ = _run_fwd(workloads.Workload(name="s", cp_size=4, layout="striped", **base))
    assert max_abs(oz, oc) < 2 * BF16_O_ATOL and max_abs(oz, o1) < 2 * BF16_O_ATOL
    assert max_abs(lz, lc) < 2 * BF16_LSE_ATOL and max_abs(lz, l1) < 2 * BF16_LSE_ATOL
    assert max_abs(os_, o1) < 2 * BF16_O_ATOL and max_abs(ls, l1) < 2 * BF16_LSE_ATOL
