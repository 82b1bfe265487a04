"""GPU parity at full size, in the launch configuration the benchmark times.

Each standard bf16 workload (S=16K GQA, S=64K GQA, the 128K-token varlen
pack, the S=256K MLA-shaped problem) runs through the C ABI exactly as the
benchmark step does: shard permutation, fused forward, D pre-pass, dK/dV and
dQ kernels, inverse permutation.  The float64 oracle then checks seeded
samples:
  * o and lse on sampled query rows for the query heads of the first and
    last GQA group (max-abs 2e-2 / 1e-3),
  * dq on the same rows (relative Frobenius 2e-2),
  * dk, dv on sampled keys near the end of their sequence, where the set of
    queries that see a key is small enough for the oracle (rel. Frobenius 2e-2),
and, over every row, the exact identities sum_j dk_j = 0 and
sum_j dv_j = sum over the group's heads of sum_i dout_i per sequence.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import BF16_GRAD_RFRO, BF16_LSE_ATOL, BF16_O_ATOL, max_abs, rel_fro

pytestmark = pytest.mark.gpu

cpa = pytest.importorskip("context_long_sequence_zigzag_gb300")


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


FULL = [
    "bf16_gqa_s16k_h32kv8_d128_c2_zigzag",
    "bf16_gqa_s64k_h32kv8_d128_c8_zigzag",
    "bf16_varlen_t128k_h16kv4_d128_c16_zigzag",
    "bf16_mla_s256k_h64_dqk192_dv128_c32_zigzag",
]


def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_parity(name):
    w = workloads.get(name)
    T = w.total_tokens
    inp = workloads.make_inputs(w, device="cuda")
    cu = inp["cu_seqlens"].tolist()
    prob = cpa.Problem(T, w.hq, w.hkv, w.d_qk, w.d_v, w.cp_size, w.layout, cu, w.causal, w.scale)
    sh = {n: cpa.cp_shard_permute(prob, inp[n]) for n in ("q", "k", "v", "dout")}
    o_s, lse_s = cpa.cp_attn_fwd(prob, sh["q"], sh["k"], sh["v"])
    dps = cpa.cp_attn_bwd_prep(prob, o_s, sh["dout"])
    dk_s, dv_s = cpa.cp_attn_bwd_dkdv(prob, sh["q"], sh["k"], sh["v"], lse_s, dps, sh["dout"])
    dq_s = cpa.cp_attn_bwd_dq(prob, sh["q"], sh["k"], sh["v"], lse_s, dps, sh["dout"])
    o, dq, dk, dv = (cpa.cp_shard_permute(prob, t, inverse=True) for t in (o_s, dq_s, dk_s, dv_s))
    perm = torch.from_numpy(oracle.shard_order(cu, w.cp_size, w.layout)).cuda()
    lse = torch.empty_like(lse_s)
    lse[:, perm] = lse_s
    torch.cuda.synchronize()
    assert cpa.cp_device_status() == 0
    del sh, o_s, dq_s, dk_s, dv_s, lse_s, dps

    # query heads of the first and last GQA group, as a sub-problem
    G = w.hq // w.hkv
    kvs = sorted({0, w.hkv - 1})
    heads = [kv * G + g for kv in kvs for g in range(G)]
    qs, dos = _f64(inp["q"][:, heads]), _f64(inp["dout"][:, heads])
    ks, vs = _f64(inp["k"][:, kvs]), _f64(inp["v"][:, kvs])
    nh = len(heads)

    # ---- forward and dq on sampled rows
    n_rows = 256 if T <= 65536 else 96
    rows = workloads.sample_rows(T, n_rows, w.seed)
    o_ref, lse_ref = oracle.attn_forward_rows(qs, ks, vs, cu, w.scale, rows, range(nh))
    rows_t = torch.from_numpy(rows).cuda()
    o_gpu = _f64(o.index_select(0, rows_t)[:, heads])
    lse_gpu = _f64(lse[heads][:, rows_t])
    assert max_abs(o_gpu, o_ref) < BF16_O_ATOL
    assert max_abs(lse_gpu, lse_ref) < BF16_LSE_ATOL
    dq_ref = oracle.attn_backward_dq_rows(qs, ks, vs, dos, cu, w.scale, rows, range(nh))
    assert rel_fro(_f64(dq.index_select(0, rows_t)[:, heads]), dq_ref) < BF16_GRAD_RFRO

    # ---- dk, dv on sampled keys near the end of sampled sequences
    rng = np.random.RandomState(w.seed + 101)
    nseq = len(cu) - 1
    seqs = sorted(rng.choice(nseq, size=min(4, nseq), replace=False).tolist())
    keys = []
    for s in seqs:
        a, b = cu[s], cu[s + 1]
        lo = max(a, b - 160)
        keys.extend(sorted(rng.choice(np.arange(lo, b), size=min(6, b - lo), replace=False).tolist()))
    keys = np.asarray(keys, dtype=np.int64)
    dk_ref, dv_ref = oracle.attn_backward_dkdv_rows(qs, ks, vs, dos, cu, w.scale, keys, range(len(kvs)))
    keys_t = torch.from_numpy(keys).cuda()
    assert rel_fro(_f64(dk.index_select(0, keys_t)[:, kvs]), dk_ref) < BF16_GRAD_RFRO
    assert rel_fro(_f64(dv.index_select(0, keys_t)[:, kvs]), dv_ref) < BF16_GRAD_RFRO

    # ---- identities over every row: sum_j dk_j = 0, sum_j dv_j = sum dout
    for s in range(nseq):
        a, b = cu[s], cu[s + 1]
        if b - a < 2:
            continue
        dks = dk[a:b].double()
        ratio = float(dks.sum(0).abs().max() / dks.abs().sum(0).max().clamp_min(1e-30))
        assert ratio < 2e-3, (s, ratio)
        want = inp["dout"][a:b].double().sum(0).view(w.hkv, G, w.d_v).sum(1)
        got = dv[a:b].double().sum(0)
        assert float((got - want).norm() / want.norm().clamp_min(1e-30)) < 1e-2, s
