"""GPU parity at full size, in the launch configuration the benchmark times.

Each standard bf16 workload (S=16K GQA, S=64K GQA, the 128K-token varlen
pack, the S=256K MLA-shaped problem) runs through the C ABI exactly as the
benchmark step does: shard permutation, fused forward, D pre-pass, dK/dV and
dQ kernels, inverse permutation.  The float64 oracle then checks seeded
samples:
  * every head group (the query heads that share one key/value head) gets
    its own 256 seeded query rows; on them o (max-abs 2e-2 and relative
    Frobenius 2e-2), lse (max-abs 1e-3) and dq (relative Frobenius 2e-2);
  * dk, dv (relative Frobenius 2e-2) on 256 seeded keys spread over the whole
    token stream, for the first and the last key/value head.  Such keys are
    seen by the queries of every later chunk of their sequence, on every
    virtual rank, so these sums run over long unmasked runs of many query
    tiles.  The oracle computes lse and D for every query row that sees them
    (row blocks, full softmax rows);
  * on the varlen pack, additionally every key of the shortest sequence;
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

ROWS_PER_GROUP = 256
KEYS = 256


def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _check_keys(name, inp, cu, w, keys, kvs, dk, dv):
    keys = np.asarray(keys, dtype=np.int64)
    dk_ref, dv_ref = oracle.attn_backward_dkdv_rows(inp["q"], inp["k"], inp["v"], inp["dout"], cu, w.scale, keys,
                                                    kvs)
    keys_t = torch.from_numpy(keys).cuda()
    for i, kv in enumerate(kvs):
        e_dk = rel_fro(_f64(dk.index_select(0, keys_t)[:, kv]), dk_ref[:, i])
        e_dv = rel_fro(_f64(dv.index_select(0, keys_t)[:, kv]), dv_ref[:, i])
        assert e_dk < BF16_GRAD_RFRO, (name, kv, e_dk)
        assert e_dv < BF16_GRAD_RFRO, (name, kv, e_dv)


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

    G = w.hq // w.hkv
    # ---- o, lse, dq: every head group, its own seeded rows
    for kv in range(w.hkv):
        heads = [kv * G + g for g in range(G)]
        rows = workloads.sample_rows(T, ROWS_PER_GROUP, w.seed + 1000 + kv)
        rows_t = torch.from_numpy(rows).cuda()
        o_ref, lse_ref = oracle.attn_forward_rows(inp["q"], inp["k"], inp["v"], cu, w.scale, rows, heads)
        o_gpu = _f64(o.index_select(0, rows_t)[:, heads])
        lse_gpu = _f64(lse[heads][:, rows_t])
        assert max_abs(o_gpu, o_ref) < BF16_O_ATOL, (kv, max_abs(o_gpu, o_ref))
        assert rel_fro(o_gpu, o_ref) < BF16_GRAD_RFRO, (kv, rel_fro(o_gpu, o_ref))
        assert max_abs(lse_gpu, lse_ref) < BF16_LSE_ATOL, (kv, max_abs(lse_gpu, lse_ref))
        dq_ref = oracle.attn_backward_dq_rows(inp["q"], inp["k"], inp["v"], inp["dout"], cu, w.scale, rows, heads)
        e_dq = rel_fro(_f64(dq.index_select(0, rows_t)[:, heads]), dq_ref)
        assert e_dq < BF16_GRAD_RFRO, (kv, e_dq)

    # ---- dk, dv: keys spread over the whole stream, first and last kv head
    kvs = sorted({0, w.hkv - 1})
    _check_keys(name, inp, cu, w, workloads.sample_rows(T, KEYS, w.seed + 101), kvs, dk, dv)
    lengths = np.diff(cu)
    if len(lengths) > 1:
        # every key of the shortest sequence: each of its 2C zigzag chunks,
        # on every virtual rank, against every query that sees it
        s = int(np.argmin(np.where(lengths >= 2 * w.cp_size, lengths, np.iinfo(np.int64).max)))
        _check_keys(name, inp, cu, w, np.arange(cu[s], cu[s + 1]), kvs, dk, dv)

    # ---- identities over every row: sum_j dk_j = 0, sum_j dv_j = sum dout
    nseq = len(cu) - 1
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
