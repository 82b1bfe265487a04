"""GPU: the library's plan checks (cp_set_debug_checks) on small problems.

With checks on, every CTA of the attention kernels first checks its own
plan entry (tile index, heads, tile and output rows, run list, run rows,
step count) against the rows of the tensors it will touch, and the host
checks every plan before uploading it.  A failed check records 0x200 | check
in the device error word and the CTA returns without touching memory;
nothing traps.  These runs must pass every check (device status 0) and still
match the float64 oracle, over the forward, the backward, one ring step
(cp_attn_block_fwd), the ring with transport and the Ulysses path, on the
tensor-core and CUDA-core kernels.
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
def _checks_on():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    prev = cpa.cp_set_debug_checks(True)
    yield
    cpa.cp_set_debug_checks(prev)


CASES = [
    dict(total_tokens=3000, hq=4, hkv=2, d_qk=128, d_v=128, cp_size=4, layout="zigzag", seqlens=(1700, 13, 1287)),
    dict(total_tokens=2048, hq=2, hkv=2, d_qk=192, d_v=128, cp_size=4, layout="zigzag", sigma=0.5),
    dict(total_tokens=2500, hq=4, hkv=1, d_qk=128, d_v=128, cp_size=3, layout="striped", seqlens=(1200, 1300)),
    dict(total_tokens=700, hq=4, hkv=2, d_qk=64, d_v=64, cp_size=4, layout="zigzag", dtype="f32",
         seqlens=(300, 3, 397)),
]


@pytest.mark.parametrize("kw", CASES, ids=lambda c: f"{c['layout']}{c['total_tokens']}_d{c['d_qk']}")
def test_all_paths_pass_their_plan_checks(kw):
    kw = dict(kw)
    dtype = kw.pop("dtype", "bf16")
    w = workloads.Workload(name="dbg", dtype=dtype, seed=71, **kw)
    f32 = dtype == "f32"
    inp = workloads.make_inputs(w)
    cu = inp["cu_seqlens"].tolist()
    perm = perm_of(cu, w.cp_size, w.layout)
    prob = cpa.Problem(w.total_tokens, w.hq, w.hkv, w.d_qk, w.d_v, w.cp_size, w.layout, cu, True, w.scale,
                       "blocked", torch.float32 if f32 else torch.bfloat16)
    q, k, v, do = (to_dev_sharded(inp[n], perm) for n in ("q", "k", "v", "dout"))
    o, lse = cpa.cp_attn_fwd(prob, q, k, v)
    dq, dk, dv = cpa.cp_attn_bwd(prob, q, k, v, o, lse, do)
    o_r, lse_r = cpa.cp_ring_attn_fwd(prob, q, k, v)
    blocks = [cpa.cp_attn_block_fwd(prob, r, (r + 1) % w.cp_size, q, k, v) for r in range(w.cp_size)]
    torch.cuda.synchronize()
    assert cpa.cp_device_status() == 0
    ref = oracle.attn_backward(inp["q"], inp["k"], inp["v"], inp["dout"], cu, w.scale)
    o_tol, l_tol = (F32_ATOL, F32_ATOL) if f32 else (BF16_O_ATOL, BF16_LSE_ATOL)
    for oo, ll in ((o, lse), (o_r, lse_r)):
        assert max_abs(f64(to_host_global(oo, perm)), ref["o"]) < o_tol
        assert max_abs(f64(lse_to_global(ll, perm)), ref["lse"]) < l_tol
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        got = f64(to_host_global(t, perm))
        if f32:
            assert max_abs(got, ref[name]) < F32_ATOL, name
        else:
            assert rel_fro(got, ref[name]) < BF16_GRAD_RFRO, name
    # one ring step per rank: the rows of rank r against the keys of rank r+1
    off = cpa.cp_shard_offsets(prob)
    for r, (op, lp) in enumerate(blocks):
        keyset = torch.zeros(w.total_tokens, dtype=torch.bool)
        keyset[perm[off[(r + 1) % w.cp_size]:off[(r + 1) % w.cp_size + 1]]] = True
        ob, lb = oracle.attn_forward_keyset(inp["q"], inp["k"], inp["v"], cu, w.scale, keyset.numpy())
        rows = perm[off[r]:off[r + 1]]
        lref = lb[:, rows.numpy()]
        lgpu = f64(lp)
        seen = lref > -1e30
        assert ((lgpu > -1e30) == seen).all()
        assert max_abs(lgpu[seen], lref[seen]) < l_tol
        assert max_abs(f64(op), ob[rows.numpy()]) < (F32_ATOL if f32 else BF16_O_ATOL)


def test_ulysses_passes_its_plan_checks():
    w = workloads.Workload(name="dbg", total_tokens=2048, hq=8, hkv=4, d_qk=128, d_v=128, cp_size=4,
                           layout="zigzag", dtype="bf16", seed=72)
    inp = workloads.make_inputs(w)
    cu = inp["cu_seqlens"].tolist()
    perm = perm_of(cu, w.cp_size, w.layout)
    prob = cpa.Problem(w.total_tokens, w.hq, w.hkv, w.d_qk, w.d_v, w.cp_size, w.layout, cu)
    q, k, v = (to_dev_sharded(inp[n], perm) for n in ("q", "k", "v"))
    o, lse = cpa.cp_ulysses_attn_fwd(prob, q, k, v)
    torch.cuda.synchronize()
    assert cpa.cp_device_status() == 0
    o_ref, lse_ref = oracle.attn_forward(inp["q"], inp["k"], inp["v"], cu, w.scale)
    assert max_abs(f64(to_host_global(o, perm)), o_ref) < BF16_O_ATOL
    assert max_abs(f64(lse_to_global(lse, perm)), lse_ref) < BF16_LSE_ATOL
