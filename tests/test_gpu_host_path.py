"""GPU: the host side of an ABI call.

Tile plans and index tables reach the device through the library's pinned
staging ring, so a call only enqueues its work: it must not wait for earlier
work on its stream (from pageable memory the runtime held a 128K-token varlen
forward's caller until the stream drained).  The ring is reused round-robin,
each region after the event behind its last copy; many calls whose plans
together exceed the ring must keep giving the same bits.
"""

import time

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

cpa = pytest.importorskip("context_long_sequence_zigzag_gb300")


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _varlen_problem():
    w = workloads.get("bf16_varlen_t128k_h16kv4_d128_c16_zigzag")
    inp = workloads.make_inputs(w, device="cuda", with_dout=False)
    cu = inp["cu_seqlens"].tolist()
    prob = cpa.Problem(w.total_tokens, w.hq, w.hkv, w.d_qk, w.d_v, w.cp_size, w.layout, cu)
    sh = {n: cpa.cp_shard_permute(prob, inp[n]) for n in ("q", "k", "v")}
    return prob, sh


def test_call_does_not_wait_for_the_stream():
    prob, sh = _varlen_problem()
    ws = cpa.workspace(prob, cpa.CP_OP_FWD)
    o, lse = cpa.cp_attn_fwd(prob, sh["q"], sh["k"], sh["v"], ws=ws)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    cpa.cp_attn_fwd(prob, sh["q"], sh["k"], sh["v"], o, lse, ws)
    torch.cuda.synchronize()
    one = time.perf_counter() - t0
    for _ in range(4):  # several forwards queued ahead of the timed call
        cpa.cp_attn_fwd(prob, sh["q"], sh["k"], sh["v"], o, lse, ws)
    t0 = time.perf_counter()
    cpa.cp_attn_fwd(prob, sh["q"], sh["k"], sh["v"], o, lse, ws)
    call = time.perf_counter() - t0
    torch.cuda.synchronize()
    assert cpa.cp_device_status() == 0
    # the call returns long before the work queued ahead of it could finish
    assert call < 0.5 * one, (call, one)


def test_staging_ring_wraps_without_changing_results():
    prob, sh = _varlen_problem()
    ws = cpa.workspace(prob, cpa.CP_OP_FWD)
    o0, lse0 = cpa.cp_attn_fwd(prob, sh["q"], sh["k"], sh["v"], ws=ws)
    torch.cuda.synchronize()
    o, lse = torch.empty_like(o0), torch.empty_like(lse0)
    # ~0.7 MB of plan per call: 80 calls pass the 32 MiB ring about twice
    for _ in range(80):
        cpa.cp_attn_fwd(prob, sh["q"], sh["k"], sh["v"], o, lse, ws)
    torch.cuda.synchronize()
    assert cpa.cp_device_status() == 0
    assert torch.equal(o, o0) and torch.equal(lse, lse0)
