"""GPU edge cases of the forward, backward and transported ring against the
float64 oracle (whole tensors, global order).

The cases are the degenerate corners of the shard map and of the kernels'
tiling: empty sequences in cu_seqlens, sequences shorter than 2C (empty
zigzag chunks on some virtual ranks), one token, 64 virtual ranks with
chunks far below a 128-row tile, GQA ratios 3:1 and 8:1, sequence isolation
without the causal mask, bf16 heads the tensor-core kernels do not take (the
CUDA-core path), a softmax scale other than 1/sqrt(d), and plans whose key
and query tiles are gathered from many run tails.  Tolerances as
everywhere: bf16 o max-abs 2e-2, lse 1e-3, gradients relative Frobenius
2e-2; fp32 max-abs 1e-5.
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


CASES = {
    "empty_sequences": dict(total_tokens=1300, hq=4, hkv=2, d_qk=128, d_v=128, cp_size=4, layout="zigzag",
                            seqlens=(0, 700, 0, 0, 600, 0)),
    "shorter_than_2C": dict(total_tokens=2010, hq=2, hkv=1, d_qk=128, d_v=128, cp_size=8, layout="zigzag",
                            seqlens=(5, 3, 1, 2001)),
    "one_token": dict(total_tokens=1, hq=2, hkv=1, d_qk=128, d_v=128, cp_size=2, layout="zigzag"),
    "c64_tiny_chunks": dict(total_tokens=4096, hq=2, hkv=1, d_qk=128, d_v=128, cp_size=64, layout="zigzag"),
    "gqa_3_to_1": dict(total_tokens=1500, hq=6, hkv=2, d_qk=128, d_v=128, cp_size=3, layout="zigzag",
                       seqlens=(900, 600)),
    "gqa_8_to_1": dict(total_tokens=1024, hq=8, hkv=1, d_qk=128, d_v=128, cp_size=2, layout="contiguous"),
    "noncausal_varlen": dict(total_tokens=1600, hq=2, hkv=2, d_qk=128, d_v=128, cp_size=4, layout="zigzag",
                             seqlens=(1000, 17, 583), causal=False),
    "bf16_cuda_core_d64": dict(total_tokens=700, hq=4, hkv=2, d_qk=64, d_v=64, cp_size=4, layout="zigzag",
                               seqlens=(400, 300)),
    "mla_heads_gqa": dict(total_tokens=1300, hq=4, hkv=2, d_qk=192, d_v=128, cp_size=4, layout="zigzag",
                          seqlens=(1000, 300), sigma=0.5),
    "f32_c16": dict(total_tokens=333, hq=2, hkv=1, d_qk=64, d_v=64, cp_size=16, layout="zigzag", dtype="f32",
                    seqlens=(200, 0, 133)),
    # gathered tiles: many run tails per tile (pieces from 1 to 127 rows, some
    # split across two tiles, some filled from rows past the tensor's end)
    "gathered_short_seqs": dict(total_tokens=4183, hq=4, hkv=2, d_qk=128, d_v=128, cp_size=4, layout="zigzag",
                                seqlens=(9, 17, 33, 65, 130, 260, 520, 1040, 2109)),
    "gathered_contiguous": dict(total_tokens=2501, hq=2, hkv=1, d_qk=128, d_v=128, cp_size=8, layout="contiguous",
                                seqlens=(1500, 700, 301)),
}

GATHERED = ("gathered_short_seqs", "gathered_contiguous", "noncausal_varlen")


def _setup(kw, scale=None):
    kw = dict(kw)
    dtype = kw.pop("dtype", "bf16")
    w = workloads.Workload(name="edge", dtype=dtype, seed=91, **kw)
    inp = workloads.make_inputs(w, with_dout=True)
    cu = inp["cu_seqlens"].tolist()
    perm = perm_of(cu, w.cp_size, w.layout)
    sc = w.scale if scale is None else scale
    prob = cpa.Problem(w.total_tokens, w.hq, w.hkv, w.d_qk, w.d_v, w.cp_size, w.layout, cu, w.causal, sc, "blocked",
                       torch.float32 if dtype == "f32" else torch.bfloat16)
    sh = {n: to_dev_sharded(inp[n], perm) for n in ("q", "k", "v", "dout")}
    return w, inp, cu, perm, prob, sh, sc, dtype == "f32"


def _check(w, inp, cu, perm, sc, f32, o, lse, grads=None):
    ref = oracle.attn_backward(inp["q"], inp["k"], inp["v"], inp["dout"], cu, sc, w.causal)
    o_tol, l_tol = (F32_ATOL, F32_ATOL) if f32 else (BF16_O_ATOL, BF16_LSE_ATOL)
    assert max_abs(f64(to_host_global(o, perm)), ref["o"]) < o_tol
    assert max_abs(f64(lse_to_global(lse, perm)), ref["lse"]) < l_tol
    if grads is not None:
        for name, t in zip(("dq", "dk", "dv"), grads):
            got = f64(to_host_global(t, perm))
            if f32:
                assert max_abs(got, ref[name]) < F32_ATOL, name
            elif float(abs(ref[name]).max()) < 1e-6:
                # a gradient that is exactly zero (one token: dS = P (dP - D) = 0)
                # leaves only rounding: compare absolutely
                assert max_abs(got, ref[name]) < 1e-3, name
            else:
                assert rel_fro(got, ref[name]) < BF16_GRAD_RFRO, name


@pytest.mark.parametrize("name", list(CASES))
def test_forward_backward_edge(name):
    w, inp, cu, perm, prob, sh, sc, f32 = _setup(CASES[name])
    if name in GATHERED:  # the tensor-core kernels run gathered tiles here
        assert sum(cpa.cp_rank_fwd_key_tiles(prob)) < sum(cpa.cp_rank_block_counts(prob))
    o, lse = cpa.cp_attn_fwd(prob, sh["q"], sh["k"], sh["v"])
    grads = cpa.cp_attn_bwd(prob, sh["q"], sh["k"], sh["v"], o, lse, sh["dout"])
    torch.cuda.synchronize()
    assert cpa.cp_device_status() == 0
    _check(w, inp, cu, perm, sc, f32, o, lse, grads)


@pytest.mark.parametrize("name", ["empty_sequences", "shorter_than_2C", "c64_tiny_chunks", "gqa_3_to_1",
                                  "noncausal_varlen", "f32_c16"])
def test_ring_with_transport_edge(name):
    w, inp, cu, perm, prob, sh, sc, f32 = _setup(CASES[name])
    o, lse = cpa.cp_ring_attn_fwd(prob, sh["q"], sh["k"], sh["v"])
    torch.cuda.synchronize()
    assert cpa.cp_device_status() == 0
    _check(w, inp, cu, perm, sc, f32, o, lse)


def test_scale_other_than_inverse_sqrt_d():
    w, inp, cu, perm, prob, sh, sc, f32 = _setup(CASES["gqa_3_to_1"], scale=0.31)
    o, lse = cpa.cp_attn_fwd(prob, sh["q"], sh["k"], sh["v"])
    grads = cpa.cp_attn_bwd(prob, sh["q"], sh["k"], sh["v"], o, lse, sh["dout"])
    torch.cuda.synchronize()
    _check(w, inp, cu, perm, sc, f32, o, lse, grads)


def test_zero_tokens_is_a_no_op():
    prob = cpa.Problem(0, 2, 1, 128, 128, 4, "zigzag", [0, 0])
    e = torch.empty(0, 2, 128, dtype=torch.bfloat16, device="cuda")
    ek = torch.empty(0, 1, 128, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    lse = torch.empty(2, 0, dtype=torch.float32, device="cuda")
    for call in (lambda: cpa.cp_attn_fwd(prob, e, ek, ek, e, lse, ws),
                 lambda: cpa.cp_attn_bwd(prob, e, ek, ek, e, lse, e, e, ek, ek, ws),
                 lambda: cpa.cp_ring_attn_fwd(prob, e, ek, ek, e, lse, ws)):
        call()
    torch.cuda.synchronize()
    assert cpa.cp_device_status() == 0
