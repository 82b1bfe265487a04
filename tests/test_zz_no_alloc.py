"""GPU: the workspace-free forward, cp_attn_fwd_noalloc, called through the C ABI.

Some callers cannot allocate device memory (a plugin whose host framework
owns every allocation and hands it only its tensors, or code on a path where
allocating is not allowed).  cp_attn_fwd_noalloc serves them: it keeps its
tile plan in a fixed 4 MiB array inside the library's device image instead
of a caller workspace.  These tests check that two calls in a row (different
problems, so the second overwrites the first one's plan) give exactly what
the workspace entry point cp_attn_fwd gives: both run the same kernel on the
same plan, so o and lse must be bit-identical.  The second plan is the
smaller one, so a stale tail of the first plan left in the array would show.
A problem whose plan does not fit is refused before any GPU work.
This file is collected last on purpose.
"""

import ctypes

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

cpa = pytest.importorskip("context_long_sequence_zigzag_gb300")


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _abi():
    lib = ctypes.CDLL(cpa.LIB_PATH)
    f = lib.cp_attn_fwd_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(cpa.cp_desc_t)] + [ctypes.c_void_p] * 6
    return f


def _problem(name, T, hq, hkv, C, layout, seqlens, seed):
    w = workloads.Workload(name=name, total_tokens=T, hq=hq, hkv=hkv, d_qk=128, d_v=128, cp_size=C,
                           layout=layout, dtype="bf16", seed=seed, backward=False, seqlens=seqlens)
    inp = workloads.make_inputs(w, device="cuda", with_dout=False)
    prob = cpa.Problem(T, hq, hkv, 128, 128, C, layout, inp["cu_seqlens"].tolist())
    return prob, inp


def test_noalloc_forward_matches_workspace_forward_twice():
    f = _abi()
    stream = torch.cuda.current_stream().cuda_stream
    cases = [
        _problem("a", 3000, 4, 2, 4, "zigzag", (1700, 13, 1287), 31),
        _problem("b", 4096, 2, 1, 2, "contiguous", None, 32),
    ]
    sizes = [cpa.cp_workspace_size(prob, cpa.CP_OP_FWD) for prob, _ in cases]
    assert sizes[1] < sizes[0], sizes
    for call, (prob, inp) in enumerate(cases):
        q, k, v = inp["q"], inp["k"], inp["v"]
        o_ref, lse_ref = cpa.cp_attn_fwd(prob, q, k, v)
        o = torch.empty_like(o_ref)
        lse = torch.empty_like(lse_ref)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        st = f(ctypes.byref(prob.desc), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
               stream)
        torch.cuda.synchronize()
        assert st == cpa.CP_OK, cpa.cp_status_string(st)
        if call > 0:  # the first call may load the module; later ones allocate nothing
            assert torch.cuda.mem_get_info()[0] == free_before
        assert cpa.cp_device_status() == 0
        assert torch.equal(o, o_ref)
        assert torch.equal(lse, lse_ref)


def test_noalloc_refuses_a_plan_beyond_its_scratch():
    f = _abi()
    # 1M tokens over 64 zigzag ranks: the plan needs far more than 4 MiB.
    T = 1 << 20
    prob = cpa.Problem(T, 1, 1, 128, 128, 64, "zigzag", [0, T])
    st = f(ctypes.byref(prob.desc), None, None, None, None, None, None)
    assert st == cpa.CP_ERR_WORKSPACE
