"""GPU: shard permutation (bit-exact), LSE merge, bounded-wait self-check."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import f64, max_abs

pytestmark = pytest.mark.gpu

cpa = pytest.importorskip("context_long_sequence_zigzag_gb300")


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _prob(T, cu, C, layout, hq=4, hkv=2, d=128, dtype=torch.bfloat16):
    return cpa.Problem(T, hq, hkv, d, d, C, layout, cu, dtype=dtype)


CASES = [
    ([4096], 4, "zigzag"),
    ([4096], 4, "contiguous"),
    ([1, 2, 7, 64, 65, 300, 5], 3, "zigzag"),
    ([1, 2, 7, 64, 65, 300, 5], 8, "contiguous"),
    (workloads.varlen_lengths(30000, 64, 9000, 11), 16, "zigzag"),
    ([5], 8, "zigzag"),  # sequence shorter than 2C: empty chunks
    ([1000], 4, "striped"),
    ([1, 2, 7, 64, 65, 300, 5], 8, "striped"),  # sequences shorter than C: ranks without tokens
]


@pytest.mark.parametrize("lengths,C,layout", CASES)
@pytest.mark.parametrize("row_elems,dtype", [(4 * 128, torch.bfloat16), (8, torch.bfloat16), (4, torch.float32),
                                             (2 * 192, torch.bfloat16)])
def test_permute_bit_exact(lengths, C, layout, row_elems, dtype):
    cu = workloads.make_cu_seqlens(lengths).tolist()
    T = cu[-1]
    p = _prob(T, cu, C, layout)
    g = torch.Generator().manual_seed(T + C)
    x = torch.randn(T, row_elems, generator=g).to(dtype)
    perm = torch.from_numpy(oracle.shard_order(cu, C, layout))
    want = x[perm]
    xd = x.cuda()
    got = cpa.cp_shard_permute(p, xd)
    torch.cuda.synchronize()
    assert torch.equal(got.cpu().view(torch.int16 if dtype == torch.bfloat16 else torch.int32),
                       want.view(torch.int16 if dtype == torch.bfloat16 else torch.int32))
    back = cpa.cp_shard_permute(p, got, inverse=True)
    assert torch.equal(back.cpu(), x)


def test_permute_large_rows_round_trip():
    # 3-D token-major tensor (q-like) over several 32 KiB pieces per chunk
    T, C = 8192, 8
    p = _prob(T, [0, T], C, "zigzag", hq=8)
    x = torch.randn(T, 8, 128, device="cuda").to(torch.bfloat16)
    s = cpa.cp_shard_permute(p, x)
    perm = torch.from_numpy(oracle.shard_order([0, T], C, "zigzag")).cuda()
    assert torch.equal(s, x.index_select(0, perm))
    assert torch.equal(cpa.cp_shard_permute(p, s, inverse=True), x)


def test_permute_rejects_bad_arguments():
    T = 256
    p = _prob(T, [0, T], 2, "zigzag")
    x = torch.zeros(T, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cpa.CpError):
        cpa.cp_shard_permute(p, x, out=x)  # in place (overlap)
    with pytest.raises(cpa.CpError):
        cpa.cp_shard_permute(p, torch.zeros(T, 3, dtype=torch.bfloat16, device="cuda"))  # 6-byte rows


@pytest.mark.parametrize("rows,hq,dv", [(1, 1, 4), (777, 3, 128), (4096, 8, 128), (100, 2, 192)])
def test_lse_merge_matches_oracle(rows, hq, dv):
    g = torch.Generator().manual_seed(rows)
    oa = torch.randn(rows, hq, dv, generator=g)
    ob = torch.randn(rows, hq, dv, generator=g)
    la = torch.randn(hq, rows, generator=g) * 4
    lb = torch.randn(hq, rows, generator=g) * 4
    # empty partials: -inf with zero output
    la[:, ::7] = -float("inf")
    oa[::7] = 0
    lb[:, ::5] = -float("inf")
    ob[::5] = 0
    wo, wl = oracle.lse_merge(f64(oa), f64(la), f64(ob), f64(lb))
    p = cpa.Problem(rows, hq, hq, 64, dv, 1, "contiguous")
    oad, lad = oa.cuda(), la.cuda()
    cpa.cp_lse_merge(p, oad, lad, ob.cuda(), lb.cuda())
    torch.cuda.synchronize()
    go, gl = f64(oad), f64(lad)
    both = np.isneginf(wl)
    assert np.array_equal(np.isneginf(gl), both)
    assert max_abs(gl[~both], wl[~both]) < 1e-5
    assert max_abs(go, wo) < 1e-5


def test_bounded_wait_returns_instead_of_hanging():
    code = cpa.cp_check_bounded_wait(20_000_000)  # 20 ms limit
    assert code == 0x100 | 0x7F
    assert cpa.cp_device_status() == 0  # the self-check leaves the word cleared
