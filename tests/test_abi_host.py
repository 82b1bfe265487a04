"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/cp_attn.h declares, validates descriptors, and its
shard map and per-rank block counts agree with the oracle's shard order."""

import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

cpa = pytest.importorskip("context_long_sequence_zigzag_gb300")


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "cp_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(cp_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_function():
    names = _declared_functions()
    assert len(names) >= 12
    lib = ctypes.CDLL(cpa.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(cpa.EXPORTED) == names


def test_status_strings():
    for s in range(6):
        assert cpa.cp_status_string(s).startswith("CP_")
    assert "unknown" in cpa.cp_status_string(99)


def _prob(**kw):
    base = dict(total_tokens=1024, hq=8, hkv=2, d_qk=128, d_v=128, cp_size=4, layout="zigzag")
    base.update(kw)
    return cpa.Problem(**base)


def test_validation():
    assert cpa.cp_validate(_prob()) == cpa.CP_OK
    assert cpa.cp_validate(_prob(hq=6, hkv=4)) == cpa.CP_ERR_INVALID_ARG
    assert cpa.cp_validate(_prob(cp_size=0)) == cpa.CP_ERR_INVALID_ARG
    assert cpa.cp_validate(_prob(d_qk=264, d_v=128)) == cpa.CP_ERR_UNSUPPORTED
    p = _prob(total_tokens=10, cu_seqlens=[0, 6, 4, 10])  # non-monotone
    assert cpa.cp_validate(p) == cpa.CP_ERR_INVALID_ARG
    p = _prob(total_tokens=11, cu_seqlens=[0, 6, 10])  # does not end at T
    assert cpa.cp_validate(p) == cpa.CP_ERR_INVALID_ARG
    p = _prob(d_qk=4, d_v=4)  # 8-byte rows violate the 16-byte rule
    assert cpa.cp_validate(p) == cpa.CP_ERR_INVALID_ARG
    p = _prob()
    p.desc.scale = float("nan")
    assert cpa.cp_validate(p) == cpa.CP_ERR_INVALID_ARG
    p = _prob()
    p.desc.layout = 7
    assert cpa.cp_validate(p) == cpa.CP_ERR_INVALID_ARG


def test_null_descriptor_and_workspace_errors():
    lib = ctypes.CDLL(cpa.LIB_PATH)
    lib.cp_validate.argtypes = [ctypes.c_void_p]
    assert lib.cp_validate(None) == cpa.CP_ERR_INVALID_ARG
    with pytest.raises(cpa.CpError):
        cpa.cp_workspace_size(_prob(hq=3, hkv=2), cpa.CP_OP_FWD)


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
@pytest.mark.parametrize("lengths", [[1000], [1, 2, 7, 64, 65, 300, 5], [4096, 31, 4097]])
@pytest.mark.parametrize("C", [1, 2, 3, 8])
def test_shard_offsets_match_oracle(layout, lengths, C):
    cu = workloads.make_cu_seqlens(lengths).tolist()
    p = _prob(total_tokens=cu[-1], cu_seqlens=cu, cp_size=C, layout=layout)
    assert cpa.cp_shard_offsets(p) == oracle.rank_offsets(cu, C, layout).tolist()


def _tile_pairs_oracle(cu, C, layout):
    """Visible 128x128 (query tile, key tile) pairs per rank, counted from the
    oracle's chunk bounds: key tiles are cut per chunk from its first row,
    except that a rank's two zigzag chunks of a sequence, adjacent in its
    shard, are cut as one run when the query tile sees both of them whole
    (every key before the tile's first query)."""
    n = C if layout == "contiguous" else 2 * C
    counts = []
    for r in range(C):
        tot = 0
        for s in range(len(cu) - 1):
            L = cu[s + 1] - cu[s]
            b = oracle.chunk_bounds(L, n)
            for ca in oracle.rank_chunks(r, C, layout):
                for t0 in range(b[ca], b[ca + 1], 128):
                    qmax = min(t0 + 128, b[ca + 1]) - 1
                    for rho in range(C):
                        runs = []  # (visible rows, whole and unmasked)
                        for cb in oracle.rank_chunks(rho, C, layout):
                            lo, hi = b[cb], b[cb + 1]
                            if hi <= lo or lo > qmax:
                                continue
                            runs.append((min(hi - lo, qmax - lo + 1), hi - 1 <= t0))
                        if layout == "zigzag" and len(runs) == 2 and runs[0][1] and runs[1][1]:
                            runs = [(runs[0][0] + runs[1][0], True)]
                        tot += sum(-(-v // 128) for v, _ in runs)
        counts.append(tot)
    return counts


@pytest.mark.parametrize("layout", ["contiguous", "zigzag"])
def test_rank_block_counts(layout):
    cu = [0, 8192]
    p = _prob(total_tokens=8192, cu_seqlens=cu, cp_size=4, layout=layout)
    got = cpa.cp_rank_block_counts(p)
    assert got == _tile_pairs_oracle(cu, 4, layout)
    if layout == "zigzag":
        assert len(set(got)) == 1  # zigzag balances the causal work
    else:
        assert got == sorted(got) and got[0] < got[-1]
    lengths = workloads.varlen_lengths(20000, 64, 4000, 3)
    cu = workloads.make_cu_seqlens(lengths).tolist()
    p = _prob(total_tokens=cu[-1], cu_seqlens=cu, cp_size=4, layout=layout)
    assert cpa.cp_rank_block_counts(p) == _tile_pairs_oracle(cu, 4, layout)


def _fwd_key_tiles_model(cu, C, layout):
    """Key tiles of the tensor-core forward per rank: as _tile_pairs_oracle,
    except that the tails (rows past the last whole 128-row step) of the
    runs a query tile sees whole and unmasked are laid back to back from
    8-row boundaries into shared key tiles, which are used where they are
    fewer than the tails."""
    n = C if layout == "contiguous" else 2 * C
    counts = []
    for r in range(C):
        tot = 0
        for s in range(len(cu) - 1):
            L = cu[s + 1] - cu[s]
            b = oracle.chunk_bounds(L, n)
            for ca in oracle.rank_chunks(r, C, layout):
                for t0 in range(b[ca], b[ca + 1], 128):
                    qmax = min(t0 + 128, b[ca + 1]) - 1
                    tails = []
                    for rho in range(C):
                        runs = []
                        for cb in oracle.rank_chunks(rho, C, layout):
                            lo, hi = b[cb], b[cb + 1]
                            if hi <= lo or lo > qmax:
                                continue
                            runs.append((min(hi - lo, qmax - lo + 1), hi - 1 <= t0))
                        if layout == "zigzag" and len(runs) == 2 and runs[0][1] and runs[1][1]:
                            runs = [(runs[0][0] + runs[1][0], True)]
                        for v, visible in runs:
                            if visible and v % 128:
                                tot += v // 128
                                tails.append(v % 128)
                            else:
                                tot += -(-v // 128)
                    gathered = -(-sum(-(-t // 8) * 8 for t in tails) // 128)
                    tot += min(gathered, len(tails))
        counts.append(tot)
    return counts


@pytest.mark.parametrize("layout", ["contiguous", "zigzag"])
def test_forward_gathers_run_tails(layout):
    lengths = workloads.varlen_lengths(20000, 64, 4000, 3)
    cu = workloads.make_cu_seqlens(lengths).tolist()
    p = _prob(total_tokens=cu[-1], cu_seqlens=cu, cp_size=4, layout=layout)
    got = cpa.cp_rank_fwd_key_tiles(p)
    assert got == _fwd_key_tiles_model(cu, 4, layout)
    assert sum(got) < sum(cpa.cp_rank_block_counts(p))
    # the CUDA-core forward (fp32) and dense shards whose runs are whole
    # 128-row steps keep one key tile per step
    f32 = _prob(total_tokens=cu[-1], cu_seqlens=cu, cp_size=4, layout=layout, dtype=torch.float32)
    assert cpa.cp_rank_fwd_key_tiles(f32) == cpa.cp_rank_block_counts(f32)
    dense = _prob(total_tokens=8192, cu_seqlens=[0, 8192], cp_size=4, layout=layout)
    assert cpa.cp_rank_fwd_key_tiles(dense) == cpa.cp_rank_block_counts(dense)


def _striped_tile_pairs(cu, C):
    """Visible (query tile, key tile) pairs per rank for striped shards, from
    global positions: rank r holds positions r, r + C, ...; a query tile of
    shard rows [t0, t1) ends at position r + C*(t1 - 1), and rank rho
    contributes its tokens at positions <= that, cut into 128-row tiles."""
    counts = []
    for r in range(C):
        tot = 0
        for s in range(len(cu) - 1):
            L = cu[s + 1] - cu[s]
            n_r = len(oracle.striped_rows(L, C, r))
            for t0 in range(0, n_r, 128):
                last = r + C * (min(t0 + 128, n_r) - 1)
                for rho in range(C):
                    n_rho = len(oracle.striped_rows(L, C, rho))
                    if last < rho or n_rho == 0:
                        continue
                    vis = min(n_rho, (last - rho) // C + 1)
                    tot += -(-vis // 128)
        counts.append(tot)
    return counts


def test_rank_block_counts_striped():
    cu = [0, 8192]
    p = _prob(total_tokens=8192, cu_seqlens=cu, cp_size=4, layout="striped")
    got = cpa.cp_rank_block_counts(p)
    assert got == _striped_tile_pairs(cu, 4)
    assert max(got) - min(got) <= 3  # striped balances the causal work
    lengths = workloads.varlen_lengths(20000, 64, 4000, 3)
    cu = workloads.make_cu_seqlens(lengths).tolist()
    p = _prob(total_tokens=cu[-1], cu_seqlens=cu, cp_size=4, layout="striped")
    assert cpa.cp_rank_block_counts(p) == _striped_tile_pairs(cu, 4)


def test_striped_permute_workspace_is_one_segment_per_token():
    cu = [0, 100, 103]
    p = _prob(total_tokens=103, cu_seqlens=cu, cp_size=4, layout="striped")
    assert cpa.cp_workspace_size(p, cpa.CP_OP_PERMUTE) >= 103 * 32


def test_workspace_sizes_positive_and_ordered():
    p = _prob()
    f = cpa.cp_workspace_size(p, cpa.CP_OP_FWD)
    b = cpa.cp_workspace_size(p, cpa.CP_OP_BWD)
    assert f > 0 and b > f
    assert cpa.cp_workspace_size(p, cpa.CP_OP_PERMUTE) >= 32
    with pytest.raises(cpa.CpError):
        cpa.cp_workspace_size(p, 99)  # no such operation


def test_linear_attention_rejected_configurations():
    # AllGather CP of the pages: contiguous pieces, one query head per KV head
    with pytest.raises(cpa.CpError) as e:
        cpa.cp_workspace_size(cpa.Problem(256, 2, 2, 64, 64, 2, "zigzag"), cpa.CP_OP_LIN_FWD)
    assert e.value.status == cpa.CP_ERR_UNSUPPORTED
    with pytest.raises(cpa.CpError) as e:
        cpa.cp_workspace_size(cpa.Problem(256, 4, 2, 64, 64, 2, "contiguous"), cpa.CP_OP_LIN_FWD)
    assert e.value.status == cpa.CP_ERR_INVALID_ARG


def test_ring_workspace_and_argument_errors():
    # two ring buffers of K and V with a slot of the longest shard per rank,
    # plus the fp32 output accumulator of a bf16 problem
    T, hq, hkv, d, C = 1000, 4, 2, 128, 4
    p = cpa.Problem(T, hq, hkv, d, d, C, "zigzag", [0, 1000])
    n = cpa.cp_workspace_size(p, cpa.CP_OP_RING_FWD)
    slot_rows = max(np.diff(cpa.cp_shard_offsets(p)))
    assert n >= 2 * C * slot_rows * hkv * 2 * d * 2 + T * hq * d * 4
    f = cpa.cp_workspace_size(cpa.Problem(T, hq, hkv, d, d, C, "zigzag", [0, 1000], dtype=__import__("torch").float32),
                              cpa.CP_OP_RING_FWD)
    assert f < n + 2 * C * slot_rows * hkv * 2 * d * 2  # fp32 accumulates in o: no extra accumulator
    lib = ctypes.CDLL(cpa.LIB_PATH)
    fn = lib.cp_ring_attn_fwd
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(cpa.cp_desc_t)] + [ctypes.c_void_p] * 6 + [ctypes.c_size_t] + [ctypes.c_void_p] * 2
    fake = 1 << 20  # aligned, never dereferenced: both errors are found before any GPU work
    assert fn(ctypes.byref(p.desc), fake, fake, None, fake, fake, fake, n, None, None) == cpa.CP_ERR_INVALID_ARG
    assert fn(ctypes.byref(p.desc), fake, fake, fake, fake, fake, fake, n - 1, None, None) == cpa.CP_ERR_WORKSPACE
    assert fn(ctypes.byref(p.desc), fake, fake, fake, fake, fake, fake + 16, n, None, None) == cpa.CP_ERR_WORKSPACE


def test_debug_checks_switch():
    prev = cpa.cp_set_debug_checks(True)
    try:
        assert cpa.cp_set_debug_checks(True) is True
        assert cpa.cp_set_debug_checks(False) is True
        assert cpa.cp_set_debug_checks(False) is False
        lib = ctypes.CDLL(cpa.LIB_PATH)
        lib.cp_set_debug_checks.argtypes = [ctypes.c_int32, ctypes.c_void_p]
        assert lib.cp_set_debug_checks(2, None) == cpa.CP_ERR_INVALID_ARG
    finally:
        cpa.cp_set_debug_checks(prev)
