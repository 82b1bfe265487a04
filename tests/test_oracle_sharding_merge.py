"""Pins for the oracle's shard order and LSE merge (CPU only)."""

import os

import numpy as np
import pytest

import oracle
from oracle.sharding import chunks_per_sequence
import workloads

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return np.random.RandomState(seed).standard_normal(shape)


def test_zigzag_matches_printed_table():
    rows = []
    with open(os.path.join(GOLDEN, "zigzag_c4_blocks.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    # 8 blocks of one token each: the sharded order lists, device by device,
    # the blocks the printed table assigns to it
    perm = oracle.shard_order([0, 8], 4, "zigzag")
    want = [b for _, b0, b1 in rows for b in (b0, b1)]
    assert perm.tolist() == want
    # and with larger blocks every block stays contiguous and in order
    perm = oracle.shard_order([0, 8 * 5], 4, "zigzag")
    want = [5 * b + t for _, b0, b1 in rows for b in (b0, b1) for t in range(5)]
    assert perm.tolist() == want


def test_contiguous_single_sequence_is_identity():
    perm = oracle.shard_order([0, 96], 4, "contiguous")
    assert perm.tolist() == list(range(96))
    assert oracle.rank_offsets([0, 96], 4, "contiguous").tolist() == [0, 24, 48, 72, 96]


@pytest.mark.parametrize("layout", ["contiguous", "zigzag"])
@pytest.mark.parametrize("C", [1, 2, 3, 8])
def test_varlen_permutation_is_bijective_and_chunked(layout, C):
    lengths = [1, 2, 7, 64, 65, 300, 5]
    cu = workloads.make_cu_seqlens(lengths).tolist()
    T = cu[-1]
    perm = oracle.shard_order(cu, C, layout)
    assert sorted(perm.tolist()) == list(range(T))
    x = _rand((T, 3), 1)
    assert np.array_equal(oracle.to_global(oracle.to_sharded(x, perm), perm), x)
    off = oracle.rank_offsets(cu, C, layout)
    assert off[0] == 0 and off[-1] == T
    n = chunks_per_sequence(C, layout)
    seq_of = np.searchsorted(np.asarray(cu), np.arange(T), side="right") - 1
    for r in range(C):
        part = perm[off[r]:off[r + 1]]
        # the rank holds, per sequence, exactly its chunks at floor(jL/n) cuts
        want = []
        for s in range(len(lengths)):
            b = oracle.chunk_bounds(lengths[s], n)
            for c in oracle.rank_chunks(r, C, layout):
                want.extend(range(cu[s] + b[c], cu[s] + b[c + 1]))
        assert part.tolist() == want
        # sequences appear in order inside the rank
        assert np.all(np.diff(seq_of[part]) >= 0)


def test_chunk_sizes_differ_by_at_most_one():
    for L in [1, 5, 16, 17, 1000, 4097]:
        for n in [2, 4, 16, 64]:
            b = oracle.chunk_bounds(L, n)
            sizes = np.diff(b)
            assert sizes.sum() == L and sizes.max() - sizes.min() <= 1


def _rank_visible_pairs(cu, C, layout):
    perm = oracle.shard_order(cu, C, layout)
    off = oracle.rank_offsets(cu, C, layout)
    seq_start = np.asarray(cu)[np.searchsorted(np.asarray(cu), perm, side="right") - 1]
    # causal visible keys of global row g: g - start(seq) + 1
    per_row = perm - seq_start + 1
    return [int(per_row[off[r]:off[r + 1]].sum()) for r in range(C)]


def test_zigzag_balances_causal_work_and_contiguous_does_not():
    # "LLM context parallel production guide", 因果 Attention 会制造 Rank 负载不均:
    # contiguous shards give later ranks more visible keys; zigzag pairing
    # equalises the per-rank visible-pair count when S is divisible by 2C.
    cu = [0, 64 * 16]
    z = _rank_visible_pairs(cu, 8, "zigzag")
    c = _rank_visible_pairs(cu, 8, "contiguous")
    assert len(set(z)) == 1
    assert c == sorted(c) and c[0] < c[-1]
    assert sum(z) == sum(c) == (64 * 16) * (64 * 16 + 1) // 2


def test_striped_worked_example():
    # "LLM context parallel production guide", 因果 Attention 会制造 Rank 负载不均
    # (striped token placement): token t of each sequence goes to rank t mod C.
    # Written out by hand for two packed sequences of 10 and 3 tokens, C = 4.
    cu = [0, 10, 13]
    want = [0, 4, 8, 10,  # rank 0: tokens 0, 4, 8 of seq 0; token 0 of seq 1
            1, 5, 9, 11,  # rank 1
            2, 6, 12,     # rank 2
            3, 7]         # rank 3: seq 1 has no token 3
    assert oracle.shard_order(cu, 4, "striped").tolist() == want
    assert oracle.rank_offsets(cu, 4, "striped").tolist() == [0, 4, 8, 11, 13]


@pytest.mark.parametrize("C", [1, 2, 3, 8])
def test_striped_varlen_permutation(C):
    lengths = [1, 2, 7, 64, 65, 300, 5]
    cu = workloads.make_cu_seqlens(lengths).tolist()
    T = cu[-1]
    perm = oracle.shard_order(cu, C, "striped")
    assert sorted(perm.tolist()) == list(range(T))
    off = oracle.rank_offsets(cu, C, "striped")
    seq_of = np.searchsorted(np.asarray(cu), np.arange(T), side="right") - 1
    pos = np.arange(T) - np.asarray(cu)[seq_of]
    for r in range(C):
        part = perm[off[r]:off[r + 1]]
        # exactly the tokens at positions = r (mod C), sequences in order,
        # positions increasing by C inside a sequence
        assert set(part.tolist()) == set(np.nonzero(pos % C == r)[0].tolist())
        assert np.all(np.diff(seq_of[part]) >= 0)
        for s in range(len(lengths)):
            ps = pos[part[seq_of[part] == s]]
            assert np.all(np.diff(ps) == C)


def test_rank_visible_pairs_closed_forms():
    # one sequence of L = C*m tokens: causal query t sees t + 1 keys
    C, m = 8, 16
    L = C * m
    striped = oracle.rank_visible_pairs([0, L], C, "striped")
    contig = oracle.rank_visible_pairs([0, L], C, "contiguous")
    zig = oracle.rank_visible_pairs([0, L], C, "zigzag")
    for r in range(C):
        # striped rank r holds t = r + C*k, k < m: sum (t + 1)
        assert striped[r] == m * (r + 1) + C * m * (m - 1) // 2
        # contiguous rank r holds t in [r*m, (r+1)*m)
        assert contig[r] == m * r * m + m * (m + 1) // 2
    assert len(set(zig.tolist())) == 1
    assert striped.sum() == contig.sum() == zig.sum() == L * (L + 1) // 2
    # striped is nearly balanced, contiguous is not
    assert striped.max() / striped.min() < 1 + 2.0 / m
    assert contig.max() / contig.min() > C
    # non-causal: every query sees its whole sequence
    cu = [0, 10, 13]
    nc = oracle.rank_visible_pairs(cu, 4, "striped", causal=False)
    assert nc.tolist() == [3 * 10 + 3, 3 * 10 + 3, 2 * 10 + 3, 2 * 10]


def test_rank_visible_pairs_agrees_with_direct_count():
    cu = workloads.make_cu_seqlens([33, 1, 90]).tolist()
    for layout in ("contiguous", "zigzag", "striped"):
        assert oracle.rank_visible_pairs(cu, 4, layout).tolist() == _rank_visible_pairs(cu, 4, layout)


# ---------------------------------------------------------------- merge

def test_merge_identity_and_equal_halves():
    o = _rand((5, 2, 3), 2)
    lse = _rand((2, 5), 3)
    empty_o = np.zeros_like(o)
    empty_l = np.full_like(lse, -np.inf)
    mo, ml = oracle.lse_merge(o, lse, empty_o, empty_l)
    np.testing.assert_allclose(mo, o, atol=0)
    np.testing.assert_allclose(ml, lse, atol=0)
    mo, ml = oracle.lse_merge(empty_o, empty_l, empty_o, empty_l)
    assert np.all(np.isneginf(ml)) and np.all(mo == 0)
    # two halves with equal statistics: lse + log 2 and the average output
    o2 = _rand((5, 2, 3), 4)
    mo, ml = oracle.lse_merge(o, lse, o2, lse)
    np.testing.assert_allclose(ml, lse + np.log(2.0), atol=1e-14)
    np.testing.assert_allclose(mo, 0.5 * (o + o2), atol=1e-14)


def test_merge_is_commutative_and_associative():
    os_ = [_rand((4, 3, 2), 10 + i) for i in range(3)]
    ls = [_rand((3, 4), 20 + i) * 3 for i in range(3)]
    a = oracle.lse_merge(*oracle.lse_merge(os_[0], ls[0], os_[1], ls[1]), os_[2], ls[2])
    b = oracle.lse_merge(os_[0], ls[0], *oracle.lse_merge(os_[1], ls[1], os_[2], ls[2]))
    c = oracle.lse_merge(os_[1], ls[1], os_[0], ls[0])
    d = oracle.lse_merge(os_[0], ls[0], os_[1], ls[1])
    np.testing.assert_allclose(a[0], b[0], atol=1e-13)
    np.testing.assert_allclose(a[1], b[1], atol=1e-13)
    np.testing.assert_allclose(c[0], d[0], atol=0)
    np.testing.assert_allclose(c[1], d[1], atol=0)


def test_merge_over_any_key_partition_equals_full_attention():
    # "LLM context parallel production guide", 核心原理: merging blockwise
    # results through their softmax statistics is exact, in any order.
    cu = [0, 37, 100]
    T = 100
    q, k, v = _rand((T, 4, 8), 40), _rand((T, 2, 8), 41), _rand((T, 2, 5), 42)
    o_full, l_full = oracle.attn_forward(q, k, v, cu, 0.3)
    rng = np.random.RandomState(43)
    for parts in (2, 3, 7):
        label = rng.randint(0, parts, size=T)
        order = rng.permutation(parts)
        o_acc = np.zeros_like(o_full)
        l_acc = np.full_like(l_full, -np.inf)
        for p in order:
            op, lp = oracle.attn_forward_keyset(q, k, v, cu, 0.3, label == p)
            o_acc, l_acc = oracle.lse_merge(o_acc, l_acc, op, lp)
        np.testing.assert_allclose(o_acc, o_full, atol=1e-13)
        np.testing.assert_allclose(l_acc, l_full, atol=1e-13)


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
def test_ring_of_shards_equals_full_attention(layout):
    # Each virtual rank merges its (q shard, kv shard) blocks in ring order
    # r, r-1, ... mod C; the result un-permuted is unsharded attention.
    lengths = [50, 3, 75]
    cu = workloads.make_cu_seqlens(lengths).tolist()
    T = cu[-1]
    C = 4
    q, k, v = _rand((T, 2, 8), 50), _rand((T, 1, 8), 51), _rand((T, 1, 4), 52)
    o_full, l_full = oracle.attn_forward(q, k, v, cu, 0.3)
    perm = oracle.shard_order(cu, C, layout)
    off = oracle.rank_offsets(cu, C, layout)
    rank_of_global = np.empty(T, dtype=np.int64)
    for r in range(C):
        rank_of_global[perm[off[r]:off[r + 1]]] = r
    for r in range(C):
        rows = perm[off[r]:off[r + 1]]
        o_acc = np.zeros((len(rows), 2, 4))
        l_acc = np.full((2, len(rows)), -np.inf)
        for step in range(C):
            src = (r - step) % C
            op, lp = oracle.attn_forward_keyset(q, k, v, cu, 0.3, rank_of_global == src)
            o_acc, l_acc = oracle.lse_merge(o_acc, l_acc, op[rows], lp[:, rows])
        np.testing.assert_allclose(o_acc, o_full[rows], atol=1e-13)
        np.testing.assert_allclose(l_acc, l_full[:, rows], atol=1e-13)
