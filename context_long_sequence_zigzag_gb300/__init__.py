"""context_long_sequence_zigzag_gb300 — Python binding of libcpattn.

Context-parallel exact causal attention on one GB300: a (packed) sequence is
cut into C context-parallel shards (contiguous, zigzag or striped); the C virtual ranks
share one GPU and the KV ring is the order in which the kernels visit the
HBM-resident KV shards.  The C ABI (``include/cp_attn.h``) is the product;
this module only marshals torch tensors into its pointers and sizes.  Every
step runs in the library's CUDA kernels; there is no fallback: importing this
module fails if ``libcpattn.so`` has not been built, and every call raises on
a non-OK status.

Functions carry the C names: ``cp_shard_permute``, ``cp_attn_block_fwd``,
``cp_lse_merge``, ``cp_attn_fwd``, ``cp_attn_bwd``, ``cp_workspace_size``,
``cp_shard_offsets``, ``cp_rank_block_counts``, ``cp_rank_fwd_key_tiles``, ``cp_device_status``,
``cp_check_bounded_wait``, ``cp_status_string``, ``cp_validate``, ``cp_ulysses_a2a``,
``cp_ulysses_attn_fwd``, ``cp_ulysses_attn_bwd``, ``cp_ring_attn_fwd``, ``cp_lin_attn_fwd``.
"""

from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcpattn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with "
        "`python context_long_sequence_zigzag_gb300/build.py` (no CPU fallback exists)")

_lib = ctypes.CDLL(LIB_PATH)

CP_OK, CP_ERR_INVALID_ARG, CP_ERR_UNSUPPORTED, CP_ERR_CUDA, CP_ERR_DEVICE_TIMEOUT, CP_ERR_WORKSPACE = range(6)
CP_LAYOUT_CONTIGUOUS, CP_LAYOUT_ZIGZAG, CP_LAYOUT_STRIPED = 0, 1, 2
CP_DT_F32, CP_DT_BF16 = 0, 1
CP_GQA_BLOCKED, CP_GQA_INTERLEAVED = 0, 1
CP_OP_FWD, CP_OP_BWD, CP_OP_BLOCK_FWD, CP_OP_PERMUTE, CP_OP_BWD_DKDV, CP_OP_BWD_DQ = 0, 1, 2, 3, 4, 5
CP_OP_ULYSSES_A2A, CP_OP_ULYSSES_FWD, CP_OP_ULYSSES_BWD, CP_OP_LIN_FWD, CP_OP_RING_FWD = 6, 7, 8, 9, 10

EXPORTED = [
    "cp_status_string", "cp_validate", "cp_workspace_size", "cp_shard_offsets",
    "cp_rank_block_counts", "cp_rank_fwd_key_tiles", "cp_shard_permute", "cp_attn_block_fwd", "cp_lse_merge",
    "cp_attn_fwd", "cp_attn_bwd", "cp_device_status", "cp_check_bounded_wait",
    "cp_attn_fwd_noalloc", "cp_attn_bwd_prep", "cp_attn_bwd_dkdv", "cp_attn_bwd_dq",
    "cp_ulysses_a2a", "cp_ulysses_attn_fwd", "cp_ulysses_attn_bwd", "cp_lin_attn_fwd", "cp_ring_attn_fwd",
    "cp_set_debug_checks",
]


class cp_desc_t(ctypes.Structure):
    _fields_ = [
        ("total_tokens", ctypes.c_int64),
        ("num_seqs", ctypes.c_int32),
        ("hq", ctypes.c_int32),
        ("hkv", ctypes.c_int32),
        ("cu_seqlens", ctypes.POINTER(ctypes.c_int32)),
        ("d_qk", ctypes.c_int32),
        ("d_v", ctypes.c_int32),
        ("cp_size", ctypes.c_int32),
        ("layout", ctypes.c_int32),
        ("causal", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("gqa", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
    ]


_P = ctypes.c_void_p
_DP = ctypes.POINTER(cp_desc_t)
_sigs = {
    "cp_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "cp_validate": (ctypes.c_int, [_DP]),
    "cp_workspace_size": (ctypes.c_int, [_DP, ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)]),
    "cp_shard_offsets": (ctypes.c_int, [_DP, ctypes.POINTER(ctypes.c_int64)]),
    "cp_rank_block_counts": (ctypes.c_int, [_DP, ctypes.POINTER(ctypes.c_int64)]),
    "cp_rank_fwd_key_tiles": (ctypes.c_int, [_DP, ctypes.POINTER(ctypes.c_int64)]),
    "cp_shard_permute": (ctypes.c_int, [_DP, _P, _P, ctypes.c_int64, ctypes.c_int32, _P, ctypes.c_size_t, _P]),
    "cp_attn_block_fwd": (ctypes.c_int, [_DP, ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P, _P, _P,
                                         ctypes.c_size_t, _P]),
    "cp_lse_merge": (ctypes.c_int, [_DP, ctypes.c_int64, _P, _P, _P, _P, _P]),
    "cp_attn_fwd": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "cp_attn_bwd": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "cp_device_status": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int32)]),
    "cp_check_bounded_wait": (ctypes.c_int, [ctypes.c_int64, ctypes.POINTER(ctypes.c_int32), _P]),
    "cp_attn_fwd_noalloc": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P]),
    "cp_attn_bwd_prep": (ctypes.c_int, [_DP, _P, _P, _P, _P]),
    "cp_attn_bwd_dkdv": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "cp_attn_bwd_dq": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "cp_ulysses_a2a": (ctypes.c_int, [_DP, _P, _P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, _P,
                                      ctypes.c_size_t, _P]),
    "cp_ulysses_attn_fwd": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "cp_lin_attn_fwd": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "cp_ulysses_attn_bwd": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "cp_ring_attn_fwd": (ctypes.c_int, [_DP, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P, _P]),
    "cp_set_debug_checks": (ctypes.c_int, [ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]),
}
for _name, (_res, _args) in _sigs.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


class CpError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {cp_status_string(status)}")


def cp_status_string(status: int) -> str:
    return _lib.cp_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != CP_OK:
        raise CpError(status, where)


class Problem:
    """Holds a cp_desc_t and the host cu_seqlens it points at.

    cu_seqlens : global-order int32 prefix sums (list / tensor), or None for
                 one sequence of ``total_tokens``.
    """

    def __init__(self, total_tokens: int, hq: int, hkv: int, d_qk: int, d_v: int, cp_size: int,
                 layout: str = "zigzag", cu_seqlens=None, causal: bool = True,
                 scale: Optional[float] = None, gqa: str = "blocked", dtype=torch.bfloat16):
        if cu_seqlens is None:
            cu = [0, int(total_tokens)]
        else:
            cu = [int(x) for x in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
        self.cu = cu
        self._cu_arr = (ctypes.c_int32 * len(cu))(*cu)
        self.torch_dtype = dtype
        self.desc = cp_desc_t(
            total_tokens=int(total_tokens), num_seqs=len(cu) - 1, hq=hq, hkv=hkv,
            cu_seqlens=ctypes.cast(self._cu_arr, ctypes.POINTER(ctypes.c_int32)),
            d_qk=d_qk, d_v=d_v, cp_size=cp_size,
            layout={"contiguous": CP_LAYOUT_CONTIGUOUS, "zigzag": CP_LAYOUT_ZIGZAG,
                    "striped": CP_LAYOUT_STRIPED}[layout],
            causal=int(bool(causal)),
            scale=float(scale if scale is not None else 1.0 / math.sqrt(d_qk)),
            gqa={"blocked": CP_GQA_BLOCKED, "interleaved": CP_GQA_INTERLEAVED}[gqa],
            dtype={torch.float32: CP_DT_F32, torch.bfloat16: CP_DT_BF16}[dtype])

    @classmethod
    def from_workload(cls, w, cu_seqlens=None) -> "Problem":
        from_cu = cu_seqlens if cu_seqlens is not None else _cu_of(w.lengths())
        return cls(w.total_tokens, w.hq, w.hkv, w.d_qk, w.d_v, w.cp_size, w.layout, from_cu,
                   w.causal, w.scale, "blocked",
                   torch.float32 if w.dtype == "f32" else torch.bfloat16)

    @property
    def ptr(self):
        return ctypes.byref(self.desc)

    @property
    def T(self) -> int:
        return int(self.desc.total_tokens)


def _cu_of(lengths):
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return cu


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if t.is_cuda and not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def cp_validate(prob: Problem) -> int:
    return _lib.cp_validate(prob.ptr)


def cp_workspace_size(prob: Problem, op: int) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.cp_workspace_size(prob.ptr, int(op), ctypes.byref(n)), "cp_workspace_size")
    return int(n.value)


def cp_shard_offsets(prob: Problem) -> list:
    arr = (ctypes.c_int64 * (prob.desc.cp_size + 1))()
    _check(_lib.cp_shard_offsets(prob.ptr, arr), "cp_shard_offsets")
    return list(arr)


def cp_rank_block_counts(prob: Problem) -> list:
    arr = (ctypes.c_int64 * prob.desc.cp_size)()
    _check(_lib.cp_rank_block_counts(prob.ptr, arr), "cp_rank_block_counts")
    return list(arr)


def cp_rank_fwd_key_tiles(prob: Problem) -> list:
    arr = (ctypes.c_int64 * prob.desc.cp_size)()
    _check(_lib.cp_rank_fwd_key_tiles(prob.ptr, arr), "cp_rank_fwd_key_tiles")
    return list(arr)


def workspace(prob: Problem, op: int, device=None) -> torch.Tensor:
    """A device buffer of cp_workspace_size bytes (256-byte aligned)."""
    n = max(cp_workspace_size(prob, op), 1)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def cp_shard_permute(prob: Problem, x: torch.Tensor, inverse: bool = False, out: Optional[torch.Tensor] = None,
                     ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Rows (first dim, T) of x from global to sharded order (inverse: back)."""
    if out is None:
        out = torch.empty_like(x)
    row_bytes = x[0].numel() * x.element_size() if x.shape[0] else x.element_size() * 16
    if ws is None:
        ws = workspace(prob, CP_OP_PERMUTE, x.device)
    _check(_lib.cp_shard_permute(prob.ptr, _ptr(x), _ptr(out), row_bytes, int(bool(inverse)), _ptr(ws),
                                 ws.numel(), _stream(stream)), "cp_shard_permute")
    return out


def cp_attn_block_fwd(prob: Problem, q_rank: int, kv_rank: int, q, k, v, o_part=None, lse_part=None,
                      ws=None, stream=None):
    off = cp_shard_offsets(prob)
    Tr = off[q_rank + 1] - off[q_rank]
    d = prob.desc
    if o_part is None:
        o_part = torch.empty(Tr, d.hq, d.d_v, dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty(d.hq, Tr, dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(prob, CP_OP_BLOCK_FWD, q.device)
    _check(_lib.cp_attn_block_fwd(prob.ptr, q_rank, kv_rank, _ptr(q), _ptr(k), _ptr(v), _ptr(o_part),
                                  _ptr(lse_part), _ptr(ws), ws.numel(), _stream(stream)), "cp_attn_block_fwd")
    return o_part, lse_part


def cp_lse_merge(prob: Problem, o_acc, lse_acc, o_part, lse_part, stream=None):
    rows = o_acc.shape[0]
    _check(_lib.cp_lse_merge(prob.ptr, rows, _ptr(o_acc), _ptr(lse_acc), _ptr(o_part), _ptr(lse_part),
                             _stream(stream)), "cp_lse_merge")
    return o_acc, lse_acc


def cp_attn_fwd(prob: Problem, q, k, v, o=None, lse=None, ws=None, stream=None):
    d = prob.desc
    if o is None:
        o = torch.empty(d.total_tokens, d.hq, d.d_v, dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(d.hq, d.total_tokens, dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(prob, CP_OP_FWD, q.device)
    _check(_lib.cp_attn_fwd(prob.ptr, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(),
                            _stream(stream)), "cp_attn_fwd")
    return o, lse


def cp_attn_bwd(prob: Problem, q, k, v, o, lse, dout, dq=None, dk=None, dv=None, ws=None, stream=None):
    if dq is None:
        dq = torch.empty_like(q)
    if dk is None:
        dk = torch.empty_like(k)
    if dv is None:
        dv = torch.empty_like(v)
    if ws is None:
        ws = workspace(prob, CP_OP_BWD, q.device)
    _check(_lib.cp_attn_bwd(prob.ptr, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                            _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(), _stream(stream)), "cp_attn_bwd")
    return dq, dk, dv


def cp_ring_attn_fwd(prob: Problem, q, k, v, o=None, lse=None, ws=None, stream=None, comm_stream=None,
                     overlap: bool = True):
    """Ring forward with explicit KV transport: C steps, each rank's block
    against the shard it holds, while the shards move one rank on through
    device-to-device copies on ``comm_stream`` (a new high-priority stream
    when None and ``overlap``, so that the copies are not queued behind the
    attention kernel's waiting CTAs; ``overlap=False`` serialises the copies
    on ``stream``)."""
    d = prob.desc
    if o is None:
        o = torch.empty(d.total_tokens, d.hq, d.d_v, dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(d.hq, d.total_tokens, dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(prob, CP_OP_RING_FWD, q.device)
    if overlap and comm_stream is None:
        comm_stream = torch.cuda.Stream(device=q.device, priority=-1)
    xs = _stream(comm_stream) if overlap else None
    _check(_lib.cp_ring_attn_fwd(prob.ptr, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(),
                                 _stream(stream), xs), "cp_ring_attn_fwd")
    return o, lse


def cp_ulysses_a2a(prob: Problem, x: torch.Tensor, inverse: bool = False, out: Optional[torch.Tensor] = None,
                   ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Ulysses all-to-all re-layout.  Forward: x [T, H, ...] in sharded order
    -> [C, T, H/C, ...] (rank r: heads r*H/C.., global token order).
    Inverse: [C, T, H/C, ...] -> [T, H, ...] sharded."""
    C = prob.desc.cp_size
    if inverse:
        heads = x.shape[2] * C
        shape = (x.shape[1], heads) + tuple(x.shape[3:])
    else:
        heads = x.shape[1]
        shape = (C, x.shape[0], heads // C) + tuple(x.shape[2:])
    head_bytes = (x[0, 0].numel() if not inverse else x[0, 0, 0].numel()) * x.element_size()
    if out is None:
        out = torch.empty(shape, dtype=x.dtype, device=x.device)
    if ws is None:
        ws = workspace(prob, CP_OP_ULYSSES_A2A, x.device)
    _check(_lib.cp_ulysses_a2a(prob.ptr, _ptr(x), _ptr(out), heads, head_bytes, int(bool(inverse)), _ptr(ws),
                               ws.numel(), _stream(stream)), "cp_ulysses_a2a")
    return out


def cp_ulysses_attn_fwd(prob: Problem, q, k, v, o=None, lse=None, ws=None, stream=None):
    """cp_attn_fwd computed the Ulysses way (all-to-all, per-rank full-sequence
    attention, all-to-all back); same inputs and outputs."""
    d = prob.desc
    if o is None:
        o = torch.empty(d.total_tokens, d.hq, d.d_v, dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(d.hq, d.total_tokens, dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(prob, CP_OP_ULYSSES_FWD, q.device)
    _check(_lib.cp_ulysses_attn_fwd(prob.ptr, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(),
                                    _stream(stream)), "cp_ulysses_attn_fwd")
    return o, lse


def cp_ulysses_attn_bwd(prob: Problem, q, k, v, o, lse, dout, dq=None, dk=None, dv=None, ws=None, stream=None):
    if dq is None:
        dq = torch.empty_like(q)
    if dk is None:
        dk = torch.empty_like(k)
    if dv is None:
        dv = torch.empty_like(v)
    if ws is None:
        ws = workspace(prob, CP_OP_ULYSSES_BWD, q.device)
    _check(_lib.cp_ulysses_attn_bwd(prob.ptr, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                                    _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(), _stream(stream)), "cp_ulysses_attn_bwd")
    return dq, dk, dv


def cp_lin_attn_fwd(prob: Problem, q, k, v, g, o=None, ws=None, stream=None):
    """Decayed linear attention with AllGather CP (contiguous pieces).
    g: float32 [hq] on the device, log of the per-head decay."""
    if o is None:
        o = torch.empty(q.shape[0], q.shape[1], v.shape[2], dtype=q.dtype, device=q.device)
    if ws is None:
        ws = workspace(prob, CP_OP_LIN_FWD, q.device)
    _check(_lib.cp_lin_attn_fwd(prob.ptr, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(o), _ptr(ws), ws.numel(),
                                _stream(stream)), "cp_lin_attn_fwd")
    return o


def cp_attn_bwd_prep(prob: Problem, o, dout, dpsum=None, stream=None):
    """D = rowsum(dout * o) per (head, row): float32 [hq, T]."""
    d = prob.desc
    if dpsum is None:
        dpsum = torch.empty(d.hq, d.total_tokens, dtype=torch.float32, device=o.device)
    _check(_lib.cp_attn_bwd_prep(prob.ptr, _ptr(o), _ptr(dout), _ptr(dpsum), _stream(stream)), "cp_attn_bwd_prep")
    return dpsum


def cp_attn_bwd_dkdv(prob: Problem, q, k, v, lse, dpsum, dout, dk=None, dv=None, ws=None, stream=None):
    if dk is None:
        dk = torch.empty_like(k)
    if dv is None:
        dv = torch.empty_like(v)
    if ws is None:
        ws = workspace(prob, CP_OP_BWD_DKDV, q.device)
    _check(_lib.cp_attn_bwd_dkdv(prob.ptr, _ptr(q), _ptr(k), _ptr(v), _ptr(lse), _ptr(dpsum), _ptr(dout), _ptr(dk),
                                 _ptr(dv), _ptr(ws), ws.numel(), _stream(stream)), "cp_attn_bwd_dkdv")
    return dk, dv


def cp_attn_bwd_dq(prob: Problem, q, k, v, lse, dpsum, dout, dq=None, ws=None, stream=None):
    if dq is None:
        dq = torch.empty_like(q)
    if ws is None:
        ws = workspace(prob, CP_OP_BWD_DQ, q.device)
    _check(_lib.cp_attn_bwd_dq(prob.ptr, _ptr(q), _ptr(k), _ptr(v), _ptr(lse), _ptr(dpsum), _ptr(dout), _ptr(dq),
                               _ptr(ws), ws.numel(), _stream(stream)), "cp_attn_bwd_dq")
    return dq


def cp_attn_fwd_noalloc(prob: Problem, q, k, v, o, lse, stream=None):
    """Forward without a workspace: the tile plan lives in the library's fixed
    device scratch (CP_NOALLOC_SCRATCH_BYTES).  o and lse are caller-owned;
    nothing is allocated here or in the library."""
    _check(_lib.cp_attn_fwd_noalloc(prob.ptr, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _stream(stream)),
           "cp_attn_fwd_noalloc")
    return o, lse


NOALLOC_SCRATCH_BYTES = 4 << 20


def cp_set_debug_checks(on: bool) -> bool:
    """Turns the plan checks on or off for later calls; returns the former setting."""
    prev = ctypes.c_int32(0)
    _check(_lib.cp_set_debug_checks(int(bool(on)), ctypes.byref(prev)), "cp_set_debug_checks")
    return bool(prev.value)


def cp_device_status(stream=None) -> int:
    code = ctypes.c_int32(0)
    st = _lib.cp_device_status(_stream(stream), ctypes.byref(code))
    if st not in (CP_OK, CP_ERR_DEVICE_TIMEOUT):
        _check(st, "cp_device_status")
    return int(code.value)


def cp_check_bounded_wait(timeout_ns: int = 20_000_000, stream=None) -> int:
    code = ctypes.c_int32(0)
    _check(_lib.cp_check_bounded_wait(int(timeout_ns), ctypes.byref(code), _stream(stream)),
           "cp_check_bounded_wait")
    return int(code.value)


__all__ = ["Problem", "CpError", "workspace", "LIB_PATH", "EXPORTED"] + EXPORTED
