"""Paged KV-cache write and paged decode attention for GB300 (sm_103a).

Thin Python layer over the C ABI of ``libpa.so`` (include/pa.h).  Every step
of the path runs in the library's CUDA kernels; this module only checks tensor
types and passes pointers, sizes and the current CUDA stream.  PyTorch serves
as the device-memory and stream provider.

    cache_write(k, v, slot_mapping, k_cache, v_cache)
    decode(q, k_cache, v_cache, block_tables, context_lens, scale, num_kv_heads) -> out
    multi_query(q, k_cache, v_cache, block_tables, context_lens, query_start, scale, num_kv_heads, max_q,
                k_new=None, v_new=None)      # with k_new / v_new: their cache write in the same launch
    copy_blocks(src_k, src_v, dst_k, dst_v, src_ids, dst_ids)   # copy-on-write, swap out / in
    BlockPool(num_blocks)                       # host block pool (untimed)
    build_slot_mapping(block_tables, context_lens, block_size)
"""
from __future__ import annotations

import ctypes
from typing import Optional

import numpy as np
import torch

from . import _native
from ._native import PAError, DecodeOptions, MATH

__all__ = ["cache_write", "copy_blocks", "decode", "decode_append", "decode_plan", "decode_plan_runs", "decode_planned", "DecodePlan", "plan_bounds", "plan_rates",
           "planned_workspace_size", "new_planned_workspace",
           "multi_query", "decode_runs", "new_runs_workspace", "gather_runs",
           "SlotPool", "decode_workspace_size", "plan_tokens_per_split", "kernel_kind",
           "new_workspace", "BlockPool",
           "build_slot_mapping", "read_device_status", "kernel_launch_count", "PAError", "lib"]

_DTYPE = {torch.float16: 0, torch.bfloat16: 1}


def lib() -> ctypes.CDLL:
    return _native.load()


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _need_cuda(name: str, t: torch.Tensor, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _opts(tokens_per_split: int, math: str, num_ctas: int = 0, timeline: Optional[torch.Tensor] = None,
          flags: int = 0) -> DecodeOptions:
    if math not in MATH:
        raise ValueError(f"math must be one of {sorted(MATH)}")
    return DecodeOptions(int(tokens_per_split), MATH[math], int(num_ctas), int(flags),
                         timeline.data_ptr() if timeline is not None else None)


def cache_write(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                v_cache: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> None:
    """k, v: [T, Hkv, D]; slot_mapping: int64 [T] (negative = skip); caches [NB, Hkv, B, D]."""
    for n, t in (("k", k), ("v", v), ("k_cache", k_cache), ("v_cache", v_cache)):
        _need_cuda(n, t, k.dtype)
    _need_cuda("slot_mapping", slot_mapping, torch.int64)
    if k.dtype not in _DTYPE:
        raise TypeError("k must be float16 or bfloat16")
    T, H, D = k.shape
    NB, H2, B, D2 = k_cache.shape
    if v.shape != k.shape or v_cache.shape != k_cache.shape or H2 != H or D2 != D or slot_mapping.numel() != T:
        raise ValueError("shape mismatch")
    rc = lib().pa_cache_write(k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), k_cache.data_ptr(),
                              v_cache.data_ptr(), T, H, D, B, NB, _DTYPE[k.dtype], _stream_ptr(stream))
    _native.check("pa_cache_write", rc)


def _pool_ptr(name: str, t: torch.Tensor, dtype=None):
    """Device memory, or pinned host memory (the library reaches it through its device view)."""
    if not isinstance(t, torch.Tensor) or not (t.is_cuda or t.is_pinned()):
        raise TypeError(f"{name} must be a CUDA tensor or a pinned host tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def copy_blocks(src_k: torch.Tensor, src_v: torch.Tensor, dst_k: torch.Tensor, dst_v: torch.Tensor,
                src_ids: torch.Tensor, dst_ids: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> None:
    """Copy whole blocks: dst[dst_ids[i]] = src[src_ids[i]] for K and V (pools [NB, Hkv, B, D]).
    Pools and ids live on the GPU or in pinned host memory; the ids are int32."""
    if src_k.dtype not in _DTYPE:
        raise TypeError("pools must be float16 or bfloat16")
    ptrs = [_pool_ptr(n, t, src_k.dtype) for n, t in (("src_k", src_k), ("src_v", src_v), ("dst_k", dst_k),
                                                     ("dst_v", dst_v))]
    sid = _pool_ptr("src_ids", src_ids, torch.int32)
    did = _pool_ptr("dst_ids", dst_ids, torch.int32)
    NBs, H, B, D = src_k.shape
    NBd = dst_k.shape[0]
    if (src_v.shape != src_k.shape or dst_k.shape[1:] != src_k.shape[1:] or dst_v.shape != dst_k.shape or
            src_ids.numel() != dst_ids.numel()):
        raise ValueError("shape mismatch")
    rc = lib().pa_copy_blocks(ptrs[0], ptrs[1], NBs, ptrs[2], ptrs[3], NBd, sid, did, src_ids.numel(), H, D, B,
                              _DTYPE[src_k.dtype], _stream_ptr(stream))
    _native.check("pa_copy_blocks", rc)


def decode_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                          max_blocks_per_seq: int, tokens_per_split: int = 0, math: str = "auto",
                          num_ctas: int = 0) -> int:
    o = _opts(tokens_per_split, math, num_ctas)
    return int(lib().pa_decode_workspace_size_ex(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                                 max_blocks_per_seq, ctypes.byref(o)))


def plan_tokens_per_split(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                          max_blocks_per_seq: int, tokens_per_split: int = 0, math: str = "auto") -> int:
    o = _opts(tokens_per_split, math)
    return _native.check("pa_decode_plan_tokens_per_split",
                         lib().pa_decode_plan_tokens_per_split(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                               block_size, max_blocks_per_seq, ctypes.byref(o)))


def kernel_kind(num_seqs: int, num_q_heads: int, num_kv_heads: int, math: str = "auto") -> int:
    """1 = split grid (CUDA cores), 2 = persistent (tensor cores), 3 = split grid (tensor cores)."""
    o = _opts(0, math)
    return _native.check("pa_decode_kernel_kind",
                         lib().pa_decode_kernel_kind(num_seqs, num_q_heads, num_kv_heads, ctypes.byref(o)))


_workspaces: dict = {}


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled decode workspace (the persistent kernel expects zeroed counters)."""
    return torch.zeros(max(int(nbytes), 16), dtype=torch.uint8, device=device or "cuda")


def _workspace(device: torch.device, nbytes: int, kind: int, num_ctas: int) -> Optional[torch.Tensor]:
    """One zeroed workspace per (device, kernel kind, CTA count): the persistent kernel's
    counters sit at an offset fixed by the CTA count and are left zero by every call."""
    if nbytes == 0:
        return None
    key = (device.index if device.index is not None else torch.cuda.current_device(), kind, num_ctas)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = new_workspace(nbytes, device)
        _workspaces[key] = ws
    return ws


def decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
           context_lens: torch.Tensor, scale: float, num_kv_heads: int, out: Optional[torch.Tensor] = None,
           workspace: Optional[torch.Tensor] = None, tokens_per_split: int = 0, math: str = "auto",
           num_ctas: int = 0, timeline: Optional[torch.Tensor] = None,
           stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Paged decode attention.  q: [S, Hq, D]; caches [NB, Hkv, B, D]; block_tables int32
    [S, max_blocks]; context_lens int32 [S].  Returns out [S, Hq, D] in q's dtype.
    ``timeline``: optional int64 CUDA tensor [num_ctas, 16] receiving the persistent kernel's trace."""
    _need_cuda("q", q)
    if q.dtype not in _DTYPE:
        raise TypeError("q must be float16 or bfloat16")
    _need_cuda("k_cache", k_cache, q.dtype)
    _need_cuda("v_cache", v_cache, q.dtype)
    _need_cuda("block_tables", block_tables, torch.int32)
    _need_cuda("context_lens", context_lens, torch.int32)
    S, Hq, D = q.shape
    NB, Hkv, B, D2 = k_cache.shape
    if Hkv != num_kv_heads or D2 != D or v_cache.shape != k_cache.shape:
        raise ValueError("cache shape does not match q / num_kv_heads")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.numel() != S:
        raise ValueError("block_tables / context_lens do not match q")
    max_blocks = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    else:
        _need_cuda("out", out, q.dtype)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    o = _opts(tokens_per_split, math, num_ctas, timeline)
    need = int(lib().pa_decode_workspace_size_ex(S, Hq, Hkv, D, B, max_blocks, ctypes.byref(o)))
    if workspace is None:
        kind = lib().pa_decode_kernel_kind(S, Hq, Hkv, ctypes.byref(o))
        workspace = _workspace(q.device, need, kind, int(num_ctas))
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib().pa_decode_ex(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                            block_tables.data_ptr(), context_lens.data_ptr(), float(scale), int(num_kv_heads),
                            S, Hq, D, B, NB, max_blocks, _DTYPE[q.dtype], ws_ptr, ws_bytes, _stream_ptr(stream),
                            ctypes.byref(o))
    _native.check("pa_decode", rc)
    return out


def decode_append(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                  v_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                  num_kv_heads: int, out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                  num_ctas: int = 0, early_reads: bool = False, timeline: Optional[torch.Tensor] = None,
                  stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Cache write of each sequence's newest token (position context_lens[s] - 1) and decode
    attention, in one launch.  k_new, v_new: [S, Hkv, D].  ``early_reads=True`` opts in to the
    early-read contract of pa_decode_append (include/pa.h): the preceding kernel in the stream
    must not write the caches, the tables or the lengths."""
    _need_cuda("q", q)
    if q.dtype not in _DTYPE:
        raise TypeError("q must be float16 or bfloat16")
    for n, t in (("k_new", k_new), ("v_new", v_new), ("k_cache", k_cache), ("v_cache", v_cache)):
        _need_cuda(n, t, q.dtype)
    _need_cuda("block_tables", block_tables, torch.int32)
    _need_cuda("context_lens", context_lens, torch.int32)
    S, Hq, D = q.shape
    NB, Hkv, B, D2 = k_cache.shape
    if Hkv != num_kv_heads or D2 != D or v_cache.shape != k_cache.shape:
        raise ValueError("cache shape does not match q / num_kv_heads")
    if k_new.shape != (S, Hkv, D) or v_new.shape != k_new.shape:
        raise ValueError("k_new / v_new must be [S, Hkv, D]")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.numel() != S:
        raise ValueError("block_tables / context_lens do not match q")
    max_blocks = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    else:
        _need_cuda("out", out, q.dtype)
    o = _opts(0, "mma", num_ctas, timeline, _native.EARLY_READS if early_reads else 0)
    need = int(lib().pa_decode_workspace_size_ex(S, Hq, Hkv, D, B, max_blocks, ctypes.byref(o)))
    if workspace is None:
        kind = lib().pa_decode_kernel_kind(S, Hq, Hkv, ctypes.byref(o))
        workspace = _workspace(q.device, need, kind, int(num_ctas))
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib().pa_decode_append(out.data_ptr(), q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
                                context_lens.data_ptr(), float(scale), int(num_kv_heads), S, Hq, D, B, NB,
                                max_blocks, _DTYPE[q.dtype], ws_ptr, ws_bytes, _stream_ptr(stream), ctypes.byref(o))
    _native.check("pa_decode_append", rc)
    return out


class DecodePlan:
    """A decode step's plan (pa_decode_plan): device bytes plus the shape it was built for."""

    def __init__(self, data: torch.Tensor, num_seqs: int, num_q_heads: int, num_kv_heads: int, block_size: int,
                 num_blocks: int, max_blocks_per_seq: int, num_ctas: int, adaptive: bool = False,
                 runs: bool = False):
        self.data = data
        self.adaptive = adaptive
        self.runs = runs
        self.num_seqs = num_seqs
        self.num_q_heads = num_q_heads
        self.num_kv_heads = num_kv_heads
        self.block_size = block_size
        self.num_blocks = num_blocks
        self.max_blocks_per_seq = max_blocks_per_seq
        self.num_ctas = num_ctas


def decode_plan(block_tables: torch.Tensor, context_lens: torch.Tensor, num_q_heads: int, num_kv_heads: int,
                block_size: int, num_blocks: int, head_dim: int = 128, plan: Optional[DecodePlan] = None,
                num_ctas: int = 0, adaptive: bool = False,
                stream: Optional[torch.cuda.Stream] = None) -> DecodePlan:
    """Build (or rebuild in place, ``plan``) the plan of a decode step: one small kernel that reads
    the block tables and lengths once for every layer's pa_decode_planned call.  ``adaptive``:
    the CTAs' shares follow the streaming rates that earlier decode_planned calls measured into
    the same plan buffer (PA_PLAN_ADAPTIVE)."""
    _need_cuda("block_tables", block_tables, torch.int32)
    _need_cuda("context_lens", context_lens, torch.int32)
    if block_tables.dim() != 2 or block_tables.shape[0] != context_lens.numel():
        raise ValueError("block_tables must be [S, max_blocks] with S = context_lens.numel()")
    S, max_blocks = block_tables.shape
    o = _opts(0, "auto", num_ctas, flags=_native.PLAN_ADAPTIVE if adaptive else 0)
    need = int(lib().pa_decode_plan_size(S, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks,
                                         ctypes.byref(o)))
    if need == 0:
        raise PAError("pa_decode_plan_size", -2)
    if plan is None or plan.data.numel() < need:
        # zeroed: an adaptive build finds no stale rates in a fresh buffer
        data = torch.zeros(need, dtype=torch.uint8, device=block_tables.device)
        plan = DecodePlan(data, S, num_q_heads, num_kv_heads, block_size, num_blocks, max_blocks, int(num_ctas),
                          adaptive)
    else:
        plan.num_seqs, plan.num_q_heads, plan.num_kv_heads = S, num_q_heads, num_kv_heads
        plan.block_size, plan.num_blocks, plan.max_blocks_per_seq, plan.num_ctas = (block_size, num_blocks,
                                                                                     max_blocks, int(num_ctas))
        plan.adaptive, plan.runs = adaptive, False
    rc = lib().pa_decode_plan(plan.data.data_ptr(), plan.data.numel(), block_tables.data_ptr(),
                              context_lens.data_ptr(), S, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                              max_blocks, _stream_ptr(stream), ctypes.byref(o))
    _native.check("pa_decode_plan", rc)
    return plan


def _plan_flags(plan: DecodePlan) -> int:
    return (_native.PLAN_ADAPTIVE if plan.adaptive else 0) | (_native.PLAN_RUNS if plan.runs else 0)


def decode_plan_runs(runs: torch.Tensor, seq_runs: torch.Tensor, num_q_heads: int, num_kv_heads: int,
                     block_size: int, num_blocks: int, max_context: int, head_dim: int = 128,
                     plan: Optional[DecodePlan] = None, num_ctas: int = 0,
                     stream: Optional[torch.cuda.Stream] = None) -> DecodePlan:
    """The plan of a decode step over contexts given as runs (block_id, slot_offset, length):
    runs int32 [R, 3], sequence s reading runs seq_runs[s] .. seq_runs[s+1]-1 (pa_decode_plan_runs).
    decode_planned then decodes each layer through it (no cache write)."""
    _need_cuda("runs", runs, torch.int32)
    _need_cuda("seq_runs", seq_runs, torch.int32)
    S = seq_runs.numel() - 1
    if S < 1 or (runs.numel() and runs.shape[-1] != 3):
        raise ValueError("seq_runs must have S + 1 entries and runs 3 columns")
    max_blocks = (int(max_context) + block_size - 1) // block_size
    o = _opts(0, "auto", num_ctas, flags=_native.PLAN_RUNS)
    need = int(lib().pa_decode_plan_size(S, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks,
                                         ctypes.byref(o)))
    if need == 0:
        raise PAError("pa_decode_plan_size", -2)
    if plan is None or plan.data.numel() < need:
        data = torch.zeros(need, dtype=torch.uint8, device=runs.device)
        plan = DecodePlan(data, S, num_q_heads, num_kv_heads, block_size, num_blocks, max_blocks, int(num_ctas),
                          False, True)
    else:
        plan.num_seqs, plan.num_q_heads, plan.num_kv_heads = S, num_q_heads, num_kv_heads
        plan.block_size, plan.num_blocks, plan.max_blocks_per_seq, plan.num_ctas = (block_size, num_blocks,
                                                                                     max_blocks, int(num_ctas))
        plan.adaptive, plan.runs = False, True
    rc = lib().pa_decode_plan_runs(plan.data.data_ptr(), plan.data.numel(),
                                   runs.data_ptr() if runs.numel() else seq_runs.data_ptr(), seq_runs.data_ptr(), S,
                                   num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, int(max_context),
                                   _stream_ptr(stream), ctypes.byref(o))
    _native.check("pa_decode_plan_runs", rc)
    return plan


def _plan_sections(plan: DecodePlan):
    o = _opts(0, "auto", plan.num_ctas, flags=_plan_flags(plan))
    ctas, b_off, r_off = ctypes.c_int(0), ctypes.c_size_t(0), ctypes.c_size_t(0)
    rc = lib().pa_decode_plan_sections(plan.num_seqs, plan.num_q_heads, plan.num_kv_heads, 128, plan.block_size,
                                       plan.max_blocks_per_seq, ctypes.byref(o), ctypes.byref(ctas),
                                       ctypes.byref(b_off), ctypes.byref(r_off))
    _native.check("pa_decode_plan_sections", rc)
    return ctas.value, b_off.value, r_off.value


def plan_bounds(plan: DecodePlan) -> torch.Tensor:
    """The plan's group bounds (int32 [2 C + 1], on the host): CTA c streams chunks
    [b[2c], b[2c+1]) forwards and [b[2c+1], b[2c+2]) backwards."""
    C, off, _ = _plan_sections(plan)
    return plan.data[off:off + 4 * (2 * C + 1)].cpu().view(torch.int32).clone()


def plan_rates(plan: DecodePlan) -> torch.Tensor:
    """The CTAs' measured streaming rates kept in an adaptive plan's buffer (float [C], host;
    weight per SM cycle, 0 = no measurement)."""
    C, _, off = _plan_sections(plan)
    return plan.data[off:off + 4 * C].cpu().view(torch.float32).clone()


def planned_workspace_size(num_ctas: int = 0) -> int:
    """Bytes of workspace pa_decode_planned needs for a plan built with ``num_ctas``."""
    o = _opts(0, "auto", num_ctas)
    return int(lib().pa_decode_planned_workspace_size(ctypes.byref(o)))


def new_planned_workspace(num_ctas: int = 0, device=None) -> torch.Tensor:
    """A pa_decode_planned workspace, filled with 0xFF bytes as the kernel expects."""
    return torch.full((max(planned_workspace_size(num_ctas), 16),), 255, dtype=torch.uint8,
                      device=device or "cuda")


def decode_planned(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, plan: DecodePlan, scale: float,
                   k_new: Optional[torch.Tensor] = None, v_new: Optional[torch.Tensor] = None,
                   out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                   early_reads: bool = False, timeline: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Decode attention of one layer through a step's plan (pa_decode_planned); with k_new / v_new
    ([S, Hkv, D]) the new token's rows are written at position L - 1 first, as decode_append."""
    _need_cuda("q", q)
    if q.dtype not in _DTYPE:
        raise TypeError("q must be float16 or bfloat16")
    _need_cuda("k_cache", k_cache, q.dtype)
    _need_cuda("v_cache", v_cache, q.dtype)
    S, Hq, D = q.shape
    NB, Hkv, B, D2 = k_cache.shape
    if (S, Hq, Hkv, B, NB) != (plan.num_seqs, plan.num_q_heads, plan.num_kv_heads, plan.block_size,
                               plan.num_blocks) or D2 != D or v_cache.shape != k_cache.shape:
        raise ValueError("q / caches do not match the plan")
    if (k_new is None) != (v_new is None):
        raise ValueError("k_new and v_new go together")
    if k_new is not None:
        for n, t in (("k_new", k_new), ("v_new", v_new)):
            _need_cuda(n, t, q.dtype)
        if k_new.shape != (S, Hkv, D) or v_new.shape != k_new.shape:
            raise ValueError("k_new / v_new must be [S, Hkv, D]")
    if out is None:
        out = torch.empty_like(q)
    else:
        _need_cuda("out", out, q.dtype)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    o = _opts(0, "auto", plan.num_ctas, timeline, (_native.EARLY_READS if early_reads else 0) | _plan_flags(plan))
    if workspace is None:
        key = ("planned", q.device.index if q.device.index is not None else torch.cuda.current_device(),
               plan.num_ctas)
        workspace = _workspaces.get(key)
        if workspace is None:
            workspace = _workspaces[key] = new_planned_workspace(plan.num_ctas, q.device)
    rc = lib().pa_decode_planned(out.data_ptr(), q.data_ptr(), k_new.data_ptr() if k_new is not None else None,
                                 v_new.data_ptr() if v_new is not None else None, k_cache.data_ptr(),
                                 v_cache.data_ptr(), plan.data.data_ptr(), plan.data.numel(), float(scale), S, Hq,
                                 Hkv, D, B, NB,
                                 plan.max_blocks_per_seq, _DTYPE[q.dtype], workspace.data_ptr(),
                                 workspace.numel() * workspace.element_size(), _stream_ptr(stream), ctypes.byref(o))
    _native.check("pa_decode_planned", rc)
    return out


def multi_query(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                context_lens: torch.Tensor, query_start: torch.Tensor, scale: float, num_kv_heads: int,
                max_q: int, out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                num_ctas: int = 0, timeline: Optional[torch.Tensor] = None,
                k_new: Optional[torch.Tensor] = None, v_new: Optional[torch.Tensor] = None,
                early_reads: bool = False, tiles: str = "tc",
                stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Several new query tokens per sequence attending causally over the paged cache.
    q: [T, Hq, D]; sequence s owns rows query_start[s] .. query_start[s+1]-1 (int32 [S+1]), its
    newest tokens; at most ``max_q`` per sequence.  See pa_multi_query in include/pa.h.
    With k_new / v_new ([T, Hkv, D], rows as q's) the same launch first writes them into the
    slots of their positions (pa_multi_query_append; ``early_reads`` as for decode_append).  ``tiles``: beyond 16 query rows per (sequence, kv head), "tc" runs the
    tcgen05 tiles of 128 rows, "mma" the mma.sync tiles of 64 rows."""
    _need_cuda("q", q)
    if q.dtype not in _DTYPE:
        raise TypeError("q must be float16 or bfloat16")
    _need_cuda("k_cache", k_cache, q.dtype)
    _need_cuda("v_cache", v_cache, q.dtype)
    _need_cuda("block_tables", block_tables, torch.int32)
    _need_cuda("context_lens", context_lens, torch.int32)
    _need_cuda("query_start", query_start, torch.int32)
    T, Hq, D = q.shape
    NB, Hkv, B, D2 = k_cache.shape
    S = context_lens.numel()
    if Hkv != num_kv_heads or D2 != D or v_cache.shape != k_cache.shape:
        raise ValueError("cache shape does not match q / num_kv_heads")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or query_start.numel() != S + 1:
        raise ValueError("block_tables / query_start do not match context_lens")
    max_blocks = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    else:
        _need_cuda("out", out, q.dtype)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    append = k_new is not None or v_new is not None
    if append:
        for n, t in (("k_new", k_new), ("v_new", v_new)):
            _need_cuda(n, t, q.dtype)
        if k_new.shape != (T, Hkv, D) or v_new.shape != k_new.shape:
            raise ValueError("k_new / v_new must be [T, Hkv, D]")
        o = _opts(0, "mma", num_ctas, timeline, _native.EARLY_READS if early_reads else 0)
    else:
        if tiles not in ("tc", "mma"):
            raise ValueError('tiles must be "tc" or "mma"')
        o = _opts(0, "mma", num_ctas, timeline, _native.PREFILL_MMA_SYNC if tiles == "mma" else 0)
    need = int(lib().pa_decode_workspace_size_ex(S, Hq, Hkv, D, B, max_blocks, ctypes.byref(o)))
    if workspace is None:
        workspace = _workspace(q.device, need, 2, int(num_ctas))
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    if append:
        rc = lib().pa_multi_query_append(
            out.data_ptr(), q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(),
            v_cache.data_ptr(), block_tables.data_ptr(), context_lens.data_ptr(), query_start.data_ptr(),
            float(scale), int(num_kv_heads), S, T, int(max_q), Hq, D, B, NB, max_blocks, _DTYPE[q.dtype], ws_ptr,
            ws_bytes, _stream_ptr(stream), ctypes.byref(o))
        _native.check("pa_multi_query_append", rc)
        return out
    rc = lib().pa_multi_query(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                              block_tables.data_ptr(), context_lens.data_ptr(), query_start.data_ptr(), float(scale),
                              int(num_kv_heads), S, T, int(max_q), Hq, D, B, NB, max_blocks, _DTYPE[q.dtype], ws_ptr,
                              ws_bytes, _stream_ptr(stream), ctypes.byref(o))
    _native.check("pa_multi_query", rc)
    return out


_runs_workspaces = {}


def _runs_workspace(device: torch.device, nbytes: int) -> torch.Tensor:
    """One pa_decode_runs workspace per device, filled with 0xFF bytes once (every completed call
    leaves it so)."""
    key = device.index if device.index is not None else torch.cuda.current_device()
    ws = _runs_workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.full((nbytes,), 255, dtype=torch.uint8, device=device)
        _runs_workspaces[key] = ws
    return ws


def new_runs_workspace(q: torch.Tensor, num_kv_heads: int, block_size: int, max_context: int) -> torch.Tensor:
    """A pa_decode_runs workspace for q's shape, filled with 0xFF bytes as the kernels expect."""
    S, Hq, D = q.shape
    need = int(lib().pa_decode_runs_workspace_size(S, Hq, num_kv_heads, D, block_size, int(max_context)))
    return torch.full((max(need, 16),), 255, dtype=torch.uint8, device=q.device)


def decode_runs(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, runs: torch.Tensor,
                seq_runs: torch.Tensor, scale: float, num_kv_heads: int, max_context: int,
                out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Decode over contexts given as runs (block_id, slot_offset, length): runs int32 [R, 3],
    sequence s reading runs seq_runs[s] .. seq_runs[s+1]-1 (int32 [S + 1]).  See pa_decode_runs."""
    _need_cuda("q", q)
    if q.dtype not in _DTYPE:
        raise TypeError("q must be float16 or bfloat16")
    _need_cuda("k_cache", k_cache, q.dtype)
    _need_cuda("v_cache", v_cache, q.dtype)
    _need_cuda("runs", runs, torch.int32)
    _need_cuda("seq_runs", seq_runs, torch.int32)
    S, Hq, D = q.shape
    NB, Hkv, B, D2 = k_cache.shape
    if Hkv != num_kv_heads or D2 != D or v_cache.shape != k_cache.shape:
        raise ValueError("cache shape does not match q / num_kv_heads")
    if seq_runs.numel() != S + 1 or (runs.numel() and runs.shape[-1] != 3):
        raise ValueError("seq_runs must have S + 1 entries and runs 3 columns")
    if out is None:
        out = torch.empty_like(q)
    else:
        _need_cuda("out", out, q.dtype)
    need = int(lib().pa_decode_runs_workspace_size(S, Hq, Hkv, D, B, int(max_context)))
    if workspace is None and need:
        workspace = _runs_workspace(q.device, need)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib().pa_decode_runs(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                              runs.data_ptr() if runs.numel() else seq_runs.data_ptr(), seq_runs.data_ptr(),
                              float(scale), int(num_kv_heads), S, Hq, D, B, NB, int(max_context), _DTYPE[q.dtype],
                              ws_ptr, ws_bytes, _stream_ptr(stream))
    _native.check("pa_decode_runs", rc)
    return out


def gather_runs(src_k: torch.Tensor, src_v: torch.Tensor, dst_k: torch.Tensor, dst_v: torch.Tensor,
                moves: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> None:
    """Row-run moves: moves int32 [M, 5] = (src_block, src_off, length, dst_block, dst_off)."""
    if src_k.dtype not in _DTYPE:
        raise TypeError("pools must be float16 or bfloat16")
    for n, t in (("src_k", src_k), ("src_v", src_v), ("dst_k", dst_k), ("dst_v", dst_v)):
        _need_cuda(n, t, src_k.dtype)
    _need_cuda("moves", moves, torch.int32)
    NBs, H, B, D = src_k.shape
    if src_v.shape != src_k.shape or dst_k.shape[1:] != src_k.shape[1:] or dst_v.shape != dst_k.shape:
        raise ValueError("shape mismatch")
    M = moves.numel() // 5
    rc = lib().pa_gather_runs(src_k.data_ptr(), src_v.data_ptr(), NBs, dst_k.data_ptr(), dst_v.data_ptr(),
                              dst_k.shape[0], moves.data_ptr(), M, H, D, B, _DTYPE[src_k.dtype], _stream_ptr(stream))
    _native.check("pa_gather_runs", rc)


class SlotPool:
    """Slotted blocks (host): nodes of up to block_size tokens packed into shared blocks."""

    def __init__(self, num_blocks: int, block_size: int):
        self._lib = lib()
        self._h = self._lib.pa_slots_create(int(num_blocks), int(block_size))
        if not self._h:
            raise ValueError("pa_slots_create failed")

    def close(self):
        if self._h:
            self._lib.pa_slots_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def alloc(self, n: int):
        """(block, offset) of a new slot of n tokens."""
        b = ctypes.c_int32(-1)
        o = ctypes.c_int32(-1)
        _native.check("pa_slots_alloc", self._lib.pa_slots_alloc(self._h, int(n), ctypes.byref(b), ctypes.byref(o)))
        return int(b.value), int(o.value)

    def release(self, block: int, offset: int, n: int) -> int:
        return _native.check("pa_slots_release", self._lib.pa_slots_release(self._h, int(block), int(offset), int(n)))

    def tail(self, block: int) -> int:
        return _native.check("pa_slots_tail", self._lib.pa_slots_tail(self._h, int(block)))

    def live(self, block: int) -> int:
        return _native.check("pa_slots_live", self._lib.pa_slots_live(self._h, int(block)))

    @property
    def num_free(self) -> int:
        return self._lib.pa_slots_num_free(self._h)


def read_device_status(clear: bool = True, stream: Optional[torch.cuda.Stream] = None) -> int:
    bits = ctypes.c_uint32(0)
    _native.check("pa_read_device_status",
                  lib().pa_read_device_status(_stream_ptr(stream), int(clear), ctypes.byref(bits)))
    return int(bits.value)


def kernel_launch_count() -> int:
    return int(lib().pa_kernel_launch_count())


# ------------------------------------------------------------------------------------------
# host block pool
# ------------------------------------------------------------------------------------------

def _i32p(a: np.ndarray):
    return a.ctypes.data_as(_native.c_i32p)


class BlockPool:
    """Free-bitmap pool with reference counts (host, untimed).  See include/pa.h."""

    def __init__(self, num_blocks: int):
        self._lib = lib()
        self._h = self._lib.pa_pool_create(int(num_blocks))
        if not self._h:
            raise ValueError("pa_pool_create failed")

    def close(self):
        if self._h:
            self._lib.pa_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def alloc(self) -> int:
        return _native.check("pa_pool_alloc", self._lib.pa_pool_alloc(self._h))

    def incref(self, block_id: int) -> int:
        return _native.check("pa_pool_incref", self._lib.pa_pool_incref(self._h, int(block_id)))

    def decref(self, block_id: int) -> int:
        return _native.check("pa_pool_decref", self._lib.pa_pool_decref(self._h, int(block_id)))

    def refcount(self, block_id: int) -> int:
        return _native.check("pa_pool_refcount", self._lib.pa_pool_refcount(self._h, int(block_id)))

    @property
    def num_free(self) -> int:
        return self._lib.pa_pool_num_free(self._h)

    @property
    def num_blocks(self) -> int:
        return self._lib.pa_pool_num_blocks(self._h)

    def assign(self, table_row: np.ndarray, context_len: int, block_size: int,
               shared_row: Optional[np.ndarray] = None, shared_blocks: int = 0) -> None:
        assert table_row.dtype == np.int32 and table_row.flags.c_contiguous
        sr = None
        if shared_blocks:
            shared_row = np.ascontiguousarray(shared_row, dtype=np.int32)
            sr = _i32p(shared_row)
        _native.check("pa_pool_assign", self._lib.pa_pool_assign(self._h, _i32p(table_row), table_row.size,
                                                                 int(context_len), int(block_size), sr,
                                                                 int(shared_blocks)))

    def append_token(self, table_row: np.ndarray, context_len: int, block_size: int):
        """Returns (slot, cow_src, cow_dst) for a token appended after context_len tokens."""
        assert table_row.dtype == np.int32 and table_row.flags.c_contiguous
        slot = ctypes.c_int64(-1)
        src = ctypes.c_int32(-1)
        dst = ctypes.c_int32(-1)
        _native.check("pa_pool_append_token",
                      self._lib.pa_pool_append_token(self._h, _i32p(table_row), table_row.size, int(context_len),
                                                     int(block_size), ctypes.byref(slot), ctypes.byref(src),
                                                     ctypes.byref(dst)))
        return int(slot.value), int(src.value), int(dst.value)

    def move_blocks(self, to: "BlockPool", table_row: np.ndarray, n: int):
        """Move the first n blocks of a sequence to pool ``to`` (swap out / in); returns the
        (src_ids, dst_ids) pairs that copy_blocks must then copy."""
        assert table_row.dtype == np.int32 and table_row.flags.c_contiguous and n <= table_row.size
        src = np.empty(max(n, 1), dtype=np.int32)
        dst = np.empty(max(n, 1), dtype=np.int32)
        _native.check("pa_pool_move_blocks", self._lib.pa_pool_move_blocks(self._h, to._h, _i32p(table_row), int(n),
                                                                           _i32p(src), _i32p(dst)))
        return src[:n], dst[:n]

    def release(self, table_row: np.ndarray, context_len: int, block_size: int) -> None:
        assert table_row.dtype == np.int32 and table_row.flags.c_contiguous
        _native.check("pa_pool_release", self._lib.pa_pool_release(self._h, _i32p(table_row), table_row.size,
                                                                   int(context_len), int(block_size)))


def build_slot_mapping(block_tables, context_lens, block_size: int) -> np.ndarray:
    """Host: slot of each sequence's newest token (context_lens[s] - 1), -1 for empty contexts."""
    bt = np.ascontiguousarray(np.asarray(block_tables.cpu() if isinstance(block_tables, torch.Tensor)
                                         else block_tables, dtype=np.int32))
    lens = np.ascontiguousarray(np.asarray(context_lens.cpu() if isinstance(context_lens, torch.Tensor)
                                           else context_lens, dtype=np.int32))
    S = lens.size
    out = np.empty(S, dtype=np.int64)
    _native.check("pa_build_slot_mapping",
                  lib().pa_build_slot_mapping(_i32p(bt), bt.shape[1] if bt.ndim == 2 else 0, _i32p(lens), S,
                                              int(block_size), out.ctypes.data_as(_native.c_i64p)))
    return out
