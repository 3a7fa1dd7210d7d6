"""CPU oracle for the paged KV cache write and paged decode attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs may import this package.  It shares
no code with the CUDA library and never imports it.

The arithmetic lives in ``pa_oracle.c`` (plain fp64 C, OpenMP over
(sequence, kv-head) pairs); this module compiles it with the host C compiler
and marshals numpy/torch CPU arrays to it.  Each entry point names the passage
it follows:

* ``locate`` / ``slot_of_token`` / ``slot_mapping`` -- the address of token t is
  (block_table[t / B], t % B): "端侧 SLM 显存保活术：在 4GB 内存板卡上实现轻量
  PagedAttention 与 KV 缓存分块", section "注意力寻址：非连续物理块的间接寻址内核";
  the new token is the last one of the context ("显存虚拟化革命：PagedAttention 内存池管理与
  显存碎片终结", §三 sequence diagram).
* ``kv_bytes_per_token`` -- the byte ledger of the first page, section "KV Cache 的物理膨胀账本".
* ``cache_write`` -- byte copy of each new (token, kv-head) row into its slot (§三 of the second page).
* ``decode`` -- out = softmax(scale * q K^T) V over the rows gathered through the
  block table, in fp64 (§五.1 kernel sketch of the second page).
* ``multi_query`` -- the same for several new query tokens per sequence, each attending
  causally up to its own position (the chunked prefill the second page's closing section
  points to).
* ``copy_blocks`` -- whole-block deep copy (§四 copy-on-write of the second page).
* ``decode_runs`` / ``gather_runs`` -- contexts given as runs (block_id, slot_offset, length)
  and row-run moves: the slotted blocks and online defragmentation of the radix-tree
  fragmentation page.

Pins (tests/test_oracle.py): exhaustive element decoding against numpy, the
pages' worked address example and byte counts, torch's fp64
``scaled_dot_product_attention`` on the unpaged data, bit-identical output under
a permutation of physical ids, closed forms (one token, zero query, equal keys,
one dominant score, two tokens), and planted mistakes that each pin must catch.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path
from typing import Optional

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "pa_oracle.c"
_BUILD = _HERE / "_build"

_c_i64 = ctypes.c_int64
_c_int = ctypes.c_int
_ptr = ctypes.c_void_p


def build(mutant: int = 0, out_dir: Optional[Path] = None, force: bool = False) -> Path:
    """Compile the oracle into a shared library and return its path."""
    out_dir = Path(out_dir) if out_dir is not None else _BUILD
    out_dir.mkdir(parents=True, exist_ok=True)
    name = "libpa_oracle.so" if mutant == 0 else f"libpa_oracle_mutant{mutant}.so"
    lib = out_dir / name
    if not force and lib.exists() and lib.stat().st_mtime >= _SRC.stat().st_mtime:
        return lib
    tmp = out_dir / (name + f".tmp{os.getpid()}")
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", str(_SRC), "-o", str(tmp), "-lm"]
    if mutant:
        cmd.insert(1, f"-DPAO_MUTANT={int(mutant)}")
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: Path):
        self.path = Path(path)
        L = ctypes.CDLL(str(self.path))
        self._L = L
        L.pao_f16_to_f64.restype = ctypes.c_double
        L.pao_f16_to_f64.argtypes = [ctypes.c_uint16]
        L.pao_bf16_to_f64.restype = ctypes.c_double
        L.pao_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.pao_decode_elems.restype = None
        L.pao_decode_elems.argtypes = [_ptr, _c_i64, _c_int, _ptr]
        L.pao_kv_bytes_per_token.restype = _c_i64
        L.pao_kv_bytes_per_token.argtypes = [_c_int, _c_int, _c_int]
        L.pao_locate.restype = None
        L.pao_locate.argtypes = [_ptr, _c_i64, _c_int, _ptr, _ptr]
        L.pao_slot_of_token.restype = _c_i64
        L.pao_slot_of_token.argtypes = [_ptr, _c_i64, _c_int]
        L.pao_slot_mapping.restype = None
        L.pao_slot_mapping.argtypes = [_ptr, _c_int, _ptr, _c_int, _c_int, _ptr]
        L.pao_cache_write.restype = None
        L.pao_cache_write.argtypes = [_ptr, _ptr, _ptr, _ptr, _ptr, _c_int, _c_int, _c_int, _c_int]
        L.pao_decode.restype = _c_int
        L.pao_decode.argtypes = [_ptr, _ptr, _ptr, _ptr, _ptr, _c_int, _ptr, ctypes.c_double,
                                 _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int]
        L.pao_copy_blocks.restype = _c_int
        L.pao_copy_blocks.argtypes = [_ptr, _ptr, _c_int, _ptr, _ptr, _c_int, _ptr, _ptr, _c_int, _c_int, _c_int,
                                      _c_int]
        L.pao_multi_query.restype = _c_int
        L.pao_multi_query.argtypes = [_ptr, _ptr, _ptr, _ptr, _ptr, _c_int, _ptr, _ptr, ctypes.c_double,
                                      _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int]
        L.pao_decode_runs.restype = _c_int
        L.pao_decode_runs.argtypes = [_ptr, _ptr, _ptr, _ptr, _ptr, _ptr, ctypes.c_double, _c_int, _c_int, _c_int,
                                      _c_int, _c_int, _c_int, _c_int, _c_int]
        L.pao_gather_runs.restype = _c_int
        L.pao_gather_runs.argtypes = [_ptr, _ptr, _c_int, _ptr, _ptr, _c_int, _ptr, _c_int, _c_int, _c_int, _c_int]
        L.pao_num_threads.restype = _c_int
        L.pao_num_threads.argtypes = []

    # -- element decoding -------------------------------------------------------------------
    def to_f64(self, bits, is_bf16: bool) -> np.ndarray:
        a = as_u16(bits)
        out = np.empty(a.shape, dtype=np.float64)
        self._L.pao_decode_elems(a.ctypes.data, a.size, int(is_bf16), out.ctypes.data)
        return out

    # -- byte ledger / addressing -----------------------------------------------------------
    def kv_bytes_per_token(self, num_kv_heads: int, head_dim: int, elem_bytes: int) -> int:
        return int(self._L.pao_kv_bytes_per_token(num_kv_heads, head_dim, elem_bytes))

    def locate(self, table_row, t: int, block_size: int):
        row = np.ascontiguousarray(np.asarray(table_row, dtype=np.int32))
        phys = ctypes.c_int32()
        off = ctypes.c_int32()
        self._L.pao_locate(row.ctypes.data, int(t), int(block_size), ctypes.byref(phys), ctypes.byref(off))
        return int(phys.value), int(off.value)

    def slot_of_token(self, table_row, t: int, block_size: int) -> int:
        row = np.ascontiguousarray(np.asarray(table_row, dtype=np.int32))
        return int(self._L.pao_slot_of_token(row.ctypes.data, int(t), int(block_size)))

    def slot_mapping(self, block_tables, context_lens, block_size: int) -> np.ndarray:
        bt = as_i32(block_tables)
        lens = as_i32(context_lens)
        S, maxb = bt.shape
        out = np.empty(S, dtype=np.int64)
        self._L.pao_slot_mapping(bt.ctypes.data, maxb, lens.ctypes.data, S, int(block_size), out.ctypes.data)
        return out

    # -- the two operations -----------------------------------------------------------------
    def cache_write(self, k, v, slots, k_cache: np.ndarray, v_cache: np.ndarray) -> None:
        """In place on the uint16 pool arrays ``k_cache``/``v_cache`` [NB, Hkv, B, D]."""
        kk, vv = as_u16(k), as_u16(v)
        sl = np.ascontiguousarray(np.asarray(slots, dtype=np.int64))
        assert k_cache.dtype == np.uint16 and k_cache.flags.c_contiguous
        assert v_cache.dtype == np.uint16 and v_cache.flags.c_contiguous
        T, H, D = kk.shape
        B = k_cache.shape[2]
        self._L.pao_cache_write(kk.ctypes.data, vv.ctypes.data, sl.ctypes.data,
                                k_cache.ctypes.data, v_cache.ctypes.data, T, H, D, B)

    def copy_blocks(self, src_k: np.ndarray, src_v: np.ndarray, dst_k: np.ndarray, dst_v: np.ndarray,
                    src_ids, dst_ids) -> int:
        """In place on the uint16 pools ``dst_k``/``dst_v`` [NB, Hkv, B, D] (they may be the
        source arrays themselves); returns how many pairs had an id outside its pool."""
        for a in (src_k, src_v, dst_k, dst_v):
            assert a.dtype == np.uint16 and a.flags.c_contiguous
        si = np.ascontiguousarray(np.asarray(src_ids, dtype=np.int32))
        di = np.ascontiguousarray(np.asarray(dst_ids, dtype=np.int32))
        assert si.shape == di.shape
        NBs, H, B, D = src_k.shape
        return int(self._L.pao_copy_blocks(src_k.ctypes.data, src_v.ctypes.data, NBs, dst_k.ctypes.data,
                                           dst_v.ctypes.data, dst_k.shape[0], si.ctypes.data, di.ctypes.data,
                                           si.size, H, B, D))

    def decode(self, q, k_cache, v_cache, block_tables, context_lens, scale: float,
               num_kv_heads: int, is_bf16: bool, num_threads: int = 0) -> np.ndarray:
        qq = as_u16(q)
        kc, vc = as_u16(k_cache), as_u16(v_cache)
        bt = as_i32(block_tables)
        lens = as_i32(context_lens)
        S, Hq, D = qq.shape
        B = kc.shape[2]
        out = np.empty((S, Hq, D), dtype=np.float64)
        rc = self._L.pao_decode(out.ctypes.data, qq.ctypes.data, kc.ctypes.data, vc.ctypes.data,
                                bt.ctypes.data, bt.shape[1], lens.ctypes.data, float(scale), S, Hq,
                                int(num_kv_heads), D, B, int(is_bf16), int(num_threads))
        if rc != 0:
            raise ValueError("oracle: arguments do not describe a valid decode problem")
        return out

    def multi_query(self, q, k_cache, v_cache, block_tables, context_lens, query_start, scale: float,
                    num_kv_heads: int, is_bf16: bool, num_threads: int = 0) -> np.ndarray:
        """Several new query tokens per sequence, causal over the paged context: q [T, Hq, D]
        with sequence s owning rows query_start[s] .. query_start[s+1]-1 (its newest tokens)."""
        qq = as_u16(q)
        kc, vc = as_u16(k_cache), as_u16(v_cache)
        bt = as_i32(block_tables)
        lens = as_i32(context_lens)
        qs = as_i32(query_start)
        T, Hq, D = qq.shape
        S = lens.size
        assert qs.size == S + 1 and int(qs[-1]) == T
        B = kc.shape[2]
        out = np.empty((T, Hq, D), dtype=np.float64)
        rc = self._L.pao_multi_query(out.ctypes.data, qq.ctypes.data, kc.ctypes.data, vc.ctypes.data,
                                     bt.ctypes.data, bt.shape[1], lens.ctypes.data, qs.ctypes.data, float(scale),
                                     S, Hq, int(num_kv_heads), D, B, int(is_bf16), int(num_threads))
        if rc != 0:
            raise ValueError("oracle: arguments do not describe a valid multi-query problem")
        return out

    def decode_runs(self, q, k_cache, v_cache, runs, seq_runs, scale: float, num_kv_heads: int, is_bf16: bool,
                    num_threads: int = 0) -> np.ndarray:
        """One query token per sequence over a context given by runs (block, slot_offset, length):
        runs int32 [R, 3], sequence s owning runs seq_runs[s] .. seq_runs[s+1]-1."""
        qq = as_u16(q)
        kc, vc = as_u16(k_cache), as_u16(v_cache)
        rr = np.ascontiguousarray(np.asarray(runs, dtype=np.int32).reshape(-1, 3))
        sr = as_i32(seq_runs)
        S, Hq, D = qq.shape
        assert sr.size == S + 1
        NB, _, B, _ = kc.shape
        out = np.empty((S, Hq, D), dtype=np.float64)
        rc = self._L.pao_decode_runs(out.ctypes.data, qq.ctypes.data, kc.ctypes.data, vc.ctypes.data, rr.ctypes.data,
                                     sr.ctypes.data, float(scale), S, Hq, int(num_kv_heads), D, B, NB, int(is_bf16),
                                     int(num_threads))
        if rc != 0:
            raise ValueError("oracle: a run leaves its block or the pool")
        return out

    def gather_runs(self, src_k: np.ndarray, src_v: np.ndarray, dst_k: np.ndarray, dst_v: np.ndarray, moves) -> int:
        """In place on the uint16 pools dst_k/dst_v; moves int32 [M, 5] = (src_block, src_off, length,
        dst_block, dst_off).  Returns how many moves were left out."""
        for a in (src_k, src_v, dst_k, dst_v):
            assert a.dtype == np.uint16 and a.flags.c_contiguous
        mv = np.ascontiguousarray(np.asarray(moves, dtype=np.int32).reshape(-1, 5))
        NBs, H, B, D = src_k.shape
        return int(self._L.pao_gather_runs(src_k.ctypes.data, src_v.ctypes.data, NBs, dst_k.ctypes.data,
                                           dst_v.ctypes.data, dst_k.shape[0], mv.ctypes.data, mv.shape[0], H, B, D))

    def num_threads(self) -> int:
        return int(self._L.pao_num_threads())


def as_u16(x) -> np.ndarray:
    """Raw 16-bit patterns of a torch fp16/bf16 tensor or numpy array, C-contiguous."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            t = x.detach().cpu().contiguous()
            if t.element_size() != 2:
                raise TypeError("expected a 16-bit tensor")
            return t.view(torch.int16).numpy().view(np.uint16)
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(x)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype.itemsize != 2:
        raise TypeError("expected 16-bit data")
    return a.view(np.uint16)


def as_i32(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().cpu().contiguous().to(torch.int32).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


_default: Optional[Oracle] = None


def get(mutant: int = 0) -> Oracle:
    """The oracle library (built on first use)."""
    global _default
    if mutant:
        return Oracle(build(mutant=mutant))
    if _default is None:
        _default = Oracle(build())
    return _default
