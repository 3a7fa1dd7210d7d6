"""Seeded synthetic inputs for paged decode attention and the paged cache write.

This module is shared by the CUDA path and by the CPU oracle, so it holds no
arithmetic of the method itself: no attention, no slot computation, no
address arithmetic.  It only draws the random structure (context lengths, a
fragmented physical pool expressed as a random permutation of block ids) and
the random values (q, the pool contents, the new token's K/V).

Shapes follow the pages:
  * cache pools ``k_cache``/``v_cache``: ``[num_blocks, num_kv_heads, block_size, head_dim]``
    -- one contiguous (block, kv-head) tile of ``block_size * head_dim``
    elements, as the paged layout of "显存虚拟化革命：PagedAttention 内存池管理与显存碎片终结",
    §三.1 "物理张量在 GPU 上的真实内存布局" keeps each physical block in one
    fixed stride of two big pool tensors;
  * ``block_tables``: int32 ``[num_seqs, max_blocks_per_seq]`` (same page, §五.1), unused
    entries hold -1;
  * ``context_lens``: int32 ``[num_seqs]``; the length counts the new token,
    whose K/V (``k_new``/``v_new``, ``[num_seqs, num_kv_heads, head_dim]``) is
    written before decode reads the cache;
  * ``q``: ``[num_seqs, num_q_heads, head_dim]``.

Values are N(0, 1) rounded to fp16 or bf16, including pool slots that no
sequence owns, so that a wrong index yields wrong numbers instead of zeros.
Structure (lengths, permutation) is always drawn on the CPU from
``torch.Generator().manual_seed(seed)``; bulk values are drawn on the
requested device from a generator seeded with the same seed.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class Workload:
    name: str
    dtype: str                    # "f16" | "bf16"
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    context_lens: torch.Tensor    # int32 [S] (CPU)
    block_tables: torch.Tensor    # int32 [S, max_blocks_per_seq] (CPU)
    scale: float
    seed: int
    # one entry per layer; every layer shares the block tables and lengths
    q: List[torch.Tensor] = field(default_factory=list)
    k_cache: List[torch.Tensor] = field(default_factory=list)
    v_cache: List[torch.Tensor] = field(default_factory=list)
    k_new: List[torch.Tensor] = field(default_factory=list)
    v_new: List[torch.Tensor] = field(default_factory=list)
    shared_prefix_blocks: int = 0  # leading table entries shared by every sequence

    @property
    def layers(self) -> int:
        return len(self.q)

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    @property
    def elem_bytes(self) -> int:
        return 2

    def kv_bytes_per_token_per_layer(self) -> int:
        """Bytes one token occupies in one layer's pools, read off the tensors."""
        kc = self.k_cache[0]
        per_token_k = kc.element_size() * kc.shape[1] * kc.shape[3]
        return 2 * per_token_k

    def block_bytes_per_layer(self) -> int:
        kc = self.k_cache[0]
        return 2 * kc.element_size() * kc.shape[1] * kc.shape[2] * kc.shape[3]

    def total_context_tokens(self) -> int:
        return int(self.context_lens.to(torch.int64).sum())


def _fill_normal(shape, dtype: torch.dtype, gen: torch.Generator, device) -> torch.Tensor:
    """N(0,1) values rounded to ``dtype``, drawn in slabs to bound fp32 scratch."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    slab = 1 << 24
    for i in range(0, flat.numel(), slab):
        n = min(slab, flat.numel() - i)
        flat[i:i + n] = torch.randn(n, generator=gen, device=device, dtype=torch.float32).to(dtype)
    return out


def _blocks_needed(lens: Sequence[int], block_size: int) -> List[int]:
    return [(int(n) + block_size - 1) // block_size for n in lens]


def make_workload(name: str, *, context_lens: Sequence[int], num_q_heads: int, num_kv_heads: int,
                  head_dim: int = 128, block_size: int = 16, dtype: str = "f16", seed: int = 0,
                  num_blocks: Optional[int] = None, pool_factor: float = 1.2,
                  max_context: Optional[int] = None, layers: int = 1,
                  shared_prefix_tokens: int = 0, device="cpu", gen: Optional[torch.Generator] = None,
                  scale: Optional[float] = None, values: bool = True) -> Workload:
    """Build one seeded workload.

    ``shared_prefix_tokens`` (a multiple of ``block_size``) makes the first
    ``shared_prefix_tokens / block_size`` table entries of every sequence name
    the same physical blocks; each ``context_lens`` entry then includes the
    prefix.  Physical ids come from a seeded random permutation of the pool,
    taken in order: the prefix first, then each sequence's private blocks.
    ``values=False`` draws only the structure (lengths, tables), no tensors.
    """
    if gen is None:
        gen = torch.Generator().manual_seed(seed)
    lens = [int(x) for x in context_lens]
    S = len(lens)
    B = block_size
    if shared_prefix_tokens % B:
        raise ValueError("shared prefix must be a whole number of blocks")
    n_prefix = shared_prefix_tokens // B
    private = _blocks_needed([max(0, n - shared_prefix_tokens) for n in lens], B)
    need = n_prefix + sum(private)
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(pool_factor * need)))
    if num_blocks < need:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {need}")
    if max_context is None:
        max_context = max(lens) if lens else 1
    max_blocks = max(1, (max_context + B - 1) // B)
    perm = torch.randperm(num_blocks, generator=gen).to(torch.int32)
    tables = torch.full((S, max_blocks), -1, dtype=torch.int32)
    prefix_ids = perm[:n_prefix]
    cursor = n_prefix
    for s in range(S):
        tables[s, :n_prefix] = prefix_ids
        k = private[s]
        tables[s, n_prefix:n_prefix + k] = perm[cursor:cursor + k]
        cursor += k
    wl = Workload(name=name, dtype=dtype, num_seqs=S, num_q_heads=num_q_heads,
                  num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=B,
                  num_blocks=num_blocks, max_blocks_per_seq=max_blocks,
                  context_lens=torch.tensor(lens, dtype=torch.int32), block_tables=tables,
                  scale=(1.0 / math.sqrt(head_dim)) if scale is None else float(scale),
                  seed=seed, shared_prefix_blocks=n_prefix)
    tdt = DTYPES[dtype]
    dev = torch.device(device)
    vgen = gen if dev.type == "cpu" else torch.Generator(device=dev).manual_seed(seed)
    for _ in range(layers if values else 0):
        wl.q.append(_fill_normal((S, num_q_heads, head_dim), tdt, vgen, dev))
        wl.k_cache.append(_fill_normal((num_blocks, num_kv_heads, B, head_dim), tdt, vgen, dev))
        wl.v_cache.append(_fill_normal((num_blocks, num_kv_heads, B, head_dim), tdt, vgen, dev))
        wl.k_new.append(_fill_normal((S, num_kv_heads, head_dim), tdt, vgen, dev))
        wl.v_new.append(_fill_normal((S, num_kv_heads, head_dim), tdt, vgen, dev))
    return wl


# --------------------------------------------------------------------------------------------
# The five named workloads.  Shapes come from the pages: the 1.1B edge model of
# "端侧 SLM 显存保活术" (24 layers, 12 q / 2 kv heads, head dim 128, fp16, 16-token
# blocks; section "KV Cache 的物理膨胀账本"), the Llama-2-7B shape of the KV-cache /
# BlockManager tutorial (32 layers x 32 heads x 128, P90 context 287; sections 2.1
# and 3.1), and the block sizes 16/32/64/128 of that tutorial's block-size table.
# --------------------------------------------------------------------------------------------

CONFIG_NAMES = {
    1: "tiny_decode_4seq_ctx7-64_gqa12x2_f16_B16",
    2: "edge1p1b_64seq_ctx16-2048_gqa12x2_f16_B16_x24layers",
    3: "llama2_7b_256seq_lognormal_p90_287_mha32_f16_B32",
    4: "longctx_16seq_ctx16384_gqa32x8_bf16_B64",
    5: "shared_prefix_128seq_1024+tail_gqa12x2_f16",
}


def _lognormal_lens(S: int, gen: torch.Generator, p90: float = 287.0, sigma: float = 0.75,
                    lo: int = 1, hi: int = 4096) -> List[int]:
    # median chosen so that exp(mu + 1.2816 sigma) = p90 (1.2816 = 90th percentile of N(0,1))
    mu = math.log(p90) - 1.2815515655446004 * sigma
    z = torch.randn(S, generator=gen, dtype=torch.float64)
    lens = torch.exp(mu + sigma * z).round().clamp(lo, hi).to(torch.int64)
    return [int(x) for x in lens]


def config(cfg: int, *, device="cpu", layers: Optional[int] = None, block_size: Optional[int] = None,
           num_seqs: Optional[int] = None, values: bool = True) -> Workload:
    """The five seeded configurations.  ``layers``/``num_seqs`` may shrink a
    config for a bounded sample; ``block_size`` picks the config-5 sweep point."""
    if cfg == 1:
        seed = 1001
        gen = torch.Generator().manual_seed(seed)
        lens = [7, 16, 33, 64]
        return make_workload(CONFIG_NAMES[1], context_lens=lens, num_q_heads=12, num_kv_heads=2,
                             block_size=16, dtype="f16", seed=seed, num_blocks=32, max_context=64,
                             layers=layers or 1, device=device, gen=gen, values=values)
    if cfg == 2:
        seed = 1002
        gen = torch.Generator().manual_seed(seed)
        S = 64
        lens = [int(x) for x in torch.randint(16, 2049, (S,), generator=gen)]
        if num_seqs is not None:
            lens = lens[:num_seqs]
        return make_workload(CONFIG_NAMES[2], context_lens=lens, num_q_heads=12, num_kv_heads=2,
                             block_size=16, dtype="f16", seed=seed, max_context=2048,
                             layers=24 if layers is None else layers, device=device, gen=gen, values=values)
    if cfg == 3:
        seed = 1003
        gen = torch.Generator().manual_seed(seed)
        lens = _lognormal_lens(256, gen)
        if num_seqs is not None:
            lens = lens[:num_seqs]
        return make_workload(CONFIG_NAMES[3], context_lens=lens, num_q_heads=32, num_kv_heads=32,
                             block_size=32, dtype="f16", seed=seed, max_context=4096,
                             layers=layers or 1, device=device, gen=gen, values=values)
    if cfg == 4:
        seed = 1004
        gen = torch.Generator().manual_seed(seed)
        S = 16 if num_seqs is None else num_seqs
        return make_workload(CONFIG_NAMES[4], context_lens=[16384] * S, num_q_heads=32,
                             num_kv_heads=8, block_size=64, dtype="bf16", seed=seed,
                             max_context=16384, layers=layers or 1, device=device, gen=gen, values=values)
    if cfg == 5:
        B = 16 if block_size is None else block_size
        if B not in (16, 32, 64, 128):
            raise ValueError("config 5 sweeps block sizes 16/32/64/128")
        seed = 1005 + B
        gen = torch.Generator().manual_seed(seed)
        S = 128
        tails = [int(x) for x in torch.randint(1, 513, (S,), generator=gen)]
        if num_seqs is not None:
            tails = tails[:num_seqs]
        lens = [1024 + t for t in tails]
        return make_workload(f"{CONFIG_NAMES[5]}_B{B}", context_lens=lens, num_q_heads=12,
                             num_kv_heads=2, block_size=B, dtype="f16", seed=seed,
                             max_context=1024 + 512, shared_prefix_tokens=1024,
                             layers=layers or 1, device=device, gen=gen, values=values)
    raise ValueError(f"unknown config {cfg}")


def to_device(wl: Workload, device) -> Workload:
    """A copy of ``wl`` whose per-layer tensors live on ``device`` (structure stays on CPU)."""
    out = Workload(**{k: getattr(wl, k) for k in ("name", "dtype", "num_seqs", "num_q_heads",
                                                   "num_kv_heads", "head_dim", "block_size",
                                                   "num_blocks", "max_blocks_per_seq",
                                                   "context_lens", "block_tables", "scale", "seed",
                                                   "shared_prefix_blocks")})
    for key in ("q", "k_cache", "v_cache", "k_new", "v_new"):
        setattr(out, key, [t.to(device) for t in getattr(wl, key)])
    return out


def multi_query_inputs(wl: Workload, new_tokens: Sequence[int], seed: int, device=None):
    """Queries for several new tokens per sequence: ``new_tokens[s]`` rows for sequence s
    (its newest tokens, already part of its context), drawn N(0, 1) in the workload's dtype.
    Returns (q [T, num_q_heads, head_dim], query_start int32 [S + 1], max new tokens)."""
    assert len(new_tokens) == wl.num_seqs
    starts = [0]
    for n in new_tokens:
        starts.append(starts[-1] + int(n))
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn((starts[-1], wl.num_q_heads, wl.head_dim), generator=gen).to(wl.torch_dtype)
    qs = torch.tensor(starts, dtype=torch.int32)
    if device is not None:
        q, qs = q.to(device), qs.to(device)
    return q, qs, max([int(n) for n in new_tokens] + [1])


def new_token_rows(wl: Workload, num_rows: int, seed: int, device=None):
    """K and V rows of ``num_rows`` new tokens ([num_rows, num_kv_heads, head_dim] each), drawn
    N(0, 1) in the workload's dtype from their own seeded generator."""
    gen = torch.Generator().manual_seed(seed)
    shape = (num_rows, wl.num_kv_heads, wl.head_dim)
    k = torch.randn(shape, generator=gen).to(wl.torch_dtype)
    v = torch.randn(shape, generator=gen).to(wl.torch_dtype)
    if device is not None:
        k, v = k.to(device), v.to(device)
    return k, v
