"""Shared helpers of the GPU parity tests: run the CUDA path and the oracle on the
same seeded workload and return what each produced."""
import numpy as np
import torch

import oracle as oracle_pkg
import paged_kv_cache_08_gb300 as pa

# Max-abs error allowed for fp16/bf16 outputs accumulated in fp32, against the fp64 oracle.
# fp16 outputs are held to the raw error |out - ref| <= TOL: half an fp16 ulp stays below 2e-3
# up to |o| < 8, and an output is a convex combination of V rows.  A bf16 value stands for every
# real number within half a unit in its last place -- up to 1.95e-3 in [0.5, 1) and 3.9e-3 in
# [1, 2) -- which no kernel can beat, so a bf16 element passes when
# |out - ref| <= TOL + ulp(out) / 2.
TOL = 2e-3


def run_cuda(wl, layer=0, tokens_per_split=0, math="auto", stream=None, num_ctas=0):
    dev = torch.device("cuda")
    kc = wl.k_cache[layer].to(dev).clone()
    vc = wl.v_cache[layer].to(dev).clone()
    bt = wl.block_tables.to(dev)
    lens = wl.context_lens.to(dev)
    slots = torch.from_numpy(pa.build_slot_mapping(wl.block_tables, wl.context_lens, wl.block_size)).to(dev)
    pa.cache_write(wl.k_new[layer].to(dev), wl.v_new[layer].to(dev), slots, kc, vc, stream=stream)
    out = pa.decode(wl.q[layer].to(dev), kc, vc, bt, lens, wl.scale, wl.num_kv_heads,
                    tokens_per_split=tokens_per_split, math=math, num_ctas=num_ctas, stream=stream)
    torch.cuda.synchronize()
    return kc, vc, out


def run_oracle(oracle, wl, layer=0):
    kc = oracle_pkg.as_u16(wl.k_cache[layer]).copy()
    vc = oracle_pkg.as_u16(wl.v_cache[layer]).copy()
    slots = oracle.slot_mapping(wl.block_tables, wl.context_lens, wl.block_size)
    oracle.cache_write(wl.k_new[layer], wl.v_new[layer], slots, kc, vc)
    ref = oracle.decode(wl.q[layer], kc, vc, wl.block_tables, wl.context_lens, wl.scale, wl.num_kv_heads,
                        wl.dtype == "bf16")
    return kc, vc, ref


def half_ulp(out: torch.Tensor) -> np.ndarray:
    """Half the spacing from |out| to the next representable magnitude of out's dtype."""
    bits = oracle_pkg.as_u16(out.detach().cpu()).astype(np.uint32) & 0x7FFF
    if out.dtype == torch.bfloat16:
        lo = (bits << 16).view(np.float32).astype(np.float64)
        hi = ((bits + 1) << 16).view(np.float32).astype(np.float64)
    else:
        lo = bits.astype(np.uint16).view(np.float16).astype(np.float64)
        hi = (bits + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    return (hi - lo) / 2


def rounding_allowance(out: torch.Tensor) -> np.ndarray:
    """Per element, the part of the output's own rounding that TOL does not cover: half an ulp
    for bf16 outputs, 0 for fp16."""
    if out.dtype != torch.bfloat16:
        return np.zeros(tuple(out.shape))
    return half_ulp(out)


def max_abs_err(out: torch.Tensor, ref: np.ndarray) -> float:
    """Largest error against the fp64 reference, less the rounding allowance of bf16 outputs
    (compare with TOL); for fp16 this is the raw max-abs error."""
    got = out.detach().float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all(), "non-finite output"
    if not ref.size:
        return 0.0
    return float(np.max(np.abs(got - ref) - rounding_allowance(out)))


def raw_max_abs_err(out: torch.Tensor, ref: np.ndarray) -> float:
    got = out.detach().float().cpu().numpy().astype(np.float64)
    return float(np.max(np.abs(got - ref))) if ref.size else 0.0


def u16(t: torch.Tensor) -> np.ndarray:
    return oracle_pkg.as_u16(t.cpu())
