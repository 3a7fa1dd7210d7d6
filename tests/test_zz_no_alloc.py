"""pa_decode_static: the allocation-free form of pa_decode.

It serves callers that cannot allocate device memory (a plugin inside a host
framework that owns the GPU's memory pool, real-time deployments that forbid
allocation after start-up): its scratch is a fixed device array inside the
library.  Called through the C ABI twice in a row, its output must match
pa_decode's (the entry point with a caller workspace) and the fp64 oracle's,
each within the parity tolerance; a problem too large for the fixed array is
refused.

This file is collected last on purpose, so that a run that stops at the first
failure has already run every other test; it does not depend on them.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_08_gb300 as pa
import workloads
from gpu_util import TOL, half_ulp, max_abs_err

pytestmark = pytest.mark.gpu


def _static_decode(wl, dev, out):
    lib = pa.lib()
    q = wl.q[0].to(dev)
    kc = wl.k_cache[0].to(dev)
    vc = wl.v_cache[0].to(dev)
    bt = wl.block_tables.to(dev)
    lens = wl.context_lens.to(dev)
    S, Hq, D = q.shape
    rc = lib.pa_decode_static(out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(),
                              lens.data_ptr(), ctypes.c_float(wl.scale), wl.num_kv_heads, S, Hq, D,
                              wl.block_size, wl.num_blocks, wl.max_blocks_per_seq,
                              1 if wl.dtype == "bf16" else 0, torch.cuda.current_stream().cuda_stream)
    return rc


def _reference(wl, dev):
    return pa.decode(wl.q[0].to(dev), wl.k_cache[0].to(dev), wl.v_cache[0].to(dev), wl.block_tables.to(dev),
                     wl.context_lens.to(dev), wl.scale, wl.num_kv_heads)


def _excess(a: torch.Tensor, b: torch.Tensor) -> float:
    d = np.abs(a.float().cpu().numpy().astype(np.float64) - b.float().cpu().numpy().astype(np.float64))
    return float(np.max(d - half_ulp(b)))


def _oracle_decode(oracle, wl):
    import oracle as oracle_pkg
    kc = oracle_pkg.as_u16(wl.k_cache[0])
    vc = oracle_pkg.as_u16(wl.v_cache[0])
    return oracle.decode(wl.q[0], kc, vc, wl.block_tables, wl.context_lens, wl.scale, wl.num_kv_heads,
                         wl.dtype == "bf16")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_static_matches_workspace_entry_point_twice(oracle, dtype):
    dev = torch.device("cuda")
    # long and short contexts, so that the persistent kernel cuts sequences between CTAs and
    # merges their pieces through the scratch counters
    wl = workloads.make_workload("no_alloc", context_lens=[1, 700, 64, 65, 2048, 0, 130, 1030, 5, 333],
                                 num_q_heads=12, num_kv_heads=2, block_size=16, dtype=dtype, seed=41,
                                 max_context=2048)
    ref = _reference(wl, dev)
    exact = _oracle_decode(oracle, wl)
    torch.cuda.synchronize()
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        rc = _static_decode(wl, dev, out)
        assert rc == 0, pa.lib().pa_status_string(rc)
        torch.cuda.synchronize()
        err = _excess(out, ref)
        assert err <= TOL, f"call {call}: max abs difference {err:.3e} beyond rounding > {TOL}"
        # against the fp64 oracle too, so that a fault both entry points share cannot pass
        err = max_abs_err(out, exact)
        assert err <= TOL, f"call {call}: max abs error against the oracle {err:.3e} > {TOL}"


def test_static_refuses_problems_beyond_its_scratch():
    dev = torch.device("cuda")
    lib = pa.lib()
    # 1024 sequences x 4096 kv heads: the persistent kernel's pieces plus one arrival counter
    # per (sequence, kv head) need more than the fixed scratch; the call must refuse before
    # launching anything
    S, Hq, Hkv, D, B, maxb = 1024, 4096, 4096, 128, 16, 4
    need = pa.decode_workspace_size(S, Hq, Hkv, D, B, maxb)
    assert need > (16 << 20)
    dummy = torch.zeros(16, dtype=torch.float16, device=dev)
    tbl = torch.zeros(16, dtype=torch.int32, device=dev)
    before = pa.kernel_launch_count()
    rc = lib.pa_decode_static(dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(),
                              tbl.data_ptr(), tbl.data_ptr(), ctypes.c_float(0.1), Hkv, S, Hq, D, B, 4, maxb, 0,
                              torch.cuda.current_stream().cuda_stream)
    assert rc == -8, pa.lib().pa_status_string(rc)
    assert pa.kernel_launch_count() == before
