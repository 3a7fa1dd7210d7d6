"""GPU parity of the paged cache write: bit-exact against the oracle's scatter,
canary rows untouched, padding slots skipped, out-of-pool slots flagged."""
import numpy as np
import pytest
import torch

import paged_kv_cache_08_gb300 as pa
import workloads
from gpu_util import u16

pytestmark = pytest.mark.gpu


def _write_both(oracle, k, v, slots, kc, vc):
    dev = torch.device("cuda")
    gk, gv = kc.to(dev).clone(), vc.to(dev).clone()
    pa.cache_write(k.to(dev), v.to(dev), torch.as_tensor(slots, dtype=torch.int64).to(dev), gk, gv)
    torch.cuda.synchronize()
    ok, ov = u16(kc).copy(), u16(vc).copy()
    oracle.cache_write(k, v, slots, ok, ov)
    return gk, gv, ok, ov


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_cache_write_bit_exact(oracle, cfg):
    wl = workloads.config(cfg, layers=1)
    slots = pa.build_slot_mapping(wl.block_tables, wl.context_lens, wl.block_size)
    gk, gv, ok, ov = _write_both(oracle, wl.k_new[0], wl.v_new[0], slots, wl.k_cache[0], wl.v_cache[0])
    assert np.array_equal(u16(gk), ok) and np.array_equal(u16(gv), ov)
    assert pa.read_device_status(clear=True) == 0


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("B", [1, 16, 48, 128])
def test_canary_and_padding(oracle, dtype, B):
    """Every slot of a canary-filled pool is written at most once; negative slots skip."""
    tdt = torch.float16 if dtype == "f16" else torch.bfloat16
    H, D, T = 3, 128, 40
    NB = max(9, (T + B - 1) // B + 2)
    g = torch.Generator().manual_seed(B)
    canary = torch.full((NB, H, B, D), 0.5, dtype=tdt)
    k = torch.randn((T, H, D), generator=g).to(tdt)
    v = torch.randn((T, H, D), generator=g).to(tdt)
    slots = torch.randperm(NB * B, generator=g)[:T].to(torch.int64)
    slots[::7] = -1                                  # padding rows
    gk, gv, ok, ov = _write_both(oracle, k, v, slots.numpy(), canary, canary)
    assert np.array_equal(u16(gk), ok) and np.array_equal(u16(gv), ov)
    untouched = np.ones((NB * B,), dtype=bool)
    untouched[slots[slots >= 0].numpy()] = False
    flat = u16(gk).reshape(NB, H, B, D).transpose(0, 2, 1, 3).reshape(NB * B, H, D)
    assert (flat[untouched] == u16(canary)[0, 0, 0, 0]).all()


def test_out_of_pool_slot_is_flagged(oracle):
    NB, H, D, B = 4, 2, 128, 16
    canary = torch.zeros((NB, H, B, D), dtype=torch.float16)
    k = torch.ones((3, H, D), dtype=torch.float16)
    slots = np.array([0, NB * B + 3, 5], dtype=np.int64)
    pa.read_device_status(clear=True)
    dev = torch.device("cuda")
    gk, gv = canary.to(dev).clone(), canary.to(dev).clone()
    pa.cache_write(k.to(dev), k.to(dev), torch.from_numpy(slots).to(dev), gk, gv)
    assert pa.read_device_status(clear=True) & 0x4
    ok = u16(canary).copy()
    ov = ok.copy()
    oracle.cache_write(k, k, np.array([0, -1, 5], np.int64), ok, ov)  # the bad row is skipped
    assert np.array_equal(u16(gk), ok)
