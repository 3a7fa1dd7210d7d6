"""GPU parity of pa_copy_blocks: copy-on-write inside the cache and swap out to / in from a
pinned host pool, bit-exact against the oracle's block copy; the copy-on-write fork of the
PagedAttention explainer page run end to end (pool bookkeeping, block copy, cache write,
decode) against the oracle; ids outside a pool flagged; pageable host memory refused."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_08_gb300 as pa
import workloads
from gpu_util import TOL, max_abs_err, u16

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(autouse=True)
def _clean_status():
    pa.read_device_status(clear=True)
    yield


def _pool(NB, H, B, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn((NB, H, B, 128), generator=g).to(DT[dtype]),
            torch.randn((NB, H, B, 128), generator=g).to(DT[dtype]))


def _pairs(NB, n, seed):
    """n (src, dst) pairs with distinct destinations that are nobody's source."""
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(NB, generator=g)
    dst = perm[:n]
    src = perm[n:][torch.randint(0, NB - n, (n,), generator=g)]
    return src.to(torch.int32), dst.to(torch.int32)


def _oracle_copy(oracle, sk, sv, dk, dv, src, dst):
    ok, ov = u16(dk).copy(), u16(dv).copy()
    same = sk is dk
    a, b = (ok, ov) if same else (u16(sk).copy(), u16(sv).copy())
    left = oracle.copy_blocks(a, b, ok, ov, src.numpy(), dst.numpy())
    return ok, ov, left


@pytest.mark.parametrize("H,B,dtype", [(2, 16, "f16"), (32, 32, "f16"), (8, 64, "bf16"), (2, 128, "f16"),
                                       (1, 16, "bf16")])
@pytest.mark.parametrize("n", [1, 7, 300])
def test_copy_within_pool_bit_exact(oracle, H, B, dtype, n):
    NB = max(2 * n + 3, 40)
    kc, vc = _pool(NB, H, B, dtype, seed=H * 1000 + B + n)
    src, dst = _pairs(NB, n, seed=n + B)
    dev = torch.device("cuda")
    gk, gv = kc.to(dev), vc.to(dev)
    pa.copy_blocks(gk, gv, gk, gv, src.to(dev), dst.to(dev))
    torch.cuda.synchronize()
    ok, ov, left = _oracle_copy(oracle, kc, vc, kc, vc, src, dst)
    assert left == 0
    assert np.array_equal(u16(gk), ok) and np.array_equal(u16(gv), ov)
    assert pa.read_device_status(clear=True) == 0


def test_copy_full_size_pool(oracle):
    """The 1.1B-shape layer pool (64 sequences, contexts up to 2048, B = 16): 1500 pairs."""
    wl = workloads.config(2, layers=1)
    kc, vc = wl.k_cache[0], wl.v_cache[0]
    src, dst = _pairs(wl.num_blocks, 1500, seed=5)
    dev = torch.device("cuda")
    gk, gv = kc.to(dev), vc.to(dev)
    before = pa.kernel_launch_count()
    pa.copy_blocks(gk, gv, gk, gv, src.to(dev), dst.to(dev))
    torch.cuda.synchronize()
    assert pa.kernel_launch_count() - before == 1
    ok, ov, _ = _oracle_copy(oracle, kc, vc, kc, vc, src, dst)
    assert np.array_equal(u16(gk), ok) and np.array_equal(u16(gv), ov)


def test_ids_outside_the_pool_are_skipped_and_flagged(oracle):
    NB, H, B = 20, 2, 16
    kc, vc = _pool(NB, H, B, "f16", seed=3)
    src = torch.tensor([1, NB, 4, -1, 6], dtype=torch.int32)
    dst = torch.tensor([10, 11, NB + 3, 12, 13], dtype=torch.int32)
    dev = torch.device("cuda")
    gk, gv = kc.to(dev), vc.to(dev)
    pa.copy_blocks(gk, gv, gk, gv, src.to(dev), dst.to(dev))
    torch.cuda.synchronize()
    assert pa.read_device_status(clear=True) & pa._native.DEV_BAD_BLOCK_ID
    ok, ov, left = _oracle_copy(oracle, kc, vc, kc, vc, src, dst)
    assert left == 3
    assert np.array_equal(u16(gk), ok) and np.array_equal(u16(gv), ov)


def test_empty_copy_launches_nothing():
    dev = torch.device("cuda")
    k = torch.zeros((4, 2, 16, 128), dtype=torch.float16, device=dev)
    ids = torch.zeros(0, dtype=torch.int32, device=dev)
    before = pa.kernel_launch_count()
    pa.copy_blocks(k, k, k, k, ids, ids)
    assert pa.kernel_launch_count() == before


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_swap_out_and_in_through_pinned_host_pool(oracle, dtype):
    """Blocks of one sequence go to a pinned host pool (0.3 x the device pool) and come back to
    other device blocks; host and device pools match the oracle bit for bit, and decode through
    the rewritten table gives the same output as before the move, bit for bit."""
    wl = workloads.make_workload(f"swap_{dtype}", context_lens=[300, 1000, 77, 513], num_q_heads=12, num_kv_heads=2,
                                 block_size=16, dtype=dtype, seed=17, max_context=1024, pool_factor=1.6)
    dev = torch.device("cuda")
    NB = wl.num_blocks
    dev_pool, host_pool = pa.BlockPool(NB), pa.BlockPool(int(0.3 * NB))
    tables = wl.block_tables.numpy().copy()
    used = sorted(set(int(x) for x in tables[tables >= 0].ravel()))
    # the device pool's bookkeeping mirrors the generated tables: hold exactly the used ids
    held = [dev_pool.alloc() for _ in range(NB)]
    for i in held:
        if i not in used:
            dev_pool.decref(i)
    kc, vc = wl.k_cache[0].to(dev), wl.v_cache[0].to(dev)
    bt, lens = wl.block_tables.to(dev), wl.context_lens.to(dev)
    out_before = pa.decode(wl.q[0].to(dev), kc, vc, bt, lens, wl.scale, wl.num_kv_heads)
    hk = torch.zeros((host_pool.num_blocks, 2, 16, 128), dtype=DT[dtype]).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    victim = 3                                  # 513 tokens: 33 blocks, within the host pool
    row = np.ascontiguousarray(tables[victim])
    n = (int(wl.context_lens[victim]) + 15) // 16
    src, dst = dev_pool.move_blocks(host_pool, row, n)
    pa.copy_blocks(kc, vc, hk, hv, torch.from_numpy(src).to(dev), torch.from_numpy(dst).to(dev))
    torch.cuda.synchronize()
    ok, ov, _ = _oracle_copy(oracle, wl.k_cache[0], wl.v_cache[0], torch.zeros_like(hk), torch.zeros_like(hv),
                             torch.from_numpy(src), torch.from_numpy(dst))
    assert np.array_equal(u16(hk), ok) and np.array_equal(u16(hv), ov)
    # swap in: the pinned ids may live in host memory too
    hsrc, hdst = host_pool.move_blocks(dev_pool, row, n)
    sid = torch.from_numpy(hsrc).pin_memory()
    did = torch.from_numpy(hdst).pin_memory()
    pa.copy_blocks(hk, hv, kc, vc, sid, did)
    torch.cuda.synchronize()
    tables[victim] = row
    bt2 = torch.from_numpy(tables).to(dev)
    out_after = pa.decode(wl.q[0].to(dev), kc, vc, bt2, lens, wl.scale, wl.num_kv_heads)
    torch.cuda.synchronize()
    assert set(hdst.tolist()).isdisjoint(set(used) - set(src.tolist())), "swap-in reused a live block"
    assert torch.equal(out_before.view(torch.int16), out_after.view(torch.int16))
    assert pa.read_device_status(clear=True) == 0


def test_pageable_host_memory_is_refused():
    dev = torch.device("cuda")
    kc = torch.zeros((4, 2, 16, 128), dtype=torch.float16, device=dev)
    host = torch.zeros((4, 2, 16, 128), dtype=torch.float16)   # pageable
    ids = torch.zeros(1, dtype=torch.int32, device=dev)
    with pytest.raises(TypeError):
        pa.copy_blocks(kc, kc, host, host, ids, ids)
    rc = pa.lib().pa_copy_blocks(kc.data_ptr(), kc.data_ptr(), 4, host.data_ptr(), host.data_ptr(), 4,
                                 ids.data_ptr(), ids.data_ptr(), 1, 2, 128, 16, 0,
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == -1


@pytest.mark.parametrize("fused", [False, True])
def test_copy_on_write_fork_end_to_end(oracle, fused):
    """Parallel sampling (§四): 6 branches forked from prompts of several lengths share the
    prompt blocks; every branch appends one token.  The pool reports the copy-on-write pairs,
    the GPU copies them, writes the new rows and decodes; the oracle does the same with its own
    block copy, cache write and decode."""
    B, H, G, D = 16, 2, 6, 128
    prompts = [37, 48, 5, 16]
    branches_per_prompt = [2, 1, 2, 1]
    NB = 64
    g = torch.Generator().manual_seed(2024)
    kc = torch.randn((NB, H, B, D), generator=g).to(torch.float16)
    vc = torch.randn((NB, H, B, D), generator=g).to(torch.float16)
    pool = pa.BlockPool(NB)
    maxb = 8
    rows, lens = [], []
    for P, nb in zip(prompts, branches_per_prompt):
        base = np.full(maxb, -1, dtype=np.int32)
        pool.assign(base, P, B)
        rows.append(base)
        lens.append(P)
        for _ in range(nb):
            r = np.full(maxb, -1, dtype=np.int32)
            pool.assign(r, P, B, shared_row=base, shared_blocks=(P + B - 1) // B)
            rows.append(r)
            lens.append(P)
    S = len(rows)
    slots, src, dst = [], [], []
    for r, L in zip(rows, lens):
        slot, s_id, d_id = pool.append_token(r, L, B)
        slots.append(slot)
        if s_id >= 0:
            src.append(s_id)
            dst.append(d_id)
    assert len(src) >= 3, "the fork must exercise copy-on-write"
    tables = torch.from_numpy(np.stack(rows))
    ctx = torch.tensor([L + 1 for L in lens], dtype=torch.int32)
    q = torch.randn((S, H * G, D), generator=g).to(torch.float16)
    k_new = torch.randn((S, H, D), generator=g).to(torch.float16)
    v_new = torch.randn((S, H, D), generator=g).to(torch.float16)
    scale = 1.0 / np.sqrt(D)
    dev = torch.device("cuda")
    gk, gv = kc.to(dev), vc.to(dev)
    s_t, d_t = torch.tensor(src, dtype=torch.int32), torch.tensor(dst, dtype=torch.int32)
    pa.copy_blocks(gk, gv, gk, gv, s_t.to(dev), d_t.to(dev))
    if fused:
        # default options: no early reads, so the append reads the copied rows only after the
        # copy kernel before it in the stream has finished
        out = pa.decode_append(q.to(dev), k_new.to(dev), v_new.to(dev), gk, gv, tables.to(dev), ctx.to(dev), scale, H)
    else:
        pa.cache_write(k_new.to(dev), v_new.to(dev), torch.tensor(slots, dtype=torch.int64).to(dev), gk, gv)
        out = pa.decode(q.to(dev), gk, gv, tables.to(dev), ctx.to(dev), scale, H)
    torch.cuda.synchronize()
    ok, ov = u16(kc).copy(), u16(vc).copy()
    assert oracle.copy_blocks(ok, ov, ok, ov, s_t.numpy(), d_t.numpy()) == 0
    oslots = oracle.slot_mapping(tables, ctx, B)
    assert list(oslots) == slots
    oracle.cache_write(k_new, v_new, oslots, ok, ov)
    ref = oracle.decode(q, ok, ov, tables, ctx, scale, H, False)
    assert np.array_equal(u16(gk), ok) and np.array_equal(u16(gv), ov)
    err = max_abs_err(out, ref)
    assert err <= TOL, f"max abs error {err:.3e}"
    assert pa.read_device_status(clear=True) == 0
