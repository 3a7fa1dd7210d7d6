"""GPU parity of the slotted-block paths: decode over contexts given as runs (block_id,
slot_offset, length) against the oracle, runs of whole blocks against the block-table decode,
row-run moves bit for bit, and compaction of slotted contexts into whole blocks (online
defragmentation) followed by the ordinary decode."""
import numpy as np
import pytest
import torch

import oracle as oracle_pkg
import paged_kv_cache_08_gb300 as pa
import workloads
from gpu_util import TOL, max_abs_err, u16

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(autouse=True)
def _clean_status():
    pa.read_device_status(clear=True)
    yield


def _slotted(lens, B, NB, seed):
    """Random runs: each sequence's context cut into pieces of random length, each piece at a
    random offset of a random block (pieces may share blocks; rows are read-only here)."""
    g = torch.Generator().manual_seed(seed)
    runs, seq_runs = [], [0]
    for L in lens:
        t = 0
        while t < L:
            ln = int(torch.randint(1, B + 1, (1,), generator=g))
            ln = min(ln, L - t)
            off = int(torch.randint(0, B - ln + 1, (1,), generator=g))
            blk = int(torch.randint(0, NB, (1,), generator=g))
            runs.append((blk, off, ln))
            t += ln
        seq_runs.append(len(runs))
    return np.array(runs, np.int32).reshape(-1, 3), np.array(seq_runs, np.int32)


def _pools(NB, H, B, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn((NB, H, B, 128), generator=g).to(DT[dtype]),
            torch.randn((NB, H, B, 128), generator=g).to(DT[dtype]))


@pytest.mark.parametrize("G,B,dtype", [(6, 16, "f16"), (1, 32, "f16"), (4, 64, "bf16"), (8, 16, "bf16"),
                                       (2, 128, "f16"), (3, 16, "f16")])
def test_decode_runs_parity(oracle, G, B, dtype):
    lens = [1, 5, 16, 77, 300, 0, 1500, 64, 129, 2049]
    Hkv = 2
    NB = 96
    kc, vc = _pools(NB, Hkv, B, dtype, seed=G * 100 + B)
    runs, seq_runs = _slotted(lens, B, NB, seed=G + B)
    g = torch.Generator().manual_seed(7 + G)
    q = torch.randn((len(lens), Hkv * G, 128), generator=g).to(DT[dtype])
    scale = 1.0 / np.sqrt(128)
    dev = torch.device("cuda")
    out = pa.decode_runs(q.to(dev), kc.to(dev), vc.to(dev), torch.from_numpy(runs).to(dev),
                         torch.from_numpy(seq_runs).to(dev), scale, Hkv, max(lens))
    torch.cuda.synchronize()
    ref = oracle.decode_runs(q, kc, vc, runs, seq_runs, scale, Hkv, dtype == "bf16")
    err = max_abs_err(out, ref)
    assert err <= TOL, f"max abs error {err:.3e}"
    assert pa.read_device_status(clear=True) == 0


def test_whole_block_runs_match_the_block_table_decode(oracle):
    wl = workloads.config(2, layers=1)
    B = wl.block_size
    tables = wl.block_tables.numpy()
    runs, seq_runs = [], [0]
    for s, L in enumerate(wl.context_lens.tolist()):
        for t0 in range(0, L, B):
            runs.append((int(tables[s, t0 // B]), 0, min(B, L - t0)))
        seq_runs.append(len(runs))
    runs = np.array(runs, np.int32)
    seq_runs = np.array(seq_runs, np.int32)
    dev = torch.device("cuda")
    out = pa.decode_runs(wl.q[0].to(dev), wl.k_cache[0].to(dev), wl.v_cache[0].to(dev), torch.from_numpy(runs).to(dev),
                         torch.from_numpy(seq_runs).to(dev), wl.scale, wl.num_kv_heads, int(wl.context_lens.max()))
    torch.cuda.synchronize()
    ref = oracle.decode(wl.q[0], wl.k_cache[0], wl.v_cache[0], wl.block_tables, wl.context_lens, wl.scale,
                        wl.num_kv_heads, False)
    assert max_abs_err(out, ref) <= TOL


def test_bad_runs_are_flagged_and_skipped(oracle):
    B, Hkv, NB = 16, 2, 10
    kc, vc = _pools(NB, Hkv, B, "f16", seed=3)
    runs = np.array([(1, 0, 16), (NB, 0, 4), (2, 10, 8), (3, 4, 5)], np.int32)   # two runs leave
    seq_runs = np.array([0, 4], np.int32)
    g = torch.Generator().manual_seed(5)
    q = torch.randn((1, 4, 128), generator=g).to(torch.float16)
    dev = torch.device("cuda")
    out = pa.decode_runs(q.to(dev), kc.to(dev), vc.to(dev), torch.from_numpy(runs).to(dev),
                         torch.from_numpy(seq_runs).to(dev), 0.1, Hkv, 64)
    torch.cuda.synchronize()
    assert pa.read_device_status(clear=True) & pa._native.DEV_BAD_BLOCK_ID
    good = runs[[0, 3]]
    ref = oracle.decode_runs(q, kc, vc, good, np.array([0, 2], np.int32), 0.1, Hkv, False)
    assert max_abs_err(out, ref) <= TOL


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_compaction_then_block_table_decode(oracle, dtype):
    """Online defragmentation: every sequence's runs moved into fresh whole blocks by
    pa_gather_runs (bit for bit against the oracle's moves), then the ordinary decode over the
    resulting block table agrees with the decode over the runs."""
    B, Hkv, G = 16, 2, 6
    lens = [5, 40, 300, 1000, 17, 129]
    NB_src = 64
    need = sum((L + B - 1) // B for L in lens)
    NB = NB_src + need
    kc, vc = _pools(NB, Hkv, B, dtype, seed=11)
    runs, seq_runs = _slotted(lens, B, NB_src, seed=12)
    maxb = max((L + B - 1) // B for L in lens)
    table = np.full((len(lens), maxb), -1, np.int32)
    moves, nxt = [], NB_src
    for s in range(len(lens)):
        t = 0
        for blk, off, ln in runs[seq_runs[s]:seq_runs[s + 1]]:
            k = 0
            while k < ln:
                if t % B == 0:
                    table[s, t // B] = nxt
                    nxt += 1
                take = min(ln - k, B - t % B)
                moves.append((blk, off + k, take, int(table[s, t // B]), t % B))
                t += take
                k += take
    moves = np.array(moves, np.int32)
    dev = torch.device("cuda")
    gk, gv = kc.to(dev), vc.to(dev)
    before = pa.kernel_launch_count()
    pa.gather_runs(gk, gv, gk, gv, torch.from_numpy(moves).to(dev))
    torch.cuda.synchronize()
    assert pa.kernel_launch_count() - before == 1
    ok, ov = u16(kc).copy(), u16(vc).copy()
    assert oracle.gather_runs(ok, ov, ok, ov, moves) == 0
    assert np.array_equal(u16(gk), ok) and np.array_equal(u16(gv), ov)
    g = torch.Generator().manual_seed(13)
    q = torch.randn((len(lens), Hkv * G, 128), generator=g).to(DT[dtype])
    lens_t = torch.tensor(lens, dtype=torch.int32)
    out = pa.decode(q.to(dev), gk, gv, torch.from_numpy(table).to(dev), lens_t.to(dev), 0.088, Hkv)
    torch.cuda.synchronize()
    ref = oracle.decode_runs(q, kc, vc, runs, seq_runs, 0.088, Hkv, dtype == "bf16")
    assert max_abs_err(out, ref) <= TOL
    assert pa.read_device_status(clear=True) == 0


@pytest.mark.parametrize("num_ctas", [1, 3, 37, 0])
@pytest.mark.parametrize("B,dtype", [(16, "f16"), (32, "bf16"), (128, "f16")])
def test_runs_plan_then_layers_with_early_reads(oracle, num_ctas, B, dtype):
    """One runs plan serves three chained layers (each layer's q is the previous layer's output,
    early reads from the second layer on); CTA counts from one to one per SM."""
    lens = [3, 64, 65, 1, 700, 0, 129, 2000, 31]
    Hkv, G, NB, layers = 2, 6, 200, 3
    runs, seq_runs = _slotted(lens, B, NB, seed=11 * B + num_ctas)
    dev = torch.device("cuda")
    pools = [_pools(NB, Hkv, B, dtype, seed=500 + l) for l in range(layers)]
    g = torch.Generator().manual_seed(3)
    q0 = torch.randn((len(lens), Hkv * G, 128), generator=g).to(DT[dtype])
    runs_d, seq_d = torch.from_numpy(runs).to(dev), torch.from_numpy(seq_runs).to(dev)
    plan = pa.decode_plan_runs(runs_d, seq_d, Hkv * G, Hkv, B, NB, max(lens), num_ctas=num_ctas)
    outs = [torch.full_like(q0.to(dev), float("nan")) for _ in range(layers)]
    q = q0.to(dev)
    for l in range(layers):
        pa.decode_planned(q, pools[l][0].to(dev), pools[l][1].to(dev), plan, 0.09, out=outs[l], early_reads=l > 0)
        q = outs[l]
    torch.cuda.synchronize()
    assert pa.read_device_status(clear=True) == 0
    oq = q0
    for l in range(layers):
        ref = oracle.decode_runs(oq, pools[l][0], pools[l][1], runs, seq_runs, 0.09, Hkv, dtype == "bf16")
        err = max_abs_err(outs[l], ref)
        assert err <= TOL, f"layer {l}: max abs error {err:.3e}"
        oq = torch.from_numpy(ref).to(DT[dtype])


def test_many_one_token_runs(oracle):
    """Contexts made of runs of one or two tokens scattered over the pool (every row its own copy)."""
    g = torch.Generator().manual_seed(21)
    lens = [int(x) for x in torch.randint(1, 400, (40,), generator=g)]
    B, NB, Hkv, G = 16, 64, 4, 2
    runs, seq_runs = [], [0]
    for L in lens:
        t = 0
        while t < L:
            ln = min(int(torch.randint(1, 3, (1,), generator=g)), L - t)
            off = int(torch.randint(0, B - ln + 1, (1,), generator=g))
            runs.append((int(torch.randint(0, NB, (1,), generator=g)), off, ln))
            t += ln
        seq_runs.append(len(runs))
    runs = np.array(runs, np.int32).reshape(-1, 3)
    seq_runs = np.array(seq_runs, np.int32)
    kc, vc = _pools(NB, Hkv, B, "f16", seed=22)
    q = torch.randn((len(lens), Hkv * G, 128), generator=g).to(torch.float16)
    dev = torch.device("cuda")
    out = pa.decode_runs(q.to(dev), kc.to(dev), vc.to(dev), torch.from_numpy(runs).to(dev),
                         torch.from_numpy(seq_runs).to(dev), 0.1, Hkv, max(lens))
    torch.cuda.synchronize()
    assert pa.read_device_status(clear=True) == 0
    ref = oracle.decode_runs(q, kc, vc, runs, seq_runs, 0.1, Hkv, False)
    assert max_abs_err(out, ref) <= TOL


def test_runs_plan_refuses_new_rows_and_block_table_launches():
    """A runs plan carries no block ids: decode_planned with new rows is refused on the host, and
    a launch that does not name PA_PLAN_RUNS flags PA_DEV_BAD_PLAN and writes nothing."""
    lens = [40, 90]
    B, NB, Hkv = 16, 32, 2
    runs, seq_runs = _slotted(lens, B, NB, seed=5)
    kc, vc = _pools(NB, Hkv, B, "f16", seed=6)
    dev = torch.device("cuda")
    q = torch.randn((2, 4, 128)).to(torch.float16).to(dev)
    plan = pa.decode_plan_runs(torch.from_numpy(runs).to(dev), torch.from_numpy(seq_runs).to(dev), 4, Hkv, B, NB,
                               max(lens))
    with pytest.raises(pa.PAError):
        pa.decode_planned(q, kc.to(dev), vc.to(dev), plan, 0.1, k_new=q[:, :Hkv].contiguous(),
                          v_new=q[:, :Hkv].contiguous())
    plan.runs = False
    out = torch.full_like(q, 7.0)
    pa.decode_planned(q, kc.to(dev), vc.to(dev), plan, 0.1, out=out)
    torch.cuda.synchronize()
    assert pa.read_device_status(clear=True) == pa._native.DEV_BAD_PLAN
    assert torch.all(out == 7.0)
