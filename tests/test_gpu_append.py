"""GPU parity of pa_decode_append (cache write of the newest token + decode, one launch).

The oracle side is the oracle's slot mapping, cache write and decode; the pools
must match bit for bit and the outputs within the parity tolerance.  A chain of
layers in which each layer's query is the previous layer's output checks the
early-read contract: the next launch may start before the previous one ends,
but must read q only after it has finished."""
import numpy as np
import pytest
import torch

import oracle as oracle_pkg
import paged_kv_cache_08_gb300 as pa
import workloads
from gpu_util import TOL, max_abs_err, run_oracle, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    pa.read_device_status(clear=True)
    yield
    assert pa.read_device_status(clear=True) == 0, "a kernel flagged a bad index"


def _append(wl, layer=0, **kw):
    dev = torch.device("cuda")
    kc = wl.k_cache[layer].to(dev).clone()
    vc = wl.v_cache[layer].to(dev).clone()
    out = pa.decode_append(wl.q[layer].to(dev), wl.k_new[layer].to(dev), wl.v_new[layer].to(dev), kc, vc,
                           wl.block_tables.to(dev), wl.context_lens.to(dev), wl.scale, wl.num_kv_heads, **kw)
    torch.cuda.synchronize()
    return kc, vc, out


def _check(oracle, wl, layer=0, **kw):
    kc, vc, out = _append(wl, layer, **kw)
    okc, ovc, ref = run_oracle(oracle, wl, layer)
    assert np.array_equal(u16(kc), okc), "k_cache differs from the oracle's"
    assert np.array_equal(u16(vc), ovc), "v_cache differs from the oracle's"
    err = max_abs_err(out, ref)
    assert err <= TOL, f"max abs error {err:.3e} > {TOL}"


@pytest.mark.parametrize("cfg,B", [(1, None), (3, None), (4, None), (5, 16), (5, 32), (5, 64), (5, 128)])
def test_append_config_parity(oracle, cfg, B):
    _check(oracle, workloads.config(cfg, block_size=B))


def test_append_config2_two_layers(oracle):
    wl = workloads.config(2, layers=2)
    for layer in range(2):
        _check(oracle, wl, layer)


@pytest.mark.parametrize("early", [True, False])
@pytest.mark.parametrize("num_ctas", [0, 1, 3, 7, 1000])
def test_append_cut_segments(oracle, num_ctas, early):
    wl = workloads.make_workload("append_cut", context_lens=[1, 700, 64, 65, 2048, 0, 130, 1030, 5, 333],
                                 num_q_heads=12, num_kv_heads=2, block_size=16, seed=23, max_context=2048)
    for _ in range(2):
        _check(oracle, wl, num_ctas=num_ctas, early_reads=early)


@pytest.mark.parametrize("B", [16, 32, 64, 128])
@pytest.mark.parametrize("G,dtype", [(1, "f16"), (6, "bf16"), (8, "f16"), (12, "f16"), (16, "bf16")])
def test_append_ragged(oracle, B, G, dtype):
    lens = [1, B - 1, B, B + 1, 63, 64, 65, 129, 300, 2 * B + 3]
    wl = workloads.make_workload(f"append_B{B}_G{G}", context_lens=lens, num_q_heads=2 * G, num_kv_heads=2,
                                 block_size=B, dtype=dtype, seed=3 * B + G, max_context=512)
    _check(oracle, wl)
    _check(oracle, wl, num_ctas=5)


@pytest.mark.parametrize("early", [True, False])
@pytest.mark.parametrize("num_ctas", [153, 199])
@pytest.mark.parametrize("G,B", [(1, 32), (2, 16), (6, 64)])
def test_append_many_segment_ends(oracle, num_ctas, early, G, B):
    """100 sequences x 8 kv heads on grids of more CTAs than SMs: at least 4 segments per CTA,
    so the launch takes the kernel built for many segment ends (weighted cut; each segment's
    new K/V rows staged in shared memory with its last chunk, or with q in the first stages).
    Two rounds check that the arrival counters reset."""
    gen = torch.Generator().manual_seed(2000 + G * B)
    lens = torch.randint(1, 300, (100,), generator=gen).tolist()
    lens[3] = lens[17] = 0
    lens[9] = 1000
    lens[25] = 64
    lens[26] = 65
    wl = workloads.make_workload(f"append_ends_G{G}_B{B}", context_lens=lens, num_q_heads=8 * G, num_kv_heads=8,
                                 block_size=B, seed=3 * G + B, max_context=1024)
    for _ in range(2):
        _check(oracle, wl, num_ctas=num_ctas, early_reads=early)


def test_append_layer_chain_reads_q_after_previous_layer(oracle):
    """Layer l + 1's query is layer l's output.  Launched back to back with early reads, each
    launch may begin while the previous one runs; q must still be read after it ends.  Output
    buffers start as NaN so that an early read of q would poison the result."""
    layers = 4
    wl = workloads.make_workload("chain", context_lens=[5, 900, 64, 2000, 333, 1], num_q_heads=12, num_kv_heads=2,
                                 block_size=16, seed=31, max_context=2048, layers=layers)
    dev = torch.device("cuda")
    bt, lens = wl.block_tables.to(dev), wl.context_lens.to(dev)
    kcs = [wl.k_cache[i].to(dev).clone() for i in range(layers)]
    vcs = [wl.v_cache[i].to(dev).clone() for i in range(layers)]
    outs = [torch.full_like(wl.q[0].to(dev), float("nan")) for _ in range(layers)]
    q = wl.q[0].to(dev)
    torch.cuda.synchronize()
    for i in range(layers):
        pa.decode_append(q, wl.k_new[i].to(dev), wl.v_new[i].to(dev), kcs[i], vcs[i], bt, lens, wl.scale,
                         wl.num_kv_heads, out=outs[i], early_reads=True)
        q = outs[i]
    torch.cuda.synchronize()
    # the oracle's own chain: each layer's query is the previous oracle output rounded to fp16
    oq = wl.q[0]
    for i in range(layers):
        okc = oracle_pkg.as_u16(wl.k_cache[i]).copy()
        ovc = oracle_pkg.as_u16(wl.v_cache[i]).copy()
        slots = oracle.slot_mapping(wl.block_tables, wl.context_lens, wl.block_size)
        oracle.cache_write(wl.k_new[i], wl.v_new[i], slots, okc, ovc)
        ref = oracle.decode(oq, okc, ovc, wl.block_tables, wl.context_lens, wl.scale, wl.num_kv_heads, False)
        assert np.array_equal(u16(kcs[i]), okc) and np.array_equal(u16(vcs[i]), ovc)
        err = max_abs_err(outs[i], ref)
        assert err <= TOL, f"layer {i}: max abs error {err:.3e}"
        oq = torch.from_numpy(ref).to(torch.float16)


def test_append_rejects_shapes_outside_the_persistent_kernel():
    wl = workloads.make_workload("g17", context_lens=[5], num_q_heads=17, num_kv_heads=1, block_size=16, seed=1)
    with pytest.raises(pa.PAError):
        _append(wl)
