"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Cache writes must match bit for bit; decode outputs within max-abs 2e-3.
Covers the five configurations at full size, split / no-split equivalence,
ragged and degenerate lengths, every supported block size and group size, both
element types, non-default streams, and the kernels' own bounds checks."""
import numpy as np
import pytest
import torch

import paged_kv_cache_08_gb300 as pa
import workloads
from gpu_util import TOL, max_abs_err, run_cuda, run_oracle, u16

pytestmark = pytest.mark.gpu


def _check(oracle, wl, layer=0, **kw):
    kc, vc, out = run_cuda(wl, layer, **kw)
    okc, ovc, ref = run_oracle(oracle, wl, layer)
    assert np.array_equal(u16(kc), okc), "k_cache differs from the oracle's scatter"
    assert np.array_equal(u16(vc), ovc), "v_cache differs from the oracle's scatter"
    err = max_abs_err(out, ref)
    assert err <= TOL, f"max abs error {err:.3e} > {TOL}"
    return err


@pytest.fixture(autouse=True)
def _clean_status():
    pa.read_device_status(clear=True)
    yield
    assert pa.read_device_status(clear=True) == 0, "a kernel flagged a bad index"


@pytest.mark.parametrize("cfg,B", [(1, None), (3, None), (4, None), (5, 16), (5, 32), (5, 64), (5, 128)])
def test_config_parity(oracle, cfg, B):
    wl = workloads.config(cfg, block_size=B)
    _check(oracle, wl)                      # the library's default path and split plan
    if cfg in (1, 4):
        _check(oracle, wl, math="fma")


def test_config2_two_layers(oracle):
    wl = workloads.config(2, layers=2)
    for layer in range(2):
        _check(oracle, wl, layer)


MATHS = ["fma", "mma", "mma_split"]


@pytest.mark.parametrize("math", MATHS)
@pytest.mark.parametrize("tps", [64, 128, 256, 0, 4096])
def test_split_lengths_agree(oracle, tps, math):
    """Many splits, the planner's choice, and one split per sequence all match the oracle."""
    wl = workloads.make_workload("splits", context_lens=[1, 63, 64, 65, 700, 1030, 2048, 5],
                                 num_q_heads=12, num_kv_heads=2, block_size=16, seed=7, max_context=2048)
    _check(oracle, wl, tokens_per_split=tps, math=math)


@pytest.mark.parametrize("math", MATHS)
@pytest.mark.parametrize("B", [16, 32, 64, 128])
@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 6, 8, 12, 16])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_ragged_lengths(oracle, B, G, dtype, math):
    if math == "fma" and G not in (1, 2, 3, 4, 6, 8):
        pytest.skip("the CUDA-core path is instantiated for G in {1, 2, 3, 4, 6, 8}")
    lens = [1, B - 1, B, B + 1, 63, 64, 65, 129, 300, 2 * B + 3]
    Hkv = 2
    wl = workloads.make_workload(f"ragged_B{B}_G{G}", context_lens=lens, num_q_heads=G * Hkv, num_kv_heads=Hkv,
                                 block_size=B, dtype=dtype, seed=B * 100 + G, max_context=512)
    _check(oracle, wl, tokens_per_split=max(B, 64) * 2, math=math)
    _check(oracle, wl, math=math)


@pytest.mark.parametrize("num_ctas", [1, 2, 3, 7, 64, 1000])
def test_persistent_ranges_and_merges(oracle, num_ctas):
    """Forced CTA counts cut sequences at arbitrary chunk boundaries; the pieces are merged by
    the last CTA to arrive.  Two calls in a row check that the arrival counters reset."""
    wl = workloads.make_workload("persist", context_lens=[1, 700, 64, 65, 2048, 0, 130, 1030, 5, 333],
                                 num_q_heads=12, num_kv_heads=2, block_size=16, seed=17, max_context=2048)
    for _ in range(2):
        _check(oracle, wl, math="mma", num_ctas=num_ctas)


@pytest.mark.parametrize("B", [16, 32, 64, 128])
@pytest.mark.parametrize("G", [1, 4, 8, 12, 16])
def test_persistent_cut_segments(oracle, B, G):
    wl = workloads.make_workload(f"pcut_B{B}_G{G}", context_lens=[B * 7 + 3, 1, 257, 64 * 5, B + 1],
                                 num_q_heads=G * 2, num_kv_heads=2, block_size=B, seed=B + G, max_context=1024)
    for ctas in (5, 11):
        _check(oracle, wl, math="mma", num_ctas=ctas)


@pytest.mark.parametrize("num_ctas", [153, 170, 199, 0])
@pytest.mark.parametrize("G,B", [(1, 32), (2, 16), (4, 64)])
def test_weighted_cut_many_short_segments(oracle, num_ctas, G, B):
    """Many short segments per CTA: 100 sequences x 8 kv heads (empty ones among them) on grids
    of more CTAs than SMs, so that two CTAs share an SM and at least 4 segments fall to each
    CTA: the cut then weighs segment ends and ranges start inside segments at other places than
    the plain cut's (the default grid of 2 CTAs per SM keeps the plain cut here).  Two calls in
    a row check that the arrival counters reset."""
    gen = torch.Generator().manual_seed(1000 + G * B)
    lens = torch.randint(0, 300, (100,), generator=gen).tolist()
    lens[3] = lens[17] = lens[99] = 0
    lens[9] = 1000
    lens[25] = 64
    wl = workloads.make_workload(f"wcut_G{G}_B{B}", context_lens=lens, num_q_heads=8 * G, num_kv_heads=8,
                                 block_size=B, seed=G + B, max_context=1024)
    for _ in range(2):
        _check(oracle, wl, math="mma", num_ctas=num_ctas)


def test_unsupported_group_is_rejected():
    wl = workloads.make_workload("g5", context_lens=[5], num_q_heads=10, num_kv_heads=2, block_size=16, seed=1)
    with pytest.raises(pa.PAError):
        run_cuda(wl, math="fma")


def test_zero_length_context(oracle):
    wl = workloads.make_workload("zero", context_lens=[0, 5, 0, 40], num_q_heads=12, num_kv_heads=2,
                                 block_size=16, seed=3, max_context=64)
    kc, vc, out = run_cuda(wl)
    _, _, ref = run_oracle(oracle, wl)
    assert not out[0].any() and not out[2].any()
    assert max_abs_err(out, ref) <= TOL


@pytest.mark.parametrize("math", MATHS)
def test_large_and_small_scores(oracle, math):
    """Scaled-up queries make the softmax peaky (running-max rescale matters)."""
    wl = workloads.make_workload("peaky", context_lens=[300, 17, 1000], num_q_heads=8, num_kv_heads=2,
                                 block_size=32, seed=11, max_context=1024, scale=1.0)
    _check(oracle, wl, tokens_per_split=128, math=math)


@pytest.mark.parametrize("scale", [0.0, -0.3])
@pytest.mark.parametrize("math", ["auto"] + MATHS)
def test_zero_and_negative_scale(oracle, scale, math):
    """Scale 0 weighs every visible token equally; a negative scale reverses the order of the
    scores, so the running maximum must be taken after scaling."""
    wl = workloads.make_workload("scale_edge", context_lens=[300, 1, 1000, 64], num_q_heads=8, num_kv_heads=2,
                                 block_size=16, seed=29, max_context=1024, scale=scale)
    _check(oracle, wl, math=math)


def test_side_stream(oracle):
    wl = workloads.make_workload("stream", context_lens=[33, 200], num_q_heads=12, num_kv_heads=2,
                                 block_size=16, seed=5, max_context=256)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        kc, vc, out = run_cuda(wl, stream=s)
    _, _, ref = run_oracle(oracle, wl)
    assert max_abs_err(out, ref) <= TOL


def test_launches_are_counted():
    wl = workloads.make_workload("count", context_lens=[10, 700], num_q_heads=12, num_kv_heads=2,
                                 block_size=16, seed=1, max_context=1024)
    before = pa.kernel_launch_count()
    run_cuda(wl, tokens_per_split=256, math="fma")
    assert pa.kernel_launch_count() - before == 3      # cache write, split pass, combine
    before = pa.kernel_launch_count()
    run_cuda(wl)
    assert pa.kernel_launch_count() - before == 2      # cache write, persistent decode


@pytest.mark.parametrize("math", MATHS)
def test_bad_block_id_is_flagged_not_faulted(oracle, math):
    """A table entry outside the pool: the kernel skips the copy and sets a status bit;
    other sequences are unaffected."""
    wl = workloads.make_workload("badid", context_lens=[40, 40], num_q_heads=12, num_kv_heads=2,
                                 block_size=16, seed=9, max_context=64)
    dev = torch.device("cuda")
    bt = wl.block_tables.clone()
    bt[1, 0] = wl.num_blocks + 5                        # out of range
    kc = wl.k_cache[0].to(dev)
    vc = wl.v_cache[0].to(dev)
    out = pa.decode(wl.q[0].to(dev), kc, vc, bt.to(dev), wl.context_lens.to(dev), wl.scale, wl.num_kv_heads,
                    math=math)
    bits = pa.read_device_status(clear=True)
    assert bits & 0x1
    got = out[0].float().cpu().numpy()
    # no cache write ran here, so compare sequence 0 with the oracle on the unwritten cache
    ref0 = oracle.decode(wl.q[0], wl.k_cache[0], wl.v_cache[0], wl.block_tables, wl.context_lens, wl.scale,
                         wl.num_kv_heads, False)
    assert np.max(np.abs(got - ref0[0])) <= TOL


@pytest.mark.parametrize("math", MATHS)
def test_bad_context_is_flagged(oracle, math):
    wl = workloads.make_workload("badctx", context_lens=[40, 20], num_q_heads=12, num_kv_heads=2,
                                 block_size=16, seed=2, max_context=64)
    dev = torch.device("cuda")
    lens = wl.context_lens.clone()
    lens[1] = 10_000                                    # longer than the table can hold
    pa.decode(wl.q[0].to(dev), wl.k_cache[0].to(dev), wl.v_cache[0].to(dev), wl.block_tables.to(dev),
              lens.to(dev), wl.scale, wl.num_kv_heads, math=math)
    assert pa.read_device_status(clear=True) & 0x2
