"""GPU parity of the planned decode path: pa_decode_plan once per step, then pa_decode_planned
per layer (decode alone, or with the new token's cache write), against the fp64 oracle.

The plan cuts the chunk list into two ranges per CTA, one streamed forwards and one backwards;
segments cut between the two groups of a CTA meet in shared memory, segments cut between CTAs
are combined by one named CTA from partials published in the workspace.  CTA counts from 1 to
the SM count, ragged lengths around the 64-token chunk and the block, every group size up to 8,
both element types and every block size cover each of those roles; a chain of layers with early
reads checks that q is read only after the preceding layer ends."""
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


def _planned(wl, layer=0, append=True, num_ctas=0, rounds=1):
    dev = torch.device("cuda")
    kc = wl.k_cache[layer].to(dev).clone()
    vc = wl.v_cache[layer].to(dev).clone()
    bt, lens = wl.block_tables.to(dev), wl.context_lens.to(dev)
    plan = pa.decode_plan(bt, lens, wl.num_q_heads, wl.num_kv_heads, wl.block_size, wl.num_blocks,
                          num_ctas=num_ctas)
    outs = []
    for _ in range(rounds):
        out = torch.full_like(wl.q[layer].to(dev), float("nan"))
        kw = dict(k_new=wl.k_new[layer].to(dev), v_new=wl.v_new[layer].to(dev)) if append else {}
        pa.decode_planned(wl.q[layer].to(dev), kc, vc, plan, wl.scale, out=out, **kw)
        outs.append(out)
    torch.cuda.synchronize()
    return kc, vc, outs


def _check(oracle, wl, layer=0, append=True, num_ctas=0, rounds=1):
    kc, vc, outs = _planned(wl, layer, append, num_ctas, rounds)
    if append:
        okc, ovc, ref = run_oracle(oracle, wl, layer)
        assert np.array_equal(u16(kc), okc), "k_cache differs from the oracle's"
        assert np.array_equal(u16(vc), ovc), "v_cache differs from the oracle's"
    else:
        okc = oracle_pkg.as_u16(wl.k_cache[layer])
        ovc = oracle_pkg.as_u16(wl.v_cache[layer])
        ref = oracle.decode(wl.q[layer], okc, ovc, wl.block_tables, wl.context_lens, wl.scale, wl.num_kv_heads,
                            wl.dtype == "bf16")
        assert np.array_equal(u16(kc), okc) and np.array_equal(u16(vc), ovc), "decode alone wrote the cache"
    for i, out in enumerate(outs):
        err = max_abs_err(out, ref)
        assert err <= TOL, f"round {i}: max abs error {err:.3e} > {TOL}"


@pytest.mark.parametrize("append", [True, False])
@pytest.mark.parametrize("cfg,B", [(1, None), (3, None), (4, None), (5, 16), (5, 32), (5, 64), (5, 128)])
def test_planned_config_parity(oracle, cfg, B, append):
    _check(oracle, workloads.config(cfg, block_size=B), append=append)


def test_planned_config2_two_layers(oracle):
    wl = workloads.config(2, layers=2)
    for layer in range(2):
        _check(oracle, wl, layer)


@pytest.mark.parametrize("num_ctas", [1, 2, 3, 5, 7, 16, 37, 151, 0])
def test_planned_cta_counts(oracle, num_ctas):
    """From one CTA (every segment in two groups) to one per SM (segments cut between CTAs,
    several pieces each); two rounds check that the published-partial flags are reset."""
    wl = workloads.make_workload("plan_ctas", context_lens=[1, 700, 64, 65, 2048, 0, 130, 1030, 5, 333, 4000, 17],
                                 num_q_heads=12, num_kv_heads=2, block_size=16, seed=29, max_context=4096)
    _check(oracle, wl, num_ctas=num_ctas, rounds=2)


@pytest.mark.parametrize("B", [16, 32, 64, 128])
@pytest.mark.parametrize("G,dtype", [(1, "f16"), (2, "bf16"), (4, "bf16"), (6, "f16"), (8, "f16")])
def test_planned_ragged(oracle, B, G, dtype):
    lens = [1, B - 1, B, B + 1, 63, 64, 65, 129, 300, 2 * B + 3, 0, 1500]
    wl = workloads.make_workload(f"plan_B{B}_G{G}", context_lens=lens, num_q_heads=2 * G, num_kv_heads=2,
                                 block_size=B, dtype=dtype, seed=5 * B + G, max_context=1536)
    for num_ctas in (0, 3):
        _check(oracle, wl, num_ctas=num_ctas)


@pytest.mark.parametrize("num_ctas", [0, 9])
def test_planned_tiny_problem_leaves_groups_empty(oracle, num_ctas):
    """Fewer chunks than groups: most CTAs own nothing, and a segment's span can cross CTAs
    without chunks."""
    wl = workloads.make_workload("plan_tiny", context_lens=[70, 3, 0, 200], num_q_heads=8, num_kv_heads=4,
                                 block_size=32, seed=8, max_context=256)
    _check(oracle, wl, num_ctas=num_ctas, rounds=2)


def test_planned_many_short_segments(oracle):
    """300 sequences x 8 kv heads of 1..300 tokens: many segment ends per group."""
    gen = torch.Generator().manual_seed(77)
    lens = torch.randint(1, 300, (300,), generator=gen).tolist()
    lens[5] = lens[50] = 0
    wl = workloads.make_workload("plan_short", context_lens=lens, num_q_heads=16, num_kv_heads=8, block_size=16,
                                 seed=78, max_context=512)
    _check(oracle, wl, rounds=2)


@pytest.mark.parametrize("num_ctas", [0, 37])
def test_planned_many_short_segments_one_row_per_head(oracle, num_ctas):
    """128 sequences x 8 kv heads with one query row each (the plan's weights fitted for that
    case), contexts of 1..300 tokens: many segment ends per group, segments cut between CTAs."""
    gen = torch.Generator().manual_seed(91)
    lens = torch.randint(1, 300, (128,), generator=gen).tolist()
    lens[7] = 0
    wl = workloads.make_workload("plan_short_g1", context_lens=lens, num_q_heads=8, num_kv_heads=8, block_size=32,
                                 seed=92, max_context=320)
    _check(oracle, wl, num_ctas=num_ctas, rounds=2)


def test_planned_layer_chain_with_early_reads(oracle):
    """Layer l + 1's query is layer l's output and every launch after the first asks for early
    reads: the plan and cached rows may be read while the previous layer runs, q only after it.
    Outputs start as NaN so that an early read of q would show."""
    layers = 4
    wl = workloads.make_workload("plan_chain", context_lens=[5, 900, 64, 2000, 333, 1, 1200], num_q_heads=12,
                                 num_kv_heads=2, block_size=16, seed=31, max_context=2048, layers=layers)
    dev = torch.device("cuda")
    bt, lens = wl.block_tables.to(dev), wl.context_lens.to(dev)
    kcs = [wl.k_cache[i].to(dev).clone() for i in range(layers)]
    vcs = [wl.v_cache[i].to(dev).clone() for i in range(layers)]
    outs = [torch.full_like(wl.q[0].to(dev), float("nan")) for _ in range(layers)]
    k_new = [wl.k_new[i].to(dev) for i in range(layers)]
    v_new = [wl.v_new[i].to(dev) for i in range(layers)]
    q = wl.q[0].to(dev)
    torch.cuda.synchronize()
    plan = pa.decode_plan(bt, lens, wl.num_q_heads, wl.num_kv_heads, wl.block_size, wl.num_blocks)
    for i in range(layers):
        # the launch right after the plan must not read early
        pa.decode_planned(q, kcs[i], vcs[i], plan, wl.scale, k_new=k_new[i], v_new=v_new[i], out=outs[i],
                          early_reads=i > 0)
        q = outs[i]
    torch.cuda.synchronize()
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


def test_plan_rebuilt_in_place_follows_new_lengths(oracle):
    """A plan rebuilt into the same buffer after every sequence grew by one token (inside the
    blocks it already holds) serves the next step, as a fresh plan would."""
    wl = workloads.make_workload("plan_grow", context_lens=[63, 64, 127, 500], num_q_heads=6, num_kv_heads=1,
                                 block_size=16, seed=12, max_context=640)
    dev = torch.device("cuda")
    bt = wl.block_tables.to(dev)
    plan = pa.decode_plan(bt, (wl.context_lens - 1).to(dev), wl.num_q_heads, wl.num_kv_heads, wl.block_size,
                          wl.num_blocks)
    first = pa.decode_planned(wl.q[0].to(dev), wl.k_cache[0].to(dev), wl.v_cache[0].to(dev), plan, wl.scale)
    pa.decode_plan(bt, wl.context_lens.to(dev), wl.num_q_heads, wl.num_kv_heads, wl.block_size, wl.num_blocks,
                   plan=plan)
    out = pa.decode_planned(wl.q[0].to(dev), wl.k_cache[0].to(dev), wl.v_cache[0].to(dev), plan, wl.scale)
    torch.cuda.synchronize()
    okc = oracle_pkg.as_u16(wl.k_cache[0])
    ovc = oracle_pkg.as_u16(wl.v_cache[0])
    for lens, got in ((wl.context_lens - 1, first), (wl.context_lens, out)):
        ref = oracle.decode(wl.q[0], okc, ovc, wl.block_tables, lens, wl.scale, wl.num_kv_heads, False)
        assert max_abs_err(got, ref) <= TOL


def test_plan_for_another_grid_is_refused_on_the_device():
    """A plan built for another CTA count: the kernel writes nothing and flags PA_DEV_BAD_PLAN."""
    wl = workloads.make_workload("plan_bad", context_lens=[100, 200], num_q_heads=4, num_kv_heads=2, block_size=16,
                                 seed=3, max_context=256)
    dev = torch.device("cuda")
    plan = pa.decode_plan(wl.block_tables.to(dev), wl.context_lens.to(dev), 4, 2, 16, wl.num_blocks, num_ctas=6)
    plan.num_ctas = 5   # launch another grid with the same bytes (large enough for it)
    out = torch.full_like(wl.q[0].to(dev), 7.0)
    pa.decode_planned(wl.q[0].to(dev), wl.k_cache[0].to(dev), wl.v_cache[0].to(dev), plan, wl.scale, out=out)
    torch.cuda.synchronize()
    assert pa.read_device_status(clear=True) == pa._native.DEV_BAD_PLAN
    assert torch.all(out == 7.0)


def test_planned_rejects_groups_above_8():
    wl = workloads.make_workload("plan_g12", context_lens=[5], num_q_heads=12, num_kv_heads=1, block_size=16, seed=1)
    dev = torch.device("cuda")
    with pytest.raises(pa.PAError):
        pa.decode_plan(wl.block_tables.to(dev), wl.context_lens.to(dev), 12, 1, 16, wl.num_blocks)


def test_adaptive_plan_follows_measured_rates(oracle):
    """Adaptive plans rebuilt into one buffer between launches: the first build cuts equal
    shares, later ones cut by the rates the launches measured; every launch stays correct and
    the measured rates are positive and finite."""
    wl = workloads.make_workload("plan_adapt", context_lens=[5, 900, 64, 2000, 333, 1, 1200, 700, 4000],
                                 num_q_heads=12, num_kv_heads=2, block_size=16, seed=41, max_context=4096)
    dev = torch.device("cuda")
    bt, lens = wl.block_tables.to(dev), wl.context_lens.to(dev)
    okc = oracle_pkg.as_u16(wl.k_cache[0])
    ovc = oracle_pkg.as_u16(wl.v_cache[0])
    ref = oracle.decode(wl.q[0], okc, ovc, wl.block_tables, wl.context_lens, wl.scale, wl.num_kv_heads, False)
    for num_ctas in (0, 7):
        plan = None
        bounds = []
        for it in range(6):
            plan = pa.decode_plan(bt, lens, wl.num_q_heads, wl.num_kv_heads, wl.block_size, wl.num_blocks,
                                  plan=plan, num_ctas=num_ctas, adaptive=True)
            for _ in range(3):
                out = pa.decode_planned(wl.q[0].to(dev), wl.k_cache[0].to(dev), wl.v_cache[0].to(dev), plan,
                                        wl.scale)
                torch.cuda.synchronize()
                err = max_abs_err(out, ref)
                assert err <= TOL, f"ctas {num_ctas}, build {it}: max abs error {err:.3e}"
            bounds.append(pa.plan_bounds(plan).tolist())
        rates = pa.plan_rates(plan)
        assert rates.numel() == (bounds[0].__len__() - 1) // 2
        r = rates[rates > 0]
        assert r.numel() > 0 and torch.isfinite(r).all()
        # the list length grows by the cuts that fall inside chunks (at most one per group bound)
        assert all(b[0] == 0 and b == sorted(b) and abs(b[-1] - bounds[0][-1]) < len(b) for b in bounds)


def test_adaptive_plan_used_without_the_flag_is_refused_on_the_device():
    """The layout of an adaptive plan differs: a launch that does not name PA_PLAN_ADAPTIVE finds
    another slot count in the plan's header, writes nothing and flags PA_DEV_BAD_PLAN."""
    wl = workloads.make_workload("plan_mismatch", context_lens=[100, 2000, 700], num_q_heads=8, num_kv_heads=2,
                                 block_size=16, seed=4, max_context=2048)
    dev = torch.device("cuda")
    plan = pa.decode_plan(wl.block_tables.to(dev), wl.context_lens.to(dev), 8, 2, 16, wl.num_blocks, adaptive=True)
    plan.adaptive = False
    out = torch.full_like(wl.q[0].to(dev), 7.0)
    pa.decode_planned(wl.q[0].to(dev), wl.k_cache[0].to(dev), wl.v_cache[0].to(dev), plan, wl.scale, out=out)
    torch.cuda.synchronize()
    assert pa.read_device_status(clear=True) == pa._native.DEV_BAD_PLAN
    assert torch.all(out == 7.0)


def test_adaptive_chain_in_a_graph_never_gives_up_a_wait(oracle):
    """Adaptive plans rebuilt every step change the cut from step to step; in a chained graph the
    cross-CTA folds then race with the words they clear (a fold must not clear a row's (m, l)
    while another thread of the row still polls it).  480 chained launches must leave the
    status word clean, and the last step must match the oracle."""
    layers, steps = 6, 80
    wl = workloads.config(2, layers=layers)
    dev = torch.device("cuda")
    bt, lens = wl.block_tables.to(dev), wl.context_lens.to(dev)
    kcs = [wl.k_cache[i].to(dev) for i in range(layers)]
    vcs = [wl.v_cache[i].to(dev) for i in range(layers)]
    qs = [wl.q[i].to(dev) for i in range(layers)]
    outs = [torch.empty_like(qs[0]) for _ in range(layers)]
    ws = pa.new_planned_workspace(0, dev)
    plan = pa.decode_plan(bt, lens, wl.num_q_heads, wl.num_kv_heads, wl.block_size, wl.num_blocks, adaptive=True)

    def step():
        pa.decode_plan(bt, lens, wl.num_q_heads, wl.num_kv_heads, wl.block_size, wl.num_blocks, plan=plan,
                       adaptive=True)
        q = qs[0]
        for i in range(layers):
            pa.decode_planned(q, kcs[i], vcs[i], plan, wl.scale, out=outs[i], workspace=ws, early_reads=i > 0)
            q = outs[i]
    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    pa.read_device_status(clear=True)
    for _ in range(steps):
        g.replay()
    torch.cuda.synchronize()
    assert pa.read_device_status(clear=True) == 0
    oq = wl.q[0]
    for i in range(layers):
        ref = oracle.decode(oq, oracle_pkg.as_u16(wl.k_cache[i]), oracle_pkg.as_u16(wl.v_cache[i]),
                            wl.block_tables, wl.context_lens, wl.scale, wl.num_kv_heads, False)
        err = max_abs_err(outs[i], ref)
        assert err <= TOL, f"layer {i}: max abs error {err:.3e}"
        oq = torch.from_numpy(ref).to(torch.float16)
