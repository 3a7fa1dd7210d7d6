"""GPU parity of pa_multi_query_append: the cache write of several new tokens per sequence and
their causal attention over the paged cache, in one launch.

The oracle side writes the same rows with its own slot arithmetic and cache write, then runs
its several-token attention; the pools must match bit for bit and the outputs within the
parity tolerance.  New tokens that straddle a 64-token chunk or a block, sequences cut between
CTAs and early reads in a chain of layers are covered."""
import numpy as np
import pytest
import torch

import oracle as oracle_pkg
import paged_kv_cache_08_gb300 as pa
import workloads
from gpu_util import TOL, max_abs_err, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    pa.read_device_status(clear=True)
    yield
    assert pa.read_device_status(clear=True) == 0, "a kernel flagged a bad index"


def _oracle_step(oracle, wl, layer, q, k_new, v_new, qs):
    """The oracle's cache write of row query_start[s] + i at position L - n + i, then attention."""
    kc = oracle_pkg.as_u16(wl.k_cache[layer]).copy()
    vc = oracle_pkg.as_u16(wl.v_cache[layer]).copy()
    tables = wl.block_tables.numpy()
    lens = wl.context_lens.numpy()
    starts = qs.numpy()
    slots = np.full(starts[-1], -1, dtype=np.int64)
    for s in range(wl.num_seqs):
        n = int(starts[s + 1] - starts[s])
        for i in range(n):
            slots[starts[s] + i] = oracle.slot_of_token(tables[s], int(lens[s]) - n + i, wl.block_size)
    oracle.cache_write(k_new, v_new, slots, kc, vc)
    ref = oracle.multi_query(q, kc, vc, wl.block_tables, wl.context_lens, qs, wl.scale, wl.num_kv_heads,
                             wl.dtype == "bf16")
    return kc, vc, ref


def _check(oracle, wl, new_tokens, seed, layer=0, **kw):
    dev = torch.device("cuda")
    q, qs, max_q = workloads.multi_query_inputs(wl, new_tokens, seed)
    k_new, v_new = workloads.new_token_rows(wl, q.shape[0], seed + 1)
    kc = wl.k_cache[layer].to(dev).clone()
    vc = wl.v_cache[layer].to(dev).clone()
    out = pa.multi_query(q.to(dev), kc, vc, wl.block_tables.to(dev), wl.context_lens.to(dev), qs.to(dev), wl.scale,
                         wl.num_kv_heads, max_q, k_new=k_new.to(dev), v_new=v_new.to(dev), **kw)
    torch.cuda.synchronize()
    okc, ovc, ref = _oracle_step(oracle, wl, layer, q, k_new, v_new, qs)
    assert np.array_equal(u16(kc), okc), "k_cache differs from the oracle's"
    assert np.array_equal(u16(vc), ovc), "v_cache differs from the oracle's"
    err = max_abs_err(out, ref)
    assert err <= TOL, f"max abs error {err:.3e}"
    return out


@pytest.mark.parametrize("G,n,dtype", [(6, 2, "f16"), (4, 4, "bf16"), (1, 16, "f16"), (8, 2, "bf16"),
                                       (2, 8, "f16"), (1, 5, "bf16"), (3, 3, "f16")])
@pytest.mark.parametrize("B", [16, 64, 128])
def test_multi_query_append_parity(oracle, G, n, dtype, B):
    # 70 with n up to 16 straddles the first chunk boundary; 2B + 3 a block boundary
    lens = [n, 70, 129, 64 + n, 300, 1000, 17, 2 * B + 3]
    wl = workloads.make_workload(f"mqa_G{G}_n{n}", context_lens=lens, num_q_heads=2 * G, num_kv_heads=2,
                                 block_size=B, dtype=dtype, seed=11 * G + n + B, max_context=1024)
    new = [min(n, L) for L in lens]
    new[2] = 1
    new[6] = 0
    _check(oracle, wl, new, seed=n * 10 + G)


@pytest.mark.parametrize("early", [True, False])
@pytest.mark.parametrize("num_ctas", [1, 3, 7, 40, 0])
def test_multi_query_append_cut_sequences(oracle, num_ctas, early):
    lens = [65, 130, 3, 2048, 700, 129, 16]
    wl = workloads.make_workload("mqa_cut", context_lens=lens, num_q_heads=4, num_kv_heads=4, block_size=16,
                                 seed=61, max_context=2048)
    _check(oracle, wl, [16, 16, 3, 16, 9, 16, 16], seed=62, num_ctas=num_ctas, early_reads=early)


def test_one_new_token_is_decode_append():
    """One new token per sequence: the same pools and bit-identical outputs as pa_decode_append."""
    wl = workloads.config(2, layers=1)
    dev = torch.device("cuda")
    q = wl.q[0].to(dev)
    bt, lens = wl.block_tables.to(dev), wl.context_lens.to(dev)
    kc1, vc1 = wl.k_cache[0].to(dev).clone(), wl.v_cache[0].to(dev).clone()
    kc2, vc2 = kc1.clone(), vc1.clone()
    kn, vn = wl.k_new[0].to(dev), wl.v_new[0].to(dev)
    dec = pa.decode_append(q, kn, vn, kc1, vc1, bt, lens, wl.scale, wl.num_kv_heads)
    qs = torch.arange(wl.num_seqs + 1, dtype=torch.int32, device=dev)
    mq = pa.multi_query(q, kc2, vc2, bt, lens, qs, wl.scale, wl.num_kv_heads, 1, k_new=kn, v_new=vn)
    torch.cuda.synchronize()
    assert torch.equal(kc1.view(torch.int16), kc2.view(torch.int16))
    assert torch.equal(vc1.view(torch.int16), vc2.view(torch.int16))
    assert torch.equal(dec.view(torch.int16), mq.view(torch.int16))


def test_multi_query_append_layer_chain(oracle):
    """Layer l + 1's queries are layer l's outputs.  Launched back to back with early reads,
    each launch may start while the previous one runs; it must still read q, k_new and v_new
    only after that one ends.  Outputs start as NaN so that an early read would show."""
    layers = 4
    lens = [5, 900, 64, 2000, 333, 20]
    new = [4, 4, 4, 1, 3, 4]
    wl = workloads.make_workload("mqa_chain", context_lens=lens, num_q_heads=8, num_kv_heads=2, block_size=16,
                                 seed=71, max_context=2048, layers=layers)
    dev = torch.device("cuda")
    bt, lens_d = wl.block_tables.to(dev), wl.context_lens.to(dev)
    q0, qs, max_q = workloads.multi_query_inputs(wl, new, seed=72)
    rows = [workloads.new_token_rows(wl, q0.shape[0], seed=80 + i) for i in range(layers)]
    kcs = [wl.k_cache[i].to(dev).clone() for i in range(layers)]
    vcs = [wl.v_cache[i].to(dev).clone() for i in range(layers)]
    outs = [torch.full_like(q0.to(dev), float("nan")) for _ in range(layers)]
    q, qs_d = q0.to(dev), qs.to(dev)
    torch.cuda.synchronize()
    for i in range(layers):
        pa.multi_query(q, kcs[i], vcs[i], bt, lens_d, qs_d, wl.scale, wl.num_kv_heads, max_q, out=outs[i],
                       k_new=rows[i][0].to(dev), v_new=rows[i][1].to(dev), early_reads=True)
        q = outs[i]
    torch.cuda.synchronize()
    oq = q0
    for i in range(layers):
        okc, ovc, ref = _oracle_step(oracle, wl, i, oq, rows[i][0], rows[i][1], qs)
        assert np.array_equal(u16(kcs[i]), okc) and np.array_equal(u16(vcs[i]), ovc)
        err = max_abs_err(outs[i], ref)
        assert err <= TOL, f"layer {i}: max abs error {err:.3e}"
        oq = torch.from_numpy(ref).to(torch.float16)


def test_multi_query_append_beyond_16_rows_is_unsupported():
    """More than 16 query rows per (sequence, kv head) go to the 64-row tiles, which write no
    cache rows: the call is refused and nothing is written."""
    wl = workloads.make_workload("mqa_big", context_lens=[40, 60], num_q_heads=8, num_kv_heads=1, block_size=16,
                                 seed=5)
    dev = torch.device("cuda")
    q, qs, max_q = workloads.multi_query_inputs(wl, [4, 4], seed=6)
    k_new, v_new = workloads.new_token_rows(wl, q.shape[0], seed=7)
    kc = wl.k_cache[0].to(dev).clone()
    before = kc.clone()
    with pytest.raises(pa.PAError):
        pa.multi_query(q.to(dev), kc, wl.v_cache[0].to(dev).clone(), wl.block_tables.to(dev),
                       wl.context_lens.to(dev), qs.to(dev), wl.scale, 1, max_q, k_new=k_new.to(dev),
                       v_new=v_new.to(dev))
    torch.cuda.synchronize()
    assert torch.equal(kc.view(torch.int16), before.view(torch.int16))
