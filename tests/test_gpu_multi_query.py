"""GPU parity of pa_multi_query: several new query tokens per sequence attending causally over
the paged cache, against the oracle; one token per sequence equal to pa_decode; sequences cut
between CTAs (the causal limit can leave a piece without a visible token for some rows);
clamped counts flagged; more than 16 rows per (sequence, kv head) through the 64-row tiles."""
import numpy as np
import pytest
import torch

import paged_kv_cache_08_gb300 as pa
import workloads
from gpu_util import TOL, max_abs_err

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    pa.read_device_status(clear=True)
    yield


def _run(oracle, wl, new_tokens, seed, num_ctas=0, check_status=True, tiles="tc"):
    dev = torch.device("cuda")
    q, qs, max_q = workloads.multi_query_inputs(wl, new_tokens, seed)
    out = pa.multi_query(q.to(dev), wl.k_cache[0].to(dev), wl.v_cache[0].to(dev), wl.block_tables.to(dev),
                         wl.context_lens.to(dev), qs.to(dev), wl.scale, wl.num_kv_heads, max_q, num_ctas=num_ctas,
                         tiles=tiles)
    torch.cuda.synchronize()
    ref = oracle.multi_query(q, wl.k_cache[0], wl.v_cache[0], wl.block_tables, wl.context_lens, qs, wl.scale,
                             wl.num_kv_heads, wl.dtype == "bf16")
    err = max_abs_err(out, ref)
    assert err <= TOL, f"max abs error {err:.3e}"
    if check_status:
        assert pa.read_device_status(clear=True) == 0
    return out


@pytest.mark.parametrize("G,n,dtype", [(6, 2, "f16"), (4, 4, "bf16"), (1, 16, "f16"), (8, 2, "bf16"), (2, 8, "f16"),
                                       (1, 5, "bf16"), (3, 3, "f16")])
@pytest.mark.parametrize("B", [16, 64])
def test_multi_query_parity(oracle, G, n, dtype, B):
    lens = [n, 70, 129, 64 + n, 300, 1000, 17, 2 * B + 3]
    wl = workloads.make_workload(f"mq_G{G}_n{n}", context_lens=lens, num_q_heads=2 * G, num_kv_heads=2, block_size=B,
                                 dtype=dtype, seed=7 * G + n + B, max_context=1024)
    new = [min(n, L) for L in lens]
    new[2] = 1
    new[6] = 0          # a sequence without new tokens has no rows
    _run(oracle, wl, new, seed=n * 100 + G)


@pytest.mark.parametrize("num_ctas", [1, 3, 7, 40, 0])
def test_multi_query_cut_sequences(oracle, num_ctas):
    """Small grids cut sequences inside their last chunk, so that a piece can hold only
    positions past the causal limit of its early query rows."""
    lens = [65, 130, 3, 2048, 700, 129]
    wl = workloads.make_workload("mq_cut", context_lens=lens, num_q_heads=4, num_kv_heads=4, block_size=16,
                                 seed=51, max_context=2048)
    _run(oracle, wl, [16, 16, 3, 16, 9, 16], seed=52, num_ctas=num_ctas)


def test_one_token_per_sequence_is_decode():
    wl = workloads.config(2, layers=1)
    dev = torch.device("cuda")
    q = wl.q[0].to(dev)
    args = (wl.k_cache[0].to(dev), wl.v_cache[0].to(dev), wl.block_tables.to(dev), wl.context_lens.to(dev))
    dec = pa.decode(q, *args, wl.scale, wl.num_kv_heads)
    qs = torch.arange(wl.num_seqs + 1, dtype=torch.int32, device=dev)
    mq = pa.multi_query(q, *args, qs, wl.scale, wl.num_kv_heads, 1)
    torch.cuda.synchronize()
    assert torch.equal(dec.view(torch.int16), mq.view(torch.int16))


def test_counts_beyond_the_context_are_clamped_and_flagged(oracle):
    lens = [10, 40]
    wl = workloads.make_workload("mq_bad", context_lens=lens, num_q_heads=2, num_kv_heads=1, block_size=16, seed=9)
    dev = torch.device("cuda")
    q, _, _ = workloads.multi_query_inputs(wl, [4, 4], seed=3)
    qs = torch.tensor([0, 4, 8], dtype=torch.int32)
    # max_q = 2 < 4 new tokens: each sequence's first 2 rows are computed as its 2 newest tokens
    out = pa.multi_query(q.to(dev), wl.k_cache[0].to(dev), wl.v_cache[0].to(dev), wl.block_tables.to(dev),
                         wl.context_lens.to(dev), qs.to(dev), wl.scale, 1, 2)
    torch.cuda.synchronize()
    assert pa.read_device_status(clear=True) & pa._native.DEV_BAD_CONTEXT
    for s, L in enumerate(lens):
        ref = oracle.multi_query(q[4 * s:4 * s + 2], wl.k_cache[0], wl.v_cache[0], wl.block_tables[s:s + 1],
                                 wl.context_lens[s:s + 1], torch.tensor([0, 2], dtype=torch.int32), wl.scale, 1,
                                 False)
        assert max_abs_err(out[4 * s:4 * s + 2], ref) <= TOL


@pytest.mark.parametrize("G,lens,new,B,dtype", [
    (4, [40, 300, 5], [5, 5, 5], 16, "f16"),                       # 20 rows: one 64-row tile
    (6, [129, 1000, 64], [16, 16, 16], 16, "bf16"),                # 96 rows: two tiles
    (1, [100, 700, 2049], [100, 64, 100], 32, "bf16"),             # full prefill of the first
    (2, [300, 31, 500], [300, 31, 1], 16, "f16"),                  # full prefills, 600 rows
    (3, [77, 0, 513, 900, 2], [37, 0, 1, 20, 2], 64, "f16"),       # ragged, an empty sequence
    (2, [260, 1024], [70, 130], 128, "bf16"),                      # 128-token blocks
    (1, [4096, 700], [512, 300], 32, "f16"),                       # the chunked-prefill bench's shape
    (4, [1000, 129, 2000], [40, 33, 64], 64, "bf16"),              # tiles of 128 rows, a ragged last
])
@pytest.mark.parametrize("tiles", ["tc", "mma"])
def test_prefill_tiles_parity(oracle, G, lens, new, B, dtype, tiles):
    """More than 16 query rows per (sequence, kv head): tcgen05 tiles of 128 rows (accumulators in
    tensor memory) or mma.sync tiles of 64 rows."""
    wl = workloads.make_workload(f"pf_G{G}_B{B}", context_lens=lens, num_q_heads=2 * G, num_kv_heads=2,
                                 block_size=B, dtype=dtype, seed=G * 13 + B, max_context=max(lens) + B)
    assert max(new) * G > 16
    _run(oracle, wl, new, seed=G + B, tiles=tiles)


@pytest.mark.parametrize("scale", [1.0, -0.25, 0.0])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("tiles", ["tc", "mma"])
def test_prefill_peaky_zero_and_negative_scale(oracle, scale, dtype, tiles):
    """Scale 1 makes the scores peaky (the exponent base moves in later stages and O is rescaled
    in place), scale 0 weighs all visible tokens equally, a negative scale reverses their order."""
    lens = [1500, 300]
    wl = workloads.make_workload("pf_scale", context_lens=lens, num_q_heads=4, num_kv_heads=2, block_size=32,
                                 dtype=dtype, seed=31, max_context=1536, scale=scale)
    _run(oracle, wl, [200, 150], seed=32, tiles=tiles)


@pytest.mark.parametrize("tiles", ["tc", "mma"])
def test_prefill_counts_beyond_the_context_are_flagged(oracle, tiles):
    lens = [10, 40]
    wl = workloads.make_workload("pf_bad", context_lens=lens, num_q_heads=8, num_kv_heads=1, block_size=16, seed=19)
    dev = torch.device("cuda")
    q, _, _ = workloads.multi_query_inputs(wl, [12, 12], seed=4)
    qs = torch.tensor([0, 12, 24], dtype=torch.int32)
    # 12 new tokens claimed for a 10-token context: clamped to 10 and flagged
    out = pa.multi_query(q.to(dev), wl.k_cache[0].to(dev), wl.v_cache[0].to(dev), wl.block_tables.to(dev),
                         wl.context_lens.to(dev), qs.to(dev), wl.scale, 1, 12, tiles=tiles)
    torch.cuda.synchronize()
    assert pa.read_device_status(clear=True) & pa._native.DEV_BAD_CONTEXT
    ref = oracle.multi_query(q[12:24], wl.k_cache[0], wl.v_cache[0], wl.block_tables[1:2], wl.context_lens[1:2],
                             torch.tensor([0, 12], dtype=torch.int32), wl.scale, 1, False)
    assert max_abs_err(out[12:24], ref) <= TOL
    ref0 = oracle.multi_query(q[0:10], wl.k_cache[0], wl.v_cache[0], wl.block_tables[0:1], wl.context_lens[0:1],
                              torch.tensor([0, 10], dtype=torch.int32), wl.scale, 1, False)
    assert max_abs_err(out[0:10], ref0) <= TOL
