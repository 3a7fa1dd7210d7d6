"""Pins for the CPU oracle: each check ties it to something other than itself.

* element decoding: exhaustive over all 65536 bit patterns against numpy's
  float16 and the bfloat16 = upper-half-of-float32 definition;
* addressing: the worked example of the PagedAttention explainer page
  (tests/golden/address_worked_example.txt);
* byte ledger: the numbers the pages print (tests/golden/byte_ledger.txt);
* decode: torch's fp64 ``scaled_dot_product_attention`` on the unpaged data,
  bit-identical output under a permutation of physical block ids, and closed
  forms (one token, zero query, equal keys, one dominant score, two tokens);
* cache write: the worked example's slots, plus a canary fill showing that
  nothing but the addressed rows changes;
* several query tokens per sequence: torch's fp64 attention with an explicit causal mask on
  the unpaged data (full causal prefill, one token, none), and bit-for-bit the decode at one
  token per sequence;
* slotted blocks: the radix-tree page's slotted block (tests/golden/slotted_worked_example.txt)
  read through runs against torch's fp64 attention on the concatenated rows, whole-block runs
  against the block-table decode, and compaction into fresh blocks (bit for bit);
* block copy: the copy-on-write fork of the PagedAttention explainer page
  (tests/golden/cow_worked_example.txt) checked against torch's fp64 attention on
  each branch's contiguous context, and a move to another pool and back that must
  leave attention bit-identical;
* planted mistakes (``PAO_MUTANT``): every one of them must fail some pin.
"""
import math
import os
from pathlib import Path

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as oracle_pkg

GOLDEN = Path(__file__).resolve().parent / "golden"


# ------------------------------------------------------------------------------------------
# helpers (test-side input construction only)
# ------------------------------------------------------------------------------------------

def _read_golden(name):
    rows = []
    for line in (GOLDEN / name).read_text(encoding="utf-8").splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        rows.append(line.split())
    return rows


def _rand16(shape, gen, bf16=False, scale=1.0):
    x = torch.randn(shape, generator=gen, dtype=torch.float32) * scale
    return x.to(torch.bfloat16 if bf16 else torch.float16)


def _paged_problem(lens, Hq, Hkv, D, B, seed, bf16=False, pool_extra=3):
    """Contiguous per-sequence K/V and their paged copy in a randomly permuted pool.

    Returns (q, Kc list, Vc list, k_cache, v_cache, block_tables).  Unused pool
    slots are random too, so a wrong address changes the result."""
    gen = torch.Generator().manual_seed(seed)
    S = len(lens)
    nblk = [(L + B - 1) // B for L in lens]
    NB = sum(nblk) + pool_extra
    maxb = max(1, max(nblk))
    perm = torch.randperm(NB, generator=gen)
    tables = torch.full((S, maxb), -1, dtype=torch.int32)
    c = 0
    for s in range(S):
        tables[s, :nblk[s]] = perm[c:c + nblk[s]].to(torch.int32)
        c += nblk[s]
    q = _rand16((S, Hq, D), gen, bf16)
    Kc = [_rand16((Hkv, L, D), gen, bf16) for L in lens]
    Vc = [_rand16((Hkv, L, D), gen, bf16) for L in lens]
    kc = _rand16((NB, Hkv, B, D), gen, bf16)
    vc = _rand16((NB, Hkv, B, D), gen, bf16)
    for s, L in enumerate(lens):
        for t in range(L):
            p, o = int(tables[s, t // B]), t % B
            kc[p, :, o, :] = Kc[s][:, t, :]
            vc[p, :, o, :] = Vc[s][:, t, :]
    return q, Kc, Vc, kc, vc, tables


def _sdpa_fp64(q, Kc, Vc, Hkv, scale):
    """torch's attention in fp64 on the unpaged data; query head h uses kv head h // G."""
    S, Hq, D = q.shape
    G = Hq // Hkv
    out = torch.zeros((S, Hq, D), dtype=torch.float64)
    for s in range(S):
        L = Kc[s].shape[1]
        if L == 0:
            continue
        qs = q[s].to(torch.float64)[:, None, :]                      # [Hq, 1, D]
        ks = Kc[s].to(torch.float64).repeat_interleave(G, dim=0)     # [Hq, L, D]
        vs = Vc[s].to(torch.float64).repeat_interleave(G, dim=0)
        out[s] = F.scaled_dot_product_attention(qs[None], ks[None], vs[None], scale=scale)[0, :, 0, :]
    return out.numpy()


# ------------------------------------------------------------------------------------------
# pins, written as functions of an oracle so that planted mistakes can be run through them
# ------------------------------------------------------------------------------------------

def pin_f16_exhaustive(o):
    bits = np.arange(65536, dtype=np.uint16)
    got = o.to_f64(bits, is_bf16=False)
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def pin_bf16_exhaustive(o):
    bits = np.arange(65536, dtype=np.uint16)
    got = o.to_f64(bits, is_bf16=True)
    with np.errstate(invalid="ignore"):
        want = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def pin_address_worked_example(o):
    rows = _read_golden("address_worked_example.txt")
    kv = {r[0]: r[1:] for r in rows if r[0] != "token"}
    B = int(kv["block_size"][0])
    table = [int(x) for x in kv["table"]]
    for r in rows:
        if r[0] == "token":
            t, phys, off = int(r[1]), int(r[2]), int(r[3])
            assert o.locate(table, t, B) == (phys, off), r
            assert o.slot_of_token(table, t, B) == phys * B + off
    # the prompt fills the last listed block up to filled_in_last_block
    prompt = int(kv["prompt_tokens"][0])
    assert len(table) == math.ceil(prompt / B)
    assert prompt - (len(table) - 1) * B == int(kv["filled_in_last_block"][0])
    # slot of the new token, from the table and the context length that counts it
    L, phys, off = (int(x) for x in kv["new_token"])
    bt = np.full((1, 8), -1, dtype=np.int32)
    bt[0, :len(table)] = table
    assert o.slot_mapping(bt, np.array([L], np.int32), B)[0] == phys * B + off
    grown = [int(x) for x in kv["grown_table"]]
    L, phys, off = (int(x) for x in kv["new_token_after_growth"])
    bt[0, :len(grown)] = grown
    assert o.slot_mapping(bt, np.array([L], np.int32), B)[0] == phys * B + off
    # an empty context writes nothing
    assert o.slot_mapping(bt, np.array([0], np.int32), B)[0] < 0


def pin_byte_ledger(o):
    for name, hkv, d, e, tokens, layers, want in _read_golden("byte_ledger.txt"):
        got = o.kv_bytes_per_token(int(hkv), int(d), int(e)) * int(tokens) * int(layers)
        assert got == int(want), name
    # the page's rounded megabytes (KB of 1024 bytes, then /1000)
    assert round(512 * 24 * 1024 / 1024 / 1000, 1) == 12.3
    assert round(2048 * 24 * 1024 / 1024 / 1000, 1) == 49.2


def pin_decode_vs_sdpa(o):
    cases = [
        dict(lens=[1, 5, 16, 17, 40], Hq=6, Hkv=2, D=128, B=16, bf16=False),
        dict(lens=[3, 33, 64, 0, 9], Hq=8, Hkv=8, D=64, B=4, bf16=False),
        dict(lens=[70, 2, 31], Hq=12, Hkv=3, D=32, B=32, bf16=True),
    ]
    for i, c in enumerate(cases):
        q, Kc, Vc, kc, vc, bt = _paged_problem(c["lens"], c["Hq"], c["Hkv"], c["D"], c["B"], 100 + i,
                                               c["bf16"])
        scale = 1.0 / math.sqrt(c["D"])
        got = o.decode(q, kc, vc, bt, torch.tensor(c["lens"], dtype=torch.int32), scale, c["Hkv"],
                       c["bf16"])
        want = _sdpa_fp64(q, Kc, Vc, c["Hkv"], scale)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12, err_msg=str(c))


def pin_scales_vs_sdpa(o):
    """The definition softmax(scale q.k) V holds for any real scale: 0 weighs every token equally,
    a negative scale reverses the order of the scores, a scale of 1 on 128 dims makes the
    weights peaky.  Decode and several query tokens per sequence against torch's fp64 attention
    on the unpaged data."""
    lens = [1, 30, 77, 16]
    Hq, Hkv, D, B = 6, 2, 128, 16
    G = Hq // Hkv
    q, Kc, Vc, kc, vc, bt = _paged_problem(lens, Hq, Hkv, D, B, 55)
    lt = np.array(lens, np.int32)
    nq = [1, 7, 3, 16]
    qm = _rand16((sum(nq), Hq, D), torch.Generator().manual_seed(56))
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    for scale in (0.0, -0.3, 1.0):
        got = o.decode(q, kc, vc, bt, lt, scale, Hkv, False)
        np.testing.assert_allclose(got, _sdpa_fp64(q, Kc, Vc, Hkv, scale), rtol=0, atol=1e-12,
                                   err_msg=f"decode, scale {scale}")
        got = o.multi_query(qm, kc, vc, bt, lt, qs, scale, Hkv, False)
        for s, (L, n) in enumerate(zip(lens, nq)):
            qq = qm[qs[s]:qs[s + 1]].to(torch.float64).permute(1, 0, 2)[None]
            kk = Kc[s].to(torch.float64).repeat_interleave(G, dim=0)[None]
            vv = Vc[s].to(torch.float64).repeat_interleave(G, dim=0)[None]
            mask = torch.arange(L)[None, :] <= torch.arange(L - n, L)[:, None]
            want = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale)[0].permute(1, 0, 2)
            assert np.max(np.abs(got[qs[s]:qs[s + 1]] - want.numpy())) < 1e-12, (scale, s)
    # scale 0: every visible token weighs the same, so decode is the mean of the context's V rows
    got = o.decode(q, kc, vc, bt, lt, 0.0, Hkv, False)
    for s, L in enumerate(lens):
        mean = Vc[s].to(torch.float64).mean(dim=1).repeat_interleave(G, dim=0).numpy()
        np.testing.assert_allclose(got[s], mean, rtol=0, atol=1e-12)


def pin_permutation_invariance(o):
    lens = [5, 23, 48, 1]
    Hq, Hkv, D, B = 4, 2, 128, 8
    q, Kc, Vc, kc, vc, bt = _paged_problem(lens, Hq, Hkv, D, B, 7)
    lt = torch.tensor(lens, dtype=torch.int32)
    base = o.decode(q, kc, vc, bt, lt, 0.125, Hkv, False)
    NB = kc.shape[0]
    sigma = torch.randperm(NB, generator=torch.Generator().manual_seed(8))   # new id of old block b
    kc2 = torch.empty_like(kc)
    vc2 = torch.empty_like(vc)
    kc2[sigma] = kc
    vc2[sigma] = vc
    bt2 = bt.clone()
    m = bt >= 0
    bt2[m] = sigma[bt[m].long()].to(torch.int32)
    moved = o.decode(q, kc2, vc2, bt2, lt, 0.125, Hkv, False)
    assert np.array_equal(base, moved)


def pin_closed_forms(o):
    D, B, Hkv, Hq = 16, 4, 1, 1
    gen = torch.Generator().manual_seed(11)
    # one cached token: softmax of one score is 1, so out = V[0] exactly
    q, Kc, Vc, kc, vc, bt = _paged_problem([1], Hq, Hkv, D, B, 12)
    got = o.decode(q, kc, vc, bt, torch.tensor([1], dtype=torch.int32), 0.3, Hkv, False)
    assert np.array_equal(got[0, 0], Vc[0][0, 0].to(torch.float64).numpy())
    # zero query: every score is 0, out = mean of V
    L = 13
    q, Kc, Vc, kc, vc, bt = _paged_problem([L], Hq, Hkv, D, B, 13)
    qz = torch.zeros_like(q)
    got = o.decode(qz, kc, vc, bt, torch.tensor([L], dtype=torch.int32), 0.7, Hkv, False)
    want = Vc[0][0].to(torch.float64).mean(dim=0).numpy()
    np.testing.assert_allclose(got[0, 0], want, rtol=0, atol=1e-14)
    # all keys equal: scores all equal, out = mean of V (any query)
    kc_eq = kc.clone()
    kc_eq[:] = kc[int(bt[0, 0]), :, 0:1, :]
    got = o.decode(q, kc_eq, vc, bt, torch.tensor([L], dtype=torch.int32), 0.7, Hkv, False)
    np.testing.assert_allclose(got[0, 0], want, rtol=0, atol=1e-14)
    # one dominant score: out = V[argmax] to within exp(-gap)
    qd = torch.zeros_like(q)
    qd[0, 0, 0] = 8.0
    kd = torch.zeros_like(kc)
    j = 9
    kd[int(bt[0, j // B]), 0, j % B, 0] = 8.0               # score 64 * scale for token j only
    got = o.decode(qd, kd, vc, bt, torch.tensor([L], dtype=torch.int32), 1.0, Hkv, False)
    np.testing.assert_allclose(got[0, 0], Vc[0][0, j].to(torch.float64).numpy(), rtol=0,
                               atol=1e-20 + 16 * math.exp(-64.0))
    # two tokens: p0 = 1 / (1 + exp(z1 - z0)), out = p0 V0 + (1 - p0) V1
    q, Kc, Vc, kc, vc, bt = _paged_problem([2], Hq, Hkv, D, B, 14)
    sc = 0.25
    got = o.decode(q, kc, vc, bt, torch.tensor([2], dtype=torch.int32), sc, Hkv, False)
    qv = q[0, 0].to(torch.float64)
    k0, k1 = Kc[0][0, 0].to(torch.float64), Kc[0][0, 1].to(torch.float64)
    v0, v1 = Vc[0][0, 0].to(torch.float64), Vc[0][0, 1].to(torch.float64)
    z0, z1 = sc * float(qv @ k0), sc * float(qv @ k1)
    p0 = 1.0 / (1.0 + math.exp(z1 - z0))
    np.testing.assert_allclose(got[0, 0], (p0 * v0 + (1 - p0) * v1).numpy(), rtol=0, atol=1e-14)
    # an empty context gives a zero output
    got = o.decode(q, kc, vc, bt, torch.tensor([0], dtype=torch.int32), sc, Hkv, False)
    assert not np.any(got)


def pin_cache_write(o):
    rows = _read_golden("address_worked_example.txt")
    kv = {r[0]: r[1:] for r in rows if r[0] != "token"}
    B = int(kv["block_size"][0])
    Hkv, D, NB = 2, 128, 26
    gen = torch.Generator().manual_seed(21)
    canary = np.full((NB, Hkv, B, D), 0x7BCD, dtype=np.uint16)
    kcache, vcache = canary.copy(), canary.copy()
    # two sequences: the 39-token example and the 49-token example of the golden file
    bt = np.full((2, 8), -1, dtype=np.int32)
    bt[0, :3] = [int(x) for x in kv["table"]]
    bt[1, :4] = [int(x) for x in kv["grown_table"]]
    lens = np.array([int(kv["new_token"][0]), int(kv["new_token_after_growth"][0])], np.int32)
    slots = o.slot_mapping(bt, lens, B)
    k = _rand16((2, Hkv, D), gen)
    v = _rand16((2, Hkv, D), gen)
    o.cache_write(k, v, slots, kcache, vcache)
    ku, vu = oracle_pkg.as_u16(k), oracle_pkg.as_u16(v)
    expect_k, expect_v = canary.copy(), canary.copy()
    for i, key in enumerate(("new_token", "new_token_after_growth")):
        _, phys, off = (int(x) for x in kv[key])
        expect_k[phys, :, off, :] = ku[i]
        expect_v[phys, :, off, :] = vu[i]
    assert np.array_equal(kcache, expect_k)
    assert np.array_equal(vcache, expect_v)
    # a negative slot is skipped
    kc2 = canary.copy()
    vc2 = canary.copy()
    o.cache_write(k, v, np.array([-1, -5], np.int64), kc2, vc2)
    assert np.array_equal(kc2, canary) and np.array_equal(vc2, canary)


def pin_copy_on_write_fork(o):
    """The copy-on-write example of §四: a prompt in blocks #10 (full) and #11 (partial) shared by
    branches A and B; A's append deep-copies #11 into #45 (tests/golden/cow_worked_example.txt),
    B then writes into #11 in place.  Each branch's attention must equal torch's fp64 attention
    on its own contiguous context (prompt + its token), and #45 must hold #11's rows."""
    kv = {r[0]: [int(x) for x in r[1:]] for r in _read_golden("cow_worked_example.txt")}
    b10, b11 = kv["prompt_blocks"]
    new, = kv["cow_new_block"]
    gen = torch.Generator().manual_seed(77)
    B, Hkv, G, D = 16, 2, 3, 128
    Hq = Hkv * G
    NB = 96
    P = B + 4                                   # #10 full, 4 rows in #11
    kc = oracle_pkg.as_u16(_rand16((NB, Hkv, B, D), gen)).copy()
    vc = oracle_pkg.as_u16(_rand16((NB, Hkv, B, D), gen)).copy()
    Kp = _rand16((Hkv, P, D), gen)
    Vp = _rand16((Hkv, P, D), gen)
    kp, vp = oracle_pkg.as_u16(Kp), oracle_pkg.as_u16(Vp)
    for t in range(P):
        blk = b10 if t < B else b11
        kc[blk, :, t % B, :] = kp[:, t, :]
        vc[blk, :, t % B, :] = vp[:, t, :]
    shared_k, shared_v = kc[b11].copy(), vc[b11].copy()
    # A: copy-on-write, then its token lands in the copy; B: its token lands in #11 itself
    assert o.copy_blocks(kc, vc, kc, vc, [b11], [new]) == 0
    assert np.array_equal(kc[new], shared_k) and np.array_equal(vc[new], shared_v)
    kn = _rand16((2, Hkv, D), gen)
    vn = _rand16((2, Hkv, D), gen)
    tables = np.array([[b10, new], [b10, b11]], np.int32)
    lens = np.array([P + 1, P + 1], np.int32)
    o.cache_write(kn, vn, o.slot_mapping(tables, lens, B), kc, vc)
    q = _rand16((2, Hq, D), gen)
    scale = 1.0 / math.sqrt(D)
    got = o.decode(q, kc, vc, tables, lens, scale, Hkv, False)
    Kc = [torch.cat([Kp, kn[i][:, None, :]], dim=1) for i in range(2)]
    Vc = [torch.cat([Vp, vn[i][:, None, :]], dim=1) for i in range(2)]
    want = _sdpa_fp64(q, Kc, Vc, Hkv, scale)
    assert np.max(np.abs(got - want)) < 1e-12


def pin_block_moves(o):
    """Blocks moved to another pool and back to new ids (a swap out and in): the rows arrive
    unchanged, nothing else changes, and attention through the rewritten table is bit-identical
    to attention before the move (the permutation invariance of paging)."""
    lens = [37, 64, 5]
    B, Hkv, D = 16, 2, 128
    q, Kc, Vc, kc, vc, tables = _paged_problem(lens, 4, Hkv, D, B, seed=91, pool_extra=12)
    kc, vc = oracle_pkg.as_u16(kc).copy(), oracle_pkg.as_u16(vc).copy()
    NB = kc.shape[0]
    lens_np = np.array(lens, np.int32)
    before = o.decode(q, kc, vc, tables, lens_np, 0.1, Hkv, False)
    nb = (lens[1] + B - 1) // B
    dev_ids = [int(x) for x in tables[1, :nb]]
    host_k = np.zeros((8, Hkv, B, D), np.uint16)
    host_v = np.zeros((8, Hkv, B, D), np.uint16)
    host_ids = [5, 2, 7, 0][:nb]
    assert o.copy_blocks(kc, vc, host_k, host_v, dev_ids, host_ids) == 0
    for d, h in zip(dev_ids, host_ids):
        assert np.array_equal(host_k[h], kc[d]) and np.array_equal(host_v[h], vc[d])
    untouched = [i for i in range(8) if i not in host_ids]
    assert not host_k[untouched].any() and not host_v[untouched].any()
    used = set(int(x) for x in tables[tables >= 0].ravel())
    free = [i for i in range(NB) if i not in used]
    new_ids = free[:nb]
    kc2, vc2 = kc.copy(), vc.copy()
    assert o.copy_blocks(host_k, host_v, kc2, vc2, host_ids, new_ids) == 0
    moved = tables.numpy().copy()
    moved[1, :nb] = new_ids
    after = o.decode(q, kc2, vc2, moved, lens_np, 0.1, Hkv, False)
    assert np.array_equal(before, after)
    # an id outside its pool leaves the pair out
    kc3 = kc.copy()
    assert o.copy_blocks(kc, vc, kc3, vc.copy(), [0, NB], [NB + 1, 1]) == 2
    assert np.array_equal(kc3, kc)


def pin_multi_query_vs_sdpa(o):
    """Several new query tokens per sequence: each attends causally over the paged context up
    to its own position.  Checked against torch's fp64 attention with an explicit mask on the
    unpaged data: ragged contexts, a full causal prefill (n = L), one token (n = 1) and no new
    token (n = 0); n = 1 must also reproduce the decode bit for bit."""
    lens = [37, 16, 5, 64, 1, 20]
    nq = [4, 16, 5, 1, 1, 0]
    B, Hkv, G, D = 16, 2, 3, 128
    Hq = Hkv * G
    q1, Kc, Vc, kc, vc, tables = _paged_problem(lens, Hq, Hkv, D, B, seed=123)
    gen = torch.Generator().manual_seed(321)
    T = sum(nq)
    q = _rand16((T, Hq, D), gen)
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    scale = 1.0 / math.sqrt(D)
    got = o.multi_query(q, kc, vc, tables, np.array(lens, np.int32), qs, scale, Hkv, False)
    for s, (L, n) in enumerate(zip(lens, nq)):
        if n == 0:
            continue
        qq = q[qs[s]:qs[s + 1]].to(torch.float64).permute(1, 0, 2)[None]          # [1, Hq, n, D]
        kk = Kc[s].to(torch.float64).repeat_interleave(G, dim=0)[None]             # [1, Hq, L, D]
        vv = Vc[s].to(torch.float64).repeat_interleave(G, dim=0)[None]
        pos = torch.arange(L - n, L)[:, None]
        mask = torch.arange(L)[None, :] <= pos                                      # [n, L]
        want = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale)[0].permute(1, 0, 2)
        assert np.max(np.abs(got[qs[s]:qs[s + 1]] - want.numpy())) < 1e-12, s
    # one new token per sequence is the decode
    dec = o.decode(q1, kc, vc, tables, np.array(lens, np.int32), scale, Hkv, False)
    one = o.multi_query(q1, kc, vc, tables, np.array(lens, np.int32), np.arange(len(lens) + 1, dtype=np.int32),
                        scale, Hkv, False)
    assert np.array_equal(dec, one)


def _slotted_golden():
    kv = {}
    for r in _read_golden("slotted_worked_example.txt"):
        if r[0] == "slot":
            kv["slot_" + r[1]] = (int(r[2]), int(r[3]))
        else:
            kv[r[0]] = float(r[1]) if "." in r[1] else int(r[1])
    return kv


def pin_slotted_runs(o):
    """Contexts given as runs (block_id, slot_offset, length): the page's slotted block (Node A in
    slots 0..4, Node B in 5..12 of one 16-slot block, tests/golden/slotted_worked_example.txt),
    sequences reading a node's slot and then blocks of their own.  Attention must equal torch's
    fp64 attention on the concatenated rows; runs of whole blocks must give the block-table decode
    bit for bit; compacting the runs into fresh blocks (the page's online defragmentation) must
    give the same decode bit for bit through a plain block table."""
    kv = _slotted_golden()
    B = kv["block_size"]
    (a_off, a_len), (b_off, b_len) = kv["slot_A"], kv["slot_B"]
    assert a_off + a_len == b_off and B - (b_off + b_len) == kv["free_tail"]
    assert B - kv["lone_node_tokens"] == kv["lone_node_idle_slots"]
    # 11 / 16 = 68.75 %, which the page prints cut to one decimal
    assert math.floor(1000 * kv["lone_node_idle_slots"] / B) / 10 == kv["lone_node_idle_pct"]
    gen = torch.Generator().manual_seed(55)
    Hkv, G, D = 2, 3, 128
    Hq = Hkv * G
    NB = 24
    kc = _rand16((NB, Hkv, B, D), gen)
    vc = _rand16((NB, Hkv, B, D), gen)
    shared = 7                                   # the slotted block
    # seq 0: node A's slot, then blocks 3 and 11 (whole) and 4 tokens of block 2
    # seq 1: node B's slot, then 9 tokens of block 20; seq 2: node A only; seq 3: empty
    runs = [(shared, a_off, a_len), (3, 0, B), (11, 0, B), (2, 0, 4),
            (shared, b_off, b_len), (20, 0, 9),
            (shared, a_off, a_len)]
    seq_runs = [0, 4, 6, 7, 7]
    S = len(seq_runs) - 1
    q = _rand16((S, Hq, D), gen)
    scale = 1.0 / math.sqrt(D)
    got = o.decode_runs(q, kc, vc, runs, seq_runs, scale, Hkv, False)
    Kc, Vc = [], []
    for s in range(S):
        ks = [kc[blk, :, off:off + ln, :] for blk, off, ln in runs[seq_runs[s]:seq_runs[s + 1]]]
        vs = [vc[blk, :, off:off + ln, :] for blk, off, ln in runs[seq_runs[s]:seq_runs[s + 1]]]
        Kc.append(torch.cat(ks, dim=1) if ks else torch.zeros((Hkv, 0, D), dtype=kc.dtype))
        Vc.append(torch.cat(vs, dim=1) if vs else torch.zeros((Hkv, 0, D), dtype=vc.dtype))
    want = _sdpa_fp64(q, Kc, Vc, Hkv, scale)
    assert np.max(np.abs(got - want)) < 1e-12
    # whole-block runs are a block table
    lens = [37, 16, 64]
    q2, _, _, kc2, vc2, tables = _paged_problem(lens, Hq, Hkv, D, B, seed=56)
    r2, sr2 = [], [0]
    for s, L in enumerate(lens):
        for t0 in range(0, L, B):
            r2.append((int(tables[s, t0 // B]), 0, min(B, L - t0)))
        sr2.append(len(r2))
    dec = o.decode(q2, kc2, vc2, tables, np.array(lens, np.int32), scale, Hkv, False)
    assert np.array_equal(dec, o.decode_runs(q2, kc2, vc2, r2, sr2, scale, Hkv, False))
    # compaction: each sequence's runs moved into fresh whole blocks, then a plain table
    ku, vu = oracle_pkg.as_u16(kc).copy(), oracle_pkg.as_u16(vc).copy()
    moves, table, nxt = [], np.full((S, 8), -1, np.int32), 12
    lens3 = []
    for s in range(S):
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
        lens3.append(t)
    assert nxt <= NB and not set(range(12, nxt)) & {b for b, _, _ in runs}
    assert o.gather_runs(ku, vu, ku, vu, moves) == 0
    comp = o.decode(q, ku, vu, table, np.array(lens3, np.int32), scale, Hkv, False)
    assert np.array_equal(comp, got)
    # a move that leaves its block is left out
    assert o.gather_runs(ku, vu, ku.copy(), vu.copy(), [(0, 10, 8, 1, 0)]) == 1


PINS = [pin_f16_exhaustive, pin_bf16_exhaustive, pin_address_worked_example, pin_byte_ledger,
        pin_decode_vs_sdpa, pin_scales_vs_sdpa, pin_permutation_invariance, pin_closed_forms, pin_cache_write,
        pin_copy_on_write_fork, pin_block_moves, pin_multi_query_vs_sdpa, pin_slotted_runs]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(oracle, pin):
    pin(oracle)


# planted mistakes, compiled into separate copies of the oracle; each must fail a pin
MUTANTS = {
    1: "query head h reads kv head h % Hkv (strided groups)",
    2: "scale dropped from the scores",
    3: "offset in block is (t + 1) % B",
    4: "K used in place of V",
    5: "softmax weights not normalised",
    6: "new token taken as position L instead of L - 1",
    7: "cache rows written with a [NB][B][H][D] layout",
    8: "block copy moves kv head 0 only",
    9: "a query token does not attend to its own position",
    10: "a run's slot offset is ignored",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=[MUTANTS[m] for m in sorted(MUTANTS)])
def test_planted_mistake_is_caught(mutant, tmp_path):
    bad = oracle_pkg.Oracle(oracle_pkg.build(mutant=mutant, out_dir=tmp_path))
    caught = []
    for pin in PINS:
        try:
            pin(bad)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin noticed mutant {mutant}: {MUTANTS[mutant]}"


def test_workload_ledger_matches_pages():
    """The seeded generator's pool layout has the pages' byte ledger."""
    import workloads
    wl = workloads.config(2, layers=1, num_seqs=2)
    assert wl.kv_bytes_per_token_per_layer() == 1024
    assert wl.kv_bytes_per_token_per_layer() * 24 * 16 == 393216
    assert wl.block_bytes_per_layer() == 16 * 1024


def test_oracle_threads(oracle):
    assert oracle.num_threads() >= 1
