"""Host block pool: allocator semantics, the lifecycle of the explainer page's
sequence diagram, copy-on-write, shared prefixes, and slot mappings that match
the oracle bit for bit on every configuration (no GPU needed)."""
from pathlib import Path

import numpy as np
import pytest

import paged_kv_cache_08_gb300 as pa
import workloads

GOLDEN = Path(__file__).resolve().parent / "golden"


def _golden():
    kv = {}
    for line in (GOLDEN / "address_worked_example.txt").read_text(encoding="utf-8").splitlines():
        line = line.strip()
        if line and not line.startswith("#") and not line.startswith("token"):
            k, *rest = line.split()
            kv[k] = [int(x) for x in rest]
    return kv


def test_lowest_free_first_and_exhaustion():
    p = pa.BlockPool(40)
    ids = [p.alloc() for _ in range(40)]
    assert ids == list(range(40))
    with pytest.raises(pa.PAError) as e:
        p.alloc()
    assert e.value.code == -4                      # PA_ERR_POOL_EXHAUSTED
    assert p.decref(33) == 0 and p.decref(5) == 0
    assert p.num_free == 2
    assert p.alloc() == 5                          # lowest free bit wins
    assert p.alloc() == 33
    with pytest.raises(pa.PAError):
        p.decref(40)                               # out of range
    assert p.decref(7) == 0
    with pytest.raises(pa.PAError):
        p.decref(7)                                # already free


def test_refcounts_free_at_zero():
    p = pa.BlockPool(4)
    b = p.alloc()
    assert p.incref(b) == 2 and p.incref(b) == 3
    assert p.decref(b) == 2 and p.decref(b) == 1
    assert p.num_free == 3
    assert p.decref(b) == 0
    assert p.num_free == 4 and p.refcount(b) == 0


def test_sequence_diagram_worked_example():
    """38-token prompt in [7, 3, 12]; the next token lands in #12 at offset 6; once #12
    is full the manager appends #25 and writes at its offset 0; EOS frees them all."""
    g = _golden()
    B = g["block_size"][0]
    new_block = g["grown_table"][-1]
    p = pa.BlockPool(32)
    for _ in range(32):
        p.alloc()                                   # every block taken ...
    p.decref(new_block)                             # ... but #25, the next one handed out
    row = np.full(8, -1, dtype=np.int32)
    row[:3] = g["table"]
    L, phys, off = g["new_token"]
    slot, cs, cd = p.append_token(row, L - 1, B)    # context before the append = L - 1
    assert (slot, cs, cd) == (phys * B + off, -1, -1)
    L2, phys2, off2 = g["new_token_after_growth"]
    slot, cs, cd = p.append_token(row, L2 - 1, B)
    assert (slot, cs, cd) == (phys2 * B + off2, -1, -1)
    assert list(row[:4]) == g["grown_table"]
    assert p.num_free == 0
    p.release(row, L2, B)
    assert p.num_free == 4
    assert list(row[:4]) == [-1] * 4


def test_copy_on_write_fork():
    """Two branches share a prompt (reference count 2).  Appending into a shared,
    partly filled block copies it first; a full shared block is left alone."""
    B = 16
    p = pa.BlockPool(16)
    a = np.full(4, -1, dtype=np.int32)
    p.assign(a, 20, B)                             # blocks [0, 1], 4 tokens in block 1
    b = np.full(4, -1, dtype=np.int32)
    p.assign(b, 20, B, shared_row=a, shared_blocks=2)
    assert list(b[:2]) == list(a[:2]) and p.refcount(a[0]) == 2 and p.refcount(a[1]) == 2
    slot, src, dst = p.append_token(a, 20, B)
    assert src == 1 and dst == a[1] and dst not in (0, 1)
    assert slot == dst * B + 4
    assert p.refcount(1) == 1 and p.refcount(dst) == 1
    slot, src, dst = p.append_token(b, 20, B)      # now the sole owner: no copy
    assert (src, dst) == (-1, -1) and slot == 1 * B + 4
    # full shared prompt blocks ([10, 11] pattern): new tokens go to fresh blocks
    c = np.full(4, -1, dtype=np.int32)
    p.assign(c, 32, B)
    d = np.full(4, -1, dtype=np.int32)
    p.assign(d, 32, B, shared_row=c, shared_blocks=2)
    _, s1, _ = p.append_token(c, 32, B)
    _, s2, _ = p.append_token(d, 32, B)
    assert s1 == -1 and s2 == -1 and c[2] != d[2]
    assert p.refcount(c[0]) == 2 and p.refcount(c[1]) == 2


def _cow_golden():
    kv = {}
    for line in (GOLDEN / "cow_worked_example.txt").read_text(encoding="utf-8").splitlines():
        line = line.strip()
        if line and not line.startswith("#"):
            k, *rest = line.split()
            kv[k] = [int(x) for x in rest]
    return kv


def _pool_with_prompt(prompt_len, B, keep_free):
    """A pool in which other sequences hold every block below 96 except the prompt's two
    blocks and `keep_free`, so that lowest-free allocation hands out the page's ids."""
    g = _cow_golden()
    b10, b11 = g["prompt_blocks"]
    p = pa.BlockPool(128)
    held = [p.alloc() for _ in range(96)]
    for i in keep_free:
        p.decref(i)
    row = np.full(4, -1, dtype=np.int32)
    row[:2] = [b10, b11]                               # the prompt owns #10 and #11 (count 1 each)
    branch = np.full(4, -1, dtype=np.int32)
    p.assign(branch, prompt_len, B, shared_row=row, shared_blocks=2)   # fork: count 2 each
    return p, row, branch, held


def test_copy_on_write_worked_example_ids():
    """§四 of the PagedAttention explainer page, with its block numbers
    (tests/golden/cow_worked_example.txt)."""
    g = _cow_golden()
    b10, b11 = g["prompt_blocks"]
    B = 16
    # the flowchart: the prompt fills #10 and #11, each branch's next token opens a block of its own
    free = [g["figure_table_A"][2]] + list(range(g["figure_table_B"][2], 96))
    p, A, Bt, _ = _pool_with_prompt(2 * B, B, free)
    assert p.refcount(b10) == g["shared_refcount"][0] and p.refcount(b11) == g["shared_refcount"][0]
    _, src, _ = p.append_token(A, 2 * B, B)
    _, src2, _ = p.append_token(Bt, 2 * B, B)
    assert (src, src2) == (-1, -1)
    assert list(A[:3]) == g["figure_table_A"] and list(Bt[:3]) == g["figure_table_B"]
    assert p.refcount(b10) == 2 and p.refcount(b11) == 2
    # the numbered steps: #11 holds 4 tokens when A appends, so A copies it into #45 first
    p, A, Bt, _ = _pool_with_prompt(B + 4, B, [g["cow_new_block"][0]])
    slot, src, dst = p.append_token(A, B + 4, B)
    assert (src, dst) == (b11, g["cow_new_block"][0])
    assert list(A[:2]) == [b10, g["cow_new_block"][0]] and slot == dst * B + 4
    assert p.refcount(b11) == g["refcount_after_cow"][0] and p.refcount(dst) == 1
    slot, src, dst = p.append_token(Bt, B + 4, B)     # B is now #11's only owner: no copy
    assert (src, dst) == (-1, -1) and slot == b11 * B + 4


def test_move_blocks_swap_out_and_in():
    """Swap a sequence out to a host pool of 0.3 x the device pool and back (the tutorial's
    §3.4 sizing): pairs for the copy, freed and allocated blocks, shared blocks kept."""
    dev = pa.BlockPool(40)
    host = pa.BlockPool(12)                          # 0.3 x 40
    B = 16
    a = np.full(8, -1, dtype=np.int32)
    dev.assign(a, 70, B)                             # 5 blocks: 0..4
    b = np.full(8, -1, dtype=np.int32)
    dev.assign(b, 40, B, shared_row=a, shared_blocks=2)   # shares 0, 1; owns 5
    before = a.copy()
    src, dst = dev.move_blocks(host, a, 5)
    assert list(src) == list(before[:5]) and list(dst) == [0, 1, 2, 3, 4]
    assert list(a[:5]) == list(dst)
    assert dev.refcount(0) == 1 and dev.refcount(1) == 1      # still held by b
    assert [dev.refcount(i) for i in (2, 3, 4)] == [0, 0, 0]
    assert host.num_free == 7
    src2, dst2 = host.move_blocks(dev, a, 5)          # swap in: lowest free device blocks
    assert list(src2) == [0, 1, 2, 3, 4] and list(dst2) == [2, 3, 4, 6, 7]
    assert host.num_free == 12
    # too few free blocks: nothing changes
    small = pa.BlockPool(2)
    row = a.copy()
    with pytest.raises(pa.PAError) as e:
        dev.move_blocks(small, row, 5)
    assert e.value.code == -4 and np.array_equal(row, a) and small.num_free == 2
    # an entry that is not allocated in the source pool
    bad = np.array([39, -1], dtype=np.int32)
    with pytest.raises(pa.PAError) as e:
        dev.move_blocks(host, bad, 1)
    assert e.value.code == -6


def test_assign_failure_leaves_pool_unchanged():
    p = pa.BlockPool(3)
    row = np.full(8, -1, dtype=np.int32)
    with pytest.raises(pa.PAError):
        p.assign(row, 4 * 16, 16)
    assert p.num_free == 3


@pytest.mark.parametrize("cfg,B", [(1, None), (2, None), (3, None), (4, None), (5, 16), (5, 32), (5, 64),
                                   (5, 128)])
def test_slot_mapping_matches_oracle(oracle, cfg, B):
    wl = workloads.config(cfg, block_size=B, values=False)
    got = pa.build_slot_mapping(wl.block_tables, wl.context_lens, wl.block_size)
    want = oracle.slot_mapping(wl.block_tables, wl.context_lens, wl.block_size)
    assert np.array_equal(got, want)
    assert (got >= 0).all()


def test_pool_builds_config5_shared_prefix_tables():
    """The pool reproduces config 5's structure: one set of prefix blocks with a
    reference per sequence (plus the resident one), private tails."""
    wl = workloads.config(5, block_size=32, values=False)
    B, S = wl.block_size, wl.num_seqs
    n_prefix = 1024 // B
    p = pa.BlockPool(wl.num_blocks)
    prefix = np.full(wl.max_blocks_per_seq, -1, dtype=np.int32)
    p.assign(prefix, 1024, B)                       # resident prefix owner
    rows = np.full((S, wl.max_blocks_per_seq), -1, dtype=np.int32)
    for s in range(S):
        p.assign(rows[s], int(wl.context_lens[s]), B, shared_row=prefix, shared_blocks=n_prefix)
    for b in prefix[:n_prefix]:
        assert p.refcount(int(b)) == S + 1
    tails = rows[:, n_prefix:]
    used = tails[tails >= 0]
    assert len(set(used.tolist())) == used.size     # tail blocks are private
    slots = pa.build_slot_mapping(rows, wl.context_lens, B)
    assert not np.isin(slots // B, prefix[:n_prefix]).any()   # no write lands in the shared prefix


def _slotted_golden():
    kv = {}
    for line in (GOLDEN / "slotted_worked_example.txt").read_text(encoding="utf-8").splitlines():
        line = line.strip()
        if line and not line.startswith("#"):
            k, *rest = line.split()
            kv[k if k != "slot" else "slot_" + rest[0]] = rest if k != "slot" else [int(x) for x in rest[1:]]
    return kv


def test_slotted_blocks_worked_example():
    """The radix-tree page's slotted block (tests/golden/slotted_worked_example.txt): Node A (5
    tokens) at offset 0 and Node B (8) at offset 5 of one 16-slot block, 3 slots left; a node
    that does not fit the tail opens a fresh block; one that fits takes the tail."""
    g = _slotted_golden()
    B = int(g["block_size"][0])
    p = pa.SlotPool(8, B)
    a_off, a_len = g["slot_A"]
    b_off, b_len = g["slot_B"]
    assert p.alloc(a_len) == (0, a_off)
    assert p.alloc(b_len) == (0, b_off)
    assert B - p.tail(0) == int(g["free_tail"][0])
    assert p.alloc(4) == (1, 0)            # 4 > 3 free slots: a fresh block
    assert p.alloc(3) == (0, 13)           # fills block 0
    assert p.live(0) == 3 and p.num_free == 6
    # releasing a middle slot does not make its space reusable while the block has live slots
    assert p.release(0, b_off, b_len) == 2
    assert p.alloc(2) == (1, 4)
    assert p.release(0, a_off, a_len) == 1 and p.release(0, 13, 3) == 0
    assert p.num_free == 7 and p.tail(0) == 0
    assert p.alloc(16) == (0, 0)           # the emptied block is whole again
    with pytest.raises(pa.PAError):
        p.release(0, 0, 17)
    with pytest.raises(pa.PAError):
        p.alloc(17)
    small = pa.SlotPool(1, B)
    small.alloc(16)
    with pytest.raises(pa.PAError) as e:
        small.alloc(1)
    assert e.value.code == -4
