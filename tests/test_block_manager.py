"""The host block manager (free list, reference counts, per-sequence block
lists; allocate / free_sequence / share_prefix / copy-on-write as the
"paged-attention-runtime" design page's BlockManager section states them) and
the device block copy that completes a copy-on-write.

CPU tests drive the manager with random operation sequences and check it
against a model that names blocks by *logical identity* (a fresh token per
allocation or copy, the same token where the page says a block is shared), so
no test predicts which physical id the manager picks.  GPU tests check the
copy kernel bit for bit, then run a decode loop whose tables, sharing and
copy-on-write come from the manager, against the oracle evaluated on an
independent contiguous layout of the same logical sequences."""
import itertools
import threading

import numpy as np
import pytest

import paged_gqa_decode_pa_gb300 as pg
from paged_gqa_decode_pa_gb300 import build as pgbuild


@pytest.fixture(scope="module", autouse=True)
def built_library():
    pgbuild.build()
    yield


class Model:
    """Logical-identity model of the manager: seqs[s] is a list of tokens."""

    def __init__(self, P, bs, S, maxblk):
        self.P, self.bs, self.S, self.maxblk = P, bs, S, maxblk
        self.seqs = [[] for _ in range(S)]
        self.fresh = itertools.count()

    def live(self):
        return {t for s in self.seqs for t in s}

    def refs(self, tok):
        return sum(s.count(tok) for s in self.seqs)

    def free(self):
        return self.P - len(self.live())


def check_against_model(bm, m: Model):
    table = bm.block_table(np.arange(m.S), m.maxblk)
    tok_to_id = {}
    for s in range(m.S):
        n = len(m.seqs[s])
        assert bm.num_seq_blocks(s) == n
        assert (table[s, n:] == -1).all()
        for i, tok in enumerate(m.seqs[s]):
            pid = int(table[s, i])
            assert 0 <= pid < m.P
            assert tok_to_id.setdefault(tok, pid) == pid  # one token, one block
    assert len(set(tok_to_id.values())) == len(tok_to_id)  # distinct tokens, distinct blocks
    for tok, pid in tok_to_id.items():
        assert bm.ref_count(pid) == m.refs(tok)
    assert bm.free_blocks() == m.free()
    used = set(tok_to_id.values())
    for pid in range(m.P):
        if pid not in used:
            assert bm.ref_count(pid) == 0


def expect(code, fn, *args):
    with pytest.raises(pg.PagedGQAError) as e:
        fn(*args)
    assert e.value.code == code


def test_page_example_share_then_copy_on_write_then_free():
    # three blocks for sequence 0, its first two shared with sequence 1
    bm = pg.BlockManager(num_blocks=8, block_size=16, max_seqs=4, max_blocks_per_seq=4)
    bm.allocate(0, 3)
    assert bm.block_table([0], 4).tolist() == [[0, 1, 2, -1]]
    bm.share_prefix(0, 1, 2)
    assert bm.block_table([1], 4).tolist() == [[0, 1, -1, -1]]
    assert [bm.ref_count(b) for b in range(3)] == [2, 2, 1]
    assert bm.free_blocks() == 5
    # a write into the shared block 0 of sequence 1 moves it to a private copy
    old, new = bm.copy_on_write(1, 0)
    assert old == 0 and new not in (0, 1, 2)
    assert bm.ref_count(0) == 1 and bm.ref_count(new) == 1
    # a write into an unshared block needs no copy
    assert bm.copy_on_write(0, 2) == (2, 2)
    # freeing sequence 0 returns the blocks whose count reaches zero
    bm.free_sequence(0)
    assert [bm.ref_count(b) for b in range(3)] == [0, 1, 0]
    assert bm.free_blocks() == 8 - 2
    bm.free_sequence(1)
    assert bm.free_blocks() == 8
    bm.close()


def test_reserve_slot_appends_at_a_block_boundary_and_copies_a_shared_tail():
    bm = pg.BlockManager(num_blocks=6, block_size=4, max_seqs=2, max_blocks_per_seq=3)
    bm.allocate(0, 1)
    assert bm.reserve_slot(0, 3) == (0, 0)       # inside its own block
    assert bm.reserve_slot(0, 4) == (1, 1)       # block boundary: one new block
    assert bm.num_seq_blocks(0) == 2
    bm.share_prefix(0, 1, 2)
    old, new = bm.reserve_slot(1, 6)             # shared tail block -> private copy
    assert old == 1 and new != 1 and bm.ref_count(1) == 1
    assert bm.reserve_slot(0, 6) == (1, 1)       # the last sharer writes in place
    expect(pg.PA_ERR_STATE, bm.reserve_slot, 0, 12)   # past max_blocks_per_seq
    expect(pg.PA_ERR_STATE, bm.reserve_slot, 0, 13)   # skips a block
    bm.close()


def test_errors_leave_the_manager_unchanged():
    m = Model(P=5, bs=16, S=3, maxblk=4)
    bm = pg.BlockManager(5, 16, 3, 4)
    bm.allocate(0, 3)
    m.seqs[0] = [next(m.fresh) for _ in range(3)]
    bm.share_prefix(0, 1, 3)
    m.seqs[1] = list(m.seqs[0])
    check_against_model(bm, m)
    expect(pg.PA_ERR_NO_BLOCKS, bm.allocate, 2, 3)      # only 2 free
    expect(pg.PA_ERR_STATE, bm.allocate, 0, 2)          # past max_blocks_per_seq
    expect(pg.PA_ERR_STATE, bm.allocate, 3, 1)          # no such sequence
    expect(pg.PA_ERR_STATE, bm.allocate, 0, -1)
    expect(pg.PA_ERR_STATE, bm.share_prefix, 0, 1, 1)   # target not empty
    expect(pg.PA_ERR_STATE, bm.share_prefix, 0, 2, 4)   # more than the source owns
    expect(pg.PA_ERR_STATE, bm.share_prefix, 0, 0, 1)
    expect(pg.PA_ERR_STATE, bm.copy_on_write, 2, 0)     # index past the list
    expect(pg.PA_ERR_STATE, bm.copy_on_write, 0, -1)
    expect(pg.PA_ERR_STATE, bm.free_sequence, -1)
    expect(pg.PA_ERR_STATE, bm.block_table, [0, 1], 2)  # 3 blocks do not fit 2 columns
    expect(pg.PA_ERR_STATE, pg.pa_bm_query, bm.handle, 7, 0)
    expect(pg.PA_ERR_STATE, pg.pa_bm_query, bm.handle, pg.PA_BM_REF_COUNT, 5)
    check_against_model(bm, m)
    bm.allocate(2, 2)                                   # uses up the free list
    m.seqs[2] = [next(m.fresh) for _ in range(2)]
    expect(pg.PA_ERR_NO_BLOCKS, bm.copy_on_write, 1, 0)  # shared, nothing free
    check_against_model(bm, m)
    bm.close()
    for bad in ((0, 16, 1, 1), (4, 0, 1, 1), (4, 16, 0, 1), (4, 16, 1, 0)):
        with pytest.raises(pg.PagedGQAError):
            pg.BlockManager(*bad)
    assert pg.lib().pa_bm_allocate(None, 0, 1) == pg.PA_ERR_STATE


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_match_the_logical_model(seed):
    rng = np.random.default_rng(seed)
    P, S, maxblk = int(rng.integers(4, 40)), int(rng.integers(2, 9)), int(rng.integers(1, 9))
    m = Model(P, 16, S, maxblk)
    bm = pg.BlockManager(P, 16, S, maxblk)
    for step in range(400):
        op = rng.integers(0, 5)
        s = int(rng.integers(0, S))
        if op == 0:
            n = int(rng.integers(0, 4))
            if len(m.seqs[s]) + n > maxblk:
                expect(pg.PA_ERR_STATE, bm.allocate, s, n)
            elif n > m.free():
                expect(pg.PA_ERR_NO_BLOCKS, bm.allocate, s, n)
            else:
                bm.allocate(s, n)
                m.seqs[s] += [next(m.fresh) for _ in range(n)]
        elif op == 1:
            bm.free_sequence(s)
            m.seqs[s] = []
        elif op == 2:
            t = int(rng.integers(0, S))
            n = int(rng.integers(0, maxblk + 1))
            if t == s or m.seqs[t] or n > len(m.seqs[s]):
                expect(pg.PA_ERR_STATE, bm.share_prefix, s, t, n)
            else:
                bm.share_prefix(s, t, n)
                m.seqs[t] = m.seqs[s][:n]
        elif op == 3:
            if not m.seqs[s]:
                expect(pg.PA_ERR_STATE, bm.copy_on_write, s, 0)
                continue
            i = int(rng.integers(0, len(m.seqs[s])))
            tok = m.seqs[s][i]
            shared = m.refs(tok) > 1
            if shared and m.free() == 0:
                expect(pg.PA_ERR_NO_BLOCKS, bm.copy_on_write, s, i)
                continue
            old, new = bm.copy_on_write(s, i)
            assert (old != new) == shared
            if shared:
                m.seqs[s][i] = next(m.fresh)
        else:
            pos = int(rng.integers(0, 16 * (len(m.seqs[s]) + 1)))
            i = pos // 16
            if i >= maxblk:
                expect(pg.PA_ERR_STATE, bm.reserve_slot, s, pos)
            elif i == len(m.seqs[s]):
                if m.free() == 0:
                    expect(pg.PA_ERR_NO_BLOCKS, bm.reserve_slot, s, pos)
                else:
                    old, new = bm.reserve_slot(s, pos)
                    assert old == new
                    m.seqs[s].append(next(m.fresh))
            else:
                tok = m.seqs[s][i]
                shared = m.refs(tok) > 1
                if shared and m.free() == 0:
                    expect(pg.PA_ERR_NO_BLOCKS, bm.reserve_slot, s, pos)
                else:
                    old, new = bm.reserve_slot(s, pos)
                    assert (old != new) == shared
                    if shared:
                        m.seqs[s][i] = next(m.fresh)
        check_against_model(bm, m)
    bm.close()


def test_concurrent_threads_keep_the_counts_consistent():
    P, S = 256, 32
    bm = pg.BlockManager(P, 16, S, 8)

    def worker(k):
        rng = np.random.default_rng(100 + k)
        for _ in range(300):
            s = 4 * k + int(rng.integers(0, 4))  # each thread owns 4 sequences
            try:
                if rng.random() < 0.5:
                    bm.allocate(s, int(rng.integers(1, 3)))
                else:
                    bm.free_sequence(s)
            except pg.PagedGQAError as e:
                assert e.code in (pg.PA_ERR_STATE, pg.PA_ERR_NO_BLOCKS)

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    table = bm.block_table(np.arange(S), 8)
    ids = table[table >= 0]
    assert len(set(ids.tolist())) == ids.size  # nothing handed out twice
    assert bm.free_blocks() == P - ids.size
    for pid in ids:
        assert bm.ref_count(int(pid)) == 1
    bm.close()


def test_copy_blocks_rejects_bad_arguments_before_any_cuda_call():
    L = pg.lib()
    import ctypes

    s = pg.pa_shape(0, 2, 2, 128, 16, 1, 8, pg.PA_BF16)
    FAKE = 1 << 20
    assert L.pa_copy_blocks(None, FAKE, FAKE, FAKE, 1, None, None) == pg.PA_ERR_NULL
    assert L.pa_copy_blocks(ctypes.byref(s), FAKE, FAKE, None, 1, None, None) == pg.PA_ERR_NULL
    assert L.pa_copy_blocks(ctypes.byref(s), FAKE + 2, FAKE, FAKE, 1, None, None) == pg.PA_ERR_ALIGN
    assert L.pa_copy_blocks(ctypes.byref(s), FAKE, FAKE, FAKE, -1, None, None) == pg.PA_ERR_SHAPE
    bad = pg.pa_shape(0, 2, 2, 12, 16, 1, 8, pg.PA_BF16)
    assert L.pa_copy_blocks(ctypes.byref(bad), FAKE, FAKE, FAKE, 1, None, None) == pg.PA_ERR_SHAPE
    assert L.pa_copy_blocks(ctypes.byref(s), FAKE, FAKE, None, 0, None, None) == pg.PA_OK


# ------------------------------------------------------------------ GPU


def _pool(rng, P, bs, Hkv, d):
    import torch

    bits = rng.integers(0, 1 << 16, size=(P, bs, Hkv, d), dtype=np.uint16)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def _bits(t):
    import torch

    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.gpu
def test_copy_blocks_bit_exact_and_bad_ids_flagged():
    import torch

    rng = np.random.default_rng(11)
    P, bs, Hkv, d = 40, 16, 4, 128
    k, v = _pool(rng, P, bs, Hkv, d), _pool(rng, P, bs, Hkv, d)
    k0, v0 = _bits(k), _bits(v)
    perm = rng.permutation(P)
    src, dst = perm[:12], perm[12:24]  # destinations distinct, never a source
    pairs = torch.from_numpy(np.stack([src, dst], 1).astype(np.int32)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pg.pa_copy_blocks(k, v, pairs, status)
    torch.cuda.synchronize()
    k1, v1 = _bits(k), _bits(v)
    ek, ev = k0.copy(), v0.copy()
    ek[dst], ev[dst] = k0[src], v0[src]
    assert np.array_equal(k1, ek) and np.array_equal(v1, ev)
    assert int(status.item()) == 0
    # an out-of-range id copies nothing and sets the status bit
    bad = torch.tensor([[0, P], [-1, 3], [5, 6]], dtype=torch.int32, device="cuda")
    pg.pa_copy_blocks(k, v, bad, status)
    torch.cuda.synchronize()
    k2 = _bits(k)
    ek[6] = k1[5]
    assert np.array_equal(k2, ek)
    assert int(status.item()) == pg.PA_STATUS_BAD_BLOCK


def _oracle_on_contiguous_layout(seqs_k, seqs_v, q, lens, bs, scale):
    """The oracle over the logical sequences laid out one after another (a
    plain table independent of the manager's placement)."""
    import oracle

    B = len(lens)
    maxblk = max(1, max(-(-int(n) // bs) for n in lens))
    Hkv, d = seqs_k[0].shape[1:]
    kp = np.zeros((B * maxblk, bs, Hkv, d), np.uint16)
    vp = np.zeros_like(kp)
    table = np.arange(B * maxblk, dtype=np.int32).reshape(B, maxblk)
    for b, n in enumerate(lens):
        flat_k = kp[b * maxblk:(b + 1) * maxblk].reshape(maxblk * bs, Hkv, d)
        flat_v = vp[b * maxblk:(b + 1) * maxblk].reshape(maxblk * bs, Hkv, d)
        flat_k[:n], flat_v[:n] = seqs_k[b][:n], seqs_v[b][:n]
    return oracle.decode(q, kp, vp, table, np.asarray(lens, np.int32), scale, "bf16")


@pytest.mark.gpu
@pytest.mark.parametrize("fused", [True, False])
def test_decode_loop_with_prefix_sharing_and_copy_on_write_matches_oracle(fused):
    import torch
    from _helpers import assert_close
    from paged_gqa_decode_pa_gb300 import workloads as wl

    rng = np.random.default_rng(21 + fused)
    H, Hkv, d, bs, P, S, maxblk = 16, 2, 128, 16, 96, 6, 12
    scale = d ** -0.5
    bm = pg.BlockManager(P, bs, S, maxblk)
    k_pool = torch.zeros((P, bs, Hkv, d), dtype=torch.bfloat16, device="cuda")
    v_pool = torch.zeros_like(k_pool)

    def rows(n):
        return wl.to_bits(rng.standard_normal((n, Hkv, d), dtype=np.float32), "bf16")

    def write_rows(s, start, kk, vv):  # prefill plumbing: place rows by the table
        t = bm.block_table([s], maxblk)[0]
        for i in range(kk.shape[0]):
            pos = start + i
            blk = int(t[pos // bs])
            k_pool[blk, pos % bs] = torch.from_numpy(kk[i].view(np.int16)).view(torch.bfloat16)
            v_pool[blk, pos % bs] = torch.from_numpy(vv[i].view(np.int16)).view(torch.bfloat16)

    # sequence 0 holds a 40-token prefix (2.5 blocks); 1..4 share all three of
    # its blocks, the partial one included; 5 is independent
    logical_k, logical_v = {}, {}
    pk, pv = rows(40), rows(40)
    bm.allocate(0, 3)
    write_rows(0, 0, pk, pv)
    logical_k[0], logical_v[0] = pk.copy(), pv.copy()
    for s in range(1, 5):
        bm.share_prefix(0, s, 3)
        logical_k[s], logical_v[s] = pk.copy(), pv.copy()
    bm.allocate(5, 2)
    k5, v5 = rows(25), rows(25)
    write_rows(5, 0, k5, v5)
    logical_k[5], logical_v[5] = k5, v5
    assert bm.ref_count(2) == 5 and bm.free_blocks() == P - 5

    active = [0, 1, 2, 3, 4, 5]
    copies = 0
    for step in range(24):
        if step == 10:
            # sequence 2 ends; a new request reuses its id and shares all of
            # sequence 1's blocks, so both must copy the tail on their next write
            bm.free_sequence(2)
            n1 = logical_k[1].shape[0]
            bm.share_prefix(1, 2, -(-n1 // bs))
            logical_k[2], logical_v[2] = logical_k[1].copy(), logical_v[1].copy()
        lens = [logical_k[s].shape[0] for s in active]
        pairs = []
        for s, n in zip(active, lens):
            old, new = bm.reserve_slot(s, n)
            if old != new:
                pairs.append((old, new))
        copies += len(pairs)
        if pairs:
            pg.pa_copy_blocks(k_pool, v_pool,
                              torch.tensor(pairs, dtype=torch.int32, device="cuda"))
        table = torch.from_numpy(bm.block_table(active, maxblk)).cuda()
        seqlens = torch.tensor(lens, dtype=torch.int32, device="cuda")
        B = len(active)
        qb = wl.to_bits(rng.standard_normal((B, H, d), dtype=np.float32), "bf16")
        kn, vn = rows(B), rows(B)
        q = torch.from_numpy(qb.view(np.int16)).view(torch.bfloat16).cuda()
        ktn = torch.from_numpy(kn.view(np.int16)).view(torch.bfloat16).cuda()
        vtn = torch.from_numpy(vn.view(np.int16)).view(torch.bfloat16).cuda()
        out = torch.full((B, H, d), float("nan"), dtype=torch.float32, device="cuda")
        ws = pg.alloc_workspace(pg.shape_of(q, k_pool, table))
        if fused:
            pg.pa_decode_append(q, ktn, vtn, k_pool, v_pool, table, seqlens, scale, out, ws)
        else:
            pg.pa_cache_append(ktn, vtn, k_pool, v_pool, table, seqlens, ws)
            pg.pa_decode(q, k_pool, v_pool, table, seqlens + 1, scale, out, ws)
        assert pg.pa_read_status(ws) == 0
        for i, s in enumerate(active):
            logical_k[s] = np.concatenate([logical_k[s], kn[i:i + 1]])
            logical_v[s] = np.concatenate([logical_v[s], vn[i:i + 1]])
        ref = _oracle_on_contiguous_layout([logical_k[s] for s in active],
                                           [logical_v[s] for s in active], qb,
                                           [n + 1 for n in lens], bs, scale)
        assert_close(out.cpu().numpy().astype(np.float64), ref, f"step {step}")
    # five sharers of the partial block 2 each wrote into it: four copies; the
    # re-shared sequences 1 and 2 copy once more
    assert copies == 4 + 1
    # the pool, read back through the manager's tables, holds every sequence
    kb, vb = _bits(k_pool), _bits(v_pool)
    table = bm.block_table(active, maxblk)
    for i, s in enumerate(active):
        n = logical_k[s].shape[0]
        blocks = table[i, :-(-n // bs)]
        assert (blocks >= 0).all()
        got_k = kb[blocks].reshape(-1, Hkv, d)[:n]
        got_v = vb[blocks].reshape(-1, Hkv, d)[:n]
        assert np.array_equal(got_k, logical_k[s]) and np.array_equal(got_v, logical_v[s])
    live = set(table[table >= 0].tolist())
    assert bm.free_blocks() == P - len(live)
    bm.close()
