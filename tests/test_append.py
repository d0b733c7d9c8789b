"""pa_cache_append bit for bit against the oracle's slot rule, and a captured
CUDA graph of (append -> decode) replayed after in-place input changes."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_pa_gb300 as pg
from paged_gqa_decode_pa_gb300 import workloads as wl
from _helpers import assert_close, run_oracle

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "p5_worked_example.json")


def bits_of(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def test_append_lands_in_the_pages_slots_bit_for_bit():
    g = json.load(open(GOLDEN))
    w = wl.p5_example(seed=201)
    q, k, v, t, sl = w.torch_tensors("cuda")
    rng = np.random.default_rng(2)
    k_new = wl.to_bits(rng.standard_normal((w.B, w.Hkv, w.d), dtype=np.float32), "f16")
    v_new = wl.to_bits(rng.standard_normal((w.B, w.Hkv, w.d), dtype=np.float32), "f16")
    kn = torch.from_numpy(k_new.view(np.int16)).view(torch.float16).cuda()
    vn = torch.from_numpy(v_new.view(np.int16)).view(torch.float16).cuda()
    ws = pg.alloc_workspace(pg.shape_of(q, k, t))
    pg.pa_cache_append(kn, vn, k, v, t, sl, ws)
    assert pg.pa_read_status(ws) == 0
    kc, vc, slots, rc = oracle.append(k_new, v_new, w.k_cache, w.v_cache, w.block_table,
                                      w.cache_seqlens)
    assert rc == 0 and slots.tolist() == g["expected_append_slot"]
    assert np.array_equal(bits_of(k), kc)
    assert np.array_equal(bits_of(v), vc)


def test_append_without_a_slot_sets_status_and_writes_nothing():
    w = wl.p5_example(seed=202)
    w.cache_seqlens = np.array([30, 128, 96], np.int32)  # no column / unmapped column
    q, k, v, t, sl = w.torch_tensors("cuda")
    kn = torch.ones((w.B, w.Hkv, w.d), dtype=torch.float16, device="cuda")
    ws = pg.alloc_workspace(pg.shape_of(q, k, t))
    before_k = bits_of(k).copy()
    pg.pa_cache_append(kn, kn, k, v, t, sl, ws)
    assert pg.pa_read_status(ws) & pg.PA_STATUS_NO_SLOT
    after = bits_of(k)
    changed = np.argwhere((after != before_k).any(axis=(2, 3)))
    assert changed.tolist() == [[2, 30]]  # only sequence 0 had a slot


def test_append_then_decode_matches_oracle_with_bf16_and_long_rows():
    w = wl.random_workload([31, 32, 33, 0], H=16, Hkv=4, d=256, bs=32, dtype="bf16", seed=3,
                           maxblk=3)
    # give every sequence a mapped block for its next position
    q, k, v, t, sl = w.torch_tensors("cuda")
    rng = np.random.default_rng(4)
    k_new = wl.to_bits(rng.standard_normal((w.B, w.Hkv, w.d), dtype=np.float32), "bf16")
    v_new = wl.to_bits(rng.standard_normal((w.B, w.Hkv, w.d), dtype=np.float32), "bf16")
    table = w.block_table.copy()
    free = w.num_blocks
    extra = 0
    for b in range(w.B):
        pos = int(w.cache_seqlens[b])
        if table[b, pos // 32] < 0:
            table[b, pos // 32] = free + extra
            extra += 1
    P = w.num_blocks + extra
    kpool = np.concatenate([w.k_cache, np.zeros((extra,) + w.k_cache.shape[1:], np.uint16)])
    vpool = np.concatenate([w.v_cache, np.zeros((extra,) + w.v_cache.shape[1:], np.uint16)])
    w.k_cache, w.v_cache, w.block_table, w.num_blocks = kpool, vpool, table, P
    q, k, v, t, sl = w.torch_tensors("cuda")
    kn = torch.from_numpy(k_new.view(np.int16)).view(torch.bfloat16).cuda()
    vn = torch.from_numpy(v_new.view(np.int16)).view(torch.bfloat16).cuda()
    ws = pg.alloc_workspace(pg.shape_of(q, k, t))
    pg.pa_cache_append(kn, vn, k, v, t, sl, ws)
    sl += 1  # the caller advances the lengths
    out = torch.empty((w.B, w.H, w.d), dtype=torch.float32, device="cuda")
    pg.pa_decode(q, k, v, t, sl, w.scale, out, ws)
    assert pg.pa_read_status(ws) == 0
    kc, vc, _, rc = oracle.append(k_new, v_new, w.k_cache, w.v_cache, table, w.cache_seqlens)
    assert rc == 0
    ref = oracle.decode(w.q, kc, vc, table, w.cache_seqlens + 1, w.scale, "bf16")
    assert_close(out.cpu().numpy().astype(np.float64), ref, "append then decode")


def test_captured_graph_replays_with_inputs_changed_in_place():
    w = wl.random_workload([700, 1500, 64, 3000], H=32, Hkv=8, d=128, bs=32, dtype="bf16",
                           seed=5, maxblk=100, extra_blocks=8)
    q, k, v, t, sl = w.torch_tensors("cuda")
    out = torch.zeros((w.B, w.H, w.d), dtype=torch.float32, device="cuda")
    shape = pg.shape_of(q, k, t)
    ws = pg.alloc_workspace(shape)
    kn = torch.zeros((w.B, w.Hkv, w.d), dtype=torch.bfloat16, device="cuda")
    vn = torch.zeros_like(kn)
    stream = torch.cuda.Stream()
    # first call outside the capture (one-time setup), then capture
    with torch.cuda.stream(stream):
        pg.pa_decode(q, k, v, t, sl, w.scale, out, ws)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        pg.pa_cache_append(kn, vn, k, v, t, sl, ws)
        pg.pa_decode(q, k, v, t, sl, w.scale, out, ws)
    rng = np.random.default_rng(6)
    for step in range(3):
        # new query and new (shorter) lengths, written in place
        q.copy_(torch.from_numpy(wl.to_bits(rng.standard_normal(q.shape, dtype=np.float32),
                                            "bf16").view(np.int16)).view(torch.bfloat16))
        # strictly shorter than the lengths the table was built for, so every
        # appended position has a mapped block
        lens = np.array([699 - step, 1499 - 7 * step, 63 - step, 2999 - 100 * step], np.int32)
        sl.copy_(torch.from_numpy(lens))
        graph.replay()
        torch.cuda.synchronize()
        w.q = bits_of(q)
        w.cache_seqlens = lens
        w.k_cache = bits_of(k)
        w.v_cache = bits_of(v)
        assert_close(out.cpu().numpy().astype(np.float64), run_oracle(w), f"replay {step}")
    assert pg.pa_read_status(ws) == 0


# ------------------------------------------------- fused append-and-attend


def with_room(w, rng):
    """Give every sequence a mapped block for position len (the new token)."""
    table = w.block_table.copy()
    extra = 0
    for b in range(w.B):
        pos = int(w.cache_seqlens[b])
        if pos // w.block_size < table.shape[1] and table[b, pos // w.block_size] < 0:
            table[b, pos // w.block_size] = w.num_blocks + extra
            extra += 1
    if extra:
        pad = wl.to_bits(rng.standard_normal((extra,) + w.k_cache.shape[1:], dtype=np.float32),
                         w.dtype)
        w.k_cache = np.concatenate([w.k_cache, pad])
        w.v_cache = np.concatenate([w.v_cache, pad])
    w.block_table = table
    w.num_blocks += extra
    return w


def fused_vs_oracle(w, opts=None, seed=0):
    rng = np.random.default_rng(seed)
    k_new = wl.to_bits(rng.standard_normal((w.B, w.Hkv, w.d), dtype=np.float32), w.dtype)
    v_new = wl.to_bits(rng.standard_normal((w.B, w.Hkv, w.d), dtype=np.float32), w.dtype)
    q, k, v, t, sl = w.torch_tensors("cuda")
    tdt = k.dtype
    kn = torch.from_numpy(k_new.view(np.int16)).view(tdt).cuda()
    vn = torch.from_numpy(v_new.view(np.int16)).view(tdt).cuda()
    out = torch.full((w.B, w.H, w.d), float("nan"), dtype=torch.float32, device="cuda")
    ws = pg.alloc_workspace(pg.shape_of(q, k, t), opts)
    pg.pa_decode_append(q, kn, vn, k, v, t, sl, w.scale, out, ws, opts)
    status = pg.pa_read_status(ws)
    kc, vc, _, rc = oracle.append(k_new, v_new, w.k_cache, w.v_cache, w.block_table,
                                  w.cache_seqlens)
    return out.cpu().numpy().astype(np.float64), status, bits_of(k), bits_of(v), kc, vc, rc


@pytest.mark.parametrize("mode", ["mma", "simt"])
def test_fused_append_on_the_page_example(mode):
    g = json.load(open(GOLDEN))
    w = wl.p5_example(seed=301)
    got, st, kb, vb, kc, vc, rc = fused_vs_oracle(w, pg.options(compute=mode), seed=1)
    assert st == 0 and rc == 0
    assert np.array_equal(kb, kc) and np.array_equal(vb, vc)
    changed = np.argwhere((kb != w.k_cache).any(axis=(2, 3)))
    assert sorted(map(tuple, changed.tolist())) == sorted(map(tuple, g["expected_append_slot"]))
    ref = oracle.decode(w.q, kc, vc, w.block_table, w.cache_seqlens + 1, w.scale, w.dtype)
    assert_close(got, ref, "fused append, page example")


FUSED = [
    # lengths chosen so new tokens land at row 0 of a new block, at a 16-row
    # tile boundary, mid-tile, at the last row of a block, and as the very
    # first token of a sequence
    ("bs16_d128_g8", dict(lens=[0, 15, 16, 31, 32, 100, 999], H=16, Hkv=2, d=128, bs=16,
                          dtype="bf16")),
    ("bs32_d64_g7_f16", dict(lens=[1, 31, 32, 47, 48, 64, 2000], H=14, Hkv=2, d=64, bs=32,
                             dtype="f16")),
    ("bs64_d256_g6", dict(lens=[63, 64, 65, 80, 3000], H=12, Hkv=2, d=256, bs=64, dtype="bf16")),
    ("bs32_d128_g4", dict(lens=list(wl.serving_mix_lengths(7, 12) // 8), H=32, Hkv=8, d=128,
                          bs=32, dtype="bf16", outlier_frac=0.01)),
]


@pytest.mark.parametrize("mode", ["mma", "simt"])
@pytest.mark.parametrize("name,kw", FUSED, ids=[f[0] for f in FUSED])
def test_fused_append_matches_append_then_decode(name, kw, mode):
    kw = dict(kw)
    lens = kw.pop("lens")
    rng = np.random.default_rng(len(name))
    maxblk = max((n + 1 + kw["bs"] - 1) // kw["bs"] for n in lens) + 1
    for opts in (pg.options(compute=mode), pg.options(compute=mode, num_ctas=5),
                 pg.options(compute=mode, partition_tokens=kw["bs"] * 2)):
        w = with_room(wl.random_workload(lens, seed=len(name) + 3, maxblk=maxblk, **kw), rng)
        got, st, kb, vb, kc, vc, rc = fused_vs_oracle(w, opts, seed=5)
        assert st == 0 and rc == 0, (st, rc)
        assert np.array_equal(kb, kc) and np.array_equal(vb, vc)
        ref = oracle.decode(w.q, kc, vc, w.block_table, w.cache_seqlens + 1, w.scale, w.dtype)
        assert_close(got, ref, f"fused {name} {mode}")
        # the first token of an empty sequence: its output is v_new exactly
        for b, n in enumerate(lens):
            if n == 0:
                for h in range(w.H):
                    vrow = wl.from_bits(vc[w.block_table[b, 0], 0, h // w.G], w.dtype)
                    np.testing.assert_allclose(got[b, h], vrow, rtol=0, atol=1e-6)


def test_fused_append_without_a_slot():
    w = wl.random_workload([10, 48, 5], H=8, Hkv=2, d=64, bs=16, dtype="bf16", seed=9, maxblk=3)
    # sequence 1 is full (48 = 3 blocks x 16): no position for a new token;
    # sequence 2's block for position 5 is unmapped
    w.block_table[2, 0] = -1
    got, st, kb, vb, kc, vc, rc = fused_vs_oracle(w, seed=2)
    assert st & pg.PA_STATUS_BAD_SEQLEN and st & pg.PA_STATUS_NO_SLOT
    assert st & pg.PA_STATUS_BAD_BLOCK
    assert np.isnan(got[1]).all() and np.isnan(got[2]).all()
    # sequence 0 is appended and attended normally
    assert np.array_equal(kb[w.block_table[0, 0], 10], kc[w.block_table[0, 0], 10])
    ref = oracle.decode(w.q[[0]], kc, vc, w.block_table[[0]], np.array([11], np.int32), w.scale,
                        w.dtype)[0]
    assert_close(got[0], ref, "sequence with a slot")
    # nothing else in the pools changed
    diff = np.argwhere((kb != w.k_cache).any(axis=(2, 3)))
    assert diff.tolist() == [[int(w.block_table[0, 0]), 10]]
