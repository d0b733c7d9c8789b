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
