"""Pins of the float64 oracle against facts that do not come from the oracle.

Each test names what fixes the expected value: the Hugging Face decoding-path
worked example (tests/golden/p5_worked_example.json), IEEE/numpy decoding of
16-bit patterns, torch's scaled_dot_product_attention (a library routine) on
contiguous layouts, closed forms, and invariants of softmax attention.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_pa_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "p5_worked_example.json")


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def f16(x):
    return np.asarray(x, dtype=np.float16).view(np.uint16)


# ---------------------------------------------------------------- widening


def test_widen_fp16_matches_numpy_for_every_pattern():
    # numpy's float16 is IEEE binary16; compare all 65536 patterns.
    lib_vals = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    for bits in range(65536):
        ref = float(lib_vals[bits])
        got = oracle.widen(bits, "f16")
        if math.isnan(ref):
            assert math.isnan(got), hex(bits)
        else:
            assert got == ref, hex(bits)
    assert oracle.widen(0x0001, "f16") == 2.0 ** -24
    assert oracle.widen(0x7BFF, "f16") == 65504.0


def test_widen_bf16_known_patterns():
    assert oracle.widen(0x3F80, "bf16") == 1.0
    assert oracle.widen(0xC0A0, "bf16") == -5.0
    assert oracle.widen(0x0001, "bf16") == 2.0 ** -133
    assert oracle.widen(0x7F7F, "bf16") == float(np.float32(3.3895313892515355e38))
    t = torch.tensor([0.1, -3.75, 1e-30, 12345.0]).to(torch.bfloat16)
    for v, b in zip(t.float().tolist(), t.view(torch.int16).numpy().view(np.uint16).tolist()):
        assert oracle.widen(b, "bf16") == v


# ---------------------------------------------------- page's worked example


def tagged_p5(dtype="f16"):
    g = golden()
    w = wl.p5_example(seed=11, dtype=dtype)
    P, bs, Hkv, d = w.k_cache.shape
    w.k_cache[...] = 0  # +0.0 in both fp16 and bf16
    p = np.arange(P)[:, None, None, None]
    r = np.arange(bs)[None, :, None, None]
    j = np.arange(Hkv)[None, None, :, None]
    k = np.arange(d)[None, None, None, :]
    sign = np.where(k % 2 == 0, 1.0, -1.0)
    tags = sign * (32 * p + r) * (2.0 ** j)
    w.v_cache[...] = wl.to_bits(tags.astype(np.float32), dtype)
    assert w.block_table.tolist() == g["facts_from_the_page"]["block_table"]
    assert w.cache_seqlens.tolist() == g["facts_from_the_page"]["cache_seqlens"]
    assert w.block_size == g["facts_from_the_page"]["block_size"]
    return w, g


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_p5_example_reads_exactly_the_rows_the_page_names(dtype):
    w, g = tagged_p5(dtype)
    out = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens, w.scale, dtype)
    G = w.G
    sign = np.where(np.arange(w.d) % 2 == 0, 1.0, -1.0)
    for b, (num, den) in enumerate(g["expected_tag_mean_exact"]):
        for h in range(w.H):
            expect = sign * (num / den) * 2.0 ** (h // G)
            np.testing.assert_allclose(out[b, h], expect, rtol=0, atol=1e-12)


def test_p5_example_ignores_rows_it_must_not_read():
    w, g = tagged_p5()
    clean = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens, w.scale,
                          "f16")
    # random keys too, so that poisoned rows would change the weights
    w2 = wl.p5_example(seed=12)
    base = oracle.decode(w2.q, w2.k_cache, w2.v_cache, w2.block_table, w2.cache_seqlens,
                         w2.scale, "f16")
    nr = g["rows_never_read"]
    for wk in (w, w2):
        for blk in nr["whole_blocks"]:
            wk.k_cache[blk] = wl.nan_bits("f16")
            wk.v_cache[blk] = wl.nan_bits("f16")
        wk.k_cache[2, nr["block_2_rows_from"]:] = wl.nan_bits("f16")
        wk.v_cache[2, nr["block_2_rows_from"]:] = wl.nan_bits("f16")
        wk.k_cache[6, nr["block_6_rows_from"]:] = wl.nan_bits("f16")
        wk.v_cache[6, nr["block_6_rows_from"]:] = wl.nan_bits("f16")
    poisoned = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens,
                             w.scale, "f16")
    assert np.array_equal(poisoned, clean)
    poisoned2 = oracle.decode(w2.q, w2.k_cache, w2.v_cache, w2.block_table, w2.cache_seqlens,
                              w2.scale, "f16")
    assert np.array_equal(poisoned2, base)
    # the generator's own read mask agrees with the page
    mask = wl.p5_example().read_mask()
    assert not mask[[1, 4, 7]].any()
    assert mask[2, :30].all() and not mask[2, 30:].any()
    assert mask[6, :6].all() and not mask[6, 6:].any()
    assert mask[[0, 3, 5]].all()


def test_p5_append_slots_match_the_page():
    g = golden()
    w = wl.p5_example(seed=13)
    rng = np.random.default_rng(0)
    k_new = f16(rng.standard_normal((w.B, w.Hkv, w.d)))
    v_new = f16(rng.standard_normal((w.B, w.Hkv, w.d)))
    kc, vc, slots, rc = oracle.append(k_new, v_new, w.k_cache, w.v_cache, w.block_table,
                                      w.cache_seqlens)
    assert rc == 0
    assert slots.tolist() == g["expected_append_slot"]
    changed = np.argwhere((kc != w.k_cache).any(axis=(2, 3)))
    assert sorted(map(tuple, changed.tolist())) == sorted(map(tuple, g["expected_append_slot"]))
    for b, (p, r) in enumerate(g["expected_append_slot"]):
        assert np.array_equal(kc[p, r], k_new[b])
        assert np.array_equal(vc[p, r], v_new[b])


def test_append_without_a_slot_is_reported():
    w = wl.p5_example(seed=14)
    sl = np.array([30, 128, 70], dtype=np.int32)  # 128 = 4 blocks * 32: no column left
    k_new = np.zeros((w.B, w.Hkv, w.d), np.uint16)
    kc, vc, slots, rc = oracle.append(k_new, k_new, w.k_cache, w.v_cache, w.block_table, sl)
    assert rc == -2 and slots[1].tolist() == [-1, -1]
    sl = np.array([30, 32, 96], dtype=np.int32)  # 96 -> table column 3 is -1
    kc, vc, slots, rc = oracle.append(k_new, k_new, w.k_cache, w.v_cache, w.block_table, sl)
    assert rc == -3 and slots[2].tolist() == [-1, -1] and slots[0].tolist() == [2, 30]


# ------------------------------------------------------ closed forms


def test_single_token_returns_its_value_row():
    w = wl.random_workload([1, 1, 1], H=8, Hkv=2, d=64, bs=16, dtype="bf16", seed=21,
                           extra_blocks=3)
    out = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens, w.scale,
                        "bf16")
    for b in range(w.B):
        p = w.block_table[b, 0]
        for h in range(w.H):
            v = wl.from_bits(w.v_cache[p, 0, h // w.G], "bf16").astype(np.float64)
            assert np.array_equal(out[b, h], v)


def test_identical_keys_give_the_mean_of_values():
    w = wl.random_workload([37, 100], H=4, Hkv=4, d=64, bs=16, dtype="f16", seed=22)
    w.k_cache[:] = w.k_cache[0, 0, 0][None, None, None, :]
    out = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens, w.scale,
                        "f16")
    for b in range(w.B):
        n = int(w.cache_seqlens[b])
        rows = [wl.from_bits(w.v_cache[w.block_table[b, t // 16], t % 16], "f16")
                for t in range(n)]
        mean = np.mean(np.stack(rows).astype(np.float64), axis=0)  # [Hkv, d]
        for h in range(w.H):
            np.testing.assert_allclose(out[b, h], mean[h], rtol=0, atol=1e-12)


@pytest.mark.parametrize("a", [0.75, 40.0, 1000.0, 8000.0])
def test_two_tokens_follow_the_logistic_closed_form(a):
    # q = a * e0, K rows carry c0, c1 in dim 0 only: s_t = scale * a * c_t.
    d, bs = 64, 16
    w = wl.random_workload([2], H=1, Hkv=1, d=d, bs=bs, dtype="f16", seed=23)
    q = np.zeros((1, 1, d), np.float32)
    q[0, 0, 0] = a
    w.q = f16(q)
    c = (1.5, -2.25)
    p = w.block_table[0, 0]
    kz = np.zeros((bs, 1, d), np.float32)
    kz[0, 0, 0], kz[1, 0, 0] = c
    w.k_cache[p] = f16(kz)
    scale = 0.125
    out = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens, scale, "f16")
    s0, s1 = scale * a * c[0], scale * a * c[1]
    w0 = 1.0 / (1.0 + math.exp(min(s1 - s0, 700.0)))
    v0 = wl.from_bits(w.v_cache[p, 0, 0], "f16").astype(np.float64)
    v1 = wl.from_bits(w.v_cache[p, 1, 0], "f16").astype(np.float64)
    expect = w0 * v0 + (1.0 - w0) * v1
    assert np.isfinite(out).all()
    np.testing.assert_allclose(out[0, 0], expect, rtol=1e-13, atol=1e-13)


def test_empty_sequence_gives_zero():
    w = wl.random_workload([0, 5], H=4, Hkv=2, d=64, bs=16, dtype="bf16", seed=24, maxblk=2)
    out = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens, w.scale,
                        "bf16")
    assert np.array_equal(out[0], np.zeros((4, 64)))
    assert np.abs(out[1]).sum() > 0


# ------------------------------------------------- a library routine


def contiguous_workload(lens, H, Hkv, d, bs, dtype, seed):
    """Sequence b owns physical blocks [b*maxblk, (b+1)*maxblk) in order."""
    w = wl.random_workload(lens, H, Hkv, d, bs, dtype=dtype, seed=seed)
    maxblk = w.max_blocks_per_seq
    B = w.B
    P = B * maxblk
    rng = np.random.default_rng(seed + 7)
    w.k_cache = wl.to_bits(rng.standard_normal((P, bs, Hkv, d), dtype=np.float32), dtype)
    w.v_cache = wl.to_bits(rng.standard_normal((P, bs, Hkv, d), dtype=np.float32), dtype)
    table = np.full((B, maxblk), -1, np.int32)
    for b in range(B):
        nb = (int(w.cache_seqlens[b]) + bs - 1) // bs
        table[b, :nb] = np.arange(b * maxblk, b * maxblk + nb)
    w.block_table = table
    w.num_blocks = P
    return w


@pytest.mark.parametrize("H,Hkv,d,bs,dtype", [
    (4, 2, 64, 32, "f16"), (14, 2, 64, 16, "f16"), (24, 4, 256, 16, "bf16"),
    (8, 8, 128, 16, "bf16"), (32, 8, 128, 32, "bf16"), (6, 1, 64, 16, "f16"),
])
def test_matches_torch_sdpa_on_contiguous_layout(H, Hkv, d, bs, dtype):
    lens = [1, 17, bs * 3, 150]
    w = contiguous_workload(lens, H, Hkv, d, bs, dtype, seed=31 + H + d)
    out = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens, w.scale,
                        dtype)
    G = H // Hkv
    maxblk = w.max_blocks_per_seq
    for b, n in enumerate(lens):
        kk = wl.from_bits(w.k_cache[b * maxblk:(b + 1) * maxblk], dtype)
        vv = wl.from_bits(w.v_cache[b * maxblk:(b + 1) * maxblk], dtype)
        kk = torch.from_numpy(kk.reshape(maxblk * bs, Hkv, d)[:n]).double()
        vv = torch.from_numpy(vv.reshape(maxblk * bs, Hkv, d)[:n]).double()
        # [heads, tokens, d]; query head h reads kv head h // G
        kk = kk.permute(1, 0, 2).repeat_interleave(G, dim=0)
        vv = vv.permute(1, 0, 2).repeat_interleave(G, dim=0)
        qq = torch.from_numpy(wl.from_bits(w.q[b], dtype)).double()[:, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=w.scale)
        np.testing.assert_allclose(out[b], ref[:, 0, :].numpy(), rtol=1e-11, atol=1e-12)


# ----------------------------------------------------------- invariants


def test_permuting_physical_blocks_with_the_table_changes_nothing():
    w = wl.random_workload([33, 64, 1, 200], H=8, Hkv=2, d=128, bs=16, dtype="bf16", seed=41,
                           extra_blocks=5)
    base = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens, w.scale,
                         "bf16")
    perm = np.random.default_rng(1).permutation(w.num_blocks)  # new id of old block
    k2 = np.empty_like(w.k_cache)
    v2 = np.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    t2 = np.where(w.block_table >= 0, perm[np.maximum(w.block_table, 0)], -1).astype(np.int32)
    out = oracle.decode(w.q, k2, v2, t2, w.cache_seqlens, w.scale, "bf16")
    assert np.array_equal(out, base)


def test_adding_a_vector_to_every_key_changes_nothing():
    # keys are small multiples of 1/16 and u = 0.5: k + u is exact in fp16
    w = wl.random_workload([50, 9], H=4, Hkv=2, d=64, bs=16, dtype="f16", seed=42)
    rng = np.random.default_rng(3)
    kq = rng.integers(-16, 16, size=w.k_cache.shape).astype(np.float32) / 16
    w.k_cache = f16(kq)
    base = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens, w.scale,
                         "f16")
    u = np.full(w.d, 0.5, np.float32)
    u[::3] = -1.0
    w.k_cache = f16(kq + u)
    out = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens, w.scale,
                        "f16")
    np.testing.assert_allclose(out, base, rtol=0, atol=1e-12)


def test_output_is_linear_in_values():
    w = wl.random_workload([70, 3], H=4, Hkv=2, d=64, bs=32, dtype="f16", seed=43)
    rng = np.random.default_rng(4)
    v1 = rng.integers(-64, 64, size=w.v_cache.shape).astype(np.float32)
    v2 = rng.integers(-64, 64, size=w.v_cache.shape).astype(np.float32)
    outs = []
    for v in (v1, v2, v1 + 2 * v2):
        outs.append(oracle.decode(w.q, w.k_cache, f16(v), w.block_table, w.cache_seqlens,
                                  w.scale, "f16"))
    np.testing.assert_allclose(outs[2], outs[0] + 2 * outs[1], rtol=1e-12, atol=1e-10)


def test_query_heads_read_the_kv_head_of_their_group():
    w = wl.random_workload([40, 77], H=12, Hkv=3, d=64, bs=16, dtype="bf16", seed=44)
    G = w.G
    # same query in every head of a group -> same output within the group
    for b in range(w.B):
        for j in range(w.Hkv):
            w.q[b, j * G:(j + 1) * G] = w.q[b, j * G]
    out = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens, w.scale,
                        "bf16")
    for b in range(w.B):
        for j in range(w.Hkv):
            for g in range(1, G):
                assert np.array_equal(out[b, j * G + g], out[b, j * G])
    # changing kv head 1 changes exactly the heads of group 1
    v2 = w.v_cache.copy()
    v2[:, :, 1, :] = wl.to_bits(np.ones((w.num_blocks, w.block_size, w.d), np.float32), "bf16")
    out2 = oracle.decode(w.q, w.k_cache, v2, w.block_table, w.cache_seqlens, w.scale, "bf16")
    changed = np.abs(out2 - out).sum(axis=2) > 0  # [B, H]
    expect = np.zeros_like(changed)
    expect[:, G:2 * G] = True
    assert np.array_equal(changed, expect)


# ----------------------------------------------------------- split-KV merge


@pytest.mark.parametrize("piece", [512, 100, 1])
def test_split_pieces_combined_equal_the_unsplit_result(piece):
    w = wl.random_workload([1500, 513, 7], H=6, Hkv=1, d=64, bs=16, dtype="bf16", seed=51,
                           outlier_frac=0.05, outlier_scale=8.0)
    full = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens, w.scale,
                         "bf16")
    for b in range(w.B):
        n = int(w.cache_seqlens[b])
        for h in (0, 5):
            ms, ls, accs = [], [], []
            for t0 in range(0, n, piece):
                m, l, a = oracle.partial(w.q, w.k_cache, w.v_cache, w.block_table,
                                         w.cache_seqlens, w.scale, "bf16", b, h, t0,
                                         min(n, t0 + piece))
                ms.append(m)
                ls.append(l)
                accs.append(a)
            m, l, a = oracle.combine(ms, ls, np.stack(accs))
            np.testing.assert_allclose(a / l, full[b, h], rtol=1e-12, atol=1e-12)


def test_combine_has_an_identity_and_ignores_order():
    w = wl.random_workload([300], H=2, Hkv=1, d=64, bs=16, dtype="f16", seed=52)
    parts = [oracle.partial(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens,
                            w.scale, "f16", 0, 1, t0, t0 + 60) for t0 in range(0, 300, 60)]
    ms = [p[0] for p in parts]
    ls = [p[1] for p in parts]
    accs = np.stack([p[2] for p in parts])
    m, l, a = oracle.combine(ms, ls, accs)
    order = [3, 0, 4, 1, 2]
    m2, l2, a2 = oracle.combine([ms[i] for i in order], [ls[i] for i in order], accs[order])
    assert m == m2
    np.testing.assert_allclose(a2 / l2, a / l, rtol=1e-13, atol=1e-14)
    # empty piece is the identity
    e = oracle.partial(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens, w.scale,
                       "f16", 0, 1, 10, 10)
    assert e[0] == -math.inf and e[1] == 0.0 and not e[2].any()
    m3, l3, a3 = oracle.combine([e[0]] + ms, [e[1]] + ls, np.vstack([e[2][None], accs]))
    assert m3 == m and l3 == l and np.array_equal(a3, a)


def test_large_scores_stay_finite_and_agree_between_forms():
    w = wl.random_workload([3000], H=4, Hkv=1, d=128, bs=32, dtype="bf16", seed=53,
                           outlier_frac=0.01, outlier_scale=64.0)
    full = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens, w.scale,
                         "bf16")
    assert np.isfinite(full).all()
    for h in range(4):
        parts = [oracle.partial(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens,
                                w.scale, "bf16", 0, h, t0, min(3000, t0 + 512))
                 for t0 in range(0, 3000, 512)]
        m, l, a = oracle.combine([p[0] for p in parts], [p[1] for p in parts],
                                 np.stack([p[2] for p in parts]))
        np.testing.assert_allclose(a / l, full[0, h], rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------- errors


def test_refuses_unmapped_entries_inside_a_sequence():
    w = wl.p5_example(seed=61)
    t = w.block_table.copy()
    t[2, 1] = -1
    with pytest.raises(oracle.OracleError):
        oracle.decode(w.q, w.k_cache, w.v_cache, t, w.cache_seqlens, w.scale, "f16")
    t[2, 1] = 8  # == P
    with pytest.raises(oracle.OracleError):
        oracle.decode(w.q, w.k_cache, w.v_cache, t, w.cache_seqlens, w.scale, "f16")
    sl = w.cache_seqlens.copy()
    sl[0] = 129  # > 4 blocks * 32
    with pytest.raises(oracle.OracleError):
        oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, sl, w.scale, "f16")
    sl[0] = -1
    with pytest.raises(oracle.OracleError):
        oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, sl, w.scale, "f16")


def test_pairs_subset_matches_full_output():
    w = wl.random_workload([90, 33, 250], H=8, Hkv=4, d=64, bs=16, dtype="bf16", seed=62)
    full = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens, w.scale,
                         "bf16")
    pairs = np.array([[2, 7], [0, 0], [1, 3]], np.int32)
    sub = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens, w.scale,
                        "bf16", pairs=pairs)
    for i, (b, h) in enumerate(pairs):
        assert np.array_equal(sub[i], full[b, h])


# ------------------------------------------- several query tokens per sequence

VARLEN = os.path.join(os.path.dirname(__file__), "golden", "hf_varlen_example.json")


def varlen_example(dtype):
    g = json.load(open(VARLEN))["facts_from_the_page"]
    H, Hkv, d, bs = 4, 2, 64, 16
    cu_q = np.array(g["cu_seq_lens_q"], np.int32)
    cu_k = np.array(g["cu_seq_lens_k"], np.int32)
    lens = np.diff(cu_k).astype(np.int32)
    table = np.array([[-1], [1], [2]], np.int32)
    P = 3
    k = np.zeros((P, bs, Hkv, d), np.uint16)  # +0.0
    vals = np.zeros((P, bs, Hkv, d), np.float32)
    sign = np.where(np.arange(d) % 2 == 0, 1.0, -1.0)
    for kidx, req in enumerate(g["k_request_index"]):
        t = kidx - cu_k[req]                      # position inside its request
        blk = table[req, t // bs]
        for j in range(Hkv):
            vals[blk, t % bs, j] = sign * (kidx + 1) * 2.0 ** j
    v = wl.to_bits(vals, dtype)
    rng = np.random.default_rng(5)
    q = wl.to_bits(rng.standard_normal((int(cu_q[-1]), H, d)).astype(np.float32), dtype)
    return g, q, cu_q, k, v, table, lens, H, Hkv, d


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_example_assigns_rows_to_the_pages_requests(dtype, causal):
    g, q, cu_q, k, v, table, lens, H, Hkv, d = varlen_example(dtype)
    gold = json.load(open(VARLEN))
    assert q.shape[0] == g["q_shape_tokens"] and int(lens.sum()) == g["k_shape_tokens"]
    out = oracle.decode_multi(q, cu_q, causal, k, v, table, lens, 0.125, dtype)
    want = gold["expected_tag_per_row_causal" if causal else "expected_tag_per_row_noncausal"]
    G = H // Hkv
    sign = np.where(np.arange(d) % 2 == 0, 1.0, -1.0)
    for r in range(q.shape[0]):
        for h in range(H):
            np.testing.assert_allclose(out[r, h], sign * want[r] * 2.0 ** (h // G), rtol=1e-12,
                                       atol=0)
    if not causal:
        # the row -> request map the page draws, read back from the tags
        tag_of_request = {0: 0, 1: 1, 2: 5}
        got = [next(b for b, t in tag_of_request.items() if t == want[r]) for r in range(14)]
        assert got == g["q_request_index"]


def packed_queries(rng, lens_q, H, d, dtype):
    cu = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    q = wl.to_bits(rng.standard_normal((int(cu[-1]), H, d)).astype(np.float32), dtype)
    return cu, q


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Hkv,d", [(8, 2, 64), (6, 3, 128), (8, 1, 64)])
def test_multi_matches_torch_sdpa_with_an_explicit_mask(causal, H, Hkv, d):
    rng = np.random.default_rng(H * 10 + d + causal)
    bs, dtype = 16, "bf16"
    lens_k = [37, 5, 64, 1]
    lens_q = [4, 5, 3, 2]       # sequence 1 and 3 have more queries than the
    w = contiguous_workload(lens_k, H, Hkv, d, bs, dtype, seed=7)  # early ones can see
    cu, q = packed_queries(rng, lens_q, H, d, dtype)
    out = oracle.decode_multi(q, cu, causal, w.k_cache, w.v_cache, w.block_table,
                              w.cache_seqlens, w.scale, dtype)
    G = H // Hkv
    qf = torch.from_numpy(wl.from_bits(q, dtype)).double()
    for b, (nk, nq) in enumerate(zip(lens_k, lens_q)):
        kf = torch.from_numpy(wl.from_bits(
            w.k_cache[w.block_table[b]].reshape(-1, Hkv, d)[:nk], dtype)).double()
        vf = torch.from_numpy(wl.from_bits(
            w.v_cache[w.block_table[b]].reshape(-1, Hkv, d)[:nk], dtype)).double()
        qq = qf[cu[b]:cu[b + 1]].permute(1, 0, 2)              # [H, nq, d]
        kk = kf.permute(1, 0, 2).repeat_interleave(G, dim=0)   # [H, nk, d]
        vv = vf.permute(1, 0, 2).repeat_interleave(G, dim=0)
        i = torch.arange(nq)[:, None]
        t = torch.arange(nk)[None, :]
        mask = (t < nk - nq + i + 1) if causal else torch.ones(nq, nk, dtype=torch.bool)
        seen = mask.any(dim=1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qq[:, seen], kk, vv, attn_mask=mask[seen], scale=w.scale)
        got = torch.from_numpy(out[cu[b]:cu[b + 1]]).permute(1, 0, 2)
        np.testing.assert_allclose(got[:, seen].numpy(), ref.numpy(), rtol=1e-10, atol=1e-12)
        assert (got[:, ~seen] == 0).all()  # queries that see no key give 0


def test_causal_query_equals_a_single_token_decode_on_the_prefix():
    # query i of n_q attends to exactly the first k_len - n_q + i + 1 tokens
    rng = np.random.default_rng(17)
    w = wl.random_workload([70, 33], H=8, Hkv=2, d=64, bs=16, dtype="f16", seed=9)
    lens_q = [6, 4]
    cu, q = packed_queries(rng, lens_q, w.H, w.d, "f16")
    out = oracle.decode_multi(q, cu, True, w.k_cache, w.v_cache, w.block_table,
                              w.cache_seqlens, w.scale, "f16")
    for b in range(2):
        for i in range(lens_q[b]):
            r = cu[b] + i
            n = int(w.cache_seqlens[b]) - lens_q[b] + i + 1
            one = oracle.decode(q[r][None], w.k_cache, w.v_cache, w.block_table[[b]],
                                np.array([n], np.int32), w.scale, "f16")
            np.testing.assert_array_equal(out[r], one[0])


def test_multi_rejects_bad_cumulative_lengths_and_rows_outside_sequences_are_zero():
    w = wl.random_workload([20, 9], H=4, Hkv=2, d=64, bs=16, dtype="f16", seed=3)
    rng = np.random.default_rng(1)
    q = wl.to_bits(rng.standard_normal((6, 4, 64)).astype(np.float32), "f16")
    for bad in ([0, 3, 2], [0, 3, 7], [-1, 2, 4]):
        with pytest.raises(oracle.OracleError):
            oracle.decode_multi(q, bad, True, w.k_cache, w.v_cache, w.block_table,
                                w.cache_seqlens, w.scale, "f16")
    out = oracle.decode_multi(q, [1, 3, 4], False, w.k_cache, w.v_cache, w.block_table,
                              w.cache_seqlens, w.scale, "f16")
    assert (out[0] == 0).all() and (out[4:] == 0).all() and (out[1:4] != 0).any()
    pairs = np.array([[2, 3], [4, 0], [1, 1]], np.int32)
    sub = oracle.decode_multi(q, [1, 3, 4], False, w.k_cache, w.v_cache, w.block_table,
                              w.cache_seqlens, w.scale, "f16", pairs=pairs)
    np.testing.assert_array_equal(sub, out[pairs[:, 0], pairs[:, 1]])
