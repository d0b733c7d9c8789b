"""GPU path vs the float64 oracle, element by element, through the C ABI.

Tolerance (fp16/bf16 inputs, fp32 output): max|err| <= 2e-3 and
mean|err| <= 2e-4.  Index handling is checked bit for bit by poisoning every
pool slot no valid token maps to with NaN: the output must not change in a
single bit.
"""
import math
import zlib

import numpy as np
import pytest
import torch

import paged_gqa_decode_pa_gb300 as pg
from paged_gqa_decode_pa_gb300 import workloads as wl
from _helpers import assert_close, run_gpu, run_oracle, sample_pairs

pytestmark = pytest.mark.gpu

MODES = ["mma", "simt"]


@pytest.fixture(scope="module", autouse=True)
def built_library():
    from paged_gqa_decode_pa_gb300 import build

    build.build()
    pg.lib()
    yield


# ------------------------------------------------ the page's worked example


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("part,ctas", [(0, 0), (0, 1), (0, 5), (32, 0), (32, 3), (64, 2)])
def test_p5_example(mode, dtype, part, ctas):
    w = wl.p5_example(seed=101, dtype=dtype)
    got, st = run_gpu(w, pg.options(partition_tokens=part, compute=mode, num_ctas=ctas))
    assert st == 0
    assert_close(got, run_oracle(w), f"p5 {mode} {dtype} part={part} ctas={ctas}")


@pytest.mark.parametrize("mode", MODES)
def test_p5_example_poisoned_rows_change_no_bit(mode):
    for part, ctas in [(0, 0), (0, 4), (32, 0)]:
        o = pg.options(partition_tokens=part, compute=mode, num_ctas=ctas)
        clean, _ = run_gpu(wl.p5_example(seed=102), o)
        dirty, st = run_gpu(wl.p5_example(seed=102, poison=True), o)
        assert st == 0
        assert np.array_equal(clean, dirty)


def test_p5_tagged_values_give_the_row_means():
    # keys zero, values tagged by (block, row): out = mean of the tags of the
    # rows the page says each sequence reads
    w = wl.p5_example(seed=103)
    P, bs, Hkv, d = w.k_cache.shape
    w.k_cache[...] = 0
    p = np.arange(P)[:, None, None, None]
    r = np.arange(bs)[None, :, None, None]
    j = np.arange(Hkv)[None, None, :, None]
    k = np.arange(d)[None, None, None, :]
    tags = np.where(k % 2 == 0, 1.0, -1.0) * (32 * p + r) * 2.0 ** j
    w.v_cache[...] = wl.to_bits(tags.astype(np.float32), "f16")
    for mode in MODES:
        got, st = run_gpu(w, pg.options(compute=mode))
        assert st == 0
        for b, mean in enumerate([78.5, 15.5, 10351 / 70]):
            for h in range(w.H):
                expect = np.where(np.arange(d) % 2 == 0, 1.0, -1.0) * mean * 2.0 ** (h // w.G)
                np.testing.assert_allclose(got[b, h], expect, rtol=2e-6, atol=0)


# ------------------------------------------------------- seeded workloads


@pytest.mark.parametrize("mode", MODES)
def test_qwen2_b8_g7_d64(mode):
    w = wl.qwen2_b8_g7_d64()
    ref = run_oracle(w)
    for part in (0, 512):
        got, st = run_gpu(w, pg.options(partition_tokens=part, compute=mode))
        assert st == 0
        assert_close(got, ref, f"qwen2 {mode} part={part}")


SMALL = [
    # (name, kwargs) -- reduced versions of the large settings, several tiles
    # and a ragged tail each
    ("long_ctx_10k_g6_d256", dict(lens=[10_007], H=24, Hkv=4, d=256, bs=16, dtype="bf16")),
    ("prefix_b8_g8_d128", dict(lens=[512, 777, 1024, 2049, 3000, 513, 4096, 600], H=64, Hkv=8,
                               d=128, bs=16, dtype="bf16", shared_prefix_blocks=32)),
    ("serving_b24_g4_d128", dict(lens=list(wl.serving_mix_lengths(5, 24) // 4 + 1), H=32,
                                 Hkv=8, d=128, bs=32, dtype="bf16", outlier_frac=0.01,
                                 outlier_scale=8.0)),
    ("mha_g1_d128_bs64", dict(lens=[1, 63, 64, 65, 1000], H=4, Hkv=4, d=128, bs=64,
                              dtype="f16")),
    ("g8_d64_bs32_f16", dict(lens=[5, 31, 32, 33, 700], H=16, Hkv=2, d=64, bs=32, dtype="f16")),
    ("g3_d256_bs32_bf16", dict(lens=[1, 40, 333], H=6, Hkv=2, d=256, bs=32, dtype="bf16")),
    ("g5_d64_bs16_bf16", dict(lens=[17, 0, 250, 16], H=10, Hkv=2, d=64, bs=16, dtype="bf16")),
]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("name,kw", SMALL, ids=[s[0] for s in SMALL])
def test_reduced_settings(name, kw, mode):
    kw = dict(kw)
    lens = kw.pop("lens")
    w = wl.random_workload(lens, seed=zlib.crc32(name.encode()) % 1000, name=name, **kw)
    ref = run_oracle(w)
    for part, ctas in [(0, 0), (0, 7), (512, 0), (kw["bs"] * 2, 0)]:
        got, st = run_gpu(w, pg.options(partition_tokens=part, compute=mode, num_ctas=ctas))
        assert st == 0
        assert_close(got, ref, f"{name} {mode} part={part} ctas={ctas}")


def test_more_merged_segments_than_the_preloaded_descriptors():
    """With many short rows and a large grid, most rows continue past a split
    CTA: more than 512 segments have pieces to merge, so the merge CTAs'
    search for their segment runs past the descriptor chunks it preloads."""
    rng = np.random.default_rng(77)
    lens = rng.integers(600, 1200, 400).astype(np.int32)
    w = wl.random_workload(lens, H=4, Hkv=2, d=64, bs=16, dtype="f16", seed=78)
    o = pg.options(num_ctas=1200)
    s = pg.pa_shape(w.B, w.H, w.Hkv, w.d, w.block_size, w.max_blocks_per_seq, w.num_blocks,
                    pg.PA_F16)
    merged = sum(pg.pa_plan_merge(s, o, lens, 1200, c) is not None for c in range(1200))
    assert merged > 512
    got, st = run_gpu(w, o)
    assert st == 0
    assert_close(got, run_oracle(w), "1200 CTAs")


@pytest.mark.parametrize("mode", MODES)
def test_poison_and_determinism_on_ragged_batch(mode):
    lens = [1, 15, 16, 17, 100, 0, 255, 1024]
    kw = dict(H=16, Hkv=4, d=128, bs=16, dtype="bf16", extra_blocks=7)
    o = pg.options(compute=mode, num_ctas=13)
    clean, _ = run_gpu(wl.random_workload(lens, seed=5, **kw), o)
    again, _ = run_gpu(wl.random_workload(lens, seed=5, **kw), o)
    dirty, st = run_gpu(wl.random_workload(lens, seed=5, poison=True, **kw), o)
    assert st == 0
    assert np.array_equal(clean, again)
    assert np.array_equal(clean, dirty)
    assert np.array_equal(clean[5], np.zeros_like(clean[5]))  # empty sequence


@pytest.mark.parametrize("layout", ["v_below_k", "same_buffer"])
def test_pool_placement_does_not_matter(layout):
    # K and V normally come in one copy per tile through a map spanning both
    # pools; it must give the same result when the V pool sits below the K
    # pool, and the two-map path must serve K and V sharing one buffer.
    w = wl.random_workload([300, 77, 1, 512], H=8, Hkv=2, d=128, bs=32, dtype="bf16", seed=31)
    ref_w = wl.random_workload([300, 77, 1, 512], H=8, Hkv=2, d=128, bs=32, dtype="bf16", seed=31)
    if layout == "same_buffer":
        w.v_cache = w.k_cache.copy()
        ref_w.v_cache = ref_w.k_cache.copy()
    q, k, v, t, sl = w.torch_tensors("cuda")
    if layout == "v_below_k":
        both = torch.empty((2,) + tuple(k.shape), dtype=k.dtype, device="cuda")
        both[0].copy_(v)
        both[1].copy_(k)
        v, k = both[0], both[1]
        assert v.data_ptr() < k.data_ptr()
    else:
        v = k
    out = torch.full((w.B, w.H, w.d), float("nan"), dtype=torch.float32, device="cuda")
    ws = pg.alloc_workspace(pg.shape_of(q, k, t))
    pg.pa_decode(q, k, v, t, sl, w.scale, out, ws)
    assert pg.pa_read_status(ws) == 0
    assert_close(out.cpu().numpy().astype(np.float64), run_oracle(ref_w), layout)


def test_empty_and_full_sequences():
    # all empty; and one sequence that fills every table column
    w = wl.random_workload([0, 0, 0], H=8, Hkv=2, d=64, bs=16, dtype="f16", seed=7, maxblk=3)
    got, st = run_gpu(w)
    assert st == 0 and np.array_equal(got, np.zeros_like(got))
    w = wl.random_workload([48, 3], H=8, Hkv=2, d=64, bs=16, dtype="f16", seed=8, maxblk=3)
    got, st = run_gpu(w)
    assert st == 0
    assert_close(got, run_oracle(w), "full table row")


@pytest.mark.parametrize("G", [1, 2, 3, 5, 6, 7, 8])
def test_every_group_size_over_one_cache(G):
    """The same cache, table and lengths read by G = 1..8 query heads per kv
    head: every group size the library takes, odd ones included."""
    base = wl.random_workload([1, 15, 16, 17, 300, 0, 1000, 129], H=8, Hkv=4, d=128, bs=16,
                              dtype="bf16", seed=41, poison=True, outlier_frac=0.02)
    w = wl.with_group(base, G, seed=50 + G)
    assert w.H == 4 * G
    for opts in (None, pg.options(num_ctas=7)):
        got, st = run_gpu(w, opts)
        assert st == 0
        assert_close(got, run_oracle(w), f"G={G}")


def test_simt_and_mma_agree():
    w = wl.random_workload([3000, 1, 77], H=24, Hkv=4, d=256, bs=16, dtype="bf16", seed=9)
    a, _ = run_gpu(w, pg.options(compute="mma"))
    b, _ = run_gpu(w, pg.options(compute="simt"))
    assert np.abs(a - b).max() <= 2 * 2e-3


# ------------------------------------------------------------ data errors


def test_bad_block_entry_poisons_only_its_group_and_sets_status():
    w = wl.random_workload([100, 200, 50], H=8, Hkv=2, d=64, bs=16, dtype="bf16", seed=11)
    ref = run_oracle(w)
    w.block_table[1, 3] = -1  # inside sequence 1's length
    for mode in MODES:
        got, st = run_gpu(w, pg.options(compute=mode))
        assert st & pg.PA_STATUS_BAD_BLOCK
        assert np.isnan(got[1]).all()
        assert_close(got[[0, 2]], ref[[0, 2]], "untouched sequences")
    w.block_table[1, 3] = w.num_blocks  # out of range
    got, st = run_gpu(w, pg.options(num_ctas=5))
    assert st & pg.PA_STATUS_BAD_BLOCK and np.isnan(got[1]).all()


def test_bad_seqlen_poisons_its_sequence_and_sets_status():
    w = wl.random_workload([100, 200, 50], H=8, Hkv=2, d=64, bs=16, dtype="bf16", seed=12)
    ref = run_oracle(w)
    for bad in (-5, w.max_blocks_per_seq * w.block_size + 1):
        w2 = wl.random_workload([100, 200, 50], H=8, Hkv=2, d=64, bs=16, dtype="bf16", seed=12)
        w2.cache_seqlens[2] = bad
        got, st = run_gpu(w2)
        assert st & pg.PA_STATUS_BAD_SEQLEN
        assert np.isnan(got[2]).all()
        assert_close(got[:2], ref[:2], "other sequences")
    # status is sticky until read, then cleared
    got, st = run_gpu(w)
    assert st == 0


# ------------------------------------------------------------ full sizes


FULL = ["long_ctx_100k_g6_d256", "prefix_share_b64_g8_d128", "serving_mix_b256_g4_d128"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_settings_sampled(name):
    w = wl.make(name)
    pairs = sample_pairs(w, 48, seed=1)
    ref = run_oracle(w, pairs=pairs)
    for opts in (pg.options(), pg.options(partition_tokens=512)):
        got, st = run_gpu(w, opts)
        assert st == 0
        assert np.isfinite(got).all()
        sub = got[pairs[:, 0], pairs[:, 1]]
        assert_close(sub, ref, name)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("scale", [-0.2, 0.0])
def test_negative_and_zero_scale(mode, scale):
    """A negative scale turns the softmax towards the smallest q.k; a zero
    scale weighs every visible key the same (the mean of V)."""
    w = wl.random_workload([300, 17, 1000, 64], H=16, Hkv=4, d=128, bs=16, dtype="bf16", seed=71)
    w.scale = scale
    for opts in (pg.options(compute=mode), pg.options(compute=mode, num_ctas=7)):
        got, st = run_gpu(w, opts)
        assert st == 0
        assert_close(got, run_oracle(w), f"scale {scale} {mode}")


@pytest.mark.parametrize("G", [1, 8])
def test_one_long_sequence_among_many_short_ones(G):
    """Many more rows than split CTAs, but one segment holding most of the
    keys: it spans most of the persistent grid, so its merge folds well over
    a hundred pieces (more than one batch of loads)."""
    lens = [1] * 300 + [40000] + [3] * 100
    w = wl.random_workload(lens, H=G, Hkv=1, d=128, bs=16, dtype="bf16", seed=81 + G,
                           poison=True)
    got, st = run_gpu(w)
    assert st == 0
    assert_close(got, run_oracle(w), f"one long sequence, G={G}")
    again, _ = run_gpu(w)
    assert np.array_equal(got, again)
