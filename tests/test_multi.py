"""Several query tokens per sequence (pa_decode_multi) against the oracle.

Packed query rows and cumulative query counts follow the varlen path of the
Hugging Face "Paged attention" page; keys come from the paged cache, the query
tokens being each sequence's last positions (causal or not)."""
import ctypes
import json
import os

import numpy as np
import pytest

import oracle
import paged_gqa_decode_pa_gb300 as pg
from paged_gqa_decode_pa_gb300 import build as pgbuild
from paged_gqa_decode_pa_gb300 import workloads as wl

VARLEN = os.path.join(os.path.dirname(__file__), "golden", "hf_varlen_example.json")


@pytest.fixture(scope="module", autouse=True)
def built_library():
    pgbuild.build()
    yield


# ------------------------------------------------------------------ host


def shape(B=3, H=8, Hkv=2, d=128, bs=16, maxblk=8, P=16, dtype=pg.PA_BF16):
    return pg.pa_shape(B, H, Hkv, d, bs, maxblk, P, dtype)


FAKE = 1 << 20


def call_multi(s, opts=None, q=FAKE, cu=FAKE, total_q=8, max_q=4, ws_bytes=1 << 30):
    L = pg.lib()
    return L.pa_decode_multi(ctypes.byref(s), ctypes.byref(opts) if opts else None, q, cu,
                             total_q, max_q, 1, FAKE, FAKE, FAKE, FAKE, 0.1, FAKE, FAKE,
                             ws_bytes, None)


def test_multi_rejects_bad_arguments_before_any_cuda_call():
    s = shape()
    assert call_multi(s, max_q=0) == pg.PA_ERR_SHAPE
    assert call_multi(s, max_q=pg.PA_MAX_QUERY_TOKENS + 1) == pg.PA_ERR_SHAPE
    assert call_multi(s, total_q=-1) == pg.PA_ERR_SHAPE
    assert call_multi(s, cu=None) == pg.PA_ERR_NULL
    assert call_multi(s, cu=FAKE + 4) == pg.PA_ERR_ALIGN
    assert call_multi(s, q=None) == pg.PA_ERR_NULL
    assert call_multi(s, pg.options(compute="simt", num_ctas=8)) == pg.PA_ERR_OPTION
    assert call_multi(s, pg.options(num_ctas=8), ws_bytes=64) == pg.PA_ERR_WORKSPACE
    # nothing to do: no sequences, or no query rows
    assert call_multi(shape(B=0), q=None, cu=None) == pg.PA_OK
    assert call_multi(s, total_q=0) == pg.PA_OK


def test_workspace_grows_with_query_groups():
    o = pg.options(num_ctas=304)
    s = shape(B=64, H=32, Hkv=8, d=128, bs=32, maxblk=256, P=20000)  # G = 4
    one = pg.pa_workspace_size(s, o)
    # 16 columns per pass at d = 128: four tokens of four heads in one group
    assert pg.pa_workspace_size_multi(s, 4, o) > one
    # fixed partitions: slots scale with the groups per sequence
    of = pg.options(num_ctas=304, partition_tokens=512)
    g1 = pg.pa_workspace_size_multi(s, 4, of)    # 1 group
    g3 = pg.pa_workspace_size_multi(s, 12, of)   # two rows of 32 columns (warp pairs)
    assert g3 > 2.5 * g1
    # above 16 columns a row holds 32 (warp pairs): 5 to 8 tokens of G = 4 are one row of 32
    # columns, 9 tokens are two
    g5, g8, g9 = (pg.pa_workspace_size_multi(s, n, of) for n in (5, 8, 9))
    assert g5 == g8 and 1.8 * g1 < g8 < 2.2 * g1 and 1.8 * g8 < g9 < 2.2 * g8


# ------------------------------------------------------------------ GPU


def run_multi(w, opts=None, max_q=None, prefill_nan=True, total_q=None):
    import torch

    q, k, v, t, sl = w.torch_tensors("cuda")
    cu = torch.from_numpy(w.cu_q).cuda()
    mq = max_q or w.max_q
    if total_q is not None and total_q != q.shape[0]:
        raise ValueError("packed q already has total_q rows")
    out = torch.full((q.shape[0], w.H, w.d), float("nan") if prefill_nan else 0.0,
                     dtype=torch.float32, device="cuda")
    ws = pg.alloc_workspace_multi(pg.shape_multi(q, k, t), mq, opts)
    pg.pa_decode_multi(q, cu, mq, w.causal, k, v, t, sl, w.scale, out, ws, opts)
    status = pg.pa_read_status(ws)
    return out.cpu().numpy().astype(np.float64), status


def oracle_multi(w, pairs=None):
    return oracle.decode_multi(w.q, w.cu_q, w.causal, w.k_cache, w.v_cache, w.block_table,
                               w.cache_seqlens, w.scale, w.dtype, pairs=pairs)


def covered_rows(w):
    return np.arange(int(w.cu_q[0]), int(w.cu_q[-1]))


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_example_of_the_page(dtype, causal):
    from _helpers import assert_close

    g = json.load(open(VARLEN))
    facts = g["facts_from_the_page"]
    lens_k = np.diff(facts["cu_seq_lens_k"]).astype(np.int32)
    lens_q = np.diff(facts["cu_seq_lens_q"]).astype(np.int32)
    H, Hkv, d, bs = 4, 2, 64, 16
    w = wl.random_workload(lens_k, H, Hkv, d, bs, dtype=dtype, seed=3, maxblk=1)
    w.k_cache[...] = 0
    vals = np.zeros(w.v_cache.shape, np.float32)
    sign = np.where(np.arange(d) % 2 == 0, 1.0, -1.0)
    for kidx, req in enumerate(facts["k_request_index"]):
        tpos = kidx - facts["cu_seq_lens_k"][req]
        blk = w.block_table[req, tpos // bs]
        for j in range(Hkv):
            vals[blk, tpos % bs, j] = sign * (kidx + 1) * 2.0 ** j
    w.v_cache[...] = wl.to_bits(vals, dtype)
    w = wl.with_query_tokens(w, lens_q, seed=4, causal=causal)
    got, status = run_multi(w, max_q=facts["max_length_q"])
    assert status == 0
    want = g["expected_tag_per_row_causal" if causal else "expected_tag_per_row_noncausal"]
    G = H // Hkv
    exp = np.array([[sign * want[r] * 2.0 ** (h // G) for h in range(H)] for r in range(14)])
    assert_close(got, exp, "varlen example")
    assert_close(got, oracle_multi(w), "varlen example vs oracle")


CASES = [
    # lens_k, lens_q, H, Hkv, d, bs, dtype
    ([300, 17, 1, 64, 513], [4, 3, 1, 4, 2], 16, 4, 128, 16, "bf16"),     # G=4: one group
    ([129, 40, 700], [1, 5, 2], 8, 1, 64, 32, "f16"),                     # G=8: tq=2, 3 groups
    ([260, 33, 5, 90], [7, 2, 6, 1], 6, 2, 128, 16, "bf16"),              # G=3: tq=5, 2 groups
    ([200, 64, 31], [3, 1, 2], 12, 2, 256, 16, "bf16"),                   # d=256: 8 columns
    ([2, 3, 50, 0], [5, 3, 1, 2], 4, 4, 64, 16, "f16"),                   # fewer keys than queries
    ([1000, 2500], [16, 9], 8, 8, 128, 64, "bf16"),                       # G=1: 16 tokens a pass
    ([500, 77, 1200, 9], [8, 8, 5, 3], 16, 4, 128, 32, "bf16"),          # G=4, 8 tokens: warp pairs
    ([900, 40], [20, 13], 8, 2, 128, 16, "f16"),                          # pairs, 3 groups of 8 tokens
    ([300, 64, 2000], [4, 2, 3], 14, 2, 64, 16, "f16"),                   # G=7, d=64: 28 columns
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("opts", [None, dict(num_ctas=5), dict(partition_tokens=64, num_ctas=7)])
def test_random_shapes_match_the_oracle(case, causal, opts):
    from _helpers import assert_close

    lens_k, lens_q, H, Hkv, d, bs, dtype = CASES[case]
    if opts and opts.get("partition_tokens") and opts["partition_tokens"] % bs:
        opts = dict(opts, partition_tokens=bs * 4)
    w = wl.random_workload(lens_k, H, Hkv, d, bs, dtype=dtype, seed=40 + case, poison=True,
                           outlier_frac=0.02)
    w = wl.with_query_tokens(w, lens_q, seed=50 + case, causal=causal)
    got, status = run_multi(w, pg.options(**opts) if opts else None)
    assert status == 0
    ref = oracle_multi(w)
    assert_close(got, ref, f"case {case}")


@pytest.mark.gpu
def test_rows_outside_the_sequences_are_not_written_and_larger_max_q_changes_nothing():
    import torch
    from _helpers import assert_close

    w = wl.random_workload([77, 150], 8, 2, 128, 16, dtype="bf16", seed=8)
    w = wl.with_query_tokens(w, [3, 2], seed=9)
    # two spare rows before and after the packed queries
    q = np.concatenate([w.q[:2] * 0, w.q, w.q[:2] * 0])
    w.q = q
    w.cu_q = w.cu_q + 2
    got, status = run_multi(w)
    assert status == 0
    assert np.isnan(got[:2]).all() and np.isnan(got[-2:]).all()
    ref = oracle_multi(w)
    assert_close(got[2:-2], ref[2:-2], "packed rows")
    again, _ = run_multi(w, max_q=40)  # 10 groups per sequence, most of them empty
    assert_close(again[2:-2], ref[2:-2], "max_q 40")


@pytest.mark.gpu
def test_one_query_token_each_matches_pa_decode():
    from _helpers import assert_close, run_gpu, run_oracle

    w = wl.random_workload([90, 1, 400, 33], 8, 2, 128, 32, dtype="bf16", seed=12)
    dec, st = run_gpu(w)
    assert st == 0
    m = wl.random_workload([90, 1, 400, 33], 8, 2, 128, 32, dtype="bf16", seed=12)
    m.cu_q = np.arange(m.B + 1, dtype=np.int32)  # q [B, H, d] is already packed
    for causal in (True, False):
        m.causal = causal
        got, st = run_multi(m)
        assert st == 0
        assert_close(got, run_oracle(w), "multi q=1")
        assert np.abs(got - dec).max() <= 1e-5


@pytest.mark.gpu
def test_bad_spans_and_lengths_set_status():
    w = wl.random_workload([40, 50, 60], 4, 2, 64, 16, dtype="f16", seed=13, maxblk=4)
    w = wl.with_query_tokens(w, [2, 3, 2], seed=14)
    # with max_q = 2, sequence 1's three tokens are not a valid span; sequence
    # 2's key length is past its table
    w.cache_seqlens = np.array([40, 50, 65], np.int32)
    got, status = run_multi(w, max_q=2, prefill_nan=False)
    assert status == pg.PA_STATUS_BAD_SEQLEN
    ref = oracle.decode_multi(w.q, w.cu_q, True, w.k_cache, w.v_cache, w.block_table,
                              np.array([40, 0, 0], np.int32), w.scale, "f16")
    np.testing.assert_allclose(got[:2], ref[:2], atol=2e-3)   # sequence 0 is fine
    assert (got[2:5] == 0).all()      # sequence 1 skipped: rows not written
    assert np.isnan(got[5:7]).all()   # sequence 2: NaN


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["serving_mix_b256_q4_g4_d128", "prefix_share_b64_q2_g8_d128"])
def test_full_size_settings_on_sampled_outputs(name):
    from _helpers import assert_close

    w = wl.make(name)
    got, status = run_multi(w)
    assert status == 0
    rng = np.random.default_rng(3)
    rows = rng.integers(0, w.q.shape[0], 96)
    heads = rng.integers(0, w.H, 96)
    pairs = np.unique(np.stack([rows, heads], 1).astype(np.int32), axis=0)
    ref = oracle_multi(w, pairs=pairs)
    assert_close(got[pairs[:, 0], pairs[:, 1]], ref, name)


@pytest.mark.gpu
def test_eight_query_tokens_full_size_sampled():
    """The serving mix with 8 query tokens per sequence (rows of 32 columns,
    one warp per row: the columns are the mma's M dimension), causal."""
    from _helpers import assert_close

    base = wl.make("serving_mix_b256_g4_d128")
    w = wl.with_query_tokens(base, np.full(base.B, 8, np.int32), seed=base.seed + 2000,
                             causal=True)
    got, status = run_multi(w)
    assert status == 0
    rng = np.random.default_rng(5)
    rows = np.concatenate([[0, w.q.shape[0] - 1], rng.integers(0, w.q.shape[0], 126)])
    heads = rng.integers(0, w.H, rows.shape[0])
    pairs = np.unique(np.stack([rows, heads], 1).astype(np.int32), axis=0)
    ref = oracle_multi(w, pairs=pairs)
    assert_close(got[pairs[:, 0], pairs[:, 1]], ref, "8 query tokens")


@pytest.mark.gpu
@pytest.mark.parametrize("scale", [-0.2, 0.0, 0.7])
def test_wide_rows_take_any_scale(scale):
    """Rows of more than 16 columns apply |scale| with q negated for a
    negative scale, and a zero scale gives every visible key the same weight."""
    from _helpers import assert_close

    w = wl.random_workload([300, 40, 1000], 16, 4, 128, 16, dtype="bf16", seed=61)
    w = wl.with_query_tokens(w, [8, 5, 7], seed=62, causal=True)
    w.scale = scale
    got, status = run_multi(w)
    assert status == 0
    assert_close(got, oracle_multi(w), f"scale {scale}")


@pytest.mark.gpu
def test_wide_rows_bad_entries_poison_and_determinism():
    """Rows of 32 columns (8 tokens at G = 4): a bad table entry inside one
    sequence's length makes that sequence's rows NaN and sets the status bit,
    the other sequences match the oracle, NaN-poisoned unread rows change no
    bit, and two runs give the same bits."""
    from _helpers import assert_close

    lens_k, lens_q = [700, 90, 1500, 33], [8, 6, 8, 3]

    def make(poison):
        w = wl.random_workload(lens_k, 16, 4, 128, 16, dtype="bf16", seed=71, poison=poison,
                               outlier_frac=0.02)
        return wl.with_query_tokens(w, lens_q, seed=72, causal=True)

    clean, st = run_multi(make(False))
    assert st == 0
    poisoned, st = run_multi(make(True))
    assert st == 0
    assert np.array_equal(clean, poisoned)
    again, _ = run_multi(make(True))
    assert np.array_equal(poisoned, again)
    ref = oracle_multi(make(False))
    assert_close(clean, ref, "wide rows")
    w = make(False)
    w.block_table[2, 40] = -1  # inside sequence 2's 1500 tokens
    got, st = run_multi(w)
    assert st == pg.PA_STATUS_BAD_BLOCK
    rows2 = np.arange(int(w.cu_q[2]), int(w.cu_q[3]))
    assert np.isnan(got[rows2]).all()
    ok = np.setdiff1d(np.arange(int(w.cu_q[-1])), rows2)
    assert_close(got[ok], ref[ok], "good rows beside a bad one")
