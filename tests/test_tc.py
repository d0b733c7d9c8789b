"""The tcgen05 split kernel (compute = "tc", head_dim 128) against the oracle.

Same outputs, partial states and merge as the mma.sync kernel; 128-token
tiles, accumulators in tensor memory.  Decode (one query token) and several
query tokens per sequence, ragged and poisoned inputs, bad entries, both
split kinds, and the full-size settings on sampled outputs.
"""
import ctypes

import numpy as np
import pytest

import oracle
import paged_gqa_decode_pa_gb300 as pg
from paged_gqa_decode_pa_gb300 import build as pgbuild
from paged_gqa_decode_pa_gb300 import workloads as wl

TC = dict(compute="tc")


@pytest.fixture(scope="module", autouse=True)
def built_library():
    pgbuild.build()
    yield


# ------------------------------------------------------------------ host

FAKE = 1 << 20


def test_tc_option_is_refused_where_it_does_not_apply():
    L = pg.lib()
    # head_dim 64: no tcgen05 kernel
    s64 = pg.pa_shape(2, 8, 2, 64, 16, 8, 32, pg.PA_BF16)
    with pytest.raises(pg.PagedGQAError) as e:
        pg.pa_workspace_size(s64, pg.options(compute="tc", num_ctas=4))
    assert e.value.code == pg.PA_ERR_OPTION
    # 128: accepted, stages 2..(what fits)
    s = pg.pa_shape(2, 8, 2, 128, 16, 8, 32, pg.PA_BF16)
    assert pg.pa_workspace_size(s, pg.options(compute="tc", num_ctas=4)) > 0
    for bad in (1, 5):
        with pytest.raises(pg.PagedGQAError) as e:
            pg.pa_workspace_size(s, pg.options(compute="tc", num_ctas=4, stages=bad))
        assert e.value.code == pg.PA_ERR_OPTION
    # the fused append has no tcgen05 form
    rc = L.pa_decode_append(ctypes.byref(s), ctypes.byref(pg.options(compute="tc", num_ctas=4)),
                            FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, FAKE, FAKE, 1 << 30,
                            None)
    assert rc == pg.PA_ERR_OPTION


# ------------------------------------------------------------------ GPU


def tc_opts(**kw):
    return pg.options(**dict(TC, **kw))


DECODE = [
    # lens, H, Hkv, bs, dtype
    ([1, 15, 16, 17, 100, 0, 255, 1024, 129, 128], 16, 4, 16, "bf16"),
    ([5, 31, 32, 33, 700, 3000], 16, 2, 32, "f16"),
    ([64, 65, 127, 128, 1000, 1], 8, 8, 64, "bf16"),   # G = 1
    ([300, 17, 2], 12, 2, 16, "f16"),                    # G = 6
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", range(len(DECODE)))
@pytest.mark.parametrize("opts", [dict(), dict(num_ctas=5), dict(num_ctas=1),
                                  dict(partition_tokens=256), dict(stages=2)])
def test_decode_matches_the_oracle(case, opts):
    from _helpers import assert_close, run_gpu, run_oracle

    lens, H, Hkv, bs, dtype = DECODE[case]
    w = wl.random_workload(lens, H=H, Hkv=Hkv, d=128, bs=bs, dtype=dtype, seed=60 + case,
                           poison=True, outlier_frac=0.02)
    got, st = run_gpu(w, tc_opts(**opts))
    assert st == 0
    assert_close(got, run_oracle(w), f"tc decode case {case} {opts}")


@pytest.mark.gpu
def test_decode_is_deterministic_and_agrees_with_the_mma_kernel():
    from _helpers import run_gpu

    lens = [1, 15, 16, 17, 100, 0, 255, 1024]
    kw = dict(H=16, Hkv=4, d=128, bs=16, dtype="bf16", extra_blocks=7)
    o = tc_opts(num_ctas=13)
    a, _ = run_gpu(wl.random_workload(lens, seed=5, **kw), o)
    b, _ = run_gpu(wl.random_workload(lens, seed=5, **kw), o)
    c, st = run_gpu(wl.random_workload(lens, seed=5, poison=True, **kw), o)
    assert st == 0
    assert np.array_equal(a, b)
    assert np.array_equal(a, c)  # poisoned unused rows change no bit
    assert np.array_equal(a[5], np.zeros_like(a[5]))
    m, _ = run_gpu(wl.random_workload(lens, seed=5, **kw), pg.options(num_ctas=13))
    assert np.abs(a - m).max() <= 2e-5


@pytest.mark.gpu
def test_bad_entry_and_bad_length_set_status():
    from _helpers import run_gpu

    w = wl.random_workload([40, 300, 60], H=8, Hkv=2, d=128, bs=16, dtype="bf16", seed=9)
    w.block_table[1, 3] = -1
    got, st = run_gpu(w, tc_opts())
    assert st & pg.PA_STATUS_BAD_BLOCK
    assert np.isnan(got[1]).all() and not np.isnan(got[0]).any() and not np.isnan(got[2]).any()
    w2 = wl.random_workload([40, 50], H=8, Hkv=2, d=128, bs=16, dtype="bf16", seed=10, maxblk=4)
    w2.cache_seqlens = np.array([40, 65], np.int32)
    got2, st2 = run_gpu(w2, tc_opts())
    assert st2 & pg.PA_STATUS_BAD_SEQLEN
    assert np.isnan(got2[1]).all() and not np.isnan(got2[0]).any()


MULTI = [
    # lens_k, lens_q, H, Hkv, bs, dtype
    ([300, 17, 1, 64, 513], [4, 3, 1, 4, 2], 16, 4, 16, "bf16"),
    ([129, 40, 700], [1, 5, 2], 8, 1, 32, "f16"),
    ([260, 33, 5, 90], [7, 2, 6, 1], 6, 2, 16, "bf16"),
    ([2, 3, 50, 0], [5, 3, 1, 2], 4, 4, 16, "f16"),
    ([1000, 2500], [16, 9], 8, 8, 64, "bf16"),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", range(len(MULTI)))
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("opts", [dict(), dict(num_ctas=5), dict(partition_tokens=128, num_ctas=7)])
def test_several_query_tokens_match_the_oracle(case, causal, opts):
    import torch
    from _helpers import assert_close

    lens_k, lens_q, H, Hkv, bs, dtype = MULTI[case]
    w = wl.random_workload(lens_k, H, Hkv, 128, bs, dtype=dtype, seed=70 + case, poison=True,
                           outlier_frac=0.02)
    w = wl.with_query_tokens(w, lens_q, seed=80 + case, causal=causal)
    q, k, v, t, sl = w.torch_tensors("cuda")
    cu = torch.from_numpy(w.cu_q).cuda()
    out = torch.full((q.shape[0], w.H, w.d), float("nan"), dtype=torch.float32, device="cuda")
    o = tc_opts(**opts)
    ws = pg.alloc_workspace_multi(pg.shape_multi(q, k, t), w.max_q, o)
    pg.pa_decode_multi(q, cu, w.max_q, w.causal, k, v, t, sl, w.scale, out, ws, o)
    assert pg.pa_read_status(ws) == 0
    ref = oracle.decode_multi(w.q, w.cu_q, w.causal, w.k_cache, w.v_cache, w.block_table,
                              w.cache_seqlens, w.scale, w.dtype)
    assert_close(out.cpu().numpy().astype(np.float64), ref, f"tc multi case {case}")


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["serving_mix_b256_g4_d128", "prefix_share_b64_g8_d128",
                                  "serving_mix_b256_q4_g4_d128"])
def test_full_size_settings_on_sampled_outputs(name):
    import torch
    from _helpers import assert_close

    w = wl.make(name)
    q, k, v, t, sl = w.torch_tensors("cuda")
    rng = np.random.default_rng(4)
    if w.cu_q is None:
        out = torch.empty((w.B, w.H, w.d), dtype=torch.float32, device="cuda")
        ws = pg.alloc_workspace(pg.shape_of(q, k, t), tc_opts())
        pg.pa_decode(q, k, v, t, sl, w.scale, out, ws, tc_opts())
        rows = rng.integers(0, w.B, 96)
        pairs = np.unique(np.stack([rows, rng.integers(0, w.H, 96)], 1).astype(np.int32), axis=0)
        ref = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens, w.scale,
                            w.dtype, pairs=pairs)
    else:
        cu = torch.from_numpy(w.cu_q).cuda()
        out = torch.empty((q.shape[0], w.H, w.d), dtype=torch.float32, device="cuda")
        ws = pg.alloc_workspace_multi(pg.shape_multi(q, k, t), w.max_q, tc_opts())
        pg.pa_decode_multi(q, cu, w.max_q, w.causal, k, v, t, sl, w.scale, out, ws, tc_opts())
        rows = rng.integers(0, q.shape[0], 96)
        pairs = np.unique(np.stack([rows, rng.integers(0, w.H, 96)], 1).astype(np.int32), axis=0)
        ref = oracle.decode_multi(w.q, w.cu_q, w.causal, w.k_cache, w.v_cache, w.block_table,
                                  w.cache_seqlens, w.scale, w.dtype, pairs=pairs)
    assert pg.pa_read_status(ws) == 0
    got = out.cpu().numpy().astype(np.float64)[pairs[:, 0], pairs[:, 1]]
    assert_close(got, ref, name + " tc")
