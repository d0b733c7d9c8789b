"""The largest shapes the boundary accepts, against the oracle.

PA_MAX_BATCH sequences in one call (every output compared, on both tensor-core
kernels), one sequence with PA_MAX_QUERY_TOKENS query tokens (sampled
outputs), and PA_MAX_BATCH rows of warp-paired columns (sampled).  Ragged
short lengths, empty sequences and a long tail.
"""
import numpy as np
import pytest

import oracle
import paged_gqa_decode_pa_gb300 as pg
from paged_gqa_decode_pa_gb300 import build as pgbuild
from paged_gqa_decode_pa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built_library():
    pgbuild.build()
    yield


@pytest.mark.parametrize("d,compute", [(64, "mma"), (128, "tc")])
def test_max_batch_every_output(d, compute):
    from _helpers import assert_close, run_gpu, run_oracle

    rng = np.random.default_rng(91)
    B = pg.PA_MAX_BATCH
    lens = rng.integers(0, 80, B).astype(np.int32)
    lens[::97] = 0                 # empty sequences here and there
    lens[-1] = 3000                # and one long tail
    w = wl.random_workload(lens, H=4, Hkv=1, d=d, bs=16, dtype="bf16", seed=92, poison=True)
    got, st = run_gpu(w, pg.options(compute=compute))
    assert st == 0
    assert_close(got, run_oracle(w), f"B={B} d={d} {compute}")
    assert np.array_equal(got[lens == 0], np.zeros_like(got[lens == 0]))


def test_max_query_tokens_sampled():
    import torch
    from _helpers import assert_close

    nq = pg.PA_MAX_QUERY_TOKENS
    w = wl.random_workload([nq + 500, 40], H=8, Hkv=2, d=64, bs=32, dtype="f16", seed=93)
    w = wl.with_query_tokens(w, [nq, 3], seed=94, causal=True)
    q, k, v, t, sl = w.torch_tensors("cuda")
    cu = torch.from_numpy(w.cu_q).cuda()
    out = torch.full((q.shape[0], w.H, w.d), float("nan"), dtype=torch.float32, device="cuda")
    ws = pg.alloc_workspace_multi(pg.shape_multi(q, k, t), nq)
    pg.pa_decode_multi(q, cu, nq, True, k, v, t, sl, w.scale, out, ws)
    assert pg.pa_read_status(ws) == 0
    got = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    rng = np.random.default_rng(95)
    rows = np.concatenate([[0, 1, nq - 2, nq - 1, nq, nq + 2], rng.integers(0, q.shape[0], 120)])
    pairs = np.unique(np.stack([rows, rng.integers(0, w.H, rows.shape[0])], 1).astype(np.int32), axis=0)
    ref = oracle.decode_multi(w.q, w.cu_q, True, w.k_cache, w.v_cache, w.block_table,
                              w.cache_seqlens, w.scale, w.dtype, pairs=pairs)
    assert_close(got[pairs[:, 0], pairs[:, 1]], ref, "4096 query tokens")


@pytest.mark.parametrize("d,max_q", [(128, 8), (256, 4)])
def test_max_rows_with_warp_pairs_sampled(d, max_q):
    """PA_MAX_BATCH rows of warp-paired columns (G = 4: 32 columns at d = 128,
    16 at d = 256): the largest prefix array next to the pair layout's
    shared memory."""
    import torch
    from _helpers import assert_close

    rng = np.random.default_rng(96 + d)
    B = pg.PA_MAX_BATCH
    lens_q = rng.integers(1, max_q + 1, B).astype(np.int32)
    lens = (lens_q + rng.integers(0, 60, B)).astype(np.int32)
    lens[::89] = 0                  # empty sequences (their query tokens see no key)
    lens[-1] = 2000
    w = wl.random_workload(lens, H=8, Hkv=2, d=d, bs=16, dtype="bf16", seed=97, poison=True)
    w = wl.with_query_tokens(w, lens_q, seed=98, causal=True)
    q, k, v, t, sl = w.torch_tensors("cuda")
    cu = torch.from_numpy(w.cu_q).cuda()
    out = torch.full((q.shape[0], w.H, w.d), float("nan"), dtype=torch.float32, device="cuda")
    ws = pg.alloc_workspace_multi(pg.shape_multi(q, k, t), max_q)
    pg.pa_decode_multi(q, cu, max_q, True, k, v, t, sl, w.scale, out, ws)
    assert pg.pa_read_status(ws) == 0
    got = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    rows = np.concatenate([[0, q.shape[0] - 1], rng.integers(0, q.shape[0], 400)])
    pairs = np.unique(np.stack([rows, rng.integers(0, w.H, rows.shape[0])], 1).astype(np.int32),
                      axis=0)
    ref = oracle.decode_multi(w.q, w.cu_q, True, w.k_cache, w.v_cache, w.block_table,
                              w.cache_seqlens, w.scale, w.dtype, pairs=pairs)
    assert_close(got[pairs[:, 0], pairs[:, 1]], ref, f"{B} paired rows d={d}")
