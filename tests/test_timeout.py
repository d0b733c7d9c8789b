"""The split kernel's bounded pipeline waits, made to run out on purpose.

Every wait of the split kernel's TMA ring gives up after a time limit, sets
PA_STATUS_TIMEOUT and lets the CTA finish: it waits (bounded) for the copies
it still has in flight, and exits.  With options.stall_test = 1, warp 0 of
every CTA that has work waits for its first tile on a barrier that nothing
ever completes, so that wait runs out after options.wait_limit_us.  Nothing
faults or hangs: the step returns, reports the timeout, and the next ordinary
call on the same workspace matches the oracle.  The tcgen05 kernel is not part of this (the
option is refused there)."""
import ctypes
import time

import numpy as np
import pytest

import oracle
import paged_gqa_decode_pa_gb300 as pg
from paged_gqa_decode_pa_gb300 import build as pgbuild
from paged_gqa_decode_pa_gb300 import workloads as wl
from _helpers import assert_close, run_oracle

LIMIT_US = 2000  # the stalled wait gives up after 2 ms


@pytest.fixture(scope="module", autouse=True)
def built_library():
    pgbuild.build()
    yield


FAKE = 1 << 20


def test_options_are_checked_before_any_cuda_call():
    L = pg.lib()
    s = pg.pa_shape(3, 8, 2, 128, 16, 8, 16, pg.PA_BF16)

    def call(o):
        return L.pa_decode(ctypes.byref(s), ctypes.byref(o), FAKE, FAKE, FAKE, FAKE, FAKE, 0.1,
                           FAKE, FAKE, 1 << 30, None)

    assert call(pg.options(num_ctas=8, wait_limit_us=-1)) == pg.PA_ERR_OPTION
    assert call(pg.options(num_ctas=8, stall_test=2)) == pg.PA_ERR_OPTION
    assert call(pg.options(num_ctas=8, stall_test=1, compute="tc")) == pg.PA_ERR_OPTION


def _decode(w, opts, ws, out):
    q, k, v, t, sl = w.torch_tensors("cuda")
    pg.pa_decode(q, k, v, t, sl, w.scale, out, ws, opts)
    return pg.pa_read_status(ws)  # synchronises


CASES = [
    # (lengths, H, Hkv, d, bs, dtype, options)
    ([3000, 17, 900, 4100, 1], 32, 8, 128, 32, "bf16", {}),
    ([3000, 17, 900, 4100, 1], 32, 8, 128, 32, "bf16", {"partition_tokens": 512}),
    ([20000, 5000], 24, 4, 256, 16, "bf16", {}),
    ([700, 1300, 90], 14, 2, 64, 16, "f16", {"compute": "simt"}),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", range(len(CASES)))
def test_a_wait_that_runs_out_reports_and_leaves_the_next_call_intact(case):
    import torch

    lens, H, Hkv, d, bs, dtype, kw = CASES[case]
    w = wl.random_workload(lens, H=H, Hkv=Hkv, d=d, bs=bs, dtype=dtype, seed=900 + case)
    q, k, v, t, sl = w.torch_tensors("cuda")
    normal = pg.options(**kw)
    stalled = pg.options(**kw, wait_limit_us=LIMIT_US, stall_test=1)
    ws = pg.alloc_workspace(pg.shape_of(q, k, t), normal)
    out = torch.full((w.B, w.H, w.d), float("nan"), dtype=torch.float32, device="cuda")
    t0 = time.perf_counter()
    status = _decode(w, stalled, ws, out)
    took = time.perf_counter() - t0
    assert status & pg.PA_STATUS_TIMEOUT, f"status {status:#x}"
    assert took < 1.5, f"the stalled step took {took:.2f} s"
    # the same workspace and output buffer, an ordinary call
    out.fill_(float("nan"))
    status = _decode(w, normal, ws, out)
    assert status == 0
    assert_close(out.cpu().numpy().astype(np.float64), run_oracle(w), "after the timeout")


@pytest.mark.gpu
def test_warp_pairs_give_up_and_drain_too():
    # several query tokens per sequence with rows wider than one warp's
    # columns: warp pairs, where the upper warp releases each ring slot
    import torch

    w = wl.random_workload([2500, 800, 3100], H=32, Hkv=8, d=128, bs=32, dtype="bf16", seed=950)
    w = wl.with_query_tokens(w, [8, 8, 5], seed=951)
    q, k, v, t, sl = w.torch_tensors("cuda")
    cu = torch.from_numpy(w.cu_q).cuda()
    normal = pg.options()
    stalled = pg.options(wait_limit_us=LIMIT_US, stall_test=1)
    ws = pg.alloc_workspace_multi(pg.shape_multi(q, k, t), w.max_q, normal)
    out = torch.full((q.shape[0], w.H, w.d), float("nan"), dtype=torch.float32, device="cuda")
    pg.pa_decode_multi(q, cu, w.max_q, w.causal, k, v, t, sl, w.scale, out, ws, stalled)
    assert pg.pa_read_status(ws) & pg.PA_STATUS_TIMEOUT
    out.fill_(float("nan"))
    pg.pa_decode_multi(q, cu, w.max_q, w.causal, k, v, t, sl, w.scale, out, ws, normal)
    assert pg.pa_read_status(ws) == 0
    ref = oracle.decode_multi(w.q, w.cu_q, w.causal, w.k_cache, w.v_cache, w.block_table,
                              w.cache_seqlens, w.scale, w.dtype)
    assert_close(out.cpu().numpy().astype(np.float64), ref, "warp pairs after the timeout")
