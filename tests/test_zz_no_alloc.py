"""pa_decode_noalloc -- decode for callers that cannot allocate device memory
where they run it (a plugin whose host framework owns every device
allocation, a serving loop that fixes its memory at start-up).  Its scratch
is a fixed static array inside the library, shared by all calls.

Checked through the C ABI against pa_decode (which uses a caller-allocated
workspace) on two calls in a row with different shapes, so the second call
runs on scratch the first one left behind.  Collected last on purpose."""
import numpy as np
import pytest
import torch

import paged_gqa_decode_pa_gb300 as pg
from paged_gqa_decode_pa_gb300 import workloads as wl
from _helpers import MAX_ABS, MEAN_ABS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built_library():
    from paged_gqa_decode_pa_gb300 import build

    build.build()
    pg.lib()
    yield


def both_ways(w, opts=None):
    q, k, v, t, sl = w.torch_tensors("cuda")
    ref = torch.full((w.B, w.H, w.d), float("nan"), dtype=torch.float32, device="cuda")
    ws = pg.alloc_workspace(pg.shape_of(q, k, t), opts)
    pg.pa_decode(q, k, v, t, sl, w.scale, ref, ws, opts)
    got = torch.full_like(ref, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pg.pa_decode_noalloc(q, k, v, t, sl, w.scale, got, status, opts)
    torch.cuda.synchronize()
    assert pg.pa_read_status(ws) == 0
    assert int(status.item()) == 0
    return got.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64)


def check(got, ref):
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS


def oracle_of(w):
    import oracle

    return oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens, w.scale,
                         w.dtype)


def test_two_calls_in_a_row_match_the_workspace_entry_point():
    # first call: serving-mix shape, split across CTAs (partial states in scratch)
    a = wl.random_workload(list(wl.serving_mix_lengths(5, 24) // 2 + 1), H=32, Hkv=8, d=128,
                           bs=32, dtype="bf16", seed=77, outlier_frac=0.01)
    got, ref = both_ways(a)
    check(got, ref)
    check(got, oracle_of(a))
    # second call: different shape and fixed 512-token partitions
    b = wl.random_workload([10_007, 3, 700], H=24, Hkv=4, d=256, bs=16, dtype="bf16", seed=78)
    got, ref = both_ways(b, pg.options(partition_tokens=512))
    check(got, ref)
    check(got, oracle_of(b))


def test_status_must_be_a_device_word_of_q_s_gpu():
    # checked in the binding before the C call: the kernels would OR bits into
    # whatever address they are given
    w = wl.random_workload([40, 9], H=8, Hkv=2, d=64, bs=16, dtype="f16", seed=81)
    q, k, v, t, sl = w.torch_tensors("cuda")
    out = torch.empty((w.B, w.H, w.d), dtype=torch.float32, device="cuda")
    for bad in (torch.zeros(1, dtype=torch.int32),                  # host memory
                torch.zeros(0, dtype=torch.int32, device="cuda"),   # no element
                torch.zeros(1, dtype=torch.float32, device="cuda")):  # not an integer word
        with pytest.raises(pg.PagedGQAError):
            pg.pa_decode_noalloc(q, k, v, t, sl, w.scale, out, bad)
    with pytest.raises(pg.PagedGQAError) as e:
        pg.pa_decode_noalloc(q, k, v, t, sl, w.scale, out, None,
                             pg.options(phase=pg.PA_PHASE_SPLIT))
    assert e.value.code == pg.PA_ERR_OPTION


def test_status_bits_reach_the_callers_word_and_oversize_is_rejected():
    w = wl.random_workload([100, 200], H=8, Hkv=2, d=64, bs=16, dtype="f16", seed=79)
    w.block_table[1, 2] = -1
    q, k, v, t, sl = w.torch_tensors("cuda")
    out = torch.empty((w.B, w.H, w.d), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pg.pa_decode_noalloc(q, k, v, t, sl, w.scale, out, status)
    torch.cuda.synchronize()
    assert int(status.item()) & pg.PA_STATUS_BAD_BLOCK
    assert torch.isnan(out[1]).all() and torch.isfinite(out[0]).all()
    # fixed 16-token partitions over a 1M-token table need far more scratch
    big = wl.random_workload([5], H=8, Hkv=8, d=256, bs=16, dtype="bf16", seed=80,
                             maxblk=65536)
    q, k, v, t, sl = big.torch_tensors("cuda")
    out = torch.empty((big.B, big.H, big.d), dtype=torch.float32, device="cuda")
    with pytest.raises(pg.PagedGQAError) as e:
        pg.pa_decode_noalloc(q, k, v, t, sl, big.scale, out, None,
                             pg.options(partition_tokens=16))
    assert e.value.code == pg.PA_ERR_SCRATCH_LIMIT
