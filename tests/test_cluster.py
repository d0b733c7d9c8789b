"""The cluster kernel: a decode step with few (sequence, kv head) segments
runs as one kernel, each segment on one thread-block cluster whose CTAs fold
their partial states through distributed shared memory (no workspace round
trip, no merge kernel).  Checked against the oracle and against the
persistent split + merge path (forced with a fixed grid) on the same inputs,
including empty, one-token, block-boundary and full-table sequences, bad
table entries and lengths, NaN-poisoned unused rows, every head dimension,
block size and storage type, graph replay after the lengths change, and the
host-buffer calls whose status word the kernel publishes itself."""
import ctypes

import numpy as np
import pytest

import paged_gqa_decode_pa_gb300 as pg
from paged_gqa_decode_pa_gb300 import build as pgbuild
from paged_gqa_decode_pa_gb300 import workloads as wl
from _helpers import assert_close, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built_library():
    pgbuild.build()
    yield


def shape_of(w):
    return pg.pa_shape(w.B, w.H, w.Hkv, w.d, w.block_size, w.max_blocks_per_seq, w.num_blocks,
                       pg.PA_BF16 if w.dtype == "bf16" else pg.PA_F16)


PERSISTENT = pg.options(num_ctas=152)  # a fixed grid keeps the two-kernel path


def test_the_plan_picks_the_cluster_kernel_for_small_steps_only():
    small = shape_of(wl.make("qwen2_b8_g7_d64"))
    p = pg.pa_launch_plan(small)
    assert p["kernels"] == 1 and 1 <= p["cluster"] <= 8
    assert p["ctas"] == p["cluster"] * small.batch * small.num_kv_heads
    assert pg.pa_launch_plan(small, PERSISTENT)["kernels"] == 2
    assert pg.pa_launch_plan(small, pg.options(partition_tokens=256))["kernels"] == 2
    assert pg.pa_launch_plan(small, pg.options(compute="simt"))["kernels"] == 2
    assert pg.pa_launch_plan(small, max_q=2)["kernels"] == 2
    # the page example: every segment fits one CTA's ring
    assert pg.pa_launch_plan(shape_of(wl.make("p5_example")))["cluster"] == 1
    # large steps keep the persistent grid
    big = pg.pa_launch_plan(pg.pa_shape(256, 32, 8, 128, 32, 1024, 30000, pg.PA_BF16))
    assert big["kernels"] == 2 and big["cluster"] == 0


CASES = [
    # lens, H, Hkv, d, bs, dtype
    ([0, 1, 16, 17, 4096, 1000, 31, 2500], 14, 2, 64, 16, "f16"),
    ([0, 1, 32, 33, 2048, 700], 32, 8, 128, 32, "bf16"),
    ([5, 900, 64, 65, 3000], 24, 4, 256, 16, "bf16"),
    ([1, 63, 64, 1500], 16, 4, 128, 64, "f16"),
    ([777], 8, 1, 128, 16, "bf16"),  # one segment: G = 8
    ([3, 300, 2], 6, 6, 64, 32, "bf16"),  # G = 1
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_cluster_kernel_matches_the_oracle_and_the_two_kernel_path(case):
    lens, H, Hkv, d, bs, dtype = CASES[case]
    w = wl.random_workload(lens, H=H, Hkv=Hkv, d=d, bs=bs, dtype=dtype, seed=400 + case,
                           poison=True, outlier_frac=0.02)
    assert pg.pa_launch_plan(shape_of(w))["kernels"] == 1
    ref = run_oracle(w)
    got, st = run_gpu(w)
    assert st == 0
    assert_close(got, ref, f"cluster case {case}")
    two, st2 = run_gpu(w, PERSISTENT)
    assert st2 == 0
    assert_close(two, ref, f"two-kernel case {case}")
    # deterministic: the same bits again
    again, _ = run_gpu(w)
    assert np.array_equal(got, again)


def test_full_table_rows_and_every_ring_depth():
    w = wl.random_workload([64 * 16, 3, 64 * 16 - 1], H=8, Hkv=2, d=128, bs=16, dtype="bf16",
                           seed=420, maxblk=64)
    ref = run_oracle(w)
    for stages in (1, 2, 3):
        o = pg.options(stages=stages)
        assert pg.pa_launch_plan(shape_of(w), o)["ring"] == stages
        got, st = run_gpu(w, o)
        assert st == 0
        assert_close(got, ref, f"stages {stages}")


def test_bad_entries_and_lengths_give_nan_and_status_bits():
    w = wl.random_workload([200, 300, 50, 900], H=16, Hkv=4, d=128, bs=16, dtype="bf16",
                           seed=430)
    w.block_table[1, 5] = -1                      # inside sequence 1's length
    w.block_table[3, 2] = w.num_blocks + 7        # out of range, inside sequence 3's length
    w.block_table[2, 10] = -1                     # past sequence 2's length: never read
    assert pg.pa_launch_plan(shape_of(w))["kernels"] == 1
    got, st = run_gpu(w)
    assert st == pg.PA_STATUS_BAD_BLOCK
    assert np.isnan(got[1]).all() and np.isnan(got[3]).all()
    ok = [0, 2]
    ref = run_oracle(wl.random_workload([200, 300, 50, 900], H=16, Hkv=4, d=128, bs=16,
                                        dtype="bf16", seed=430))
    assert_close(got[ok], ref[ok], "good rows beside bad ones")
    w2 = wl.random_workload([200, 300], H=8, Hkv=2, d=64, bs=16, dtype="f16", seed=431)
    w2.cache_seqlens[1] = w2.max_blocks_per_seq * 16 + 1
    got, st = run_gpu(w2)
    assert st == pg.PA_STATUS_BAD_SEQLEN
    assert np.isnan(got[1]).all() and np.isfinite(got[0]).all()


def test_graph_replay_follows_new_lengths():
    import torch

    w = wl.random_workload([300, 1000, 17], H=16, Hkv=4, d=128, bs=16, dtype="bf16", seed=440,
                           maxblk=80)
    q, k, v, t, sl = w.torch_tensors("cuda")
    out = torch.full((w.B, w.H, w.d), float("nan"), dtype=torch.float32, device="cuda")
    ws = pg.alloc_workspace(pg.shape_of(q, k, t))
    assert pg.pa_launch_plan(pg.shape_of(q, k, t))["kernels"] == 1
    step = pg.bind_decode(q, k, v, t, sl, w.scale, out, ws)
    step()  # first call: one-time setup outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        cap = pg.bind_decode(q, k, v, t, sl, w.scale, out, ws, stream=s)
        with torch.cuda.graph(g, stream=s):
            cap()
    # lengths within each sequence's mapped blocks (19, 63 and 2 blocks of 16)
    for lens in ([300, 1000, 17], [1, 1008, 0], [304, 2, 32]):
        sl.copy_(torch.tensor(lens, dtype=torch.int32))
        w.cache_seqlens[:] = lens
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert pg.pa_read_status(ws) == 0
        assert_close(out.cpu().numpy().astype(np.float64), run_oracle(w), f"replay {lens}")


def test_host_buffer_calls_publish_each_calls_status():
    """The host-buffer calls run the cluster kernel too; its last CTA
    publishes the call's status word (and clears the device words)."""
    import torch

    w = wl.random_workload([40, 300, 60, 1000], H=16, Hkv=4, d=128, bs=16, dtype="bf16",
                           seed=450)
    assert pg.pa_launch_plan(shape_of(w))["kernels"] == 1
    q, k, v, t, sl = w.torch_tensors("cpu")
    q, t, sl = q.pin_memory(), t.pin_memory(), sl.pin_memory()
    k, v = k.cuda(), v.cuda()
    out = torch.full((w.B, w.H, w.d), float("nan"), dtype=torch.float32).pin_memory()
    ws = pg.alloc_workspace_host(pg.shape_of(q, k, t))
    step = pg.bind_decode_host(q, k, v, t, sl, w.scale, out, ws)
    assert step() == 0
    dev, st = run_gpu(w)
    assert st == 0 and np.array_equal(out.numpy().astype(np.float64), dev)
    good = t[1, 0].item()
    t[1, 0] = -1
    assert step() == pg.PA_STATUS_BAD_BLOCK
    assert torch.isnan(out[1]).all()
    t[1, 0] = good
    assert step() == 0  # the bad bit belonged to that call only
    assert np.array_equal(out.numpy().astype(np.float64), dev)
    # a status word in pageable memory gets the bits by a copy
    stw = ctypes.c_uint32(77)
    shape = pg.shape_of(q, k, t)
    rc = pg.lib().pa_decode_host(ctypes.byref(shape), None, q.data_ptr(), k.data_ptr(),
                                 v.data_ptr(), t.data_ptr(), sl.data_ptr(), w.scale,
                                 out.data_ptr(), ctypes.byref(stw), ws.data_ptr(), ws.numel(),
                                 pg._binding._stream(None))
    assert rc == pg.PA_OK and stw.value == 0
    # asynchronous calls, alternating slots
    wsa = pg.alloc_workspace_host_async(shape)
    outs = [torch.full_like(out, float("nan")).pin_memory() for _ in range(4)]
    calls = [pg.bind_decode_host_async(q, k, v, t, sl, w.scale, o, wsa, i % 2)
             for i, o in enumerate(outs)]
    for c in calls:
        c()
    torch.cuda.synchronize()
    for c, o in zip(calls, outs):
        assert c.status() == 0 and np.array_equal(o.numpy().astype(np.float64), dev)


def test_no_alloc_entry_point_on_the_cluster_kernel():
    import torch

    w = wl.random_workload([300, 7, 1200], H=14, Hkv=2, d=64, bs=16, dtype="f16", seed=460)
    assert pg.pa_launch_plan(shape_of(w))["kernels"] == 1
    q, k, v, t, sl = w.torch_tensors("cuda")
    out = torch.full((w.B, w.H, w.d), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pg.pa_decode_noalloc(q, k, v, t, sl, w.scale, out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(out.cpu().numpy().astype(np.float64), run_oracle(w), "no-alloc, cluster kernel")
