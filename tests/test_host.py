"""The host-buffer entry points (pa_decode_host, pa_decode_multi_host)
against the oracle and against the device-buffer calls: the step's q,
block table, lengths (and query offsets) come from host memory, the result
goes back to host memory, inside one call.  Pinned and pageable host
buffers, the per-call status, and a full-size setting on sampled outputs."""
import ctypes

import numpy as np
import pytest

import oracle
import paged_gqa_decode_pa_gb300 as pg
from paged_gqa_decode_pa_gb300 import build as pgbuild
from paged_gqa_decode_pa_gb300 import workloads as wl


@pytest.fixture(scope="module", autouse=True)
def built_library():
    pgbuild.build()
    yield


def host_inputs(w, pinned):
    q, k, v, t, sl = w.torch_tensors("cpu")
    if pinned:
        q, t, sl = q.pin_memory(), t.pin_memory(), sl.pin_memory()
    return q, k.cuda(), v.cuda(), t, sl


def empty_out(shape, pinned):
    import torch

    out = torch.full(shape, float("nan"), dtype=torch.float32)
    return out.pin_memory() if pinned else out


CASES = [
    # lens, H, Hkv, d, bs, dtype, opts
    ([1, 15, 16, 17, 100, 0, 255, 1024, 129, 3000], 16, 4, 128, 16, "bf16", dict()),
    ([5, 31, 32, 33, 700], 14, 2, 64, 16, "f16", dict(num_ctas=7)),
    ([300, 2, 1500], 24, 4, 256, 16, "bf16", dict(partition_tokens=256)),
    ([64, 4000, 1], 32, 8, 128, 32, "bf16", dict(compute="tc")),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("pinned", [True, False])
def test_decode_host_matches_the_oracle_and_the_device_call(case, pinned):
    import torch
    from _helpers import assert_close, run_gpu, run_oracle

    lens, H, Hkv, d, bs, dtype, kw = CASES[case]
    w = wl.random_workload(lens, H=H, Hkv=Hkv, d=d, bs=bs, dtype=dtype, seed=90 + case,
                           poison=True, outlier_frac=0.02)
    o = pg.options(**kw)
    q, k, v, t, sl = host_inputs(w, pinned)
    out = empty_out((w.B, w.H, w.d), pinned)
    ws = pg.alloc_workspace_host(pg.shape_of(q, k, t), o)
    st = pg.pa_decode_host(q, k, v, t, sl, w.scale, out, ws, o)
    assert st == 0
    got = out.numpy().astype(np.float64)
    assert_close(got, run_oracle(w), f"host case {case}")
    dev, st2 = run_gpu(w, o)
    assert st2 == 0
    assert np.array_equal(got, dev)  # same plan, same kernels, same bits
    # a second call on the same workspace gives the same bits
    out2 = empty_out((w.B, w.H, w.d), pinned)
    assert pg.pa_decode_host(q, k, v, t, sl, w.scale, out2, ws, o) == 0
    assert torch.equal(out, out2)


@pytest.mark.gpu
def test_decode_host_status_is_per_call():
    w = wl.random_workload([40, 300, 60], H=8, Hkv=2, d=128, bs=16, dtype="bf16", seed=9)
    q, k, v, t, sl = host_inputs(w, True)
    t[1, 3] = -1
    out = empty_out((w.B, w.H, w.d), True)
    ws = pg.alloc_workspace_host(pg.shape_of(q, k, t))
    st = pg.pa_decode_host(q, k, v, t, sl, w.scale, out, ws)
    assert st & pg.PA_STATUS_BAD_BLOCK
    got = out.numpy()
    assert np.isnan(got[1]).all() and not np.isnan(got[0]).any() and not np.isnan(got[2]).any()
    # the workspace's own status word was not touched
    assert pg.pa_read_status(ws) == 0
    # the next clean call reports a clean status
    t[1, 3] = w.block_table[1, 3]
    assert pg.pa_decode_host(q, k, v, t, sl, w.scale, out, ws) == 0
    assert not np.isnan(out.numpy()).any()
    # without a status pointer the bits land in the workspace's status word
    t[1, 3] = -1
    shape = pg.shape_of(q, k, t)
    rc = pg.lib().pa_decode_host(ctypes.byref(shape), None, q.data_ptr(), k.data_ptr(),
                                 v.data_ptr(), t.data_ptr(), sl.data_ptr(), w.scale,
                                 out.data_ptr(), None, ws.data_ptr(), ws.numel(),
                                 pg._binding._stream(None))
    assert rc == pg.PA_OK
    assert pg.pa_read_status(ws) & pg.PA_STATUS_BAD_BLOCK


@pytest.mark.gpu
def test_decode_host_mixes_page_locked_and_pageable_buffers():
    """Each buffer takes its own route: the SMs move page-locked ones (and
    write out into it directly), copies move the pageable ones; the result
    does not depend on the route.  A pageable status word gets the bits by a
    copy."""
    import torch

    w = wl.random_workload([1, 40, 300, 7, 900], H=16, Hkv=4, d=128, bs=16, dtype="bf16",
                           seed=21, poison=True)
    q, k, v, t, sl = host_inputs(w, True)
    ref = None
    for mix in range(4):
        qq = q if mix & 1 else q.clone()          # pageable copy when bit 0 is clear
        tt = t.clone() if mix & 2 else t
        out = empty_out((w.B, w.H, w.d), pinned=bool(mix & 2))
        ws = pg.alloc_workspace_host(pg.shape_of(qq, k, tt))
        st = ctypes.c_uint32(123)
        shape = pg.shape_of(qq, k, tt)
        rc = pg.lib().pa_decode_host(ctypes.byref(shape), None, qq.data_ptr(), k.data_ptr(),
                                     v.data_ptr(), tt.data_ptr(), sl.data_ptr(), w.scale,
                                     out.data_ptr(), ctypes.byref(st), ws.data_ptr(), ws.numel(),
                                     pg._binding._stream(None))
        assert rc == pg.PA_OK and st.value == 0
        if ref is None:
            ref = out.clone()
        assert torch.equal(out, ref), mix
    from _helpers import assert_close, run_oracle

    assert_close(ref.numpy().astype(np.float64), run_oracle(w), "mixed host buffers")


MULTI = [
    # lens_k, lens_q, H, Hkv, d, bs, dtype, causal
    ([300, 17, 1, 64, 513], [4, 3, 1, 4, 2], 16, 4, 128, 16, "bf16", True),
    ([129, 40, 700], [1, 5, 2], 8, 1, 64, 32, "f16", False),
    ([2, 3, 50, 0], [5, 3, 1, 2], 12, 2, 256, 16, "bf16", True),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", range(len(MULTI)))
@pytest.mark.parametrize("pinned", [True, False])
def test_decode_multi_host_matches_the_oracle_and_the_device_call(case, pinned):
    import torch

    from _helpers import assert_close

    lens_k, lens_q, H, Hkv, d, bs, dtype, causal = MULTI[case]
    w = wl.random_workload(lens_k, H, Hkv, d, bs, dtype=dtype, seed=100 + case, poison=True,
                           outlier_frac=0.02)
    w = wl.with_query_tokens(w, lens_q, seed=110 + case, causal=causal)
    q, k, v, t, sl = host_inputs(w, pinned)
    cu = torch.from_numpy(w.cu_q)
    if pinned:
        cu = cu.pin_memory()
    out = empty_out((q.shape[0], w.H, w.d), pinned)
    shape = pg.shape_multi(q, k, t)
    # sized for more rows than this call has: the staging of q and out comes last
    ws = pg.alloc_workspace_multi_host(shape, w.max_q, q.shape[0] + 37)
    st = pg.pa_decode_multi_host(q, cu, w.max_q, w.causal, k, v, t, sl, w.scale, out, ws)
    assert st == 0
    ref = oracle.decode_multi(w.q, w.cu_q, w.causal, w.k_cache, w.v_cache, w.block_table,
                              w.cache_seqlens, w.scale, w.dtype)
    got = out.numpy().astype(np.float64)
    assert_close(got, ref, f"multi host case {case}")
    qd, td, sld, cud = q.cuda(), t.cuda(), sl.cuda(), cu.cuda()
    outd = torch.full((q.shape[0], w.H, w.d), float("nan"), dtype=torch.float32, device="cuda")
    wsd = pg.alloc_workspace_multi(shape, w.max_q)
    pg.pa_decode_multi(qd, cud, w.max_q, w.causal, k, v, td, sld, w.scale, outd, wsd)
    assert pg.pa_read_status(wsd) == 0
    assert np.array_equal(got, outd.cpu().numpy().astype(np.float64))
    # the bound form of the same call gives the same bits
    out_b = empty_out((q.shape[0], w.H, w.d), pinned)
    step = pg.bind_decode_multi_host(q, cu, w.max_q, w.causal, k, v, t, sl, w.scale, out_b, ws)
    assert step() == 0 and step() == 0
    assert np.array_equal(got, out_b.numpy().astype(np.float64))
    # too small a workspace for this many rows is refused
    small = pg.alloc_workspace_multi_host(shape, w.max_q, q.shape[0] - 1)
    with pytest.raises(pg.PagedGQAError) as e:
        pg.pa_decode_multi_host(q, cu, w.max_q, w.causal, k, v, t, sl, w.scale, out, small)
    assert e.value.code == pg.PA_ERR_WORKSPACE


@pytest.mark.gpu
def test_full_size_serving_mix_from_host_buffers_on_sampled_outputs():
    from _helpers import assert_close, sample_pairs

    w = wl.make("serving_mix_b256_g4_d128")
    q, k, v, t, sl = host_inputs(w, True)
    out = empty_out((w.B, w.H, w.d), True)
    ws = pg.alloc_workspace_host(pg.shape_of(q, k, t))
    assert pg.pa_decode_host(q, k, v, t, sl, w.scale, out, ws) == 0
    pairs = sample_pairs(w, 96, seed=3)
    ref = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens, w.scale,
                        w.dtype, pairs=pairs)
    got = out.numpy().astype(np.float64)[pairs[:, 0], pairs[:, 1]]
    assert_close(got, ref, "serving mix from host buffers")


@pytest.mark.gpu
def test_bound_host_calls_follow_the_buffers_contents():
    """A bound call reruns on the same buffers: rewriting q, the table and
    the lengths in place between steps changes the result as pa_decode_host
    on the new contents would."""
    import torch

    w = wl.random_workload([40, 300, 60, 1000], H=16, Hkv=4, d=128, bs=16, dtype="bf16",
                           seed=31)
    q, k, v, t, sl = host_inputs(w, True)
    out = empty_out((w.B, w.H, w.d), True)
    ws = pg.alloc_workspace_host(pg.shape_of(q, k, t))
    step = pg.bind_decode_host(q, k, v, t, sl, w.scale, out, ws)
    assert step() == 0
    first = out.clone()
    # the next step: new queries, the sequences' tables and lengths permuted
    perm = [3, 0, 2, 1]
    q2 = torch.randn(q.shape, generator=torch.Generator().manual_seed(5)).to(q.dtype)
    t2, sl2 = t[perm].clone(), sl[perm].clone()
    sl2[2] = 17  # and one sequence shortened
    q.copy_(q2), t.copy_(t2), sl.copy_(sl2)
    assert step() == 0
    ref = torch.full_like(out, float("nan"))
    assert pg.pa_decode_host(q2, k, v, t2, sl2, w.scale, ref,
                             pg.alloc_workspace_host(pg.shape_of(q2, k, t2))) == 0
    assert torch.equal(out, ref) and not torch.equal(out, first)
    t[1, 0] = -1
    assert step() & pg.PA_STATUS_BAD_BLOCK
    t[1, 0] = t2[1, 0]
    assert step() == 0 and torch.equal(out, ref)


@pytest.mark.gpu
def test_decode_host_accepts_device_buffers():
    """Memory of the current device is used in place (the C ABI takes any
    mix of pageable, page-locked and device buffers); the result does not
    change."""
    import torch

    from _helpers import run_gpu

    w = wl.random_workload([3, 200, 0, 1500], H=16, Hkv=4, d=128, bs=32, dtype="bf16", seed=23,
                           poison=True)
    ref, st = run_gpu(w)
    assert st == 0
    qd, k, v, td, sld = w.torch_tensors("cuda")
    qh, _, _, th, slh = host_inputs(w, True)
    for mix in range(4):
        q = qd if mix & 1 else qh
        t, sl = (td, sld) if mix & 2 else (th, slh)
        out = (torch.full((w.B, w.H, w.d), float("nan"), device="cuda") if mix & 1
               else empty_out((w.B, w.H, w.d), True))
        ws = pg.alloc_workspace_host(pg.shape_of(q, k, t))
        stw = ctypes.c_uint32(99)
        shape = pg.shape_of(q, k, t)
        rc = pg.lib().pa_decode_host(ctypes.byref(shape), None, q.data_ptr(), k.data_ptr(),
                                     v.data_ptr(), t.data_ptr(), sl.data_ptr(), w.scale,
                                     out.data_ptr(), ctypes.byref(stw), ws.data_ptr(), ws.numel(),
                                     pg._binding._stream(None))
        assert rc == pg.PA_OK and stw.value == 0
        assert np.array_equal(out.cpu().numpy().astype(np.float64), ref), mix


# ------------------------------------------------------- asynchronous calls


def test_async_host_calls_reject_bad_slots_before_any_cuda_call():
    L = pg.lib()
    s = pg.pa_shape(3, 4, 2, 64, 32, 4, 8, pg.PA_F16)
    o = pg.options(num_ctas=8)
    F = 1 << 20
    for slot in (-1, 2):
        assert L.pa_decode_host_async(ctypes.byref(s), ctypes.byref(o), F, F, F, F, F, 0.1, F,
                                      None, slot, F, 1 << 30, None) == pg.PA_ERR_OPTION
        assert L.pa_decode_multi_host_async(ctypes.byref(s), ctypes.byref(o), F, F, 6, 2, 1, F,
                                            F, F, F, 0.1, F, None, slot, F, 1 << 30,
                                            None) == pg.PA_ERR_OPTION
    # room for two staging slots
    one = pg.pa_workspace_size_host(s, o)
    two = pg.pa_workspace_size_host_async(s, o)
    plain = pg.pa_workspace_size(s, o)
    assert two - one >= one - plain > 0
    assert L.pa_decode_host_async(ctypes.byref(s), ctypes.byref(o), F, F, F, F, F, 0.1, F, None,
                                  1, F, one, None) == pg.PA_ERR_WORKSPACE
    m1 = pg.pa_workspace_size_multi_host(s, 2, 6, o)
    m2 = pg.pa_workspace_size_multi_host_async(s, 2, 6, o)
    assert m2 - m1 >= m1 - pg.pa_workspace_size_multi(s, 2, o) > 0


def _step_inputs(w, i, pinned=True):
    """Step i's host inputs over one cache: new queries, the tables and
    lengths rotated among the sequences, one sequence shortened."""
    import torch

    q, k, v, t, sl = w.torch_tensors("cpu")
    perm = np.roll(np.arange(w.B), i)
    q = torch.randn(q.shape, generator=torch.Generator().manual_seed(1000 + i)).to(q.dtype)
    t, sl = t[perm].clone(), sl[perm].clone()
    sl[i % w.B] = max(0, int(sl[i % w.B]) - 7 * i)
    if pinned:
        q, t, sl = q.pin_memory(), t.pin_memory(), sl.pin_memory()
    return q, t, sl


ASYNC = [
    # lens, H, Hkv, d, bs, dtype, opts
    ([1, 15, 16, 17, 100, 0, 255, 1024, 129, 3000], 16, 4, 128, 16, "bf16", dict()),
    ([300, 2, 1500, 40], 24, 4, 256, 16, "bf16", dict(partition_tokens=256)),
    ([5, 31, 32, 33, 700], 14, 2, 64, 16, "f16", dict(num_ctas=7)),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", range(len(ASYNC)))
def test_async_steps_alternating_slots_match_the_device_call(case):
    """Six steps issued back to back without waiting, slots 0, 1, 0, ...,
    each with its own host buffers and inputs; after one synchronisation
    every step's output equals pa_decode's on the same inputs, bit for bit."""
    import torch

    lens, H, Hkv, d, bs, dtype, kw = ASYNC[case]
    w = wl.random_workload(lens, H=H, Hkv=Hkv, d=d, bs=bs, dtype=dtype, seed=300 + case,
                           poison=True, outlier_frac=0.02)
    o = pg.options(**kw)
    _, k, v, _, _ = host_inputs(w, True)
    steps = [_step_inputs(w, i) for i in range(6)]
    shape = pg.shape_of(steps[0][0], k, steps[0][1])
    ws = pg.alloc_workspace_host_async(shape, o)
    outs = [empty_out((w.B, w.H, w.d), True) for _ in steps]
    calls = [pg.bind_decode_host_async(q, k, v, t, sl, w.scale, out, ws, i % 2, o)
             for i, ((q, t, sl), out) in enumerate(zip(steps, outs))]
    for c in calls:
        c()
    torch.cuda.synchronize()
    wsd = pg.alloc_workspace(shape, o)
    for i, ((q, t, sl), out, c) in enumerate(zip(steps, outs, calls)):
        assert c.status() == 0, i
        ref = torch.full((w.B, w.H, w.d), float("nan"), dtype=torch.float32, device="cuda")
        pg.pa_decode(q.cuda(), k, v, t.cuda(), sl.cuda(), w.scale, ref, wsd, o)
        assert pg.pa_read_status(wsd) == 0
        assert torch.equal(out, ref.cpu()), f"step {i}"


@pytest.mark.gpu
def test_async_loop_reusing_two_buffer_sets():
    """A serving loop's shape: two buffer sets, one per slot; each step
    rewrites its set only after the step that last used it has finished
    (one synchronisation per step, a step behind).  Status bits land in the
    step's own word."""
    import torch

    w = wl.random_workload([40, 300, 60, 1000, 7], H=16, Hkv=4, d=128, bs=32, dtype="bf16",
                           seed=320)
    _, k, v, _, _ = host_inputs(w, True)
    sets = [_step_inputs(w, 0), _step_inputs(w, 1)]
    outs = [empty_out((w.B, w.H, w.d), True) for _ in range(2)]
    shape = pg.shape_of(sets[0][0], k, sets[0][1])
    ws = pg.alloc_workspace_host_async(shape)
    calls = [pg.bind_decode_host_async(q, k, v, t, sl, w.scale, outs[s], ws, s)
             for s, (q, t, sl) in enumerate(sets)]
    wsd = pg.alloc_workspace(shape)
    done = torch.cuda.Event()
    for i in range(8):
        s = i % 2
        q, t, sl = sets[s]
        nq, nt, nsl = _step_inputs(w, i)
        if i == 5:
            nt[2, 0] = -1  # a bad table entry in one step
        q.copy_(nq), t.copy_(nt), sl.copy_(nsl)
        calls[s]()
        if i > 0:
            done.synchronize()  # the previous step: check it while this one runs
            check_step(i - 1, prev, calls[1 - s], outs[1 - s], k, v, w, wsd)
        done.record()
        prev = (nq.clone(), nt.clone(), nsl.clone())
    done.synchronize()
    check_step(7, prev, calls[1], outs[1], k, v, w, wsd)


def check_step(i, inputs, call, out, k, v, w, wsd):
    import torch

    q, t, sl = inputs
    st = call.status()
    if i == 5:
        assert st & pg.PA_STATUS_BAD_BLOCK and torch.isnan(out[2]).all()
        return
    assert st == 0, i
    ref = torch.full((w.B, w.H, w.d), float("nan"), dtype=torch.float32, device="cuda")
    pg.pa_decode(q.cuda(), k, v, t.cuda(), sl.cuda(), w.scale, ref, wsd)
    assert pg.pa_read_status(wsd) == 0
    assert torch.equal(out, ref.cpu()), f"step {i}"


@pytest.mark.gpu
def test_async_multi_steps_match_the_synchronous_call():
    import torch

    w = wl.random_workload([300, 17, 1, 64, 513], H=16, Hkv=4, d=128, bs=16, dtype="bf16",
                           seed=330, poison=True)
    w = wl.with_query_tokens(w, [4, 3, 1, 4, 2], seed=331)
    q, k, v, t, sl = host_inputs(w, True)
    cu = torch.from_numpy(w.cu_q).pin_memory()
    shape = pg.shape_multi(q, k, t)
    ref = empty_out((q.shape[0], w.H, w.d), True)
    ws1 = pg.alloc_workspace_multi_host(shape, w.max_q, q.shape[0])
    assert pg.pa_decode_multi_host(q, cu, w.max_q, w.causal, k, v, t, sl, w.scale, ref, ws1) == 0
    ws = pg.alloc_workspace_multi_host_async(shape, w.max_q, q.shape[0])
    outs = [empty_out((q.shape[0], w.H, w.d), True) for _ in range(4)]
    calls = [pg.bind_decode_multi_host_async(q, cu, w.max_q, w.causal, k, v, t, sl, w.scale,
                                             outs[i], ws, i % 2) for i in range(4)]
    for c in calls:
        c()
    torch.cuda.synchronize()
    for c, out in zip(calls, outs):
        assert c.status() == 0
        assert torch.equal(out, ref)
