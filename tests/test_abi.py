"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every symbol include/pagedgqa.h declares, rejects bad arguments before it
touches CUDA, and its work split covers every unit exactly once while the
merge finds exactly the pieces that were cut."""
import ctypes
import os
import re

import numpy as np
import pytest

import paged_gqa_decode_pa_gb300 as pg
from paged_gqa_decode_pa_gb300 import build as pgbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedgqa.h")


@pytest.fixture(scope="module", autouse=True)
def built_library():
    pgbuild.build()
    yield


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert len(names) >= 10
    assert sorted(pg.EXPORTS) == names
    L = ctypes.CDLL(pg.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n
    assert pg.pa_version() == 100


def shape(B=3, H=4, Hkv=2, d=64, bs=32, maxblk=4, P=8, dtype=pg.PA_F16):
    return pg.pa_shape(B, H, Hkv, d, bs, maxblk, P, dtype)


FAKE = 1 << 20  # an aligned, non-null address; never dereferenced on these paths


def call_decode(s, opts, q=FAKE, k=FAKE, v=FAKE, t=FAKE, sl=FAKE, out=FAKE, ws=FAKE,
                ws_bytes=0, scale=0.125):
    L = pg.lib()
    return L.pa_decode(ctypes.byref(s), ctypes.byref(opts) if opts else None, q, k, v, t, sl,
                       scale, out, ws, ws_bytes, None)


def test_rejects_bad_arguments_before_any_cuda_call():
    o = pg.options(num_ctas=8)
    s = shape()
    assert call_decode(s, o, q=None) == pg.PA_ERR_NULL
    assert call_decode(s, o, ws=None) == pg.PA_ERR_NULL
    assert call_decode(s, o, out=FAKE + 4) == pg.PA_ERR_ALIGN
    assert call_decode(s, o, k=FAKE + 8) == pg.PA_ERR_ALIGN
    assert call_decode(s, o, ws_bytes=16) == pg.PA_ERR_WORKSPACE
    assert call_decode(s, o, scale=float("nan")) == pg.PA_ERR_SHAPE
    for bad in (shape(d=96), shape(bs=8), shape(bs=48), shape(H=5, Hkv=2), shape(H=18, Hkv=2),
                shape(B=-1), shape(maxblk=0), shape(P=0), shape(dtype=7)):
        assert call_decode(bad, o) == pg.PA_ERR_SHAPE
    assert call_decode(s, pg.options(partition_tokens=48, num_ctas=8)) == pg.PA_ERR_OPTION
    assert call_decode(s, pg.options(compute=9, num_ctas=8)) == pg.PA_ERR_OPTION
    assert call_decode(s, pg.options(stages=-1, num_ctas=8)) == pg.PA_ERR_OPTION
    assert call_decode(s, pg.options(stages=99, num_ctas=8)) == pg.PA_ERR_OPTION
    # an empty batch is a no-op and needs no pointers
    assert call_decode(shape(B=0), o, q=None, k=None, v=None, t=None, sl=None, out=None,
                       ws=None) == pg.PA_OK
    L = pg.lib()
    assert L.pa_cache_append(ctypes.byref(s), None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 256,
                             None) == pg.PA_ERR_NULL
    assert L.pa_cache_append(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8,
                             None) == pg.PA_ERR_WORKSPACE
    assert L.pa_read_status(None, None, None) == pg.PA_ERR_NULL
    for code in (0, -1, -2, -3, -4, -5, -6, 1, 2, 4, 8):
        assert L.pa_status_string(code).decode() != "unknown code"


def test_workspace_size_with_fixed_grid_is_host_only():
    s = shape(B=256, H=32, Hkv=8, d=128, bs=32, maxblk=1024, P=30000, dtype=pg.PA_BF16)
    a = pg.pa_workspace_size(s, pg.options(num_ctas=304))
    b = pg.pa_workspace_size(s, pg.options(num_ctas=608))
    assert b > a > 0
    # balanced split: 2 partial slots per CTA, G x (d + 2) floats each
    G = 4
    assert b - a >= 304 * 2 * G * (128 + 2) * 4
    f = pg.pa_workspace_size(s, pg.options(num_ctas=304, partition_tokens=512))
    assert f >= 256 * 8 * (32768 // 512) * G * 128 * 4


def all_units(lens, Hkv, bs):
    return {(b, j, k) for b, n in enumerate(lens) for j in range(Hkv)
            for k in range((int(n) + bs - 1) // bs)}


def check_schedule(lens, Hkv, bs, maxblk, part_tokens, C):
    s = shape(B=len(lens), H=Hkv * 2, Hkv=Hkv, d=128, bs=bs, maxblk=maxblk, P=1000,
              dtype=pg.PA_BF16)
    o = pg.options(partition_tokens=part_tokens, num_ctas=C)
    seen = set()
    pieces_of = {}
    slots = set()
    for c in range(C):
        for (b, j, k0, k1, slot) in pg.pa_plan_pieces(s, o, lens, C, c):
            assert 0 <= k0 < k1
            for k in range(k0, k1):
                assert (b, j, k) not in seen
                seen.add((b, j, k))
            pieces_of.setdefault((b, j), []).append((k0, k1, slot))
            if slot >= 0:
                assert slot not in slots
                slots.add(slot)
    assert seen == all_units(lens, Hkv, bs)
    n_slots = 2 * C if part_tokens == 0 else len(lens) * Hkv * -(-maxblk // (part_tokens // bs))
    assert all(0 <= x < n_slots for x in slots)
    nseg = C if part_tokens == 0 else len(lens) * Hkv
    merged = {}
    for seg in range(nseg):
        r = pg.pa_plan_merge(s, o, lens, C, seg)
        if r is None:
            continue
        (b, j), sl = r
        assert (b, j) not in merged
        merged[(b, j)] = sl
    for key, ps in pieces_of.items():
        ps.sort()
        if len(ps) == 1 and ps[0][2] < 0:
            assert key not in merged  # finished in one CTA, written directly
            n = (int(lens[key[0]]) + bs - 1) // bs
            assert ps[0][:2] == (0, n)
        else:
            assert all(p[2] >= 0 for p in ps)
            assert merged[key] == [p[2] for p in ps]  # block order
    assert set(merged) <= set(pieces_of)


@pytest.mark.parametrize("part", [0, 64, 512])
@pytest.mark.parametrize("C", [1, 2, 7, 64, 304])
def test_work_split_covers_each_unit_once_and_merge_finds_all_pieces(part, C):
    rng = np.random.default_rng(C * 7 + part)
    for trial in range(4):
        B = int(rng.integers(1, 40))
        lens = rng.integers(0, 3000, size=B)
        lens[rng.random(B) < 0.2] = 0
        bs = int(rng.choice([16, 32]))
        maxblk = int(-(-lens.max() // bs)) + int(rng.integers(0, 3)) if lens.max() > 0 else 1
        check_schedule(lens, int(rng.choice([1, 2, 8])), bs, max(maxblk, 1),
                       part if part % bs == 0 else 0, C)


def test_work_split_on_the_page_example():
    # the Hugging Face decoding-path example: lengths [30, 32, 70], block 32
    for C in (1, 2, 3, 4, 5, 11):
        check_schedule([30, 32, 70], 2, 32, 4, 0, C)
        check_schedule([30, 32, 70], 2, 32, 4, 32, C)


K_UNITS = {(16, 256): 13, (32, 128): 13, (16, 128): 25, (16, 64): 50}  # 200 KB / (4 bs d)


def test_balanced_split_is_even():
    # one long sequence: every CTA gets the same blocks, except that the CTA
    # where a segment begins is also charged the segment's overhead units
    lens = [100_000]
    s = shape(B=1, H=24, Hkv=4, d=256, bs=16, maxblk=6250, P=6250, dtype=pg.PA_BF16)
    C = 304
    sizes = [sum(k1 - k0 for (_, _, k0, k1, _) in pg.pa_plan_pieces(s, None, lens, C, c))
             for c in range(C)]
    assert sum(sizes) == 4 * 6250
    K = K_UNITS[(16, 256)]
    assert max(sizes) - min(sizes) <= K + 1
    assert sorted(sizes)[4] >= max(sizes) - 1  # only the 4 segment starts are short


def test_balanced_split_charges_each_segment_its_overhead():
    # 64 short sequences then one long one, 8 CTAs: the CTAs holding many
    # segment starts get fewer blocks, and every CTA's blocks plus K units per
    # segment it starts add up to the same load -- within 2K + 1, since a
    # range may begin or end inside a segment's overhead units
    lens = [64] * 64 + [40_000]
    s = shape(B=65, H=8, Hkv=1, d=128, bs=16, maxblk=2500, P=8000, dtype=pg.PA_BF16)
    K = K_UNITS[(16, 128)]
    C = 8
    loads = []
    for c in range(C):
        pieces = pg.pa_plan_pieces(s, None, lens, C, c)
        blocks = sum(k1 - k0 for (_, _, k0, k1, _) in pieces)
        starts = sum(1 for (_, _, k0, _, _) in pieces if k0 == 0)
        loads.append(blocks + K * starts)
    assert max(loads) - min(loads) <= 2 * K + 1
    first = sum(k1 - k0 for (_, _, k0, k1, _) in pg.pa_plan_pieces(s, None, lens, C, 0))
    last = sum(k1 - k0 for (_, _, k0, k1, _) in pg.pa_plan_pieces(s, None, lens, C, C - 1))
    assert first < last - 5 * K


def test_batch_limit_matches_the_header():
    s = pg.pa_shape(pg.PA_MAX_BATCH, 8, 2, 128, 16, 4, 64, pg.PA_BF16)
    assert pg.pa_workspace_size(s, pg.options(num_ctas=8)) > 0
    s.batch = pg.PA_MAX_BATCH + 1
    with pytest.raises(pg.PagedGQAError) as e:
        pg.pa_workspace_size(s, pg.options(num_ctas=8))
    assert e.value.code == pg.PA_ERR_SHAPE


def test_host_buffer_calls_reject_bad_arguments_before_any_cuda_call():
    L = pg.lib()
    o = pg.options(num_ctas=8)
    s = shape()
    st = ctypes.c_uint32(7)

    def host(s=s, opts=o, q=FAKE, t=FAKE, sl=FAKE, out=FAKE, ws=FAKE, ws_bytes=1 << 30):
        return L.pa_decode_host(ctypes.byref(s), ctypes.byref(opts) if opts else None, q, FAKE,
                                FAKE, t, sl, 0.125, out, ctypes.byref(st), ws, ws_bytes, None)

    for kw in (dict(q=None), dict(t=None), dict(sl=None), dict(out=None), dict(ws=None)):
        assert host(**kw) == pg.PA_ERR_NULL, kw
    need = pg.pa_workspace_size_host(s, o)
    assert host(ws_bytes=need - 1) == pg.PA_ERR_WORKSPACE
    assert host(opts=pg.options(num_ctas=8, phase=pg.PA_PHASE_SPLIT)) == pg.PA_ERR_OPTION
    assert host(s=shape(d=96)) == pg.PA_ERR_SHAPE
    # an empty batch is a no-op that needs no pointers and reports a clean status
    assert host(s=shape(B=0), q=None, t=None, sl=None, out=None, ws=None) == pg.PA_OK
    assert st.value == 0

    def multi(total_q=5, max_q=2, ws_bytes=1 << 30, cu=FAKE):
        return L.pa_decode_multi_host(ctypes.byref(s), ctypes.byref(o), FAKE, cu, total_q, max_q,
                                      1, FAKE, FAKE, FAKE, FAKE, 0.125, FAKE, ctypes.byref(st),
                                      FAKE, ws_bytes, None)

    assert multi(cu=None) == pg.PA_ERR_NULL
    assert multi(max_q=0) == pg.PA_ERR_SHAPE
    assert multi(total_q=-1) == pg.PA_ERR_SHAPE
    n5 = pg.pa_workspace_size_multi_host(s, 2, 5, o)
    assert multi(ws_bytes=n5 - 1) == pg.PA_ERR_WORKSPACE
    st.value = 7
    assert multi(total_q=0) == pg.PA_OK and st.value == 0


def test_host_workspace_adds_the_staging():
    s = shape(B=256, H=32, Hkv=8, d=128, bs=32, maxblk=1024, P=30000, dtype=pg.PA_BF16)
    o = pg.options(num_ctas=304)
    base, host = pg.pa_workspace_size(s, o), pg.pa_workspace_size_host(s, o)
    staged = 256 * 32 * 128 * (2 + 4) + 256 * 1024 * 4 + 256 * 4 + 4
    assert staged <= host - base <= staged + 6 * 256
    m = [pg.pa_workspace_size_multi_host(s, 4, n, o) for n in (0, 1, 1024)]
    assert m[0] >= pg.pa_workspace_size_multi(s, 4, o) + 256 * 1024 * 4
    assert m[1] - m[0] >= 32 * 128 * 6 and m[2] - m[0] >= 1024 * 32 * 128 * 6


def test_with_group_keeps_the_cache_and_draws_new_queries():
    from paged_gqa_decode_pa_gb300 import workloads as wl

    a = wl.random_workload([5, 40, 0], H=8, Hkv=2, d=64, bs=16, dtype="f16", seed=3)
    k, v, t, sl = a.k_cache.copy(), a.v_cache.copy(), a.block_table.copy(), a.cache_seqlens.copy()
    b = wl.with_group(a, 3, seed=9)
    assert b.H == 6 and b.G == 3 and b.q.shape == (3, 6, 64)
    assert np.array_equal(b.k_cache, k) and np.array_equal(b.v_cache, v)
    assert np.array_equal(b.block_table, t) and np.array_equal(b.cache_seqlens, sl)
    c = wl.with_group(wl.random_workload([5, 40, 0], H=8, Hkv=2, d=64, bs=16, dtype="f16",
                                         seed=3), 3, seed=9)
    assert np.array_equal(b.q, c.q)  # seeded
    with pytest.raises(ValueError):
        wl.with_group(c, 0)


def test_noalloc_rejects_split_or_merge_phase_before_any_cuda_call():
    L = pg.lib()
    s = shape()
    for phase in (pg.PA_PHASE_SPLIT, pg.PA_PHASE_MERGE):
        o = pg.options(num_ctas=8, phase=phase)
        assert L.pa_decode_noalloc(ctypes.byref(s), ctypes.byref(o), FAKE, FAKE, FAKE, FAKE,
                                   FAKE, 0.125, FAKE, None, None) == pg.PA_ERR_OPTION


@pytest.mark.parametrize("grid", [152, 256])
def test_noalloc_scratch_holds_the_default_split_at_the_largest_shapes(grid):
    # the bound include/pagedgqa.h states for pa_decode_noalloc: the default
    # balanced split at B = PA_MAX_BATCH, G = 8, d = 256 fits the static
    # scratch for any persistent grid of up to 256 CTAs
    limit = pg.PA_STATIC_SCRATCH_BYTES
    for dtype in (pg.PA_F16, pg.PA_BF16):
        s = shape(B=pg.PA_MAX_BATCH, H=64, Hkv=8, d=256, bs=16, maxblk=8192, P=1 << 20,
                  dtype=dtype)
        assert pg.pa_workspace_size(s, pg.options(num_ctas=grid)) <= limit
