"""Shared helpers of the GPU tests: run the library on a workload, run the
oracle on the same inputs, compare within the stated tolerance."""
import numpy as np
import torch

import oracle
import paged_gqa_decode_pa_gb300 as pg

# Tolerance for fp16/bf16 inputs with fp32 output, against the float64 oracle.
MAX_ABS = 2e-3
MEAN_ABS = 2e-4


def run_gpu(w, opts=None, out=None, ws=None, device="cuda", stream=None):
    q, k, v, t, sl = w.torch_tensors(device)
    if out is None:
        out = torch.full((w.B, w.H, w.d), float("nan"), dtype=torch.float32, device=device)
    shape = pg.shape_of(q, k, t)
    if ws is None:
        ws = pg.alloc_workspace(shape, opts, device)
    pg.pa_decode(q, k, v, t, sl, w.scale, out, ws, opts, stream)
    status = pg.pa_read_status(ws, stream)
    return out.cpu().numpy().astype(np.float64), status


def run_oracle(w, pairs=None):
    return oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens, w.scale,
                         w.dtype, pairs=pairs)


def assert_close(got, ref, what=""):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite outputs"
    err = np.abs(got - ref)
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max|err|={mx:.3g} mean|err|={mean:.3g}"
    return mx, mean


def sample_pairs(w, n, seed=0):
    rng = np.random.default_rng(seed)
    b = rng.integers(0, w.B, size=n)
    h = rng.integers(0, w.H, size=n)
    # always include the longest sequence and the first/last heads
    bl = int(np.argmax(w.cache_seqlens))
    extra = np.array([[bl, 0], [bl, w.H - 1], [0, 0], [w.B - 1, w.H - 1]])
    pairs = np.concatenate([np.stack([b, h], axis=1), extra]).astype(np.int32)
    return np.unique(pairs, axis=0)
