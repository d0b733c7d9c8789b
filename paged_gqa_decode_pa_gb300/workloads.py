"""Seeded synthetic inputs for paged GQA decode.

This module only draws inputs: sequence lengths, block tables, physical pool
layouts and N(0,1) query/key/value values rounded to the storage type.  It
holds none of the attention arithmetic, imports neither the CUDA library nor
the oracle, and is the one piece of code both sides share.

Recipe (every workload): ``numpy.random.default_rng(seed)`` drawn in the
fixed order lengths -> block permutation -> q -> K -> V (-> outlier rows);
values are float32 N(0,1) rounded to nearest-even into fp16 or bf16 and kept
as raw 16-bit patterns (``uint16``).  Pools above 2^24 elements are drawn in
chunks of whole physical blocks, chunk i from child generator i of
``rng.spawn``.

The shapes follow the settings the pages describe:
  * ``p5_example``          -- the Hugging Face "Paged attention" decoding-path
                               example (block size 32, lengths [30, 32, 70],
                               its block table verbatim), 4 query / 2 kv heads.
  * ``qwen2_b8_g7_d64``     -- Qwen2-0.5B attention shape (14 query heads,
                               2 kv heads, d=64) from the paged-attention-runtime
                               design page, 8 concurrent sequences, block 16.
  * ``long_ctx_100k_g6_d256`` -- the BI-V100 architecture page's parameters:
                               d=256, 24 query / 4 kv heads, 100,000 tokens,
                               block 16, split into 512-token partitions.
  * ``prefix_share_b64_g8_d128`` -- 64 query / 8 kv heads (G=8, the AHBM design
                               page's real-GQA case), 64 sequences whose first
                               32 logical blocks map to one shared set of
                               physical blocks (prefix sharing, design page of
                               the paged-attention runtime).
  * ``serving_mix_b256_g4_d128`` -- 256 sequences, lognormal lengths (median
                               2048, sigma 1, clipped to [1, 32768]), block 32,
                               1% of K rows scaled by 8.
"""
from __future__ import annotations

import dataclasses
import math
import os
from typing import Optional

import numpy as np

F16 = "f16"
BF16 = "bf16"

_CHUNK_ELEMS = 1 << 24  # elements per chunk for large pools


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    H: int
    Hkv: int
    d: int
    block_size: int
    max_blocks_per_seq: int
    num_blocks: int  # P, physical blocks in the pool
    dtype: str  # "f16" | "bf16"
    scale: float
    cache_seqlens: np.ndarray  # [B] int32
    block_table: np.ndarray  # [B, maxblk] int32, -1 = unallocated
    q: np.ndarray  # [B, H, d] uint16 bit patterns
    k_cache: np.ndarray  # [P, bs, Hkv, d] uint16
    v_cache: np.ndarray  # [P, bs, Hkv, d] uint16
    partition_tokens: int = 0  # the split size the setting names (0 = none)
    seed: int = 0
    # several query tokens per sequence: q is packed [total_q, H, d] and
    # sequence b owns rows cu_q[b] .. cu_q[b+1]-1 (None: one token each)
    cu_q: Optional[np.ndarray] = None
    causal: bool = True

    @property
    def max_q(self) -> int:
        return 1 if self.cu_q is None else max(1, int(np.diff(self.cu_q).max(initial=0)))

    @property
    def G(self) -> int:
        return self.H // self.Hkv

    def read_mask(self) -> np.ndarray:
        """[P, bs] bool: True where some sequence's valid tokens map."""
        mask = np.zeros((self.num_blocks, self.block_size), dtype=bool)
        bs = self.block_size
        for b in range(self.B):
            n = int(self.cache_seqlens[b])
            full, tail = divmod(n, bs)
            ids = self.block_table[b, :full]
            mask[ids[ids >= 0], :] = True
            if tail:
                p = self.block_table[b, full]
                if p >= 0:
                    mask[p, :tail] = True
        return mask

    def unique_kv_tokens(self) -> int:
        """Number of distinct (physical block, row) slots the step must read."""
        return int(self.read_mask().sum())

    def kv_bytes(self) -> int:
        """Unique K+V bytes one decode step must read (shared slots once)."""
        return self.unique_kv_tokens() * self.Hkv * self.d * 2 * 2

    def torch_tensors(self, device="cpu"):
        """(q, k_cache, v_cache, block_table, cache_seqlens) as torch tensors."""
        import torch

        tdt = torch.float16 if self.dtype == F16 else torch.bfloat16

        def cast(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(tdt).to(device)

        return (cast(self.q), cast(self.k_cache), cast(self.v_cache),
                torch.from_numpy(np.ascontiguousarray(self.block_table)).to(device),
                torch.from_numpy(np.ascontiguousarray(self.cache_seqlens)).to(device))


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to nearest-even fp16/bf16; return uint16 patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == F16:
        return x.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        import torch

        t = torch.from_numpy(x).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16)
    raise ValueError(dtype)


def from_bits(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float32 values of stored fp16/bf16 patterns."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == F16:
        return bits.view(np.float16).astype(np.float32)
    if dtype == BF16:
        return (bits.astype(np.uint32) << 16).view(np.float32)
    raise ValueError(dtype)


def nan_bits(dtype: str) -> int:
    return 0x7E00 if dtype == F16 else 0x7FC0


def _normal_bits(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    """N(0,1) float32 draws rounded into the storage type.

    Arrays up to _CHUNK_ELEMS elements are drawn from `rng` directly.  Larger
    ones are cut into chunks of whole leading-axis rows, each drawn from its
    own child generator (rng.spawn, deterministic), filled by a thread pool.
    """
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.uint16)
    rows = shape[0]
    per_row = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    if rows * per_row <= _CHUNK_ELEMS:
        out[...] = to_bits(rng.standard_normal(shape, dtype=np.float32), dtype)
        return out
    step = max(1, _CHUNK_ELEMS // max(per_row, 1))
    starts = list(range(0, rows, step))
    children = rng.spawn(len(starts))

    def fill(i):
        r0 = starts[i]
        r1 = min(rows, r0 + step)
        x = children[i].standard_normal((r1 - r0,) + shape[1:], dtype=np.float32)
        out[r0:r1] = to_bits(x, dtype)

    import concurrent.futures as cf

    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        list(ex.map(fill, range(len(starts))))
    return out


def _table_from_lengths(rng, lens, bs, maxblk, shared_prefix_blocks=0):
    """Block table for the given lengths.

    The first ``shared_prefix_blocks`` logical blocks of every row map to the
    physical blocks 0..n-1 (one shared set); every other used logical block
    gets a distinct physical block.  The distinct ids are a random
    permutation of the pool that remains, drawn without replacement, handed
    out sequence by sequence.  Unused table entries are -1.
    """
    B = len(lens)
    nblk = [(int(n) + bs - 1) // bs for n in lens]
    own = [max(0, nb - shared_prefix_blocks) for nb in nblk]
    total_own = int(sum(own))
    P = shared_prefix_blocks + total_own
    perm = rng.permutation(total_own).astype(np.int64) + shared_prefix_blocks
    table = np.full((B, maxblk), -1, dtype=np.int32)
    pos = 0
    for b in range(B):
        k = min(nblk[b], shared_prefix_blocks)
        table[b, :k] = np.arange(k, dtype=np.int32)
        table[b, k:nblk[b]] = perm[pos:pos + own[b]]
        pos += own[b]
    return table, P


def _poison(w: Workload) -> None:
    """Fill every pool slot no valid token maps to with NaN."""
    mask = w.read_mask()
    nb = nan_bits(w.dtype)
    w.k_cache[~mask] = nb
    w.v_cache[~mask] = nb


def p5_example(seed: int = 1, poison: bool = False, dtype: str = F16,
               H: int = 4, Hkv: int = 2, d: int = 64) -> Workload:
    """The Hugging Face decoding-path example: block 32, lengths [30,32,70]."""
    rng = np.random.default_rng(seed)
    lens = np.array([30, 32, 70], dtype=np.int32)
    table = np.array([[2, -1, -1, -1], [0, 1, -1, -1], [3, 5, 6, -1]], dtype=np.int32)
    P, bs, B = 8, 32, 3
    q = _normal_bits(rng, (B, H, d), dtype)
    k = _normal_bits(rng, (P, bs, Hkv, d), dtype)
    v = _normal_bits(rng, (P, bs, Hkv, d), dtype)
    w = Workload("p5_example", B, H, Hkv, d, bs, 4, P, dtype, 1.0 / math.sqrt(d),
                 lens, table, q, k, v, seed=seed)
    if poison:
        _poison(w)
    return w


def random_workload(lens, H, Hkv, d, bs, dtype=BF16, seed=0, maxblk=None,
                    shared_prefix_blocks=0, outlier_frac=0.0, outlier_scale=8.0,
                    poison=False, extra_blocks=0, name="random", scale=None,
                    partition_tokens=0) -> Workload:
    """General seeded workload with the given per-sequence lengths."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    B = int(lens.shape[0])
    need = max([(int(n) + bs - 1) // bs for n in lens] + [1])
    if maxblk is None:
        maxblk = need
    if maxblk < need:
        raise ValueError("max_blocks_per_seq smaller than the longest sequence")
    table, P = _table_from_lengths(rng, lens, bs, maxblk, shared_prefix_blocks)
    P = max(P + extra_blocks, 1)
    q = _normal_bits(rng, (B, H, d), dtype)
    k = _normal_bits(rng, (P, bs, Hkv, d), dtype)
    v = _normal_bits(rng, (P, bs, Hkv, d), dtype)
    if outlier_frac > 0:
        sel = rng.random((P, bs, Hkv)) < outlier_frac
        kf = from_bits(k[sel], dtype) * np.float32(outlier_scale)
        k[sel] = to_bits(kf, dtype)
    w = Workload(name, B, H, Hkv, d, bs, int(maxblk), int(P), dtype,
                 float(scale if scale is not None else 1.0 / math.sqrt(d)),
                 lens, table, q, k, v, partition_tokens=partition_tokens, seed=seed)
    if poison:
        _poison(w)
    return w


def qwen2_b8_g7_d64(seed: int = 2, poison: bool = False) -> Workload:
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, 4096, size=8, endpoint=True).astype(np.int32)
    return random_workload(lens, 14, 2, 64, 16, dtype=F16, seed=seed + 1000, maxblk=256,
                           poison=poison, name="qwen2_b8_g7_d64")


def long_ctx_100k_g6_d256(seed: int = 3, poison: bool = False, length: int = 100_000
                          ) -> Workload:
    lens = np.array([length], dtype=np.int32)
    return random_workload(lens, 24, 4, 256, 16, dtype=BF16, seed=seed,
                           maxblk=(length + 15) // 16, poison=poison,
                           name="long_ctx_100k_g6_d256", partition_tokens=512)


def prefix_share_b64_g8_d128(seed: int = 4, poison: bool = False) -> Workload:
    rng = np.random.default_rng(seed)
    lens = rng.integers(512, 8192, size=64, endpoint=True).astype(np.int32)
    return random_workload(lens, 64, 8, 128, 16, dtype=BF16, seed=seed + 1000, maxblk=512,
                           shared_prefix_blocks=32, poison=poison,
                           name="prefix_share_b64_g8_d128")


def serving_mix_lengths(seed: int = 5, B: int = 256) -> np.ndarray:
    rng = np.random.default_rng(seed)
    x = np.exp(math.log(2048.0) + 1.0 * rng.standard_normal(B))
    return np.clip(np.round(x), 1, 32768).astype(np.int32)


def serving_mix_b256_g4_d128(seed: int = 5, poison: bool = False, B: int = 256) -> Workload:
    lens = serving_mix_lengths(seed, B)
    return random_workload(lens, 32, 8, 128, 32, dtype=BF16, seed=seed + 1000, maxblk=1024,
                           outlier_frac=0.01, outlier_scale=8.0, poison=poison,
                           name=f"serving_mix_b{B}_g4_d128")


def serving_mix_b32_g4_d128(seed: int = 5, poison: bool = False) -> Workload:
    """The serving mix at 32 sequences (~0.4 GB of K/V, still above L2): the
    size used for detailed profiler captures."""
    return serving_mix_b256_g4_d128(seed, poison, B=32)


def with_query_tokens(w: Workload, lens_q, seed: int = 0, causal: bool = True,
                      name: Optional[str] = None) -> Workload:
    """The same cache with lens_q[b] query tokens for sequence b, packed
    (cumulative counts in cu_q) and drawn like q.  The cache lengths already
    count the query tokens: they are the last positions of each sequence."""
    rng = np.random.default_rng(seed)
    lens_q = np.asarray(lens_q, dtype=np.int32)
    if lens_q.shape != (w.B,):
        raise ValueError("one query count per sequence")
    cu = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    w.q = _normal_bits(rng, (int(cu[-1]), w.H, w.d), w.dtype)
    w.cu_q = cu
    w.causal = bool(causal)
    if name:
        w.name = name
    return w


def with_group(w: Workload, G: int, seed: int = 0, name: Optional[str] = None) -> Workload:
    """The same cache, table and lengths with G query heads per kv head
    (H = G * Hkv), the queries drawn afresh: the K/V a step reads does not
    change with G, only the heads that share it."""
    if G < 1:
        raise ValueError("G >= 1")
    rng = np.random.default_rng(seed)
    w.H = G * w.Hkv
    rows = w.B if w.cu_q is None else int(w.cu_q[-1])
    w.q = _normal_bits(rng, (rows, w.H, w.d), w.dtype)
    if name:
        w.name = name
    return w


def serving_mix_b256_q4_g4_d128(seed: int = 5, poison: bool = False) -> Workload:
    """The serving mix verifying 4 tokens per sequence (3 drafted + 1), causal."""
    w = serving_mix_b256_g4_d128(seed, poison)
    return with_query_tokens(w, np.full(w.B, 4), seed=seed + 2000,
                             name="serving_mix_b256_q4_g4_d128")


def prefix_share_b64_q2_g8_d128(seed: int = 4, poison: bool = False) -> Workload:
    """Prefix sharing with 2 query tokens per sequence, causal."""
    w = prefix_share_b64_g8_d128(seed, poison)
    return with_query_tokens(w, np.full(w.B, 2), seed=seed + 2000,
                             name="prefix_share_b64_q2_g8_d128")


WORKLOADS = {
    "p5_example": p5_example,
    "qwen2_b8_g7_d64": qwen2_b8_g7_d64,
    "long_ctx_100k_g6_d256": long_ctx_100k_g6_d256,
    "prefix_share_b64_g8_d128": prefix_share_b64_g8_d128,
    "serving_mix_b256_g4_d128": serving_mix_b256_g4_d128,
    "serving_mix_b32_g4_d128": serving_mix_b32_g4_d128,
    "serving_mix_b256_q4_g4_d128": serving_mix_b256_q4_g4_d128,
    "prefix_share_b64_q2_g8_d128": prefix_share_b64_q2_g8_d128,
}


def make(name: str, seed: Optional[int] = None, poison: bool = False) -> Workload:
    fn = WORKLOADS[name]
    return fn(poison=poison) if seed is None else fn(seed=seed, poison=poison)
