"""Seeded synthetic inputs for paged MLA decode.

This module builds inputs only: random values, their rounding to the storage
dtype (bf16 bit patterns or OCP e4m3fn codes with a per-tensor scale), block
tables, sequence lengths, query-length layouts and top-k index lists. It holds
none of the decode's arithmetic. The CUDA path and the oracle both consume
what it returns, so neither depends on the other for its inputs.

Every array is produced by ``numpy.random.default_rng(seed)``; the same seed
gives the same bytes on any machine.

Shapes follow the problem statement of the vLLM ROCm AITER MLA backend pages:
``q [tokens, heads, 576]`` (512 latent columns followed by 64 rope columns),
``kv_c_and_k_pe_cache [blocks, block_size, 576]`` whose first 512 columns are
also the values, ``block_table [requests, max_blocks]`` int32, ``seq_lens``
int32, ``qo_indptr [requests + 1]`` int32, and for the sparse variant
``topk_indices [tokens, topk]`` int32 with -1 marking an unused entry.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

HEAD_DIM = 576          # kv_lora_rank + qk_rope_head_dim
KV_LORA_RANK = 512      # value width: the first 512 columns of a cache row
ROPE_DIM = HEAD_DIM - KV_LORA_RANK
E4M3_MAX = 448.0

BF16_NAN_BITS = 0x7FC0  # quiet NaN in bf16
E4M3_NAN_CODE = 0x7F    # S.1111.111 is NaN in e4m3fn


@dataclass
class Workload:
    """One decode call's inputs, in the storage dtypes the kernels read."""

    name: str
    num_heads: int
    block_size: int
    q_dtype: str                     # "bf16" or "fp8"
    kv_dtype: str                    # "bf16" or "fp8"
    q: np.ndarray                    # uint16 bf16 bits or uint8 e4m3 codes, [T, H, 576]
    cache: np.ndarray                # same storage kind, [num_blocks, block_size, 576]
    block_table: np.ndarray          # int32 [R, max_blocks_per_req]
    seq_lens: np.ndarray             # int32 [R], KV length including the new tokens
    qo_indptr: np.ndarray | None     # int32 [R + 1]; None means one token per request
    softmax_scale: float
    q_scale: float = 1.0
    kv_scale: float = 1.0
    sinks: np.ndarray | None = None  # float32 [H], natural-log logits
    num_segments: int = 0            # 0 lets the planner choose
    # sparse variant
    req_id_per_token: np.ndarray | None = None   # int32 [T]
    topk_indices: np.ndarray | None = None       # int32 [T, topk], -1 = unused
    meta: dict = field(default_factory=dict)

    @property
    def num_reqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.cache.shape[0])

    @property
    def max_blocks_per_req(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def topk(self) -> int:
        return 0 if self.topk_indices is None else int(self.topk_indices.shape[1])

    @property
    def max_qlen(self) -> int:
        if self.qo_indptr is None:
            return 1
        return int(np.max(np.diff(self.qo_indptr))) if self.num_reqs else 0

    @property
    def sparse(self) -> bool:
        return self.topk_indices is not None


# --------------------------------------------------------------------------
# storage-dtype rounding of generated values (input construction only)
# --------------------------------------------------------------------------

def float32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bf16 (round to nearest, ties to even)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def float32_to_e4m3_codes(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values (|x| <= 448) to e4m3fn codes.

    Uses PyTorch's float8_e4m3fn cast (round to nearest even); inputs are
    clipped to +-448 first so no value turns into NaN.
    """
    import torch

    t = torch.from_numpy(np.clip(np.ascontiguousarray(x, dtype=np.float32),
                                 -E4M3_MAX, E4M3_MAX))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def _normal_storage(rng: np.random.Generator, shape, std: float, dtype: str,
                    scale: float | None = None, chunk_rows: int = 1 << 16):
    """Draw N(0, std^2) float32 values of ``shape`` and store them as ``dtype``.

    Returns (storage array, per-tensor scale). For fp8 the scale is
    amax / 448 of the drawn values unless given; the stored code is
    round(value / scale). Large tensors are drawn in row chunks so the float32
    temporaries stay small; the draw order is the row-major order either way.
    """
    shape = tuple(int(s) for s in shape)
    rows = shape[0]
    inner = shape[1:]
    out = np.empty(shape, dtype=np.uint16 if dtype == "bf16" else np.uint8)
    if dtype == "bf16":
        for a in range(0, rows, chunk_rows):
            b = min(rows, a + chunk_rows)
            v = rng.standard_normal((b - a,) + inner, dtype=np.float32) * np.float32(std)
            out[a:b] = float32_to_bf16_bits(v)
        return out, 1.0
    if dtype != "fp8":
        raise ValueError(f"unknown storage dtype {dtype!r}")
    # fp8: two passes over the same stream (a cloned generator) so the
    # per-tensor scale sees every value before any is rounded.
    if scale is None:
        probe = np.random.Generator(type(rng.bit_generator)())
        probe.bit_generator.state = rng.bit_generator.state
        amax = 0.0
        for a in range(0, rows, chunk_rows):
            b = min(rows, a + chunk_rows)
            v = probe.standard_normal((b - a,) + inner, dtype=np.float32) * np.float32(std)
            amax = max(amax, float(np.max(np.abs(v))) if v.size else 0.0)
        scale = (amax / E4M3_MAX) if amax > 0 else 1.0
    inv = np.float32(1.0 / scale)
    for a in range(0, rows, chunk_rows):
        b = min(rows, a + chunk_rows)
        v = rng.standard_normal((b - a,) + inner, dtype=np.float32) * np.float32(std)
        out[a:b] = float32_to_e4m3_codes(v * inv)
    return out, float(scale)


def _poison_value(dtype: str) -> int:
    return BF16_NAN_BITS if dtype == "bf16" else E4M3_NAN_CODE


# --------------------------------------------------------------------------
# dense (optionally multi-token) workloads
# --------------------------------------------------------------------------

def build_dense(seed: int, *, seq_lens, num_heads: int, block_size: int,
                dtype: str = "bf16", q_dtype: str | None = None,
                q_std: float = 1.0, kv_std: float = 1.0, qlens=None,
                with_sinks: bool = False, spare_blocks: int = 3,
                extra_table_cols: int = 1, num_segments: int = 0,
                softmax_scale: float = 1.0 / math.sqrt(192.0),
                poison: bool = True, name: str = "dense") -> Workload:
    """A paged dense decode batch.

    Every request owns ``cdiv(seq_len, block_size)`` physical blocks drawn
    from a random permutation of the pool, so logically adjacent blocks are
    scattered. With ``poison`` the spare blocks, the rows past ``seq_len`` in
    a request's last block, and every unused block-table entry (which points
    at a spare block) hold NaN: a kernel that reads a key it must not read
    turns its output into NaN.
    """
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    R = int(seq_lens.shape[0])
    q_dtype = q_dtype or dtype
    qlens = np.ones(R, dtype=np.int64) if qlens is None else np.asarray(qlens, dtype=np.int64)
    if np.any(qlens < 1) or np.any(seq_lens < 0):
        raise ValueError("qlens must be >= 1 and seq_lens >= 0")
    T = int(qlens.sum())
    H = int(num_heads)
    bpr = (seq_lens + block_size - 1) // block_size
    mb = int(max(1, int(bpr.max()) if R else 1)) + int(extra_table_cols)
    used = int(bpr.sum())
    nb = used + int(spare_blocks)
    perm = rng.permutation(nb).astype(np.int32)
    spare = perm[used:] if spare_blocks > 0 else perm[:1]
    bt = np.empty((R, mb), dtype=np.int32)
    pos = 0
    for r in range(R):
        n = int(bpr[r])
        bt[r, :n] = perm[pos:pos + n]
        pos += n
        fill = rng.choice(spare, size=mb - n) if spare.size else 0
        bt[r, n:] = fill
    cache, kv_scale = _normal_storage(rng, (nb, block_size, HEAD_DIM), kv_std, dtype)
    q, q_scale = _normal_storage(rng, (T, H, HEAD_DIM), q_std, q_dtype)
    if poison:
        pv = _poison_value(dtype)
        if spare_blocks > 0:
            cache[perm[used:]] = pv
        for r in range(R):
            L = int(seq_lens[r])
            n = int(bpr[r])
            if n and L % block_size:
                cache[bt[r, n - 1], L % block_size:] = pv
    sinks = rng.standard_normal(H).astype(np.float32) if with_sinks else None
    qo = None
    if np.any(qlens != 1):
        qo = np.zeros(R + 1, dtype=np.int32)
        qo[1:] = np.cumsum(qlens)
    return Workload(name=name, num_heads=H, block_size=int(block_size),
                    q_dtype=q_dtype, kv_dtype=dtype, q=q, cache=cache,
                    block_table=bt, seq_lens=seq_lens.astype(np.int32),
                    qo_indptr=qo, softmax_scale=float(softmax_scale),
                    q_scale=float(q_scale), kv_scale=float(kv_scale),
                    sinks=sinks, num_segments=int(num_segments),
                    meta={"seed": seed, "spare_blocks": np.asarray(perm[used:])})


# --------------------------------------------------------------------------
# sparse top-k workloads
# --------------------------------------------------------------------------

def build_sparse(seed: int, *, num_reqs: int, tokens_per_req: int, num_heads: int,
                 cache_tokens: int, topk: int, block_size: int = 64,
                 dtype: str = "bf16", max_pad: int = 256,
                 interspersed_rows: int = 0, spare_blocks: int = 2,
                 softmax_scale: float = 1.0 / math.sqrt(192.0),
                 num_segments: int = 0, name: str = "sparse") -> Workload:
    """A sparse top-k decode batch.

    Every request holds ``cache_tokens`` tokens in scattered blocks. Each query
    token carries ``topk`` distinct positions drawn uniformly from
    ``[0, cache_tokens)``, unsorted; a per-token count drawn from
    ``[0, max_pad)`` of trailing entries is replaced by -1. The first
    ``interspersed_rows`` tokens additionally get -1 at random interior
    positions.
    """
    rng = np.random.default_rng(seed)
    R = int(num_reqs)
    T = R * int(tokens_per_req)
    bpr = (cache_tokens + block_size - 1) // block_size
    used = R * bpr
    nb = used + int(spare_blocks)
    perm = rng.permutation(nb).astype(np.int32)
    bt = perm[:used].reshape(R, bpr).copy()
    cache, kv_scale = _normal_storage(rng, (nb, block_size, HEAD_DIM), 1.0, dtype)
    pv = _poison_value(dtype)
    cache[perm[used:]] = pv
    if cache_tokens % block_size:
        for r in range(R):
            cache[bt[r, -1], cache_tokens % block_size:] = pv
    q, q_scale = _normal_storage(rng, (T, num_heads, HEAD_DIM), 1.0, dtype)
    idx = np.empty((T, topk), dtype=np.int32)
    for t in range(T):
        idx[t] = rng.choice(cache_tokens, size=topk, replace=False).astype(np.int32)
        pad = int(rng.integers(0, max_pad)) if max_pad > 0 else 0
        if pad:
            idx[t, topk - pad:] = -1
    for t in range(min(int(interspersed_rows), T)):
        holes = rng.choice(topk, size=max(1, topk // 8), replace=False)
        idx[t, holes] = -1
    req = np.repeat(np.arange(R, dtype=np.int32), tokens_per_req)
    seq = np.full(R, cache_tokens, dtype=np.int32)
    return Workload(name=name, num_heads=int(num_heads), block_size=int(block_size),
                    q_dtype=dtype, kv_dtype=dtype, q=q, cache=cache,
                    block_table=bt, seq_lens=seq, qo_indptr=None,
                    softmax_scale=float(softmax_scale), q_scale=float(q_scale),
                    kv_scale=float(kv_scale), sinks=None,
                    num_segments=int(num_segments), req_id_per_token=req,
                    topk_indices=idx, meta={"seed": seed})


# --------------------------------------------------------------------------
# the five workload shapes (sizes can be scaled down for oracle parity)
# --------------------------------------------------------------------------

def tiny_dense(seed: int = 1) -> Workload:
    """Batch 2, 16 heads, seq_lens {37, 130}, block 16, bf16 ~N(0, 0.5^2),
    4 segments with tile 16, shuffled block table."""
    return build_dense(seed, seq_lens=[37, 130], num_heads=16, block_size=16,
                       q_std=0.5, kv_std=0.5, num_segments=4, name="tiny_dense")


def dsv3_bf16(seed: int = 2, batch: int = 64, num_heads: int = 128,
              seq_lo: int = 1024, seq_hi: int = 8192, num_segments: int = 0,
              poison: bool = True) -> Workload:
    """DeepSeek-V3-shaped bf16 decode: 128 heads, qlen 1, block 64,
    seq_lens uniform in [seq_lo, seq_hi], values ~N(0, 1)."""
    rng = np.random.default_rng(seed + 1000)
    seq = rng.integers(seq_lo, seq_hi + 1, size=batch)
    return build_dense(seed, seq_lens=seq, num_heads=num_heads, block_size=64,
                       num_segments=num_segments, poison=poison,
                       name=f"dsv3_bf16_b{batch}_h{num_heads}")


def fp8_decode(num_heads: int, seed: int = 3, batch: int = 52,
               seq_len: int = 16384, num_segments: int = 0,
               poison: bool = True) -> Workload:
    """fp8 e4m3 q and KV with per-tensor scales: qlen 1, block 64, every
    request ``seq_len`` tokens, values ~N(0, 1) before quantisation."""
    return build_dense(seed, seq_lens=[seq_len] * batch, num_heads=num_heads,
                       block_size=64, dtype="fp8", num_segments=num_segments,
                       poison=poison, name=f"fp8_b{batch}_h{num_heads}_L{seq_len}")


def mtp_sinks(seed: int = 4, batch: int = 32, num_heads: int = 128,
              median: float = 4096.0, sigma: float = 1.0, lo: int = 128,
              hi: int = 32768, num_segments: int = 0) -> Workload:
    """Multi-token causal decode with sinks: qlen uniform in {2, 3, 4},
    seq_lens lognormal(ln median, sigma) clipped to [lo, hi], bf16,
    per-head float32 sinks ~N(0, 1)."""
    rng = np.random.default_rng(seed + 1000)
    qlens = rng.integers(2, 5, size=batch)
    seq = np.clip(np.round(rng.lognormal(math.log(median), sigma, size=batch)), lo, hi)
    seq = np.maximum(seq.astype(np.int64), qlens)
    return build_dense(seed, seq_lens=seq, num_heads=num_heads, block_size=64,
                       qlens=qlens, with_sinks=True, num_segments=num_segments,
                       name=f"mtp_sinks_b{batch}_h{num_heads}")


def sparse_topk(seed: int = 5, num_reqs: int = 16, tokens_per_req: int = 8,
                num_heads: int = 128, cache_tokens: int = 65536, topk: int = 2048,
                interspersed_rows: int = 0, max_pad: int = 256,
                num_segments: int = 0) -> Workload:
    """Sparse decode: 8 tokens per request, 128 heads, bf16, a 65536-token
    cache per request at block 64, 2048 distinct indices per token with
    trailing -1 padding."""
    return build_sparse(seed, num_reqs=num_reqs, tokens_per_req=tokens_per_req,
                        num_heads=num_heads, cache_tokens=cache_tokens, topk=topk,
                        max_pad=max_pad, interspersed_rows=interspersed_rows,
                        num_segments=num_segments,
                        name=f"sparse_r{num_reqs}x{tokens_per_req}_h{num_heads}_k{topk}")


def dcp_shard_positions(w: Workload, world: int, rank: int, pad_to: int = 128):
    """Per-token logical positions one rank holds when token ``p`` of a
    request lives on rank ``p % world`` (decode context parallelism, interleave
    1), for single-token rows: ``[T, K]`` int32, -1 padded to a multiple of
    ``pad_to``, plus the request id of every token."""
    if w.qo_indptr is not None:
        raise ValueError("shard positions are built for one token per request")
    T = w.num_tokens
    lists = [np.arange(rank, int(w.seq_lens[t]), world, dtype=np.int32) for t in range(T)]
    K = max([len(l) for l in lists] + [1])
    K = -(-K // pad_to) * pad_to
    idx = np.full((T, K), -1, dtype=np.int32)
    for t, l in enumerate(lists):
        idx[t, :len(l)] = l
    return idx, np.arange(T, dtype=np.int32)
