"""Plain fp64 CPU oracle for paged MLA decode, segment partials, the segment
merge, the sparse index conversion and the sparse front end (list lengths,
fixed-width index fit).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run anything in this package.
It shares no code, header, table or helper with the CUDA library, and it
imports nothing from it.

Everything is computed in float64 from the stored bits (bf16 bit patterns or
OCP e4m3fn codes times a per-tensor scale). The decode is the unsplit
definition ``softmax(scale * q . K^T) . V`` over the keys a row may see; the
split-K segments and their merge are written out separately, step by step, so
the tests can hold each one against the unsplit definition.

Sources (vLLM pages on the ROCm AITER MLA backend):
  * "vllm.v1.attention.ops.rocm_aiter_mla_merge" -- module docstring and
    ``merge_mla_segments_triton``: the segment partition
    ``tiles_per_segment = cdiv(seq_len, NUM_SEGMENTS * TILE_SIZE)``, base-2
    partials, the natural-log LSE and the output shapes.
  * "vllm.v1.attention.backends.mla.rocm_aiter_mla_sparse" --
    ``ROCMAiterMLASparseImpl.__init__`` and ``_forward_mla`` (sinks: fp32
    ``[H]``; rows with no keys give zero output; the sink enters the
    denominator only), ``triton_convert_req_index_to_global_index`` (the
    index formula and its -1 rules).
  * "vllm/v1/attention/backends/mla/rocm_aiter_mla.py" (source listing) --
    ``_segmented_mla_page_size`` (tile rule), ``dcp_local_verify_row_lens``
    and the Gluon MTP comment in ``forward_mqa`` (row j of a qlen-token block
    sees positions ``[0, seq_len - qlen + j]``), and
    ``_forward_segmented_dcp_verify`` (the cache viewed as pages of 576-wide
    rows; the values are the first ``kv_lora_rank`` columns).

Every function here is pinned by tests/test_oracle.py against closed forms,
brute force and invariants; none is "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

HEAD_DIM = 576
KV_LORA_RANK = 512
LOG2E = 1.0 / math.log(2.0)
LN2 = math.log(2.0)


# ---------------------------------------------------------------------------
# storage decoding
# ---------------------------------------------------------------------------

def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64. A bf16 value is the upper half
    of the float32 with the same sign, exponent and leading mantissa bits."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def decode_e4m3fn(codes: np.ndarray) -> np.ndarray:
    """OCP FP8 E4M3 ("fn": finite, no infinities) codes -> float64.

    Written from the format definition: 1 sign bit, 4 exponent bits with
    bias 7, 3 mantissa bits. Exponent field 0 holds subnormals
    ``(-1)^s * 2^-6 * m/8``; otherwise ``(-1)^s * 2^(e-7) * (1 + m/8)``; the
    single pattern S.1111.111 is NaN, so the largest finite value is 448.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    sub = np.ldexp(m / 8.0, -6)
    val = sign * np.where(e == 0, sub, normal)
    return np.where((e == 15) & ((c & 0x7) == 7), np.nan, val)


def dequantize(storage: np.ndarray, dtype: str, scale: float = 1.0) -> np.ndarray:
    """Stored q or cache values -> float64 real values (value * per-tensor scale)."""
    if dtype == "bf16":
        return decode_bf16(storage) * float(scale)
    if dtype == "fp8":
        return decode_e4m3fn(storage) * float(scale)
    raise ValueError(f"unknown dtype {dtype!r}")


# ---------------------------------------------------------------------------
# page, tile and segment geometry
# ---------------------------------------------------------------------------

def tile_size_for_block(block_size: int) -> int:
    """Largest power of two that divides the block, capped at 128
    (``_segmented_mla_page_size`` in rocm_aiter_mla.py)."""
    if block_size <= 0:
        raise ValueError("block_size must be positive")
    return min(128, block_size & -block_size)


def segment_bounds(part_len: int, num_segments: int, tile_size: int):
    """The split-K partition of ``[0, part_len)``.

    ``tiles_per_segment = cdiv(part_len, num_segments * tile_size)``
    (rocm_aiter_mla_merge module docstring); segment ``s`` covers
    ``[s * tps * tile, min((s + 1) * tps * tile, part_len))`` and is empty when
    its start is at or past ``part_len``. Returns ``num_segments`` (start, end)
    pairs with ``end <= start`` for an empty segment.
    """
    span = num_segments * tile_size
    tps = -(-int(part_len) // span) if part_len > 0 else 0
    seg = tps * tile_size
    out = []
    for s in range(num_segments):
        a = s * seg
        b = min((s + 1) * seg, int(part_len))
        out.append((a, b))
    return out


def visible_len(seq_len: int, qlen: int, j: int) -> int:
    """Keys visible to row ``j`` of a ``qlen``-token causal block: positions
    ``[0, seq_len - qlen + j]`` inclusive (``dcp_local_verify_row_lens`` and
    the Gluon MTP bound ``seq_len - qlen + q_pos + 1``), clamped at zero."""
    return max(0, int(seq_len) - int(qlen) + int(j) + 1)


def dense_slots(block_table_row: np.ndarray, block_size: int, n: int) -> np.ndarray:
    """Global cache slots of logical positions ``[0, n)`` of one request:
    ``block_table[r, p // block_size] * block_size + p % block_size``."""
    p = np.arange(int(n), dtype=np.int64)
    return block_table_row[p // block_size].astype(np.int64) * block_size + p % block_size


def token_layout(num_reqs: int, qo_indptr):
    """(request, position j within the request, qlen) for every token."""
    if qo_indptr is None:
        return [(r, 0, 1) for r in range(num_reqs)]
    out = []
    for r in range(num_reqs):
        a, b = int(qo_indptr[r]), int(qo_indptr[r + 1])
        for j in range(b - a):
            out.append((r, j, b - a))
    return out


# ---------------------------------------------------------------------------
# attention over an explicit key list
# ---------------------------------------------------------------------------

def attend(q: np.ndarray, keys: np.ndarray, softmax_scale: float, sinks=None):
    """Softmax attention of ``q [H, 576]`` over ``keys [n, 576]`` (float64).

    ``s = scale * q . k`` over all 576 columns; ``m = max(max_p s_p, sink)``;
    ``Z = sum_p e^(s_p - m) + e^(sink - m)``; ``out = sum_p e^(s_p - m) v_p / Z``
    with ``v_p`` the first 512 columns of key ``p``; ``lse = m + ln Z``. The sink
    is a natural-log logit that adds mass to the denominator and no value.
    With no keys: ``out = 0`` and ``lse = -inf`` (or the sink). This equals
    the post-hoc fold in ``_forward_mla`` of the sparse impl page
    (``out * exp(lse - logaddexp(lse, sink))``, zero output for empty rows).
    """
    H = q.shape[0]
    sk = None if sinks is None else np.asarray(sinks, dtype=np.float64)
    if keys.shape[0] == 0:
        out = np.zeros((H, KV_LORA_RANK))
        lse = np.full(H, -np.inf) if sk is None else sk.copy()
        return out, lse
    s = float(softmax_scale) * (q @ keys.T)          # [H, n]
    m = s.max(axis=1)
    if sk is not None:
        m = np.maximum(m, sk)
    e = np.exp(s - m[:, None])
    z = e.sum(axis=1)
    if sk is not None:
        z = z + np.exp(sk - m)
    out = (e @ keys[:, :KV_LORA_RANK]) / z[:, None]
    lse = m + np.log(z)
    return out, lse


def _gather(cache: np.ndarray, kv_dtype: str, kv_scale: float, slots: np.ndarray):
    flat = cache.reshape(-1, HEAD_DIM)
    return dequantize(flat[np.asarray(slots, dtype=np.int64)], kv_dtype, kv_scale)


def _token_keys(t, lay, q_dtype, cache, kv_dtype, kv_scale, block_table, seq_lens,
                block_size, sparse_slots, sparse_indptr):
    """(keys of the token's partition in order, valid mask, visible count rule).

    Dense: the request's positions ``[0, seq_len)`` in logical order; a row
    sees the prefix given by ``visible_len``. Sparse: the token's slot list in
    order (global slots, -1 unused), one key per valid entry.
    """
    r, j, ql = lay[t]
    if sparse_slots is None:
        L = int(seq_lens[r])
        slots = dense_slots(block_table[r], block_size, L)
        vis = np.arange(L) < visible_len(L, ql, j)
        return slots, vis
    if sparse_indptr is None:
        lst = np.asarray(sparse_slots[t], dtype=np.int64)
    else:
        lst = np.asarray(sparse_slots[int(sparse_indptr[t]):int(sparse_indptr[t + 1])],
                         dtype=np.int64)
    return lst, lst >= 0


# ---------------------------------------------------------------------------
# the decode (unsplit definition)
# ---------------------------------------------------------------------------

def mla_decode(q, q_dtype, q_scale, cache, kv_dtype, kv_scale, block_table, seq_lens,
               softmax_scale, *, block_size=None, qo_indptr=None, sinks=None,
               sparse_slots=None, sparse_indptr=None, tokens=None):
    """Paged MLA decode, unsplit, in float64.

    Dense: token ``t`` = row ``j`` of request ``r`` sees logical positions
    ``[0, visible_len(seq_len_r, qlen_r, j))`` mapped through the block table.
    Sparse (``sparse_slots`` given): token ``t`` sees the global slots of its
    list that are >= 0; ``sparse_slots`` is ``[T, topk]`` or, with
    ``sparse_indptr [T + 1]``, one flat ragged list.
    ``tokens`` restricts the computation to a subset of token indices.
    Returns ``out [n_tokens, H, 512]`` and ``lse [n_tokens, H]`` (natural log).
    """
    q = np.asarray(q)
    T, H = q.shape[0], q.shape[1]
    bs = int(block_size if block_size is not None else cache.shape[1])
    lay = token_layout(len(seq_lens), qo_indptr) if sparse_slots is None else \
        [(None, 0, 1)] * T
    toks = range(T) if tokens is None else [int(t) for t in tokens]
    out = np.zeros((len(toks), H, KV_LORA_RANK))
    lse = np.zeros((len(toks), H))
    for i, t in enumerate(toks):
        qt = dequantize(q[t], q_dtype, q_scale)
        slots, vis = _token_keys(t, lay, q_dtype, cache, kv_dtype, kv_scale, block_table,
                                 seq_lens, bs, sparse_slots, sparse_indptr)
        keys = _gather(cache, kv_dtype, kv_scale, slots[vis])
        out[i], lse[i] = attend(qt, keys, softmax_scale, sinks)
    return out, lse


# ---------------------------------------------------------------------------
# split-K partials and their merge
# ---------------------------------------------------------------------------

def partition_lengths(seq_lens, qo_indptr=None, sparse_slots=None, sparse_indptr=None,
                      num_tokens=None):
    """Length that defines each token's partition: the request's ``seq_len``
    for dense rows (shared by all rows of a multi-token request), the
    length of the token's entry list for sparse rows."""
    if sparse_slots is not None:
        if sparse_indptr is not None:
            return np.diff(np.asarray(sparse_indptr, dtype=np.int64))
        return np.full(int(np.asarray(sparse_slots).shape[0]),
                       int(np.asarray(sparse_slots).shape[1]), dtype=np.int64)
    lay = token_layout(len(seq_lens), qo_indptr)
    return np.array([int(seq_lens[r]) for (r, _, _) in lay], dtype=np.int64)


def segment_partials(q, q_dtype, q_scale, cache, kv_dtype, kv_scale, block_table,
                     seq_lens, softmax_scale, num_segments, tile_size, *,
                     block_size=None, qo_indptr=None, sparse_slots=None,
                     sparse_indptr=None, tokens=None):
    """Per-segment base-2 partials of the split-K decode.

    For segment ``s`` of a token's partition and the keys of that segment the
    row may see: ``m2 = max_p s_p * log2(e)``, ``l = sum_p 2^(s_p log2 e - m2)``,
    ``o = sum_p 2^(s_p log2 e - m2) v_p / l`` (the output is normalised by its
    own expsum). A segment with no visible key gives ``(-inf, 0, 0)``.
    Returns ``segm_output [n, H, NS, 512]``, ``segm_max [n, H, NS]`` and
    ``segm_expsum [n, H, NS]`` (rocm_aiter_mla_merge, base-2 partials).
    """
    q = np.asarray(q)
    T, H = q.shape[0], q.shape[1]
    bs = int(block_size if block_size is not None else cache.shape[1])
    NS = int(num_segments)
    lay = token_layout(len(seq_lens), qo_indptr) if sparse_slots is None else \
        [(None, 0, 1)] * T
    toks = range(T) if tokens is None else [int(t) for t in tokens]
    so = np.zeros((len(toks), H, NS, KV_LORA_RANK))
    sm = np.full((len(toks), H, NS), -np.inf)
    se = np.zeros((len(toks), H, NS))
    for i, t in enumerate(toks):
        qt = dequantize(q[t], q_dtype, q_scale)
        slots, vis = _token_keys(t, lay, q_dtype, cache, kv_dtype, kv_scale, block_table,
                                 seq_lens, bs, sparse_slots, sparse_indptr)
        for s, (a, b) in enumerate(segment_bounds(len(slots), NS, tile_size)):
            if b <= a:
                continue
            sel = np.arange(a, b)[vis[a:b]]
            if sel.size == 0:
                continue
            keys = _gather(cache, kv_dtype, kv_scale, slots[sel])
            s2 = float(softmax_scale) * (qt @ keys.T) * LOG2E
            m2 = s2.max(axis=1)
            w = np.exp2(s2 - m2[:, None])
            l = w.sum(axis=1)
            so[i, :, s] = (w @ keys[:, :KV_LORA_RANK]) / l[:, None]
            sm[i, :, s] = m2
            se[i, :, s] = l
    return so, sm, se


def merge_segments(segm_output, segm_max, segm_expsum, part_lens, tile_size, sinks=None):
    """Merge base-2 segment partials into ``out`` and a natural-log ``lse``.

    A segment takes part when its start lies inside the token's partition
    (``segment_bounds`` from ``part_lens`` and ``tile_size``, the only extra
    inputs the merge wrapper takes) and its expsum is positive. With
    ``M = max(m2_s, sink * log2 e)`` and ``W = sum_s l_s 2^(m2_s - M)
    + 2^(sink log2 e - M)``: ``out = sum_s l_s 2^(m2_s - M) o_s / W`` and
    ``lse = ln 2 * (M + log2 W)`` (``LOGE2`` in the merge wrapper). No
    contributing segment and no sink gives ``out = 0``, ``lse = -inf``.
    """
    so = np.asarray(segm_output, dtype=np.float64)
    smx = np.asarray(segm_max, dtype=np.float64)
    sex = np.asarray(segm_expsum, dtype=np.float64)
    T, H, NS, DV = so.shape
    out = np.zeros((T, H, DV))
    lse = np.full((T, H), -np.inf)
    sk = None if sinks is None else np.asarray(sinks, dtype=np.float64) * LOG2E
    for t in range(T):
        live = [s for s, (a, b) in enumerate(segment_bounds(int(part_lens[t]), NS, tile_size))
                if a < int(part_lens[t])]
        for h in range(H):
            segs = [s for s in live if sex[t, h, s] > 0]
            cands = [smx[t, h, s] for s in segs]
            if sk is not None:
                cands.append(sk[h])
            if not cands:
                continue
            M = max(cands)
            W = 0.0
            acc = np.zeros(DV)
            for s in segs:
                w = sex[t, h, s] * 2.0 ** (smx[t, h, s] - M)
                W += w
                acc += w * so[t, h, s]
            if sk is not None:
                W += 2.0 ** (sk[h] - M)
            out[t, h] = acc / W
            lse[t, h] = LN2 * (M + math.log2(W))
    return out, lse


# ---------------------------------------------------------------------------
# sparse index conversion
# ---------------------------------------------------------------------------

def index_convert(req_id, block_table, token_indices, block_size, cu_seqlens=None,
                  out_init=None):
    """Per-request top-k positions -> global cache slots
    (``triton_convert_req_index_to_global_index``).

    ``out[t, i] = block_table[req_id[t], idx // BS] * BS + idx % BS`` with
    ``idx = token_indices[t, i]``; ``-1`` when ``idx`` is negative or when the
    block column ``idx // BS`` is not below the table's width. The page's
    out-of-bounds safety rule is read as covering the row index too: a
    request id outside the table also gives ``-1``. Block-table values
    themselves are not range-checked.

    Without ``cu_seqlens`` the result is ``[T, topk]``. With ``cu_seqlens
    [T + 1]`` the first ``cu[t + 1] - cu[t]`` converted entries of row ``t``
    are written to ``out[cu[t] + i]`` of the flat buffer ``out_init`` (a copy
    is returned; positions no row writes keep their value).
    """
    ti = np.asarray(token_indices, dtype=np.int64)
    bt = np.asarray(block_table, dtype=np.int64)
    req = np.asarray(req_id, dtype=np.int64)
    T, K = ti.shape
    cols = bt.shape[1]
    blk = np.where(ti >= 0, ti // block_size, 0)
    req_ok = (req >= 0) & (req < bt.shape[0])
    ok = (ti >= 0) & (blk < cols) & req_ok[:, None]
    rows = np.broadcast_to(np.where(req_ok, req, 0)[:, None], ti.shape)
    base = bt[rows, np.where(ok, blk, 0)]
    conv = np.where(ok, base * block_size + np.where(ti >= 0, ti % block_size, 0), -1)
    conv = conv.astype(np.int64)
    if cu_seqlens is None:
        return conv
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    out = np.array(out_init, dtype=np.int64, copy=True)
    for t in range(T):
        n = int(cu[t + 1] - cu[t])
        out[cu[t]:cu[t] + n] = conv[t, :n]
    return out


# ---------------------------------------------------------------------------
# sparse front end: per-token list lengths and the fixed-width index fit
# ---------------------------------------------------------------------------

def sparse_seqlen(query_start_loc, seq_lens, topk):
    """Per-token length of the sparse slot list and its exclusive prefix sum
    (the sparse page's metadata builder: ``generate_sparse_seqlen_triton``
    then ``torch.cumsum`` into ``paged_kv_indptr``).

    Reading (the kernel body is not on the page): token ``j`` of request
    ``r`` (``qlen = qsl[r + 1] - qsl[r]`` tokens) sees the causal prefix
    ``[0, seq_len - qlen + j]``, as the dense page's
    ``dcp_local_verify_row_lens`` has it, and can select at most ``topk`` of
    those positions: ``len = clamp(seq_len - qlen + j + 1, 0, topk)``.
    Returns ``(lens [T], indptr [T + 1])`` as int64.
    """
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    sl = np.asarray(seq_lens, dtype=np.int64)
    T = int(qsl[-1])
    lens = np.zeros(T, dtype=np.int64)
    for r in range(len(sl)):
        qlen = int(qsl[r + 1] - qsl[r])
        for j in range(qlen):
            lens[qsl[r] + j] = min(max(int(sl[r]) - qlen + j + 1, 0), int(topk))
    indptr = np.zeros(T + 1, dtype=np.int64)
    indptr[1:] = np.cumsum(lens)
    return lens, indptr


def fit_kpool_indices(token_indices, topk):
    """Fit ``[T, W]`` top-k rows (``W >= topk``) to AITER's fixed width
    ``topk`` (``fit_kpool_indices_to_aiter`` on the sparse page, which does
    so while keeping the kpool tail's live entries).

    Reading (the kernel body is not on the page): columns ``[0, topk)`` are
    the selected positions, columns ``[topk, W)`` the kpool tail; a tail
    entry is live when it is ``>= 0``. With ``n`` the number of live tail
    entries (at most ``topk`` of them, the first ones, are kept), the output
    row is the first ``topk - n`` selected entries followed by the ``n``
    live tail entries in their order. Nothing is de-duplicated. ``W ==
    topk`` returns the rows unchanged; ``W < topk`` is an error.
    """
    ti = np.asarray(token_indices, dtype=np.int64)
    T, W = ti.shape
    if W < topk:
        raise ValueError("token_indices width must be at least topk")
    out = np.empty((T, topk), dtype=np.int64)
    for t in range(T):
        live = [int(v) for v in ti[t, topk:] if v >= 0][:topk]
        n = len(live)
        out[t, :topk - n] = ti[t, :topk - n]
        out[t, topk - n:] = live
    return out


# ---------------------------------------------------------------------------
# merge of per-shard (out, lse) pairs (decode context parallelism)
# ---------------------------------------------------------------------------

def merge_lse_shards(outs, lses, sinks=None):
    """Combine the natural-log ``(out, lse)`` of W key shards of the same rows.

    The merge page says its natural-log LSE is what the cross-rank DCP merge
    consumes; with shard ``w`` holding ``out_w = sum_p e^{s_p} v_p / Z_w`` and
    ``lse_w = ln Z_w`` over its own keys: ``M = max_w lse_w``,
    ``out = sum_w e^{lse_w - M} out_w / sum_w e^{lse_w - M}``,
    ``lse = M + ln sum_w e^{lse_w - M}``. Shards with ``lse = -inf`` (no keys)
    take no part. A sink, if given, is folded once here (it adds
    ``e^{sink - M}`` to the denominator), so the shards must be decoded
    without it. ``outs [W, T, H, Dv]``, ``lses [W, T, H]``.
    """
    outs = np.asarray(outs, dtype=np.float64)
    lses = np.asarray(lses, dtype=np.float64)
    W, T, H, DV = outs.shape
    out = np.zeros((T, H, DV))
    lse = np.full((T, H), -np.inf)
    sk = None if sinks is None else np.asarray(sinks, dtype=np.float64)
    for t in range(T):
        for h in range(H):
            live = [w for w in range(W) if lses[w, t, h] > -np.inf]
            cands = [lses[w, t, h] for w in live]
            if sk is not None:
                cands.append(sk[h])
            if not cands:
                continue
            M = max(cands)
            Z = 0.0
            acc = np.zeros(DV)
            for w in live:
                e = math.exp(lses[w, t, h] - M)
                Z += e
                acc += e * outs[w, t, h]
            if sk is not None:
                Z += math.exp(sk[h] - M)
            out[t, h] = acc / Z
            lse[t, h] = M + math.log(Z)
    return out, lse


def round_robin_positions(seq_len: int, qlen: int, j: int, world: int, rank: int):
    """Logical positions a rank holds of row ``j``'s visible keys when token
    ``p`` lives on rank ``p % world`` (decode context parallelism with an
    interleave of one): ``{p < visible_len(seq_len, qlen, j) : p % world == rank}``
    (``dcp_local_verify_row_lens`` counts exactly these)."""
    n = visible_len(seq_len, qlen, j)
    return np.arange(rank, n, world, dtype=np.int64)


# ---------------------------------------------------------------------------
# q pre-step: concat of the latent and rope parts, optional e4m3 quantisation
# ---------------------------------------------------------------------------

def _e4m3_grid():
    codes = np.arange(0x00, 0x7F, dtype=np.uint8)          # +0 .. +448, NaN excluded
    vals = decode_e4m3fn(codes)
    order = np.argsort(vals, kind="stable")
    return vals[order], codes[order]


def encode_e4m3fn(x):
    """Real values -> e4m3fn codes: the nearest representable value, ties to
    the even code (mantissa LSB 0), magnitudes above 448 saturated to 448
    (static per-tensor fp8 quantisation clamps before casting), the sign kept
    (a negative value that rounds to zero gives negative zero, 0x80). NaN is
    not an input here."""
    vals, codes = _e4m3_grid()
    a = np.minimum(np.abs(np.asarray(x, dtype=np.float64)), vals[-1])
    hi = np.clip(np.searchsorted(vals, a, side="left"), 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    dlo = a - vals[lo]
    dhi = vals[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ((codes[hi] & 1) == 0))
    c = np.where(pick_hi, codes[hi], codes[lo]).astype(np.uint8)
    # the sign is kept, also for values that round to zero (negative zero 0x80)
    neg = np.signbit(np.asarray(x, dtype=np.float64))
    return np.where(neg, c | 0x80, c).astype(np.uint8)


def concat_quant_q(ql_nope, q_pe, q_scale=None):
    """``q = ql_nope || q_pe`` along the last dim (forward_mqa's concat of the
    absorbed latent query and its rope part). With ``q_scale`` the result is
    quantised to e4m3fn codes of ``q / q_scale``; without it the float values
    are returned."""
    q = np.concatenate([np.asarray(ql_nope, dtype=np.float64),
                        np.asarray(q_pe, dtype=np.float64)], axis=-1)
    if q_scale is None:
        return q
    # q / q_scale is formed in float32: the static per-tensor quantisation of
    # forward_mqa (scaled_fp8_quant with the layer's float32 q scale) divides
    # in the scale's type before rounding to e4m3, and a value on the edge
    # between two codes must round the same way here.
    scaled = (q.astype(np.float32) / np.float32(q_scale)).astype(np.float64)
    return encode_e4m3fn(scaled)
