"""Pins for the fp64 oracle: closed forms, brute force, invariants and the
worked values the pages fix. CPU only.

Each pin is chosen so that a plausible slip in the oracle (a dropped rope
term, the value columns taken from the wrong end of the row, a missing
scale, a wrong sign in the rescale, a transposed operand, an off-by-one in
the causal bound or the partition) fails at least one test here.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from paged_mla_decode_06_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _bf16(x):
    return I.float32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _single(q, cache, bt, seq, scale, **kw):
    return O.mla_decode(q, "bf16", 1.0, cache, "bf16", 1.0, bt, seq, scale, **kw)


# ---------------------------------------------------------------- decoders

def test_e4m3_decoder_matches_torch_on_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    got = O.decode_e4m3fn(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok].astype(np.float64), got[ok])
    assert np.nanmax(got) == 448.0 and np.nanmin(got) == -448.0
    assert got[1] == 2.0 ** -9  # smallest subnormal


def test_bf16_decoder_matches_torch_on_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    got = O.decode_bf16(bits)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok].astype(np.float64), got[ok])


# ---------------------------------------------------------------- geometry

def test_tile_rule_golden():
    for bs, tile in _golden_rows("tile_rule.txt"):
        assert O.tile_size_for_block(int(bs)) == int(tile)


def test_segment_partition_golden():
    for row in _golden_rows("segment_partition.txt"):
        L, ns, tile = int(row[0]), int(row[1]), int(row[2])
        want = []
        for tok in row[3:]:
            if tok == "-":
                want.append(None)
            else:
                a, b = tok.split("-")
                want.append((int(a), int(b)))
        got = [(a, b) if b > a else None for (a, b) in O.segment_bounds(L, ns, tile)]
        assert got == want, (row, got)


@pytest.mark.parametrize("L", [0, 1, 15, 16, 17, 63, 64, 65, 129, 1000, 8192, 16384])
@pytest.mark.parametrize("ns,tile", [(1, 16), (2, 64), (3, 16), (4, 64), (7, 1), (8, 128)])
def test_segment_partition_tiles_the_range(L, ns, tile):
    segs = O.segment_bounds(L, ns, tile)
    assert len(segs) == ns
    covered = []
    for a, b in segs:
        assert a % tile == 0
        if b > a:
            covered.extend(range(a, b))
    assert covered == list(range(L))


def test_causal_bound_includes_own_token():
    # a 3-token verify block over seq_len 10: the last row sees all 10 keys,
    # the first sees 8 (its own position 7 included).
    assert [O.visible_len(10, 3, j) for j in range(3)] == [8, 9, 10]
    assert O.visible_len(1, 3, 0) == 0


def test_fetch_size_golden():
    (b, n, row, total), = _golden_rows("fetch_size.txt")
    assert int(b) * int(n) * int(row) == int(total)
    assert O.HEAD_DIM == int(row)  # one e4m3 byte per column of a 576-wide row


# ---------------------------------------------------------------- closed forms

def _dense_case(seed, seq_lens, H=4, bs=16, std=1.0, qlens=None, sinks=False):
    return I.build_dense(seed, seq_lens=seq_lens, num_heads=H, block_size=bs,
                         q_std=std, kv_std=std, qlens=qlens, with_sinks=sinks)


def _run(w, **kw):
    return O.mla_decode(w.q, w.q_dtype, w.q_scale, w.cache, w.kv_dtype, w.kv_scale,
                        w.block_table, w.seq_lens, w.softmax_scale,
                        qo_indptr=w.qo_indptr, sinks=w.sinks, **kw)


def test_single_key_returns_its_value_row():
    w = _dense_case(10, [1], H=3)
    out, lse = _run(w)
    row = O.decode_bf16(w.cache[w.block_table[0, 0], 0])
    q = O.decode_bf16(w.q[0])
    assert np.array_equal(out[0], np.broadcast_to(row[:512], (3, 512)))
    s0 = w.softmax_scale * (q @ row)
    np.testing.assert_allclose(lse[0], s0, rtol=0, atol=1e-12)


def test_uniform_scores_give_mean_value_and_log_count():
    # q_nope = 0 and identical k_pe in every key: every score is the same s,
    # so out = mean of the value rows and lse = s + ln L.
    w = _dense_case(11, [23], H=2)
    q = O.decode_bf16(w.q).copy()
    q[..., :512] = 0.0
    w.q = _bf16(q)
    pe = _bf16(np.linspace(-1, 1, 64))
    flat = w.cache.reshape(-1, 576)
    slots = O.dense_slots(w.block_table[0], w.block_size, 23)
    flat[slots, 512:] = pe
    out, lse = _run(w)
    V = O.decode_bf16(flat[slots])[:, :512]
    np.testing.assert_allclose(out[0], np.broadcast_to(V.mean(0), (2, 512)), atol=1e-12)
    s = w.softmax_scale * (O.decode_bf16(w.q[0]) @ O.decode_bf16(flat[slots[0]]))
    np.testing.assert_allclose(lse[0], s + math.log(23), atol=1e-12)


def test_zero_query_gives_mean_value_and_log_count():
    w = _dense_case(12, [40], H=2)
    w.q[:] = 0
    out, lse = _run(w)
    slots = O.dense_slots(w.block_table[0], w.block_size, 40)
    V = O.decode_bf16(w.cache.reshape(-1, 576)[slots])[:, :512]
    np.testing.assert_allclose(out[0, 1], V.mean(0), atol=1e-12)
    np.testing.assert_allclose(lse[0], math.log(40), atol=1e-12)


def test_brute_force_python_loops():
    w = _dense_case(13, [5, 3], H=3, bs=2)
    out, lse = _run(w)
    flat = w.cache.reshape(-1, 576)
    for r in range(2):
        L = int(w.seq_lens[r])
        rows = []
        for p in range(L):
            slot = int(w.block_table[r, p // 2]) * 2 + p % 2
            rows.append([float(x) for x in O.decode_bf16(flat[slot])])
        for h in range(3):
            q = [float(x) for x in O.decode_bf16(w.q[r, h])]
            sc = [w.softmax_scale * sum(q[d] * k[d] for d in range(576)) for k in rows]
            m = max(sc)
            e = [math.exp(s - m) for s in sc]
            z = sum(e)
            o = [sum(e[p] * rows[p][c] for p in range(L)) / z for c in range(512)]
            assert abs(lse[r, h] - (m + math.log(z))) < 1e-10
            assert np.max(np.abs(out[r, h] - np.array(o))) < 1e-10


def test_page_permutation_invariance():
    w = _dense_case(14, [50, 17, 64], H=2, bs=16)
    out, lse = _run(w)
    rng = np.random.default_rng(0)
    nb = w.cache.shape[0]
    perm = rng.permutation(nb)          # new position of old block b is perm[b]
    cache2 = np.empty_like(w.cache)
    cache2[perm] = w.cache
    w.cache = cache2
    w.block_table = perm[w.block_table].astype(np.int32)
    out2, lse2 = _run(w)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_heads_are_independent():
    w = _dense_case(15, [33], H=4)
    out, lse = _run(w)
    q = O.decode_bf16(w.q).copy()
    q[0, 2] *= -3.0
    w.q = _bf16(q)
    out2, lse2 = _run(w)
    keep = [0, 1, 3]
    assert np.array_equal(out[:, keep], out2[:, keep])
    assert np.array_equal(lse[:, keep], lse2[:, keep])
    assert not np.allclose(out[:, 2], out2[:, 2])


def test_causal_rows_equal_single_token_decode():
    w = _dense_case(16, [9, 30], H=2, bs=4, qlens=[3, 2])
    out, lse = _run(w)
    t = 0
    for r, ql in enumerate([3, 2]):
        for j in range(ql):
            n = int(w.seq_lens[r]) - ql + j + 1
            o1, l1 = _single(w.q[t:t + 1], w.cache, w.block_table[r:r + 1],
                             np.array([n], np.int32), w.softmax_scale)
            assert np.array_equal(out[t], o1[0]) and np.array_equal(lse[t], l1[0])
            t += 1


def test_sinks_match_the_post_hoc_fold():
    # The sparse impl page folds a sink after the kernel:
    # lse' = logaddexp(lse, sink); out' = out * exp(lse - lse'); rows
    # without keys give out' = 0 and lse' = sink.
    w = _dense_case(17, [12, 0, 40], H=3, sinks=True)
    out, lse = _run(w)
    base_o, base_l = O.mla_decode(w.q, "bf16", 1.0, w.cache, "bf16", 1.0, w.block_table,
                                  w.seq_lens, w.softmax_scale)
    sink = w.sinks.astype(np.float64)
    has = (w.seq_lens > 0)[:, None]
    l0 = np.where(has, base_l, -np.inf)
    l1 = np.logaddexp(l0, sink[None, :])
    o1 = np.where(has[..., None], base_o * np.exp(l0 - l1)[..., None], 0.0)
    np.testing.assert_allclose(lse, l1, atol=1e-12)
    np.testing.assert_allclose(out, o1, atol=1e-12)
    assert np.all(out[1] == 0) and np.array_equal(lse[1], sink)


def test_minus_inf_sink_equals_no_sink():
    w = _dense_case(18, [21], H=2, sinks=True)
    w.sinks[:] = -np.inf
    out, lse = _run(w)
    w.sinks = None
    out2, lse2 = _run(w)
    np.testing.assert_allclose(out, out2, atol=1e-14)
    np.testing.assert_allclose(lse, lse2, atol=1e-14)


def test_empty_row_without_sink():
    w = _dense_case(19, [0, 5], H=2)
    out, lse = _run(w)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))


def test_fp8_inputs_compare_after_dequantisation():
    # fp8 decode equals attention over the values torch's own e4m3 cast gives
    # back, times the per-tensor scales.
    w = I.build_dense(20, seq_lens=[19, 33], num_heads=2, block_size=16, dtype="fp8")
    out, lse = _run(w)
    flat = torch.from_numpy(w.cache.reshape(-1, 576).copy()).view(torch.float8_e4m3fn)
    kv = flat.double().numpy() * w.kv_scale
    qv = torch.from_numpy(w.q.copy()).view(torch.float8_e4m3fn).double().numpy() * w.q_scale
    for r in range(2):
        slots = O.dense_slots(w.block_table[r], 16, int(w.seq_lens[r]))
        o, l = O.attend(qv[r], kv[slots], w.softmax_scale)
        np.testing.assert_allclose(out[r], o, atol=1e-12)
        np.testing.assert_allclose(lse[r], l, atol=1e-12)


# ---------------------------------------------------------------- split-K + merge

@pytest.mark.parametrize("ns", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("tile", [1, 16, 64])
def test_merge_of_any_split_equals_unsplit(ns, tile):
    w = _dense_case(21 + ns, [1, 37, 130, 0, 64], H=2, bs=16, sinks=(ns % 2 == 0))
    out, lse = _run(w)
    so, sm, se = O.segment_partials(w.q, "bf16", 1.0, w.cache, "bf16", 1.0, w.block_table,
                                    w.seq_lens, w.softmax_scale, ns, tile)
    pl = O.partition_lengths(w.seq_lens)
    mo, ml = O.merge_segments(so, sm, se, pl, tile, sinks=w.sinks)
    np.testing.assert_allclose(mo, out, atol=1e-12)
    np.testing.assert_allclose(ml, lse, atol=1e-12)


def test_merge_causal_rows_share_the_request_partition():
    w = _dense_case(30, [40, 7], H=2, bs=8, qlens=[4, 3], sinks=True)
    out, lse = _run(w)
    so, sm, se = O.segment_partials(w.q, "bf16", 1.0, w.cache, "bf16", 1.0, w.block_table,
                                    w.seq_lens, w.softmax_scale, 4, 8, qo_indptr=w.qo_indptr)
    pl = O.partition_lengths(w.seq_lens, w.qo_indptr)
    assert list(pl) == [40] * 4 + [7] * 3
    mo, ml = O.merge_segments(so, sm, se, pl, 8, sinks=w.sinks)
    np.testing.assert_allclose(mo, out, atol=1e-12)
    np.testing.assert_allclose(ml, lse, atol=1e-12)


def test_merge_single_segment_is_identity():
    rng = np.random.default_rng(3)
    so = rng.standard_normal((3, 2, 1, 512))
    sm = rng.standard_normal((3, 2, 1)) * 4
    se = rng.uniform(0.5, 30, (3, 2, 1))
    out, lse = O.merge_segments(so, sm, se, np.array([5, 9, 100]), 16)
    np.testing.assert_allclose(out, so[:, :, 0], atol=1e-14)
    np.testing.assert_allclose(lse, math.log(2) * sm[..., 0] + np.log(se[..., 0]), atol=1e-12)


def test_merge_ignores_segments_outside_the_partition():
    # seq 37 with 4 segments of tile 16: [0,16) [16,32) [32,37) and an empty
    # fourth segment, whose partial slot may hold anything.
    rng = np.random.default_rng(4)
    so = rng.standard_normal((1, 1, 4, 512))
    sm = rng.standard_normal((1, 1, 4))
    se = rng.uniform(1, 2, (1, 1, 4))
    so[0, 0, 3] = np.nan
    sm[0, 0, 3] = np.nan
    se[0, 0, 3] = np.nan
    out, lse = O.merge_segments(so, sm, se, np.array([37]), 16)
    w = se[0, 0, :3] * 2.0 ** (sm[0, 0, :3] - sm[0, 0, :3].max())
    np.testing.assert_allclose(out[0, 0], (w[:, None] * so[0, 0, :3]).sum(0) / w.sum(),
                               atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], math.log(2) * sm[0, 0, :3].max() + math.log(w.sum()),
                               atol=1e-12)


def test_merge_of_all_empty_rows():
    so = np.zeros((2, 3, 4, 512))
    sm = np.full((2, 3, 4), -np.inf)
    se = np.zeros((2, 3, 4))
    out, lse = O.merge_segments(so, sm, se, np.array([0, 0]), 16)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    sinks = np.array([0.5, -1.0, 2.0])
    out, lse = O.merge_segments(so, sm, se, np.array([0, 0]), 16, sinks=sinks)
    assert np.all(out == 0)
    np.testing.assert_allclose(lse, np.broadcast_to(sinks, (2, 3)), atol=1e-14)


def test_partials_of_fully_masked_causal_segment():
    # row 0 of a 4-token block over seq 8 sees 5 keys; with 2 segments of
    # tile 4 the second segment [4, 8) holds one visible key for row 0.
    w = _dense_case(31, [8], H=1, bs=4, qlens=[4])
    so, sm, se = O.segment_partials(w.q, "bf16", 1.0, w.cache, "bf16", 1.0, w.block_table,
                                    w.seq_lens, w.softmax_scale, 4, 2, qo_indptr=w.qo_indptr)
    # tile 2, 4 segments: [0,2) [2,4) [4,6) [6,8); row 0 sees [0,5)
    assert se[0, 0, 3] == 0 and np.isneginf(sm[0, 0, 3])
    assert se[0, 0, 2] == 1.0   # exactly one visible key: weight 2^0


# ---------------------------------------------------------------- sparse

def _brute_convert(req, bt, ti, bs):
    T, K = ti.shape
    out = [[0] * K for _ in range(T)]
    for t in range(T):
        for i in range(K):
            idx = int(ti[t, i])
            if idx < 0 or idx // bs >= bt.shape[1] or not 0 <= int(req[t]) < bt.shape[0]:
                out[t][i] = -1
            else:
                out[t][i] = int(bt[int(req[t]), idx // bs]) * bs + idx % bs
    return np.array(out, dtype=np.int64)


def test_index_convert_brute_force_and_edges():
    rng = np.random.default_rng(7)
    bt = rng.integers(0, 1000, size=(3, 5)).astype(np.int32)
    req = np.array([0, 2, 1, 2], dtype=np.int32)
    ti = rng.integers(-3, 6 * 16, size=(4, 256)).astype(np.int32)
    ti[0, 0] = -1
    ti[0, 1] = 5 * 16 - 1      # last valid column, last offset
    ti[0, 2] = 5 * 16          # first out-of-bounds column
    ti[1, :4] = [0, 15, 16, -7]
    got = O.index_convert(req, bt, ti, 16)
    want = _brute_convert(req, bt, ti, 16)
    assert np.array_equal(got, want)
    assert got[0, 0] == -1 and got[0, 2] == -1 and got[1, 3] == -1
    assert got[0, 1] == int(bt[0, 4]) * 16 + 15


def test_index_convert_request_outside_table():
    bt = np.arange(8, dtype=np.int32).reshape(2, 4)
    ti = np.array([[0, 17, -1, 63], [5, 6, 7, 8]], dtype=np.int32)
    got = O.index_convert(np.array([2, -1], dtype=np.int32), bt, ti, 16)
    assert np.all(got == -1)
    got = O.index_convert(np.array([1, 0], dtype=np.int32), bt, ti, 16)
    assert got.tolist() == [[4 * 16, 5 * 16 + 1, -1, 7 * 16 + 15], [5, 6, 7, 8]]


def test_index_convert_ragged_output():
    rng = np.random.default_rng(8)
    bt = rng.integers(0, 50, size=(2, 4)).astype(np.int32)
    req = np.array([0, 1, 1], dtype=np.int32)
    ti = rng.integers(-1, 64, size=(3, 128)).astype(np.int32)
    cu = np.array([0, 100, 100, 228], dtype=np.int32)
    init = np.full(3 * 128, 12345, dtype=np.int64)
    got = O.index_convert(req, bt, ti, 16, cu_seqlens=cu, out_init=init)
    dense = _brute_convert(req, bt, ti, 16)
    assert np.array_equal(got[:100], dense[0, :100])
    assert np.array_equal(got[100:228], dense[2, :128])
    assert np.all(got[228:] == 12345)


def test_sparse_over_dense_slots_equals_dense():
    w = _dense_case(40, [45, 3], H=2, bs=16)
    out, lse = _run(w)
    T = 2
    K = 64
    slots = np.full((T, K), -1, dtype=np.int64)
    for r in range(2):
        s = O.dense_slots(w.block_table[r], 16, int(w.seq_lens[r]))
        slots[r, :len(s)] = s
    so, sl = O.mla_decode(w.q, "bf16", 1.0, w.cache, "bf16", 1.0, None, None,
                          w.softmax_scale, sparse_slots=slots)
    assert np.array_equal(so, out) and np.array_equal(sl, lse)


def test_sparse_slot_order_does_not_matter():
    w = I.sparse_topk(seed=41, num_reqs=2, tokens_per_req=2, num_heads=2,
                      cache_tokens=300, topk=128, interspersed_rows=1)
    slots = O.index_convert(w.req_id_per_token, w.block_table, w.topk_indices, w.block_size)
    out, lse = O.mla_decode(w.q, "bf16", 1.0, w.cache, "bf16", 1.0, None, None,
                            w.softmax_scale, sparse_slots=slots)
    rng = np.random.default_rng(1)
    perm = rng.permutation(slots.shape[1])
    out2, lse2 = O.mla_decode(w.q, "bf16", 1.0, w.cache, "bf16", 1.0, None, None,
                              w.softmax_scale, sparse_slots=slots[:, perm])
    np.testing.assert_allclose(out, out2, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, atol=1e-12)
    assert np.isfinite(out).all()


def test_sparse_ragged_list_equals_padded_list():
    w = I.sparse_topk(seed=42, num_reqs=1, tokens_per_req=3, num_heads=2,
                      cache_tokens=200, topk=128, max_pad=0)
    slots = O.index_convert(w.req_id_per_token, w.block_table, w.topk_indices, w.block_size)
    lens = [128, 5, 60]
    cu = np.concatenate([[0], np.cumsum(lens)])
    flat = np.concatenate([slots[t, :lens[t]] for t in range(3)])
    padded = np.full_like(slots, -1)
    for t in range(3):
        padded[t, :lens[t]] = slots[t, :lens[t]]
    a = O.mla_decode(w.q, "bf16", 1.0, w.cache, "bf16", 1.0, None, None, w.softmax_scale,
                     sparse_slots=flat, sparse_indptr=cu)
    b = O.mla_decode(w.q, "bf16", 1.0, w.cache, "bf16", 1.0, None, None, w.softmax_scale,
                     sparse_slots=padded)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ---------------------------------------------------------------- shard (DCP) merge

@pytest.mark.parametrize("world", [1, 2, 3, 4])
def test_round_robin_shards_merge_to_the_unsplit_decode(world):
    w = _dense_case(50 + world, [1, 9, 40, 130], H=3, bs=16, qlens=[1, 3, 2, 1], sinks=True)
    out, lse = _run(w)
    lay = O.token_layout(len(w.seq_lens), w.qo_indptr)
    T = w.num_tokens
    outs = np.zeros((world, T, 3, 512))
    lses = np.zeros((world, T, 3))
    for rank in range(world):
        K = 256
        slots = np.full((T, K), -1, dtype=np.int64)
        for t, (r, j, ql) in enumerate(lay):
            pos = O.round_robin_positions(int(w.seq_lens[r]), ql, j, world, rank)
            slots[t, :len(pos)] = O.dense_slots(w.block_table[r], w.block_size,
                                                int(w.seq_lens[r]))[pos]
        outs[rank], lses[rank] = O.mla_decode(w.q, "bf16", 1.0, w.cache, "bf16", 1.0, None,
                                              None, w.softmax_scale, sparse_slots=slots)
    mo, ml = O.merge_lse_shards(outs, lses, sinks=w.sinks)
    np.testing.assert_allclose(mo, out, atol=1e-12)
    np.testing.assert_allclose(ml, lse, atol=1e-12)


def test_shard_merge_closed_forms():
    rng = np.random.default_rng(5)
    o = rng.standard_normal((1, 2, 3, 512))
    l = rng.standard_normal((1, 2, 3))
    mo, ml = O.merge_lse_shards(o, l)        # one shard: identity
    np.testing.assert_allclose(mo, o[0], atol=1e-14)
    np.testing.assert_allclose(ml, l[0], atol=1e-14)
    o2 = np.stack([o[0], o[0]])
    l2 = np.stack([l[0], l[0]])
    mo, ml = O.merge_lse_shards(o2, l2)      # two equal shards: same out, lse + ln 2
    np.testing.assert_allclose(mo, o[0], atol=1e-14)
    np.testing.assert_allclose(ml, l[0] + math.log(2), atol=1e-12)
    l3 = np.stack([l[0], np.full_like(l[0], -np.inf)])
    mo, ml = O.merge_lse_shards(np.stack([o[0], np.full_like(o[0], np.nan)]), l3)
    np.testing.assert_allclose(mo, o[0], atol=1e-14)   # an empty shard is ignored
    mo, ml = O.merge_lse_shards(np.zeros((2, 1, 1, 512)), np.full((2, 1, 1), -np.inf))
    assert np.all(mo == 0) and np.isneginf(ml).all()


# ---------------------------------------------------------------- q pre-step

def test_e4m3_encoder_matches_torch_rounding():
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.standard_normal(20000) * 40, rng.uniform(-448, 448, 20000),
                        rng.standard_normal(5000) * 1e-2, [0.0, -0.0, 448.0, -448.0]])
    x = x.astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.encode_e4m3fn(x)
    assert np.array_equal(got, ref)        # signed zeros included


def test_e4m3_encoder_ties_saturation_and_round_trip():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = O.decode_e4m3fn(codes)
    back = O.encode_e4m3fn(vals)
    assert np.array_equal(O.decode_e4m3fn(back), vals)      # every value is its own code
    assert O.encode_e4m3fn(np.array([1000.0, -1e9]))[0] == 0x7E  # saturate to +448
    assert O.encode_e4m3fn(np.array([-1e9]))[0] == 0xFE
    # 1 + 1/16 lies halfway between 1 (code 0x38, even) and 1.125 (0x39): ties to even
    assert O.encode_e4m3fn(np.array([1.0625]))[0] == 0x38
    assert O.encode_e4m3fn(np.array([1.1875]))[0] == 0x3A   # between 1.125 (odd) and 1.25
    assert list(O.encode_e4m3fn(np.array([0.0, -0.0, -1e-6]))) == [0x00, 0x80, 0x80]


def test_concat_quant_q():
    rng = np.random.default_rng(12)
    a = rng.standard_normal((2, 3, 512))
    b = rng.standard_normal((2, 3, 64))
    q = O.concat_quant_q(a, b)
    assert q.shape == (2, 3, 576) and np.array_equal(q[..., :512], a) and np.array_equal(q[..., 512:], b)
    codes = O.concat_quant_q(a, b, q_scale=0.05)
    np.testing.assert_allclose(O.decode_e4m3fn(codes) * 0.05, q, rtol=0.07, atol=0.05 * 2 ** -9)


# ---------------------------------------------------------------- sparse front end

def test_sparse_seqlen_golden():
    rows = _golden_rows("sparse_seqlen.txt")
    want_lens = [int(v) for v in rows[0][1:]]
    want_indptr = [int(v) for v in rows[1][1:]]
    seq = [5, 300, 2, 0, 130]
    qlens = [1, 3, 2, 1, 4]
    qsl = np.concatenate([[0], np.cumsum(qlens)])
    lens, indptr = O.sparse_seqlen(qsl, seq, 128)
    assert lens.tolist() == want_lens
    assert indptr.tolist() == want_indptr


def test_sparse_seqlen_matches_dense_visible_rows():
    # the same causal bound as the dense multi-token rows, capped at topk
    rng = np.random.default_rng(21)
    seq = rng.integers(0, 700, size=40)
    qlens = rng.integers(1, 5, size=40)
    qsl = np.concatenate([[0], np.cumsum(qlens)])
    for topk in (128, 512, 2048):
        lens, indptr = O.sparse_seqlen(qsl, seq, topk)
        assert indptr[0] == 0 and np.array_equal(np.diff(indptr), lens)
        t = 0
        for r in range(40):
            for j in range(int(qlens[r])):
                assert lens[t] == min(O.visible_len(int(seq[r]), int(qlens[r]), j), topk)
                t += 1
        # within a request consecutive tokens see one more position each
        for r in range(40):
            seg = lens[qsl[r]:qsl[r + 1]]
            assert np.all(np.diff(seg) <= 1) and np.all(np.diff(seg) >= 0)
            assert np.all((seg >= 0) & (seg <= topk))


def test_fit_kpool_golden():
    rows = [" ".join(r) for r in _golden_rows("fit_kpool.txt")]
    for line in rows:
        a, b = line.split("|")
        row = np.array([int(v) for v in a.split()])
        want = [int(v) for v in b.split()]
        got = O.fit_kpool_indices(row[None, :], 4)
        assert got[0].tolist() == want, line


def test_fit_kpool_invariants_and_edges():
    rng = np.random.default_rng(22)
    T, topk, W = 50, 128, 192
    ti = rng.integers(0, 10000, size=(T, W))
    ti[rng.random((T, W)) < 0.3] = -1
    out = O.fit_kpool_indices(ti, topk)
    assert out.shape == (T, topk)
    for t in range(T):
        live = [v for v in ti[t, topk:] if v >= 0]
        n = len(live)
        assert out[t, topk - n:].tolist() == live           # every live tail entry, in order
        assert out[t, :topk - n].tolist() == ti[t, :topk - n].tolist()  # a prefix of the selection
    # width == topk: unchanged; width < topk: error; more live tail than topk: the first topk
    assert np.array_equal(O.fit_kpool_indices(ti[:, :topk], topk), ti[:, :topk])
    with pytest.raises(ValueError):
        O.fit_kpool_indices(ti[:, :100], topk)
    wide = np.concatenate([np.full((2, 4), 7), np.arange(12).reshape(2, 6)], axis=1)
    assert O.fit_kpool_indices(wide, 4).tolist() == [[0, 1, 2, 3], [6, 7, 8, 9]]
