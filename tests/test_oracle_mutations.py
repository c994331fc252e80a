"""Planted mistakes in the oracle must fail its pins.

Each case swaps one oracle function for a plausible wrong version (on the
CPU, for the duration of the test only) and checks that the pin written to
catch that mistake fails.
"""
import numpy as np
import pytest

import oracle.mla_oracle as M
import tests.test_oracle as P


def _attend_without_rope(q, keys, scale, sinks=None):
    return _orig_attend(q[:, :512], keys[:, :512], scale, sinks)


def _attend_values_from_tail(q, keys, scale, sinks=None):
    out, lse = _orig_attend(q, keys, scale, sinks)
    if keys.shape[0] == 0:
        return out, lse
    s = scale * (q @ keys.T)
    e = np.exp(s - s.max(axis=1, keepdims=True))
    return (e @ keys[:, 64:]) / e.sum(axis=1)[:, None], lse


def _attend_sink_scaled(q, keys, scale, sinks=None):
    return _orig_attend(q, keys, scale, None if sinks is None else np.asarray(sinks) * scale)


def _visible_off_by_one(seq_len, qlen, j):
    return max(0, int(seq_len) - int(qlen) + int(j))


def _bounds_floor(part_len, ns, tile):
    span = ns * tile
    tps = max(1, int(part_len) // span) if part_len > 0 else 0
    return [(s * tps * tile, min((s + 1) * tps * tile, int(part_len))) for s in range(ns)]


def _merge_wrong_base(so, sm, se, pl, tile, sinks=None):
    return _orig_merge(so, np.asarray(sm) * np.log(2.0), se, pl, tile, sinks)


def _convert_no_oob(req, bt, ti, bs, cu_seqlens=None, out_init=None):
    ti = np.asarray(ti, dtype=np.int64)
    bt = np.asarray(bt, dtype=np.int64)
    blk = np.clip(np.where(ti >= 0, ti // bs, 0), 0, bt.shape[1] - 1)
    base = bt[np.asarray(req)[:, None], blk]
    return np.where(ti >= 0, base * bs + np.where(ti >= 0, ti % bs, 0), -1)


def _seqlen_without_own_token(qsl, seq, topk):
    qsl = np.asarray(qsl, dtype=np.int64)
    lens = []
    for r in range(len(seq)):
        q = int(qsl[r + 1] - qsl[r])
        lens += [min(max(int(seq[r]) - q + j, 0), topk) for j in range(q)]
    lens = np.array(lens, dtype=np.int64)
    return lens, np.concatenate([[0], np.cumsum(lens)])


def _fit_keeps_whole_tail(ti, topk):
    ti = np.asarray(ti, dtype=np.int64)
    tail = ti[:, topk:][:, :topk]
    n = tail.shape[1]
    return np.concatenate([ti[:, :topk - n], tail], axis=1)


_orig_attend = M.attend
_orig_merge = M.merge_segments

CASES = [
    ("attend", _attend_without_rope, P.test_brute_force_python_loops),
    ("attend", _attend_values_from_tail, P.test_single_key_returns_its_value_row),
    ("attend", _attend_sink_scaled, P.test_sinks_match_the_post_hoc_fold),
    ("visible_len", _visible_off_by_one, P.test_causal_bound_includes_own_token),
    ("segment_bounds", _bounds_floor, P.test_segment_partition_golden),
    ("merge_segments", _merge_wrong_base, P.test_merge_single_segment_is_identity),
    ("index_convert", _convert_no_oob, P.test_index_convert_brute_force_and_edges),
    ("sparse_seqlen", _seqlen_without_own_token, P.test_sparse_seqlen_golden),
    ("fit_kpool_indices", _fit_keeps_whole_tail, P.test_fit_kpool_golden),
]


@pytest.mark.parametrize("name,bad,pin", CASES, ids=[f"{c[0]}-{c[1].__name__}" for c in CASES])
def test_planted_mistake_is_caught(monkeypatch, name, bad, pin):
    monkeypatch.setattr(M, name, bad)
    monkeypatch.setattr(P.O, name, bad)
    with pytest.raises(AssertionError):
        pin()
