"""Host-side checks of the C ABI: the library loads, exports every entry point
declared in include/*.h, plans problems, and rejects bad arguments with the
documented status before launching anything. No GPU needed: every call here
either stays on the host or fails validation before a launch.
"""
import ctypes
import glob
import os
import re

import numpy as np

import pytest

from paged_mla_decode_06_gb300 import binding as B
from paged_mla_decode_06_gb300 import build as BUILD

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    BUILD.build()
    return B.load_library()


def _declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        names.update(re.findall(r"MLA_API\s+[\w\s\*]+?\b(mla_\w+)\s*\(", src))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = _declared_symbols()
    assert {"mla_decode_plan", "mla_decode_fwd", "mla_decode_segments", "mla_merge_segments",
            "mla_sparse_index_convert"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_struct_sizes_match_the_header(lib):
    assert ctypes.sizeof(B.Problem) == 17 * 4
    # 17 problem ints + 14 plan ints (+ 4 bytes of padding) + 5 size_t; the
    # library asserts the same size at compile time
    assert ctypes.sizeof(B.Plan) == 168


def test_status_strings(lib):
    for code, name in [(0, "MLA_OK"), (1, "MLA_ERR_INVALID_ARG"), (2, "MLA_ERR_UNSUPPORTED"),
                       (3, "MLA_ERR_WORKSPACE"), (4, "MLA_ERR_CUDA"), (5, "MLA_ERR_DEVICE_STATUS")]:
        assert lib.mla_status_string(code).decode() == name
    assert lib.mla_version() >= 100


def _dense_problem(**kw):
    base = dict(num_tokens=64, num_reqs=64, num_heads=128, block_size=64, num_blocks=5000,
                max_blocks_per_req=130, max_seq_len=8192, num_sms=152)
    base.update(kw)
    return B.make_problem(**base)


def test_plan_dense_defaults(lib):
    plan = B.mla_decode_plan(_dense_problem())
    assert plan.tile_size == 64
    assert plan.kernel == 4 and plan.rows_per_cta == 128 and plan.row_tiles == 1
    assert plan.grid_x == 2 and plan.grid_z == 64 and plan.grid_y == plan.num_segments
    assert plan.workspace_bytes >= 256 and plan.status_offset == 0
    assert 1 <= plan.num_segments <= 16
    if plan.num_segments > 1:
        th = 64 * 128
        assert plan.workspace_bytes >= th * plan.num_segments * (512 + 2) * 4
        assert plan.segm_max_offset % 256 == 0 and plan.segm_expsum_offset % 256 == 0


def test_plan_tile_rule_golden(lib):
    rows = [l.split() for l in open(os.path.join(ROOT, "tests", "golden", "tile_rule.txt"))
            if l.strip() and not l.startswith("#")]
    for bs, tile in rows:
        bs = int(bs)
        plan = B.mla_decode_plan(_dense_problem(block_size=bs, max_blocks_per_req=9000,
                                                max_seq_len=8192, num_blocks=10000))
        assert plan.tile_size == int(tile), bs


def test_plan_explicit_segments_and_small_heads(lib):
    plan = B.mla_decode_plan(_dense_problem(num_heads=16, num_segments=4, num_tokens=2,
                                            num_reqs=2, block_size=16, max_seq_len=130,
                                            max_blocks_per_req=10))
    assert plan.num_segments == 4 and plan.tile_size == 16
    assert plan.rows_per_cta == 16 and plan.row_tiles == 1


def test_plan_multi_token_rows(lib):
    plan = B.mla_decode_plan(_dense_problem(num_tokens=96, num_reqs=32, max_qlen=4,
                                            max_seq_len=8192))
    assert plan.row_tiles == 4 and plan.grid_x == 8  # 4 tokens x 128 heads / 128-row pairs
    plan = B.mla_decode_plan(_dense_problem(num_tokens=96, num_reqs=32, max_qlen=4,
                                            max_seq_len=8192, kernel=B.MLA_KERNEL_WARP_MMA))
    assert plan.row_tiles == 8  # 4 tokens x 128 heads / 64 rows


def test_plan_sparse(lib):
    plan = B.mla_decode_plan(B.make_problem(num_tokens=128, num_heads=128, block_size=64,
                                            num_blocks=16384, topk=2048, num_sms=152))
    assert plan.tile_size == 64 and plan.grid_z == 128


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim_override=512), B.MLA_ERR_UNSUPPORTED),
    (dict(num_heads=129), B.MLA_ERR_UNSUPPORTED),
    (dict(num_heads=0), B.MLA_ERR_INVALID_ARG),
    (dict(block_size=0), B.MLA_ERR_INVALID_ARG),
    (dict(num_segments=65), B.MLA_ERR_INVALID_ARG),
    (dict(topk=100, num_reqs=0), B.MLA_ERR_UNSUPPORTED),
    (dict(max_seq_len=100000), B.MLA_ERR_INVALID_ARG),
    (dict(max_qlen=0), B.MLA_ERR_INVALID_ARG),
    (dict(mixed_dtype=True), B.MLA_ERR_UNSUPPORTED),
    (dict(kernel=2, block_size=16, max_blocks_per_req=600), B.MLA_ERR_UNSUPPORTED),
    (dict(kernel=3), B.MLA_ERR_UNSUPPORTED),              # rows-as-N: e4m3 only
    (dict(kernel=3, dtype="fp8", num_tokens=128, max_qlen=2),
     B.MLA_ERR_UNSUPPORTED),                              # rows-as-N: 256 rows > 128
    (dict(kernel=3, dtype="fp8", num_heads=16, block_size=16, max_blocks_per_req=600),
     B.MLA_ERR_UNSUPPORTED),                              # rows-as-N: block size not 64k
    (dict(kernel=4), B.MLA_ERR_INVALID_ARG),
])
def test_plan_rejects(lib, kw, status):
    kw = dict(kw)
    hd = kw.pop("head_dim_override", None)
    mixed = kw.pop("mixed_dtype", False)
    prob = _dense_problem(**kw)
    if hd is not None:
        prob.head_dim = hd
    if mixed:
        prob.kv_dtype = B.MLA_DTYPE_FP8_E4M3
    plan = B.Plan()
    assert lib.mla_decode_plan(ctypes.byref(prob), ctypes.byref(plan)) == status
    assert lib.mla_decode_plan(None, ctypes.byref(plan)) == B.MLA_ERR_INVALID_ARG


FAKE = 0x10000  # aligned, never dereferenced: every call below fails validation first


def _fwd(lib, plan, **over):
    args = dict(q=FAKE, kv=FAKE, bt=FAKE, bts=130, seq=FAKE, qo=None, slots=None, sind=None,
                sc=0.07, qs=1.0, ks=1.0, sinks=None, ws=FAKE, wsb=1 << 40, out=FAKE, lse=FAKE)
    args.update(over)
    return lib.mla_decode_fwd(ctypes.byref(plan), args["q"], args["kv"], args["bt"], args["bts"],
                              args["seq"], args["qo"], args["slots"], args["sind"], args["sc"],
                              args["qs"], args["ks"], args["sinks"], args["ws"], args["wsb"],
                              args["out"], args["lse"], None)


@pytest.mark.parametrize("over,status", [
    (dict(q=None), B.MLA_ERR_INVALID_ARG),
    (dict(kv=FAKE + 8), B.MLA_ERR_INVALID_ARG),          # misaligned cache
    (dict(bt=None), B.MLA_ERR_INVALID_ARG),
    (dict(bts=10), B.MLA_ERR_INVALID_ARG),               # stride < max_blocks_per_req
    (dict(seq=None), B.MLA_ERR_INVALID_ARG),
    (dict(slots=FAKE), B.MLA_ERR_INVALID_ARG),           # sparse list on a dense plan
    (dict(sinks=FAKE), B.MLA_ERR_INVALID_ARG),           # sinks not announced in the problem
    (dict(out=None), B.MLA_ERR_INVALID_ARG),
    (dict(lse=FAKE + 2), B.MLA_ERR_INVALID_ARG),
    (dict(qs=0.0), B.MLA_ERR_INVALID_ARG),
    (dict(sc=float("nan")), B.MLA_ERR_INVALID_ARG),
    (dict(sc=-0.07), B.MLA_ERR_INVALID_ARG),
])
def test_fwd_rejects_bad_arguments(lib, over, status):
    plan = B.mla_decode_plan(_dense_problem(num_segments=1))
    assert _fwd(lib, plan, **over) == status


def test_fwd_rejects_small_workspace(lib):
    plan = B.mla_decode_plan(_dense_problem(num_segments=4))
    assert plan.workspace_bytes > 0
    assert _fwd(lib, plan, wsb=plan.workspace_bytes - 1) == B.MLA_ERR_WORKSPACE
    plan1 = B.mla_decode_plan(_dense_problem(num_segments=1))
    assert plan1.workspace_bytes == 256
    assert _fwd(lib, plan1, ws=None) == B.MLA_ERR_WORKSPACE
    assert _fwd(lib, plan, ws=None) == B.MLA_ERR_WORKSPACE
    assert _fwd(lib, plan, ws=FAKE + 128) == B.MLA_ERR_INVALID_ARG


def test_fwd_requires_qo_indptr_for_multi_token(lib):
    plan = B.mla_decode_plan(_dense_problem(num_tokens=96, num_reqs=32, max_qlen=4,
                                            num_segments=1))
    assert _fwd(lib, plan) == B.MLA_ERR_INVALID_ARG


def test_fwd_sparse_rejects_qo_indptr(lib):
    plan = B.mla_decode_plan(B.make_problem(num_tokens=128, num_heads=128, block_size=64,
                                            num_blocks=16384, topk=2048, num_sms=152,
                                            num_segments=1))
    assert _fwd(lib, plan, slots=FAKE, qo=FAKE) == B.MLA_ERR_INVALID_ARG
    assert _fwd(lib, plan, slots=None) == B.MLA_ERR_INVALID_ARG


def test_merge_rejects(lib):
    f = lib.mla_merge_segments
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 8, 0, 512, 16, None, 0, FAKE, FAKE, None) == B.MLA_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 8, 2, 500, 16, None, 0, FAKE, FAKE, None) == B.MLA_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 8, 2, 512, 16, None, 1, FAKE, FAKE, None) == B.MLA_ERR_UNSUPPORTED
    assert f(None, FAKE, FAKE, FAKE, 4, 8, 2, 512, 16, None, 0, FAKE, FAKE, None) == B.MLA_ERR_INVALID_ARG
    assert f(FAKE + 4, FAKE, FAKE, FAKE, 4, 8, 2, 512, 16, None, 0, FAKE, FAKE, None) == B.MLA_ERR_INVALID_ARG
    # zero tokens: nothing to do, nothing launched
    assert f(None, None, None, None, 0, 8, 2, 512, 16, None, 0, None, None, None) == B.MLA_OK


def test_index_convert_rejects(lib):
    f = lib.mla_sparse_index_convert
    assert f(FAKE, FAKE, 4, 8, 8, FAKE, 2048, 16, 2000, 64, None, FAKE, None) == B.MLA_ERR_INVALID_ARG
    assert f(FAKE, FAKE, 4, 8, 8, FAKE, 2048, 16, 2048, 0, None, FAKE, None) == B.MLA_ERR_INVALID_ARG
    assert f(FAKE, FAKE, 4, 8, 4, FAKE, 2048, 16, 2048, 64, None, FAKE, None) == B.MLA_ERR_INVALID_ARG
    assert f(FAKE, FAKE, 4, 8, 8, FAKE, 1024, 16, 2048, 64, None, FAKE, None) == B.MLA_ERR_INVALID_ARG
    assert f(None, FAKE, 4, 8, 8, FAKE, 2048, 16, 2048, 64, None, FAKE, None) == B.MLA_ERR_INVALID_ARG
    assert f(FAKE + 1, FAKE, 4, 8, 8, FAKE, 2048, 16, 2048, 64, None, FAKE, None) == B.MLA_ERR_INVALID_ARG
    assert f(None, None, 4, 8, 8, None, 2048, 0, 2048, 64, None, None, None) == B.MLA_OK


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(B, "_lib", None)
    with pytest.raises(RuntimeError, match="not found"):
        B.load_library(str(tmp_path / "nope.so"))


def test_merge_lse_rejects(lib):
    f = lib.mla_merge_lse
    assert f(FAKE, FAKE, 0, 4, 8, 512, None, FAKE, FAKE, None) == B.MLA_ERR_INVALID_ARG
    assert f(FAKE, FAKE, 2, 4, 8, 500, None, FAKE, FAKE, None) == B.MLA_ERR_INVALID_ARG
    assert f(None, FAKE, 2, 4, 8, 512, None, FAKE, FAKE, None) == B.MLA_ERR_INVALID_ARG
    assert f(FAKE + 8, FAKE, 2, 4, 8, 512, None, FAKE, FAKE, None) == B.MLA_ERR_INVALID_ARG
    assert f(None, None, 2, 0, 8, 512, None, None, None, None) == B.MLA_OK


def test_concat_quant_q_rejects(lib):
    f = lib.mla_concat_quant_q
    args = [FAKE, 512 * 8, 512, FAKE, 64 * 8, 64, 4, 8]
    assert f(*args, 7, 1.0, FAKE, None) == B.MLA_ERR_INVALID_ARG
    assert f(*args, 1, 0.0, FAKE, None) == B.MLA_ERR_INVALID_ARG
    assert f(FAKE, 512 * 8, 500, FAKE, 64 * 8, 64, 4, 8, 0, 1.0, FAKE, None) == B.MLA_ERR_INVALID_ARG
    assert f(FAKE + 4, 512 * 8, 512, FAKE, 64 * 8, 64, 4, 8, 0, 1.0, FAKE, None) == B.MLA_ERR_INVALID_ARG
    assert f(None, 512 * 8, 512, FAKE, 64 * 8, 64, 4, 8, 0, 1.0, FAKE, None) == B.MLA_ERR_INVALID_ARG
    assert f(None, 0, 0, None, 0, 0, 0, 8, 0, 1.0, None, None) == B.MLA_OK


# ---------------------------------------------------------------- balanced schedule

def test_plan_balanced_schedule(lib):
    plan = B.mla_decode_plan(_dense_problem())
    assert plan.schedule == 1 and plan.num_segments == 1 and plan.kernel == 4
    assert plan.split_items == 152 and plan.max_items == 64 + 76
    slots_rows = plan.split_items * 128
    assert plan.segm_output_offset % 256 == 0 and plan.segm_max_offset % 256 == 0
    assert plan.segm_max_offset - plan.segm_output_offset >= slots_rows * 512 * 4
    assert plan.segm_expsum_offset - plan.segm_max_offset >= slots_rows * 4
    assert plan.workspace_bytes >= plan.segm_expsum_offset + slots_rows * 4
    assert plan.workspace_bytes <= 64 << 20  # fits the static scratch of mla_decode_fwd_static
    # an explicit segment count or the warp-MMA kernel keeps the uniform partition
    assert B.mla_decode_plan(_dense_problem(num_segments=4)).schedule == 0
    assert B.mla_decode_plan(_dense_problem(kernel=B.MLA_KERNEL_WARP_MMA)).schedule == 0


@pytest.mark.parametrize("heads,qlen,rows", [(16, 1, 16), (20, 1, 32), (32, 1, 32), (48, 1, 48),
                                             (64, 1, 64), (16, 4, 64), (20, 3, 64), (1, 1, 16)])
def test_plan_rows_as_n(lib, heads, qlen, rows):
    """e4m3 requests of at most 64 query rows go to the rows-as-N kernel (one
    CTA per row tile, one worker per SM under the balanced schedule, partial
    slots of tile_rows rows); wider ones stay on the CTA pair."""
    prob = _dense_problem(dtype="fp8", num_heads=heads, num_tokens=64 * qlen, max_qlen=qlen)
    plan = B.mla_decode_plan(prob)
    assert plan.kernel == 5 and plan.rows_per_cta == rows and plan.row_tiles == 1
    assert plan.tile_rows == rows and plan.grid_x == 1
    assert plan.schedule == 1 and plan.split_items == 2 * 152 and plan.max_items == 64 + 152
    slot_rows = plan.split_items * rows
    assert plan.segm_max_offset - plan.segm_output_offset >= slot_rows * 512 * 4
    assert plan.workspace_bytes >= plan.segm_expsum_offset + slot_rows * 4
    assert plan.workspace_bytes <= 64 << 20
    # the CTA pair and the warp-MMA kernel can still be asked for
    assert B.mla_decode_plan(_dense_problem(dtype="fp8", num_heads=heads, num_tokens=64 * qlen,
                                            max_qlen=qlen, kernel=B.MLA_KERNEL_TCGEN05)).kernel == 4
    # more rows go to the CTA pair
    wide = B.mla_decode_plan(_dense_problem(dtype="fp8", num_heads=128, num_tokens=128, max_qlen=2))
    assert wide.kernel == 4


@pytest.mark.parametrize("heads,qlen,rows", [(96, 1, 48), (128, 1, 64), (65, 1, 48), (40, 3, 64),
                                             (33, 2, 48)])
def test_plan_rows_as_n_cluster(lib, heads, qlen, rows):
    """65..128 query rows: one row tile on a cluster of two CTAs of equal row
    counts (one pass over the keys for all heads), a worker per two SMs, and
    partial slots of the whole tile."""
    prob = _dense_problem(dtype="fp8", num_heads=heads, num_tokens=64 * qlen, max_qlen=qlen)
    plan = B.mla_decode_plan(prob)
    assert plan.kernel == 5 and plan.rows_per_cta == rows and plan.tile_rows == 2 * rows
    assert plan.row_tiles == 1 and plan.grid_x == 2
    assert plan.schedule == 1 and plan.split_items == 2 * 76 and plan.max_items == 64 + 76
    slot_rows = plan.split_items * 2 * rows
    assert plan.segm_max_offset - plan.segm_output_offset >= slot_rows * 512 * 4
    assert plan.workspace_bytes >= plan.segm_expsum_offset + slot_rows * 4
    uniform = B.mla_decode_plan(_dense_problem(dtype="fp8", num_heads=heads, num_tokens=64 * qlen,
                                               max_qlen=qlen, num_segments=3))
    assert uniform.schedule == 0 and uniform.kernel == 5 and uniform.grid_x == 2
    assert uniform.grid_y == 3 and uniform.tile_rows == 2 * rows


def test_schedule_stages_reject_bad_arguments(lib):
    plan = B.mla_decode_plan(_dense_problem())
    uniform = B.mla_decode_plan(_dense_problem(num_segments=4))
    wsb = plan.workspace_bytes
    sched = lambda p, **k: lib.mla_decode_schedule(ctypes.byref(p), k.get("seq", FAKE), None, None,
                                                   k.get("ws", FAKE), k.get("wsb", wsb), None)
    assert sched(uniform) == B.MLA_ERR_INVALID_ARG
    assert sched(plan, ws=None) == B.MLA_ERR_WORKSPACE
    assert sched(plan, wsb=wsb - 1) == B.MLA_ERR_WORKSPACE
    assert sched(plan, ws=FAKE + 64) == B.MLA_ERR_INVALID_ARG
    assert sched(plan, seq=None) == B.MLA_ERR_INVALID_ARG
    items = lambda p, **k: lib.mla_decode_items(
        ctypes.byref(p), FAKE, FAKE, FAKE, 130, FAKE, None, None, None, 0.07, 1.0, 1.0, None,
        k.get("ws", FAKE), k.get("wsb", wsb), k.get("out", FAKE), FAKE, None)
    assert items(uniform) == B.MLA_ERR_INVALID_ARG
    assert items(plan, wsb=16) == B.MLA_ERR_WORKSPACE
    assert items(plan, out=None) == B.MLA_ERR_INVALID_ARG
    merge = lambda p, **k: lib.mla_merge_items(ctypes.byref(p), None, k.get("sinks"), FAKE,
                                               k.get("wsb", wsb), FAKE, FAKE, None)
    assert merge(uniform) == B.MLA_ERR_INVALID_ARG
    assert merge(plan, wsb=0) == B.MLA_ERR_WORKSPACE
    assert merge(plan, sinks=FAKE) == B.MLA_ERR_INVALID_ARG   # sinks not announced


# ---------------------------------------------------------------- sparse front end

def test_sparse_seqlen_rejects_bad_arguments(lib):
    f = lambda **k: lib.mla_sparse_seqlen(k.get("qsl", FAKE), k.get("seq", FAKE), k.get("R", 4),
                                          k.get("T", 8), k.get("topk", 128), k.get("lens"),
                                          k.get("indptr", FAKE), None)
    assert f(topk=0) == B.MLA_ERR_INVALID_ARG
    assert f(R=-1) == B.MLA_ERR_INVALID_ARG
    assert f(indptr=None) == B.MLA_ERR_INVALID_ARG
    assert f(indptr=FAKE + 2) == B.MLA_ERR_INVALID_ARG
    assert f(qsl=None) == B.MLA_ERR_INVALID_ARG
    assert f(seq=None) == B.MLA_ERR_INVALID_ARG
    assert f(lens=FAKE + 1) == B.MLA_ERR_INVALID_ARG
    assert f(T=1 << 20, topk=1 << 12) == B.MLA_ERR_UNSUPPORTED


def test_fit_kpool_rejects_bad_arguments(lib):
    f = lambda **k: lib.mla_fit_kpool_indices(k.get("ti", FAKE), k.get("tis", 320), k.get("T", 8),
                                              k.get("W", 320), k.get("topk", 256),
                                              k.get("out", FAKE + (1 << 20)), k.get("os", 256), None)
    assert f(W=128) == B.MLA_ERR_INVALID_ARG          # width < topk
    assert f(topk=0) == B.MLA_ERR_INVALID_ARG
    assert f(tis=300) == B.MLA_ERR_INVALID_ARG        # row stride < width
    assert f(os=200) == B.MLA_ERR_INVALID_ARG         # row stride < topk
    assert f(out=FAKE + 64) == B.MLA_ERR_INVALID_ARG  # overlaps the input rows
    assert f(ti=None) == B.MLA_ERR_INVALID_ARG
    assert f(T=0) == B.MLA_OK                         # nothing to launch


def test_plan_random_problems_are_consistent(lib):
    """Random valid problems: the plan succeeds and its launch shape and
    workspace layout hold together; random invalid ones are refused."""
    rng = np.random.default_rng(123)
    for _ in range(400):
        sparse = rng.random() < 0.3
        heads = int(rng.integers(1, 129))
        bs = int(rng.choice([1, 16, 48, 64, 128, 256]))
        sms = int(rng.choice([2, 16, 100, 152]))
        ns = int(rng.choice([0, 0, 1, 3, 16]))
        if sparse:
            T = int(rng.integers(1, 3000))
            prob = B.make_problem(num_tokens=T, num_heads=heads, block_size=bs, num_blocks=1000,
                                  topk=128 * int(rng.integers(1, 17)), num_segments=ns, num_sms=sms,
                                  dtype="bf16")
            units = T
        else:
            R = int(rng.integers(1, 2000))
            qlen = int(rng.integers(1, 5))
            mb = int(rng.integers(1, 300))
            prob = B.make_problem(num_tokens=R * qlen, num_reqs=R, num_heads=heads, block_size=bs,
                                  num_blocks=100000, max_blocks_per_req=mb,
                                  max_seq_len=int(rng.integers(0, mb * bs + 1)), max_qlen=qlen,
                                  num_segments=ns, num_sms=sms,
                                  dtype=str(rng.choice(["bf16", "fp8"])))
            units = R
        plan = B.mla_decode_plan(prob)
        assert plan.num_segments >= 1 and plan.tile_size >= 1 and plan.row_tiles >= 1
        assert plan.grid_x >= 1 and plan.grid_y >= 1 and plan.grid_z == units
        assert plan.workspace_bytes >= 256 and plan.workspace_bytes % 256 == 0
        rn_ok = (not sparse and prob.kv_dtype == B.MLA_DTYPE_FP8_E4M3 and bs % 64 == 0
                 and heads * prob.max_qlen <= 128)
        if rn_ok:  # the planner's first choice wherever it can run
            rows = heads * prob.max_qlen
            cl = 2 if rows > 64 else 1
            assert plan.kernel == 5 and plan.row_tiles == 1 and plan.grid_x == cl
            assert plan.rows_per_cta == max(16, -(-(-(-rows // cl)) // 16) * 16)
            assert plan.tile_rows == cl * plan.rows_per_cta
        elif plan.kernel == 4:
            assert plan.tile_rows == plan.rows_per_cta == 128
        if plan.schedule == 1:
            assert plan.kernel in (4, 5) and ns == 0 and plan.num_segments == 1
            pairs = plan.kernel == 4 or plan.tile_rows > plan.rows_per_cta
            workers = min(1024, max(1, sms // 2) if pairs else sms)
            per_cut = plan.row_tiles if plan.kernel == 4 else 1  # a cut splits every tile of a unit
            assert plan.split_items == 2 * workers * per_cut
            assert plan.max_items == units * plan.row_tiles + workers * per_cut
            rows = plan.split_items * plan.tile_rows
            assert plan.segm_output_offset >= 512 + plan.max_items * 32
            assert plan.segm_max_offset >= plan.segm_output_offset + rows * 512 * 4
            assert plan.segm_expsum_offset >= plan.segm_max_offset + rows * 4
            assert plan.workspace_bytes >= plan.segm_expsum_offset + rows * 4
        elif plan.num_segments > 1:
            th = prob.num_tokens * heads
            assert plan.segm_max_offset >= plan.segm_output_offset + th * plan.num_segments * 512 * 4
            assert plan.workspace_bytes >= plan.segm_expsum_offset + th * plan.num_segments * 4
        # the same problem with one field broken is refused
        bad = B.make_problem(num_tokens=prob.num_tokens, num_reqs=prob.num_reqs, num_heads=heads,
                             block_size=bs, num_blocks=prob.num_blocks,
                             max_blocks_per_req=prob.max_blocks_per_req, max_seq_len=prob.max_seq_len,
                             max_qlen=prob.max_qlen, topk=prob.topk, num_sms=sms,
                             num_segments=int(rng.choice([-1, 65])))
        out = B.Plan()
        assert lib.mla_decode_plan(ctypes.byref(bad), ctypes.byref(out)) == B.MLA_ERR_INVALID_ARG


def test_workspace_status_rejects_bad_arguments(lib):
    plan = B.mla_decode_plan(_dense_problem())
    assert plan.wait_limit_us == 0  # the planner leaves the default (2 s)
    code = ctypes.c_int32(7)
    f = lib.mla_workspace_status
    assert f(None, FAKE, ctypes.byref(code), 0, None) == B.MLA_ERR_INVALID_ARG
    assert f(ctypes.byref(plan), None, ctypes.byref(code), 0, None) == B.MLA_ERR_INVALID_ARG
    assert f(ctypes.byref(plan), FAKE, None, 0, None) == B.MLA_ERR_INVALID_ARG
    assert f(ctypes.byref(plan), FAKE + 64, ctypes.byref(code), 0, None) == B.MLA_ERR_INVALID_ARG
    assert code.value == 7  # nothing written on a refused call
