"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Small cases are compared element by element on every token; the full-size
workloads, in the launch configuration the benchmark times, are compared on
sampled tokens the oracle computes one by one. Tolerances: bf16 output
max-abs 1e-2, fp8 output 2e-2, LSE 1e-3 absolute, index conversion
bit-exact. Caches carry NaN in every slot the decode must not read.
"""
import numpy as np
import pytest
import torch

import oracle as O
from paged_mla_decode_06_gb300 import binding as B
from paged_mla_decode_06_gb300 import build as BUILD
from paged_mla_decode_06_gb300 import inputs as I
from tests.gpu_helpers import assert_close, oracle_slots, run_gpu, run_oracle, visible_keys
from tests.test_schedule_rule import cut_rule, ranked_list

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    BUILD.build()
    B.load_library()


# ---------------------------------------------------------------- index conversion

def _convert_case(seed, T, topk, rows, cols, bs):
    rng = np.random.default_rng(seed)
    bt = rng.integers(0, 1 << 14, size=(rows, cols)).astype(np.int32)
    req = rng.integers(0, rows, size=T).astype(np.int32)
    ti = rng.integers(-2, cols * bs + 3 * bs, size=(T, topk)).astype(np.int32)
    ti[:, -1] = cols * bs - 1       # last valid position
    ti[0, :8] = -1
    if T > 2:
        req[2] = rows                # request outside the table
        req[1] = -1
    return req, bt, ti


@pytest.mark.parametrize("T,topk,rows,cols,bs", [
    (5, 128, 3, 7, 16), (33, 256, 9, 40, 64), (128, 2048, 16, 1024, 64), (7, 384, 4, 13, 48)])
def test_index_convert_bit_exact(T, topk, rows, cols, bs):
    req, bt, ti = _convert_case(T + topk, T, topk, rows, cols, bs)
    want = O.index_convert(req, bt, ti, bs)
    dev = torch.device("cuda")
    out = torch.full((T, topk), 7, dtype=torch.int32, device=dev)
    B.mla_sparse_index_convert(torch.from_numpy(req).to(dev), torch.from_numpy(bt).to(dev),
                               torch.from_numpy(ti).to(dev), block_size=bs, out=out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().astype(np.int64), want)


def test_index_convert_ragged_bit_exact():
    T, topk = 9, 256
    req, bt, ti = _convert_case(3, T, topk, 5, 20, 64)
    rng = np.random.default_rng(4)
    lens = rng.integers(0, topk + 1, size=T)
    lens[0], lens[1] = 0, topk
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    init = np.full(T * topk, 99, dtype=np.int64)
    want = O.index_convert(req, bt, ti, 64, cu_seqlens=cu, out_init=init)
    dev = torch.device("cuda")
    out = torch.full((T * topk,), 99, dtype=torch.int32, device=dev)
    B.mla_sparse_index_convert(torch.from_numpy(req).to(dev), torch.from_numpy(bt).to(dev),
                               torch.from_numpy(ti).to(dev), block_size=64,
                               cu_seqlens=torch.from_numpy(cu).to(dev), out=out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().astype(np.int64), want)


def test_index_convert_strided_inputs():
    T, topk = 6, 128
    req, bt, ti = _convert_case(5, T, topk, 4, 10, 16)
    want = O.index_convert(req, bt, ti, 16)
    dev = torch.device("cuda")
    bt_wide = torch.zeros((4, 17), dtype=torch.int32, device=dev)
    bt_wide[:, :10] = torch.from_numpy(bt).to(dev)
    ti_wide = torch.zeros((T, 200), dtype=torch.int32, device=dev)
    ti_wide[:, :topk] = torch.from_numpy(ti).to(dev)
    out = torch.empty((T, topk), dtype=torch.int32, device=dev)
    B.mla_sparse_index_convert(torch.from_numpy(req).to(dev), bt_wide[:, :10], ti_wide[:, :topk],
                               block_size=16, out=out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().astype(np.int64), want)


# ---------------------------------------------------------------- merge kernel

@pytest.mark.parametrize("sinks", [False, True])
@pytest.mark.parametrize("ns,tile", [(1, 16), (4, 16), (5, 64), (16, 1)])
def test_merge_kernel_matches_oracle(ns, tile, sinks):
    rng = np.random.default_rng(ns * 10 + tile + sinks)
    T, H = 7, 12
    lens = np.array([0, 1, 17, 64, 65, 300, 5000], dtype=np.int32)
    # partial outputs are weighted means of values: magnitudes of order one
    so = (rng.standard_normal((T, H, ns, 512)) * 0.5).astype(np.float32)
    sm = (rng.standard_normal((T, H, ns)) * 6).astype(np.float32)
    se = rng.uniform(0.5, 40, (T, H, ns)).astype(np.float32)
    for t in range(T):
        for s, (a, b) in enumerate(O.segment_bounds(int(lens[t]), ns, tile)):
            if a >= lens[t]:                  # dead segment: garbage the merge must skip
                so[t, :, s] = np.nan
                sm[t, :, s] = np.nan
                se[t, :, s] = np.nan
    se[5, 3, 0] = 0.0                          # a fully masked live segment
    sm[5, 3, 0] = -np.inf
    so[5, 3, 0] = 0.0
    sk = rng.standard_normal(H).astype(np.float32) if sinks else None
    ref_o, ref_l = O.merge_segments(so.astype(np.float64), sm, se, lens, tile, sinks=sk)
    dev = torch.device("cuda")
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    B.mla_merge_segments(torch.from_numpy(so).to(dev), torch.from_numpy(sm).to(dev),
                         torch.from_numpy(se).to(dev), torch.from_numpy(lens).to(dev),
                         tile_size=tile, sinks=None if sk is None else torch.from_numpy(sk).to(dev),
                         out=out, lse=lse)
    torch.cuda.synchronize()
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    # the merge itself only rounds: fp32 accumulation and the bf16 output
    assert np.isfinite(o).all()
    assert np.max(np.abs(o - ref_o) / (np.abs(ref_o) + 1e-3)) < 1e-2
    assert_close(o, l, ref_o, ref_l, "bf16", "merge")


# ---------------------------------------------------------------- dense decode

def test_tiny_dense_full_parity():
    w = I.tiny_dense()
    out, lse, dw = run_gpu(w)
    assert dw.plan.num_segments == 4 and dw.plan.tile_size == 16
    ref_o, ref_l = run_oracle(w)
    assert_close(out, lse, ref_o, ref_l, "bf16", "tiny dense")


def test_tiny_dense_segment_partials():
    w = I.tiny_dense()
    dw = B.DeviceWorkload(w)
    T, H, NS = w.num_tokens, w.num_heads, dw.plan.num_segments
    dev = dw.device
    so = torch.empty((T, H, NS, 512), dtype=torch.float32, device=dev)
    sm = torch.empty((T, H, NS), dtype=torch.float32, device=dev)
    se = torch.empty((T, H, NS), dtype=torch.float32, device=dev)
    B.mla_decode_segments(dw.plan, dw.q, dw.cache, block_table=dw.block_table,
                          seq_lens=dw.seq_lens, softmax_scale=w.softmax_scale,
                          segm_output=so, segm_max=sm, segm_expsum=se)
    torch.cuda.synchronize()
    ro, rm, re = O.segment_partials(w.q, "bf16", 1.0, w.cache, "bf16", 1.0, w.block_table,
                                    w.seq_lens, w.softmax_scale, NS, dw.plan.tile_size)
    so, sm, se = so.cpu().numpy(), sm.cpu().numpy(), se.cpu().numpy()
    assert np.array_equal(np.isneginf(sm), np.isneginf(rm))
    assert np.array_equal(se == 0, re == 0)
    live = re > 0
    assert np.max(np.abs(sm[live] - rm[live])) < 1e-3
    assert np.max(np.abs(se[live] / re[live] - 1)) < 5e-3
    assert np.max(np.abs(so - ro)) < 1e-2
    # merging the GPU partials with the oracle merge gives the unsplit result
    mo, ml = O.merge_segments(so, sm, se, O.partition_lengths(w.seq_lens), dw.plan.tile_size)
    uo, ul = run_oracle(w)
    assert_close(mo, ml, uo, ul, "bf16", "oracle merge of gpu partials")


KERNELS = [B.MLA_KERNEL_WARP_MMA, B.MLA_KERNEL_TCGEN05]
KIDS = ["mma", "tcgen05"]


@pytest.mark.parametrize("kernel", KERNELS, ids=KIDS)
@pytest.mark.parametrize("ns", [0, 1, 2, 3, 7])
def test_dsv3_shaped_bf16(ns, kernel):
    w = I.dsv3_bf16(batch=6, seq_lo=1024, seq_hi=2100, num_segments=ns)
    out, lse, dw = run_gpu(w, kernel=kernel)
    ref_o, ref_l = run_oracle(w)
    assert_close(out, lse, ref_o, ref_l, "bf16", f"dsv3 ns={dw.plan.num_segments} k={kernel}")


@pytest.mark.parametrize("heads", [1, 16, 64, 100, 128])
def test_tcgen05_head_counts_and_short_rows(heads):
    # lengths around the 64-key chunk, an empty row, and a segment split
    w = I.build_dense(60 + heads, seq_lens=[0, 1, 63, 64, 65, 127, 128, 129, 700],
                      num_heads=heads, block_size=64, num_segments=3)
    out, lse, dw = run_gpu(w, kernel=B.MLA_KERNEL_TCGEN05)
    assert dw.plan.kernel == 4
    ref_o, ref_l = run_oracle(w)
    assert_close(out, lse, ref_o, ref_l, "bf16", f"tcgen05 H={heads}", keys=visible_keys(w))


@pytest.mark.parametrize("case", ["dense", "multi_token", "sparse", "one_long", "many_units"])
def test_balanced_schedule_items(case):
    """The planner's balanced schedule (tensor-core kernel, segments left to
    the planner): read the work list back from the workspace and check that
    the pieces of every (unit, row tile) cover its key groups once and in
    order, items come longest first, split pieces own distinct partial slots
    within the budget, the items fit the grid, the output matches the oracle,
    and a second decode and merge over the same list give the same bits.
    The pieces equal the cut rule's (host model), and the row tiles of a
    multi-token request are cut at the same keys and listed side by side."""
    if case == "dense":
        w = I.build_dense(71, seq_lens=[0, 1, 129, 700, 3000, 9000, 257], num_heads=128,
                          block_size=64, num_segments=0)
        lens, tiles = w.seq_lens, np.ones(w.num_reqs, dtype=np.int64)
    elif case == "multi_token":
        w = I.build_dense(72, seq_lens=[5000, 40, 2600], num_heads=128, block_size=64,
                          qlens=[4, 1, 3], with_sinks=True, num_segments=0)
        q = np.diff(w.qo_indptr)
        lens, tiles = w.seq_lens, -(-q * 128 // 128)
    elif case == "one_long":       # one request cut into pieces on every pair
        w = I.build_dense(73, seq_lens=[60000], num_heads=128, block_size=64, num_segments=0)
        lens, tiles = w.seq_lens, np.ones(1, dtype=np.int64)
    elif case == "many_units":     # more units than the schedule block's threads: the binned path
        rng = np.random.default_rng(74)
        lens = rng.integers(0, 700, size=300)
        lens[:3] = [0, 1, 4000]
        w = I.build_dense(74, seq_lens=lens.tolist(), num_heads=128, block_size=64, num_segments=0)
        lens, tiles = w.seq_lens, np.ones(len(lens), dtype=np.int64)
    else:
        w = I.sparse_topk(num_reqs=2, tokens_per_req=3, cache_tokens=4096, topk=1024,
                          max_pad=300, num_segments=0)
        lens, tiles = np.full(w.num_tokens, 1024), np.ones(w.num_tokens, dtype=np.int64)
    out, lse, dw = run_gpu(w, kernel=B.MLA_KERNEL_TCGEN05)
    plan = dw.plan
    assert plan.schedule == 1 and plan.num_segments == 1
    ws = dw.workspace.cpu().numpy()
    n = int(ws[256:260].view(np.int32)[0])
    items = ws[512:512 + 32 * n].view(np.int32).reshape(n, 8)
    tab_off = 512 + -(-plan.max_items * 32 // 256) * 256
    tab = ws[tab_off:tab_off + 8 * len(lens) * plan.row_tiles].view(np.int32).reshape(
        len(lens), plan.row_tiles, 2)
    sizes = (items[:, 3] - items[:, 2]) // 128
    assert np.all(np.diff(sizes) <= 0), "items not longest first"
    split = False
    slots = []
    for u in range(len(lens)):
        g = -(-int(lens[u]) // 128)
        for t in range(int(tiles[u])):
            mine = items[(items[:, 0] == u) & (items[:, 1] == t)]
            mine = mine[np.argsort(mine[:, 2])]
            k = len(mine)
            assert k == max(1, tab[u, t, 1]) and k >= 1
            assert mine[0, 2] == 0 and mine[-1, 3] == g * 128
            assert np.array_equal(mine[1:, 2], mine[:-1, 3])
            if k > 1:
                split = True
                assert sorted(mine[:, 4].tolist()) == list(range(tab[u, t, 0], tab[u, t, 0] + k))
                slots += mine[:, 4].tolist()
            else:
                assert mine[0, 4] == -1 and tab[u, t, 0] == -1
    assert n == sum(max(1, int(tab[u, t, 1])) for u in range(len(lens)) for t in range(int(tiles[u])))
    # the host model of the rule gives the same pieces, row by row
    groups = [-(-int(x) // 128) for x in lens]
    per_cut = plan.row_tiles
    rows_m, pieces_m, _ = cut_rule(groups, [int(t) for t in tiles], plan.split_items // (2 * per_cut))
    r = 0
    for u in range(len(lens)):
        for t in range(int(tiles[u])):
            mine = items[(items[:, 0] == u) & (items[:, 1] == t)]
            mine = mine[np.argsort(mine[:, 2])]
            assert ((mine[:, 3] - mine[:, 2]) // 128).tolist() == pieces_m[r], (u, t)
            r += 1
    # at most 256 units: the device's list is the host model's, item by item
    # (pieces by size, ties in unit order; the sparse units are its tokens)
    if len(lens) <= 256:
        want = ranked_list(groups, [int(t) for t in tiles], plan.split_items // (2 * per_cut))
        got = [(int(a), int(b), int(c), int(d), int(e)) for a, b, c, d, e in items[:, :5]]
        assert got == want
    # a piece's row tiles are consecutive items
    for i in range(n):
        u, t, kb = items[i, 0], items[i, 1], items[i, 2]
        if t > 0:
            assert items[i - 1, 0] == u and items[i - 1, 1] == t - 1 and items[i - 1, 2] == kb
    assert len(set(slots)) == len(slots) and all(0 <= s < plan.split_items for s in slots)
    assert n <= plan.max_items
    assert split or case == "sparse" or n == sum(int(t) for t in tiles)
    ref_o, ref_l = run_oracle(w)
    assert_close(out, lse, ref_o, ref_l, "bf16", f"balanced {case}", keys=visible_keys(w))
    # the list again from the same lengths: the same items, and in the same
    # order when the units fit the schedule block's threads (pieces ranked by
    # a key; the binned path for more units orders equal sizes by atomics)
    B.mla_decode_schedule(plan, seq_lens=None if w.sparse else dw.seq_lens, qo_indptr=dw.qo_indptr,
                          workspace=dw.workspace)
    torch.cuda.synchronize()
    items2 = dw.workspace.cpu().numpy()[512:512 + 32 * n].view(np.int32).reshape(n, 8)
    if len(lens) <= 256:
        assert np.array_equal(items2, items)
    else:
        assert sorted(map(tuple, items2.tolist())) == sorted(map(tuple, items.tolist()))
    # the same work list serves a second decode: identical bits
    dw.out.zero_()
    dw.lse.zero_()
    B.mla_decode_items(plan, dw.q, dw.cache, block_table=None if w.sparse else dw.block_table,
                       seq_lens=None if w.sparse else dw.seq_lens, qo_indptr=dw.qo_indptr,
                       sparse_slots=dw.slots, softmax_scale=w.softmax_scale, sinks=dw.sinks,
                       workspace=dw.workspace, out=dw.out, lse=dw.lse)
    B.mla_merge_items(plan, qo_indptr=dw.qo_indptr, sinks=dw.sinks, workspace=dw.workspace,
                      out=dw.out, lse=dw.lse)
    torch.cuda.synchronize()
    assert dw.status() == 0
    assert np.array_equal(dw.out.float().cpu().numpy(), out)
    assert np.array_equal(dw.lse.cpu().numpy(), lse)


def test_tcgen05_segment_partials():
    w = I.build_dense(61, seq_lens=[1, 70, 300, 1000], num_heads=128, block_size=64,
                      num_segments=4)
    dw = B.DeviceWorkload(w, kernel=B.MLA_KERNEL_TCGEN05)
    T, H, NS = w.num_tokens, w.num_heads, dw.plan.num_segments
    dev = dw.device
    so = torch.full((T, H, NS, 512), 7.0, dtype=torch.float32, device=dev)
    sm = torch.full((T, H, NS), 7.0, dtype=torch.float32, device=dev)
    se = torch.full((T, H, NS), 7.0, dtype=torch.float32, device=dev)
    B.mla_decode_segments(dw.plan, dw.q, dw.cache, block_table=dw.block_table,
                          seq_lens=dw.seq_lens, softmax_scale=w.softmax_scale,
                          segm_output=so, segm_max=sm, segm_expsum=se)
    torch.cuda.synchronize()
    ro, rm, re = O.segment_partials(w.q, "bf16", 1.0, w.cache, "bf16", 1.0, w.block_table,
                                    w.seq_lens, w.softmax_scale, NS, dw.plan.tile_size)
    so, sm, se = so.cpu().numpy(), sm.cpu().numpy(), se.cpu().numpy()
    assert np.array_equal(np.isneginf(sm), np.isneginf(rm))
    live = re > 0
    assert np.array_equal(se > 0, live)
    assert np.max(np.abs(sm[live] - rm[live])) < 1e-3
    assert np.max(np.abs(se[live] / re[live] - 1)) < 5e-3
    assert np.max(np.abs(so - ro)) < 1e-2


@pytest.mark.parametrize("kernel", KERNELS, ids=KIDS)
@pytest.mark.parametrize("heads", [16, 32, 48, 64, 96, 128])
def test_fp8_heads(heads, kernel):
    w = I.fp8_decode(heads, batch=3, seq_len=2048, num_segments=2)
    out, lse, _ = run_gpu(w, kernel=kernel)
    ref_o, ref_l = run_oracle(w)
    assert_close(out, lse, ref_o, ref_l, "fp8", f"fp8 H={heads}")


@pytest.mark.parametrize("kernel", KERNELS, ids=KIDS)
@pytest.mark.parametrize("ns", [0, 1, 4])
def test_multi_token_with_sinks(ns, kernel):
    w = I.mtp_sinks(batch=6, median=700, lo=128, hi=2048, num_segments=ns)
    out, lse, _ = run_gpu(w, kernel=kernel)
    ref_o, ref_l = run_oracle(w)
    assert_close(out, lse, ref_o, ref_l, "bf16", "mtp+sinks")


@pytest.mark.parametrize("heads,bs,ns,sinks", [
    (1, 16, 1, False), (5, 16, 4, True), (16, 16, 3, False), (20, 8, 2, True),
    (48, 16, 1, True), (128, 16, 5, False)])
def test_edge_lengths(heads, bs, ns, sinks):
    seq = [0, 1, 15, 16, 17, 63, 64, 65, 200]
    w = I.build_dense(77 + heads, seq_lens=seq, num_heads=heads, block_size=bs,
                      with_sinks=sinks, num_segments=ns)
    out, lse, _ = run_gpu(w)
    ref_o, ref_l = run_oracle(w)
    assert_close(out, lse, ref_o, ref_l, "bf16", "edge lengths", keys=visible_keys(w))
    if not sinks:
        assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))


@pytest.mark.parametrize("bs", [1, 8, 48, 128, 256])
def test_block_sizes(bs):
    w = I.build_dense(90 + bs, seq_lens=[3, 300, 513], num_heads=16, block_size=bs,
                      num_segments=0)
    out, lse, dw = run_gpu(w)
    assert dw.plan.tile_size == O.tile_size_for_block(bs)
    ref_o, ref_l = run_oracle(w)
    assert_close(out, lse, ref_o, ref_l, "bf16", f"block {bs}", keys=visible_keys(w))


def test_multi_token_rows_and_short_sequences():
    # qlen larger than 1 with a sequence shorter than the block: the first
    # rows see very few keys.
    w = I.build_dense(5, seq_lens=[4, 2, 9], num_heads=128, block_size=64, qlens=[4, 2, 3],
                      with_sinks=False, num_segments=2)
    out, lse, _ = run_gpu(w)
    ref_o, ref_l = run_oracle(w)
    assert_close(out, lse, ref_o, ref_l, "bf16", "short mtp", keys=visible_keys(w))


# ---------------------------------------------------------------- sparse decode

@pytest.mark.parametrize("kernel", KERNELS, ids=KIDS)
@pytest.mark.parametrize("ns", [0, 1, 4])
def test_sparse_small(ns, kernel):
    w = I.sparse_topk(num_reqs=3, tokens_per_req=4, cache_tokens=4096, topk=512,
                      interspersed_rows=2, max_pad=64, num_segments=ns)
    out, lse, dw = run_gpu(w, kernel=kernel)
    assert np.array_equal(dw.slots.cpu().numpy().astype(np.int64), oracle_slots(w))
    ref_o, ref_l = run_oracle(w)
    assert_close(out, lse, ref_o, ref_l, "bf16", "sparse")


@pytest.mark.parametrize("kernel", KERNELS, ids=KIDS)
@pytest.mark.parametrize("ns", [1, 3])
def test_sparse_invalid_chunks_nan_rows(ns, kernel):
    """Slot lists with whole 64-key chunks of -1, a token with a single valid
    slot, one with none, and every cache row that no valid slot names set to
    NaN: unused rows must not reach the output (softmax weight 0 times NaN)."""
    w = I.sparse_topk(num_reqs=2, tokens_per_req=2, cache_tokens=2048, topk=256, max_pad=0)
    slots = oracle_slots(w).astype(np.int32)
    slots[0, 64:128] = -1             # one aligned chunk without a valid key
    slots[0, 200:] = -1               # a ragged tail of -1
    keep = slots[1, 137]
    slots[1, :] = -1
    slots[1, 137] = keep              # a single valid key
    slots[2, :] = -1                  # none at all
    slots[3, 1:64:2] = -1             # every other key of the first chunk
    valid = np.unique(slots[slots >= 0])
    flat_cache = w.cache.reshape(-1, w.cache.shape[-1])
    poison = np.ones(flat_cache.shape[0], dtype=bool)
    poison[valid] = False
    flat_cache[poison] = 0x7FC0       # bf16 quiet NaN
    lens = np.full(4, 256)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    flat = slots.reshape(-1).copy()
    dw = B.DeviceWorkload(w, num_segments=ns, kernel=kernel)
    dev = dw.device
    B.mla_decode_fwd(dw.plan, dw.q, dw.cache, sparse_slots=torch.from_numpy(flat).to(dev),
                     sparse_indptr=torch.from_numpy(cu).to(dev), softmax_scale=w.softmax_scale,
                     workspace=dw.workspace, out=dw.out, lse=dw.lse)
    torch.cuda.synchronize()
    ref_o, ref_l = O.mla_decode(w.q, "bf16", 1.0, w.cache, "bf16", 1.0, None, None,
                                w.softmax_scale, sparse_slots=flat, sparse_indptr=cu)
    assert dw.status() == 0
    out = dw.out.float().cpu().numpy()
    assert not np.isnan(out).any()
    assert_close(out, dw.lse.cpu().numpy(), ref_o, ref_l, "bf16", "sparse invalid chunks",
                 keys=visible_keys(w, slots=flat, indptr=cu))


@pytest.mark.parametrize("kernel", KERNELS, ids=KIDS)
def test_sparse_ragged_indptr(kernel):
    w = I.sparse_topk(num_reqs=2, tokens_per_req=3, cache_tokens=2048, topk=256, max_pad=0)
    slots = oracle_slots(w)
    lens = np.array([256, 0, 17, 128, 255, 1])
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    flat = np.concatenate([slots[t, :lens[t]] for t in range(6)]).astype(np.int32)
    dw = B.DeviceWorkload(w, num_segments=3, kernel=kernel)
    dev = dw.device
    B.mla_decode_fwd(dw.plan, dw.q, dw.cache, sparse_slots=torch.from_numpy(flat).to(dev),
                     sparse_indptr=torch.from_numpy(cu).to(dev), softmax_scale=w.softmax_scale,
                     workspace=dw.workspace, out=dw.out, lse=dw.lse)
    torch.cuda.synchronize()
    ref_o, ref_l = O.mla_decode(w.q, "bf16", 1.0, w.cache, "bf16", 1.0, None, None,
                                w.softmax_scale, sparse_slots=flat, sparse_indptr=cu)
    assert dw.status() == 0
    assert_close(dw.out.float().cpu().numpy(), dw.lse.cpu().numpy(), ref_o, ref_l, "bf16",
                 "sparse ragged", keys=visible_keys(w, slots=flat, indptr=cu))


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("kernel", KERNELS, ids=KIDS)
def test_rerun_and_page_permutation_are_bit_identical(kernel):
    w = I.dsv3_bf16(batch=5, seq_lo=300, seq_hi=1500, num_segments=3)
    out1, lse1, _ = run_gpu(w, kernel=kernel)
    out2, lse2, _ = run_gpu(w, kernel=kernel)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)
    rng = np.random.default_rng(9)
    perm = rng.permutation(w.num_blocks)
    cache2 = np.empty_like(w.cache)
    cache2[perm] = w.cache
    w.cache = cache2
    w.block_table = perm[w.block_table].astype(np.int32)
    out3, lse3, _ = run_gpu(w, kernel=kernel)
    assert np.array_equal(out1, out3) and np.array_equal(lse1, lse3)


@pytest.mark.parametrize("kernel", KERNELS, ids=KIDS)
def test_side_stream_and_graph_replay(kernel):
    w = I.dsv3_bf16(batch=4, seq_lo=200, seq_hi=900, num_segments=2)
    ref_o, ref_l = run_oracle(w)
    dw = B.DeviceWorkload(w, kernel=kernel)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dw.forward()
        dw.forward()
    torch.cuda.synchronize()
    assert_close(dw.out.float().cpu().numpy(), dw.lse.cpu().numpy(), ref_o, ref_l, "bf16",
                 "side stream")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dw.forward()
    # replay with shorter sequences written into the same device buffer
    w2 = I.dsv3_bf16(batch=4, seq_lo=200, seq_hi=900, num_segments=2)
    w2.seq_lens = np.maximum(w.seq_lens - 37, 1).astype(np.int32)
    dw.seq_lens.copy_(torch.from_numpy(w2.seq_lens))
    dw.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    ro2, rl2 = run_oracle(w2)
    assert_close(dw.out.float().cpu().numpy(), dw.lse.cpu().numpy(), ro2, rl2, "bf16",
                 "graph replay")


def test_balanced_schedule_graph_replay():
    """The balanced call (schedule, decode, merge; the last two programmatic
    dependents of the launch before them) captured in a CUDA graph and
    replayed with other lengths in the same device buffer: the work list is
    rebuilt from the new lengths inside the graph."""
    w = I.dsv3_bf16(batch=6, seq_lo=300, seq_hi=3000, num_segments=0)
    dw = B.DeviceWorkload(w, kernel=B.MLA_KERNEL_TCGEN05)
    assert dw.plan.schedule == 1
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dw.forward()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dw.forward()
    w2 = I.dsv3_bf16(batch=6, seq_lo=300, seq_hi=3000, num_segments=0)
    # shorter by different amounts (inside every request's blocks): another work list
    w2.seq_lens = np.maximum(w.seq_lens - np.array([101, 900, 13, 500, 1700, 64]), 1).astype(np.int32)
    dw.seq_lens.copy_(torch.from_numpy(w2.seq_lens))
    dw.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert dw.status() == 0
    ro2, rl2 = run_oracle(w2)
    assert_close(dw.out.float().cpu().numpy(), dw.lse.cpu().numpy(), ro2, rl2, "bf16",
                 "balanced graph replay")


# ---------------------------------------------------------------- full-size workloads

def _sampled(w, tokens, ns=None):
    out, lse, dw = run_gpu(w, num_segments=ns)
    ref_o, ref_l = run_oracle(w, tokens=tokens)
    return out[tokens], lse[tokens], ref_o, ref_l, dw


@pytest.mark.parametrize("kernel", KERNELS, ids=KIDS)
def test_full_dsv3_bf16_sampled(kernel):
    w = I.dsv3_bf16()
    order = np.argsort(w.seq_lens)
    tokens = sorted({int(order[0]), int(order[-1]), 5, 31, 63})
    out, lse, dw = run_gpu(w, kernel=kernel)
    ro, rl = run_oracle(w, tokens=tokens)
    assert_close(out[tokens], lse[tokens], ro, rl, "bf16",
                 f"full dsv3 ns={dw.plan.num_segments} k={kernel}")


@pytest.mark.parametrize("kernel", [B.MLA_KERNEL_AUTO, B.MLA_KERNEL_TCGEN05], ids=["auto", "pair"])
@pytest.mark.parametrize("heads", [96, 128])
def test_fp8_planner_path_split_rows(heads, kernel):
    # e4m3 above 64 heads under the balanced schedule: the planner's default
    # (the rows-as-N kernel, a cluster of two CTAs per request) and the CTA pair;
    # 6 requests x 4096 keys on 76-152 workers split every row
    w = I.fp8_decode(heads, batch=6, seq_len=4096, num_segments=0)
    out, lse, dw = run_gpu(w, kernel=kernel)
    assert dw.plan.schedule == 1
    assert dw.plan.kernel == (5 if kernel == B.MLA_KERNEL_AUTO else 4)
    ref_o, ref_l = run_oracle(w)
    assert_close(out, lse, ref_o, ref_l, "fp8", f"fp8 planner path H={heads} kernel={dw.plan.kernel}")


@pytest.mark.parametrize("heads", [16, 128])
def test_full_fp8_sampled(heads):
    w = I.fp8_decode(heads)
    out, lse, ro, rl, _ = _sampled(w, [0, 25, 51])
    assert_close(out, lse, ro, rl, "fp8", f"full fp8 H={heads}")


def test_full_mtp_sinks_sampled():
    w = I.mtp_sinks()
    T = w.num_tokens
    out, lse, ro, rl, _ = _sampled(w, [0, 1, T // 2, T - 1])
    assert_close(out, lse, ro, rl, "bf16", "full mtp+sinks")


def test_full_sparse_sampled():
    w = I.sparse_topk(interspersed_rows=1)
    out, lse, dw = run_gpu(w)
    slots = oracle_slots(w)
    assert np.array_equal(dw.slots.cpu().numpy().astype(np.int64), slots)
    tokens = [0, 1, 64, 127]
    ro, rl = run_oracle(w, tokens=tokens, slots=slots)
    assert_close(out[tokens], lse[tokens], ro, rl, "bf16", "full sparse")


# ---------------------------------------------------------------- q pre-step

@pytest.mark.parametrize("fp8", [False, True])
def test_concat_quant_q_bit_exact(fp8):
    rng = np.random.default_rng(21)
    T, H = 9, 20
    nope = I.float32_to_bf16_bits(rng.standard_normal((T, H, 512)).astype(np.float32) * 3)
    pe = I.float32_to_bf16_bits(rng.standard_normal((T, H, 64)).astype(np.float32) * 3)
    nope[0, 0, :4] = I.float32_to_bf16_bits(np.array([1e6, -1e6, 0.0, -0.0], np.float32))
    dev = torch.device("cuda")
    # strided views: the latent and rope parts live in one wider buffer
    big = torch.zeros((T, H, 640), dtype=torch.int16)
    big[..., :512] = torch.from_numpy(nope.view(np.int16))
    big[..., 576:640] = torch.from_numpy(pe.view(np.int16))
    big = big.to(dev).view(torch.bfloat16)
    a, b = big[..., :512], big[..., 576:640]
    scale = 0.0371
    if fp8:
        out = torch.empty((T, H, 576), dtype=torch.uint8, device=dev)
        B.mla_concat_quant_q(a, b, out=out, q_scale=scale)
        want = O.concat_quant_q(O.decode_bf16(nope), O.decode_bf16(pe), q_scale=scale)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), want)
    else:
        out = torch.empty((T, H, 576), dtype=torch.bfloat16, device=dev)
        B.mla_concat_quant_q(a, b, out=out)
        torch.cuda.synchronize()
        want = O.concat_quant_q(O.decode_bf16(nope), O.decode_bf16(pe))
        assert np.array_equal(out.float().cpu().numpy().astype(np.float64), want)


# ---------------------------------------------------------------- sparse front end

@pytest.mark.parametrize("topk", [128, 2048])
def test_sparse_seqlen_bit_exact(topk):
    rng = np.random.default_rng(topk)
    R = 37
    seq = rng.integers(0, 3 * topk, size=R).astype(np.int32)
    seq[:3] = [0, 1, topk]
    qlens = rng.integers(0, 5, size=R)
    qsl = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    T = int(qsl[-1]) + 2                   # two tokens past the last request: length 0
    want_lens, want_ptr = O.sparse_seqlen(qsl, seq, topk)
    want_lens = np.concatenate([want_lens, [0, 0]])
    want_ptr = np.concatenate([want_ptr, [want_ptr[-1]] * 2])
    dev = torch.device("cuda")
    lens = torch.full((T,), -7, dtype=torch.int32, device=dev)
    ptr = torch.full((T + 1,), -7, dtype=torch.int32, device=dev)
    B.mla_sparse_seqlen(torch.from_numpy(qsl).to(dev), torch.from_numpy(seq).to(dev), topk=topk,
                        indptr=ptr, lens=lens)
    torch.cuda.synchronize()
    assert np.array_equal(lens.cpu().numpy(), want_lens)
    assert np.array_equal(ptr.cpu().numpy(), want_ptr)


def test_sparse_seqlen_tokens_before_the_first_request():
    # query_start_loc need not start at 0: the tokens before it have no list
    qsl = np.array([3, 5, 9, 10], dtype=np.int32)
    seq = np.array([4, 300, 2], dtype=np.int32)
    want_lens, want_ptr = O.sparse_seqlen(qsl, seq, 128)
    dev = torch.device("cuda")
    lens = torch.full((10,), -7, dtype=torch.int32, device=dev)
    ptr = torch.full((11,), -7, dtype=torch.int32, device=dev)
    B.mla_sparse_seqlen(torch.from_numpy(qsl).to(dev), torch.from_numpy(seq).to(dev), topk=128,
                        indptr=ptr, lens=lens)
    torch.cuda.synchronize()
    assert np.array_equal(lens.cpu().numpy(), want_lens)
    assert np.array_equal(ptr.cpu().numpy(), want_ptr)
    assert np.all(want_lens[:3] == 0)


def test_sparse_seqlen_many_tokens():
    rng = np.random.default_rng(5)
    R = 3000
    seq = rng.integers(0, 5000, size=R).astype(np.int32)
    qlens = rng.integers(1, 5, size=R)
    qsl = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    want_lens, want_ptr = O.sparse_seqlen(qsl, seq, 2048)
    dev = torch.device("cuda")
    ptr = torch.empty((int(qsl[-1]) + 1,), dtype=torch.int32, device=dev)
    B.mla_sparse_seqlen(torch.from_numpy(qsl).to(dev), torch.from_numpy(seq).to(dev), topk=2048,
                        indptr=ptr)
    torch.cuda.synchronize()
    assert np.array_equal(ptr.cpu().numpy(), want_ptr)


@pytest.mark.parametrize("T,topk,W", [(33, 128, 128), (40, 256, 320), (7, 128, 700), (200, 2048, 2112)])
def test_fit_kpool_bit_exact(T, topk, W):
    rng = np.random.default_rng(T + W)
    ti = rng.integers(0, 1 << 20, size=(T, W)).astype(np.int32)
    ti[rng.random((T, W)) < 0.35] = -1
    ti[0, topk:] = -1                      # no live tail
    if W > topk:
        ti[1, topk:] = np.arange(W - topk)  # every tail entry live
    want = O.fit_kpool_indices(ti, topk)
    dev = torch.device("cuda")
    wide = torch.zeros((T, W + 5), dtype=torch.int32, device=dev)   # strided input
    wide[:, :W] = torch.from_numpy(ti).to(dev)
    out_wide = torch.full((T, topk + 3), 99, dtype=torch.int32, device=dev)
    B.mla_fit_kpool_indices(wide[:, :W], topk=topk, out=out_wide[:, :topk])
    torch.cuda.synchronize()
    got = out_wide.cpu().numpy()
    assert np.array_equal(got[:, :topk], want)
    assert np.all(got[:, topk:] == 99)


def test_sparse_front_end_pipeline():
    """Indexer rows wider than topk -> fit -> per-token lengths -> ragged index
    conversion -> decode over the ragged lists, against the same chain of
    oracle functions."""
    w = I.sparse_topk(num_reqs=3, tokens_per_req=3, cache_tokens=2048, topk=256, max_pad=0)
    T, topk, W = w.num_tokens, 256, 256 + 48
    rng = np.random.default_rng(31)
    seq = np.array([100, 2048, 700], dtype=np.int32)
    qsl = np.array([0, 3, 6, 9], dtype=np.int32)
    ti = np.full((T, W), -1, dtype=np.int32)
    for t in range(T):
        r, j = t // 3, t % 3
        vis = int(seq[r]) - 3 + j + 1
        k = min(vis, topk)
        ti[t, :k] = rng.choice(vis, size=k, replace=False)
        tail = np.arange(max(0, vis - 40), vis)[::-1][:40]
        ti[t, topk:topk + len(tail)] = tail
        ti[t, topk + rng.integers(0, 48, size=10)] = -1
    fitted = O.fit_kpool_indices(ti, topk)
    lens, ptr = O.sparse_seqlen(qsl, seq, topk)
    flat = O.index_convert(w.req_id_per_token, w.block_table, fitted, w.block_size, cu_seqlens=ptr,
                           out_init=np.full(T * topk, -1, dtype=np.int64))[:int(ptr[-1])]
    ref_o, ref_l = O.mla_decode(w.q, "bf16", 1.0, w.cache, "bf16", 1.0, None, None, w.softmax_scale,
                                sparse_slots=flat, sparse_indptr=ptr)
    dw = B.DeviceWorkload(w, kernel=B.MLA_KERNEL_TCGEN05)
    dev = dw.device
    d_fit = torch.empty((T, topk), dtype=torch.int32, device=dev)
    B.mla_fit_kpool_indices(torch.from_numpy(ti).to(dev), topk=topk, out=d_fit)
    d_ptr = torch.empty((T + 1,), dtype=torch.int32, device=dev)
    B.mla_sparse_seqlen(torch.from_numpy(qsl).to(dev), torch.from_numpy(seq).to(dev), topk=topk,
                        indptr=d_ptr)
    d_flat = torch.full((T * topk,), -1, dtype=torch.int32, device=dev)
    B.mla_sparse_index_convert(dw.req_id, dw.block_table, d_fit, block_size=w.block_size,
                               cu_seqlens=d_ptr, out=d_flat)
    B.mla_decode_fwd(dw.plan, dw.q, dw.cache, sparse_slots=d_flat, sparse_indptr=d_ptr,
                     softmax_scale=w.softmax_scale, workspace=dw.workspace, out=dw.out, lse=dw.lse)
    torch.cuda.synchronize()
    assert dw.status() == 0
    assert np.array_equal(d_ptr.cpu().numpy(), ptr)
    assert np.array_equal(d_flat.cpu().numpy()[:int(ptr[-1])].astype(np.int64), flat)
    assert_close(dw.out.float().cpu().numpy(), dw.lse.cpu().numpy(), ref_o, ref_l, "bf16",
                 "sparse front end", keys=visible_keys(w, slots=flat, indptr=ptr))
