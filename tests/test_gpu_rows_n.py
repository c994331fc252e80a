"""The tcgen05 decode kernel with the query rows as the MMA N dimension (e4m3
cache, block size a multiple of 64, at most 128 query rows per request: one
CTA up to 64, a cluster of two sharing each key box above), through the C
ABI, against the fp64 oracle: head counts 1..128, multi-token causal rows
with sinks, edge lengths, block sizes, the split-K partials, the uniform and
the balanced partitions, the balanced work list itself against its rule,
workers running many items in turn, reruns and page permutations
(bit-equal), CUDA-graph replay, and the full-size e4m3 batch on sampled
tokens. Caches hold NaN in every slot the decode must not read."""
import numpy as np
import pytest
import torch

import oracle as O
from paged_mla_decode_06_gb300 import binding as B
from paged_mla_decode_06_gb300 import build as BUILD
from paged_mla_decode_06_gb300 import inputs as I
from tests.gpu_helpers import assert_close, run_gpu, run_oracle, visible_keys
from tests.test_schedule_rule import contiguous_rule

pytestmark = pytest.mark.gpu

RN = B.MLA_KERNEL_TCGEN05_ROWS_N
EDGE = [0, 1, 63, 64, 65, 127, 128, 129, 700, 3000]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    BUILD.build()
    B.load_library()


def _rows(heads, qlen=1):
    """(rows per CTA, CTAs per row tile) of the planner."""
    n = heads * qlen
    cl = 2 if n > 64 else 1
    return -(-(-(-n // cl)) // 16) * 16, cl


@pytest.mark.parametrize("ns", [0, 1, 3])
@pytest.mark.parametrize("heads", [1, 8, 16, 20, 32, 48, 64, 65, 96, 112, 128])
def test_rows_n_head_counts(heads, ns):
    w = I.build_dense(200 + heads, seq_lens=EDGE, num_heads=heads, block_size=64, dtype="fp8",
                      num_segments=ns)
    out, lse, dw = run_gpu(w, kernel=RN)
    rows, cl = _rows(heads)
    assert dw.plan.kernel == 5 and dw.plan.rows_per_cta == rows and dw.plan.tile_rows == cl * rows
    assert dw.plan.schedule == (1 if ns == 0 else 0)
    ref_o, ref_l = run_oracle(w)
    assert_close(out, lse, ref_o, ref_l, "fp8", f"rows-as-N H={heads} ns={ns}", keys=visible_keys(w))
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))


@pytest.mark.parametrize("ns", [0, 2])
@pytest.mark.parametrize("heads,qlens", [(16, [1, 2, 3, 4, 4]), (8, [2, 4, 3]), (20, [3, 1, 2]),
                                         (32, [4, 1, 2, 3, 4]), (40, [3, 1, 2]), (24, [1, 4, 1])])
def test_rows_n_multi_token_with_sinks(heads, qlens, ns):
    """Causal rows of 2-4 tokens; with 65..128 rows a request of fewer tokens
    leaves the second CTA of the cluster some or all rows empty."""
    seq = [900, 2500, 300, 4, 5000][:len(qlens)]
    w = I.build_dense(230 + heads, seq_lens=seq, num_heads=heads, block_size=64, dtype="fp8",
                      qlens=qlens, with_sinks=True, num_segments=ns)
    out, lse, dw = run_gpu(w, kernel=RN)
    assert dw.plan.rows_per_cta == _rows(heads, max(qlens))[0]
    ref_o, ref_l = run_oracle(w)
    assert_close(out, lse, ref_o, ref_l, "fp8", f"rows-as-N mtp H={heads}", keys=visible_keys(w))


@pytest.mark.parametrize("bs", [64, 128, 256])
def test_rows_n_block_sizes(bs):
    w = I.build_dense(240 + bs, seq_lens=[5, 300, 1537, 4100], num_heads=16, block_size=bs,
                      dtype="fp8", num_segments=0)
    out, lse, dw = run_gpu(w)
    assert dw.plan.kernel == 5
    ref_o, ref_l = run_oracle(w)
    assert_close(out, lse, ref_o, ref_l, "fp8", f"rows-as-N block {bs}", keys=visible_keys(w))


@pytest.mark.parametrize("heads", [16, 64, 96])
def test_rows_n_segment_partials(heads):
    w = I.build_dense(250 + heads, seq_lens=[1, 70, 300, 1000, 2049], num_heads=heads,
                      block_size=64, dtype="fp8", num_segments=4)
    dw = B.DeviceWorkload(w, kernel=RN)
    T, H, NS = w.num_tokens, w.num_heads, dw.plan.num_segments
    dev = dw.device
    so = torch.full((T, H, NS, 512), 7.0, dtype=torch.float32, device=dev)
    sm = torch.full((T, H, NS), 7.0, dtype=torch.float32, device=dev)
    se = torch.full((T, H, NS), 7.0, dtype=torch.float32, device=dev)
    B.mla_decode_segments(dw.plan, dw.q, dw.cache, block_table=dw.block_table,
                          seq_lens=dw.seq_lens, softmax_scale=w.softmax_scale, q_scale=w.q_scale,
                          kv_scale=w.kv_scale, segm_output=so, segm_max=sm, segm_expsum=se)
    torch.cuda.synchronize()
    ro, rm, re = O.segment_partials(w.q, "fp8", w.q_scale, w.cache, "fp8", w.kv_scale,
                                    w.block_table, w.seq_lens, w.softmax_scale, NS,
                                    dw.plan.tile_size)
    so, sm, se = so.cpu().numpy(), sm.cpu().numpy(), se.cpu().numpy()
    assert np.array_equal(np.isneginf(sm), np.isneginf(rm))
    live = re > 0
    assert np.array_equal(se > 0, live)
    assert np.max(np.abs(sm[live] - rm[live])) < 1e-3
    assert np.max(np.abs(se[live] / re[live] - 1)) < 1e-2
    assert np.max(np.abs(so - ro)) < 2e-2
    # the oracle merge of the GPU partials gives the unsplit result
    mo, ml = O.merge_segments(so, sm, se, O.partition_lengths(w.seq_lens), dw.plan.tile_size)
    uo, ul = run_oracle(w)
    assert_close(mo, ml, uo, ul, "fp8", "oracle merge of rows-as-N partials", keys=visible_keys(w))


def test_rows_n_rerun_and_page_permutation_bit_identical():
    w = I.fp8_decode(32, batch=5, seq_len=3000, num_segments=0)
    out1, lse1, _ = run_gpu(w)
    out2, lse2, _ = run_gpu(w)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)
    rng = np.random.default_rng(9)
    perm = rng.permutation(w.num_blocks)
    cache2 = np.empty_like(w.cache)
    cache2[perm] = w.cache
    w.cache = cache2
    w.block_table = perm[w.block_table].astype(np.int32)
    out3, lse3, _ = run_gpu(w)
    assert np.array_equal(out1, out3) and np.array_equal(lse1, lse3)


def test_rows_n_balanced_graph_replay():
    w = I.build_dense(260, seq_lens=[3000, 700, 12000, 129], num_heads=16, block_size=64,
                      dtype="fp8", num_segments=0)
    dw = B.DeviceWorkload(w, kernel=RN)
    assert dw.plan.schedule == 1
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dw.forward()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dw.forward()
    w.seq_lens = np.array([2900, 640, 11000, 1], dtype=np.int32)
    dw.seq_lens.copy_(torch.from_numpy(w.seq_lens))
    dw.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert dw.status() == 0
    ref_o, ref_l = run_oracle(w)
    assert_close(dw.out.float().cpu().numpy(), dw.lse.cpu().numpy(), ref_o, ref_l, "fp8",
                 "rows-as-N graph replay", keys=visible_keys(w))


def _work_list(dw, units):
    """Items, per-worker first items and the unit table read back from the
    workspace (layout as the header documents it)."""
    plan = dw.plan
    ws = dw.workspace.cpu().numpy()
    n = int(ws[256:260].view(np.int32)[0])
    items = ws[512:512 + 32 * n].view(np.int32).reshape(n, 8)
    tab_off = 512 + -(-plan.max_items * 32 // 256) * 256
    tab = ws[tab_off:tab_off + 8 * units * plan.row_tiles].view(np.int32).reshape(units, plan.row_tiles, 2)
    wf_off = tab_off + -(-units * plan.row_tiles * 8 // 256) * 256
    workers = plan.split_items // 2
    first = ws[wf_off:wf_off + 4 * (workers + 1)].view(np.int32)
    return items, first, tab


@pytest.mark.parametrize("case", ["many_short", "mixed", "cluster", "one_long", "fewer_groups"])
def test_rows_n_work_list_and_item_runs(case):
    """The device's work list equals the contiguous rule exactly (items in
    sequence order, a cut at every multiple of W, each worker's first item),
    and the decode over it, where workers run several items one after
    another (empty requests among them), matches the oracle."""
    rng = np.random.default_rng(300 + len(case))
    heads, qlens = 16, None
    if case == "many_short":      # about four items per worker, empty rows between
        seq = rng.integers(0, 700, size=600)
        seq[::37] = 0
    elif case == "mixed":
        seq = np.concatenate([rng.integers(1, 200, size=100), [30000, 0, 12000], rng.integers(1, 5000, size=40)])
    elif case == "cluster":       # a cluster of two per row tile
        heads = 96
        seq = rng.integers(0, 3000, size=150)
    elif case == "one_long":      # one request cut on every worker
        seq = np.array([70000])
    else:                         # fewer key groups than workers
        heads, qlens = 20, [1, 3, 2]
        seq = np.array([300, 5, 90])
    w = I.build_dense(310 + len(case), seq_lens=[int(x) for x in seq], num_heads=heads, block_size=64,
                      dtype="fp8", qlens=qlens, num_segments=0)
    out, lse, dw = run_gpu(w, kernel=RN)
    plan = dw.plan
    assert plan.schedule == 1 and plan.kernel == 5
    units = len(w.seq_lens)
    items, first, tab = _work_list(dw, units)
    qn = np.diff(w.qo_indptr) if w.qo_indptr is not None else np.ones(units, dtype=np.int64)
    tiles = [int(-(-int(q) * heads // plan.tile_rows)) for q in qn]
    groups = [int(-(-int(x) // 128)) for x in w.seq_lens]
    want, want_first, _ = contiguous_rule(groups, tiles, plan.split_items // 2)
    got = [(int(a), int(b), int(c) // 128, int(d) // 128, int(e)) for a, b, c, d, e in items[:, :5]]
    assert got == want
    assert np.array_equal(first, np.array(want_first, dtype=np.int32))
    ref_o, ref_l = run_oracle(w)
    assert_close(out, lse, ref_o, ref_l, "fp8", f"rows-as-N work list {case}", keys=visible_keys(w))


@pytest.mark.parametrize("heads", [16, 32, 48, 64, 96, 128])
def test_rows_n_full_fp8_sampled(heads):
    """The benchmark's e4m3 batch (52 requests x 16384 keys) on the planner's
    default launch, sampled tokens against the oracle."""
    w = I.fp8_decode(heads)
    out, lse, dw = run_gpu(w)
    assert dw.plan.kernel == 5 and dw.plan.schedule == 1
    tokens = [0, 25, 51]
    ref_o, ref_l = run_oracle(w, tokens=tokens)
    assert_close(out[tokens], lse[tokens], ref_o, ref_l, "fp8", f"full fp8 rows-as-N H={heads}")
