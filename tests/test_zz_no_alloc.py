"""mla_decode_fwd_static: the decode on the library's file-scope device scratch
(no caller workspace) agrees with mla_decode_fwd on the same inputs and with
the fp64 oracle on sampled tokens, over calls in a row on different
workloads and partitions (uniform split-K, and the balanced schedule, whose
work list and partial slots are the largest use of the scratch), and
rejects plans larger than the scratch before touching the device.

Collected last on purpose: it must hold both alone in a fresh process and
after every other test has run in the same process.
"""
import ctypes

import numpy as np
import pytest

from paged_mla_decode_06_gb300 import binding as B
from paged_mla_decode_06_gb300 import build as BUILD
from paged_mla_decode_06_gb300 import inputs as I

STATIC_SCRATCH_BYTES = 64 << 20  # MLA_STATIC_SCRATCH_BYTES in include/mla_decode.h


def test_static_rejects_plans_beyond_the_scratch():
    BUILD.build()
    lib = B.load_library()
    prob = B.make_problem(num_tokens=64, num_reqs=64, num_heads=128, block_size=64,
                          num_blocks=5000, max_blocks_per_req=130, max_seq_len=8192,
                          num_segments=16, num_sms=152)
    plan = B.mla_decode_plan(prob)
    assert plan.workspace_bytes > STATIC_SCRATCH_BYTES
    st = lib.mla_decode_fwd_static(ctypes.byref(plan), None, None, None, 0, None, None, None,
                                   None, 1.0, 1.0, 1.0, None, None, None, None, None)
    assert st == 3  # MLA_ERR_WORKSPACE, before any device call
    assert lib.mla_status_string(st).decode() == "MLA_ERR_WORKSPACE"


def _static_vs_fwd(w, num_segments, tokens):
    import torch

    from tests.gpu_helpers import TOL_LSE, TOL_OUT, assert_close, run_oracle

    dw = B.DeviceWorkload(w, num_segments=num_segments)
    assert 0 < dw.plan.workspace_bytes <= STATIC_SCRATCH_BYTES
    if num_segments:
        assert dw.plan.num_segments > 1  # the partials live in the scratch
    else:
        assert dw.plan.schedule == 1     # work list, unit table and partial slots in the scratch
    if w.sparse:
        dw.convert()
    dw.forward(convert=False)
    torch.cuda.synchronize()
    assert dw.status() == 0
    ref_out = dw.out.float().cpu().numpy()
    ref_lse = dw.lse.cpu().numpy()

    out = torch.full_like(dw.out, float("nan"))
    lse = torch.full_like(dw.lse, float("nan"))
    status = torch.full((1,), -1, dtype=torch.int32, device=dw.device)
    B.mla_decode_fwd_static(
        dw.plan, dw.q, dw.cache,
        block_table=None if w.sparse else dw.block_table,
        seq_lens=None if w.sparse else dw.seq_lens, qo_indptr=dw.qo_indptr,
        sparse_slots=dw.slots, softmax_scale=w.softmax_scale, q_scale=w.q_scale,
        kv_scale=w.kv_scale, sinks=dw.sinks, out=out, lse=lse, status_out=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got_out = out.float().cpu().numpy()
    got_lse = lse.cpu().numpy()
    assert np.isfinite(got_out).all()
    err = float(np.max(np.abs(got_out - ref_out)))
    assert err <= TOL_OUT[w.kv_dtype], f"{w.name}: max |static - fwd| = {err:.3e}"
    ninf = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(got_lse), ninf)
    lerr = float(np.max(np.abs(got_lse[~ninf] - ref_lse[~ninf]))) if (~ninf).any() else 0.0
    assert lerr <= TOL_LSE, f"{w.name}: max |static lse - fwd lse| = {lerr:.3e}"
    # and against the fp64 oracle on sampled tokens
    or_o, or_l = run_oracle(w, tokens=tokens)
    assert_close(got_out[tokens], got_lse[tokens], or_o, or_l, w.kv_dtype, f"{w.name} static vs oracle")


@pytest.mark.gpu
def test_static_matches_fwd_on_calls_in_a_row():
    BUILD.build()
    # first call: DeepSeek-V3-shaped bf16 decode, 4 segments
    _static_vs_fwd(I.dsv3_bf16(seed=21, batch=8, seq_lo=700, seq_hi=5000), num_segments=4,
                   tokens=[0, 7])
    # second call, same scratch: multi-token rows with sinks, 3 segments,
    # a different partial layout than the first call left behind
    _static_vs_fwd(I.mtp_sinks(seed=22, batch=4, median=2000.0, hi=6000), num_segments=3,
                   tokens=[0, 5])
    # third: the planner's default for 128 heads, the balanced schedule on the
    # CTA-pair kernel (~41 MB of work list and partial slots)
    _static_vs_fwd(I.dsv3_bf16(seed=23, batch=64, seq_lo=1024, seq_hi=8192), num_segments=0,
                   tokens=[0, 31, 63])
    # fourth: e4m3 at 16 heads, the balanced schedule on the rows-as-N kernel
    _static_vs_fwd(I.fp8_decode(16, seed=24, batch=12, seq_len=8192), num_segments=0,
                   tokens=[0, 11])
