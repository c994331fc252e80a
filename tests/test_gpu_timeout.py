"""Failure detection without a GPU fault: a decode whose bounded internal
waits are given a 1 microsecond limit (plan.wait_limit_us) gives up, records
a code in its workspace status word and exits; the call returns, the status
query reports it, and the next calls (a fresh workspace, and the same
workspace once cleared) decode correctly. Nothing here faults, traps or
hangs the GPU: the waits are bounded and the kernel drains what it issued."""
import numpy as np
import pytest
import torch

from paged_mla_decode_06_gb300 import binding as B
from paged_mla_decode_06_gb300 import build as BUILD
from paged_mla_decode_06_gb300 import inputs as I
from tests.gpu_helpers import assert_close, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    BUILD.build()
    B.load_library()


@pytest.mark.parametrize("heads", [16, 128])
def test_bounded_wait_runs_out_and_is_reported(heads):
    """16 heads: one CTA per worker; 128 heads: clusters of two CTAs whose
    key boxes are multicast, where a CTA that gives up must still drain every
    box its peer armed on it before either exits."""
    w = I.fp8_decode(heads, batch=4, seq_len=4096)
    dw = B.DeviceWorkload(w)
    assert dw.plan.kernel == 5  # the rows-as-N kernel, balanced schedule
    assert dw.plan.tile_rows == (2 if heads > 64 else 1) * dw.plan.rows_per_cta
    assert B.mla_workspace_status(dw.plan, dw.workspace) == 0
    dw.plan.wait_limit_us = 1
    dw.forward()                # returns: the kernel gives up and exits
    torch.cuda.synchronize()
    code = B.mla_workspace_status(dw.plan, dw.workspace)
    assert code != 0
    tokens = [0, 3]
    ref_o, ref_l = run_oracle(w, tokens=tokens)
    # a fresh workspace with the default limit decodes correctly
    fresh = B.DeviceWorkload(w)
    fresh.forward()
    torch.cuda.synchronize()
    assert fresh.status() == 0
    assert_close(fresh.out.float().cpu().numpy()[tokens], fresh.lse.cpu().numpy()[tokens],
                 ref_o, ref_l, "fp8", "after a timed-out call")
    # the old workspace, once cleared, serves the next call
    assert B.mla_workspace_status(dw.plan, dw.workspace, clear=True) == code
    assert B.mla_workspace_status(dw.plan, dw.workspace) == 0
    dw.plan.wait_limit_us = 0
    dw.forward()
    torch.cuda.synchronize()
    assert B.mla_workspace_status(dw.plan, dw.workspace) == 0
    assert_close(dw.out.float().cpu().numpy()[tokens], dw.lse.cpu().numpy()[tokens],
                 ref_o, ref_l, "fp8", "cleared workspace")


def test_bounded_wait_runs_out_on_the_cta_pair():
    """The CTA-pair kernel (bf16, balanced schedule): with a 1 microsecond
    limit the score and value CTAs give up, drain their copies to each other
    and their MMAs, and exit; the next call with the default limit decodes
    correctly."""
    w = I.build_dense(91, seq_lens=[3000, 700, 129, 4100], num_heads=128, block_size=64, num_segments=0)
    dw = B.DeviceWorkload(w, kernel=B.MLA_KERNEL_TCGEN05)
    assert dw.plan.kernel == 4 and dw.plan.schedule == 1
    dw.plan.wait_limit_us = 1
    dw.forward()
    torch.cuda.synchronize()
    code = B.mla_workspace_status(dw.plan, dw.workspace, clear=True)
    assert code != 0
    dw.plan.wait_limit_us = 0
    dw.forward()
    torch.cuda.synchronize()
    assert B.mla_workspace_status(dw.plan, dw.workspace) == 0
    ref_o, ref_l = run_oracle(w)
    assert_close(dw.out.float().cpu().numpy(), dw.lse.cpu().numpy(), ref_o, ref_l, "bf16",
                 "CTA pair after a timed-out call")
