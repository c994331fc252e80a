"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and the oracle on the same seeded inputs, and compare them."""
import numpy as np
import torch

import oracle as O
from paged_mla_decode_06_gb300 import binding as B

TOL_OUT = {"bf16": 1e-2, "fp8": 2e-2}
TOL_LSE = 1e-3
# Rows that see only a handful of keys of unit-variance values lie outside
# the specified workloads (whose outputs average hundreds of keys). There one
# p rounded to bf16 (relative error <= 2^-9) moves the output by up to
# 2^-9 * max|v|, and rounding the output to bf16 adds up to 2^-8 * |out|:
# for |v|, |out| <= 4.5 that is 0.009 + 0.018 < 3e-2.
TOL_FEW_KEYS = 3e-2


def run_gpu(w, num_segments=None, stream=None, kernel=B.MLA_KERNEL_AUTO):
    dw = B.DeviceWorkload(w, num_segments=num_segments, kernel=kernel)
    dw.forward(stream=stream)
    torch.cuda.synchronize()
    assert dw.status() == 0, f"device status word {dw.status()}"
    return dw.out.float().cpu().numpy(), dw.lse.cpu().numpy(), dw


def oracle_slots(w):
    return O.index_convert(w.req_id_per_token, w.block_table, w.topk_indices, w.block_size)


def run_oracle(w, tokens=None, slots=None):
    if w.sparse:
        if slots is None:
            slots = oracle_slots(w)
        return O.mla_decode(w.q, w.q_dtype, w.q_scale, w.cache, w.kv_dtype, w.kv_scale,
                            None, None, w.softmax_scale, sparse_slots=slots, sinks=w.sinks,
                            tokens=tokens)
    return O.mla_decode(w.q, w.q_dtype, w.q_scale, w.cache, w.kv_dtype, w.kv_scale,
                        w.block_table, w.seq_lens, w.softmax_scale, block_size=w.block_size,
                        qo_indptr=w.qo_indptr, sinks=w.sinks, tokens=tokens)


def assert_close(out, lse, ref_out, ref_lse, dtype="bf16", what="", tol=None):
    tol = TOL_OUT[dtype] if tol is None else tol
    assert out.shape == ref_out.shape, (out.shape, ref_out.shape)
    assert np.isfinite(out).all(), f"{what}: non-finite output"
    err = float(np.max(np.abs(out - ref_out))) if out.size else 0.0
    assert err <= tol, f"{what}: max |out - oracle| = {err:.3e} > {tol}"
    ninf = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), ninf), f"{what}: -inf lse pattern differs"
    assert not np.isnan(lse).any(), f"{what}: NaN lse"
    if (~ninf).any():
        lerr = float(np.max(np.abs(lse[~ninf] - ref_lse[~ninf])))
        assert lerr <= TOL_LSE, f"{what}: max |lse - oracle| = {lerr:.3e} > {TOL_LSE}"
    return err
