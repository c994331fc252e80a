"""Decode context parallelism emulated on one GPU, all through the C ABI:
the KV of every request is split round-robin over W "ranks" (token p on rank
p % W); each rank's positions go through mla_sparse_index_convert and a
sparse mla_decode_fwd without sinks; mla_merge_lse combines the W (out, lse)
pairs and folds the sinks once. The result must match the oracle's unsplit
decode."""
import numpy as np
import pytest
import torch

import oracle as O
from paged_mla_decode_06_gb300 import binding as B
from paged_mla_decode_06_gb300 import build as BUILD
from paged_mla_decode_06_gb300 import inputs as I
from tests.gpu_helpers import assert_close, visible_keys

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    BUILD.build()
    B.load_library()


def _shard_decode(w, dw, world, rank, kernel):
    dev = dw.device
    idx, req = I.dcp_shard_positions(w, world, rank)
    T, K = idx.shape
    slots = torch.empty((T, K), dtype=torch.int32, device=dev)
    B.mla_sparse_index_convert(torch.from_numpy(req).to(dev), dw.block_table,
                               torch.from_numpy(idx).to(dev), block_size=w.block_size, out=slots)
    prob = B.make_problem(num_tokens=T, num_heads=w.num_heads, block_size=w.block_size,
                          num_blocks=w.num_blocks, topk=K, dtype=w.kv_dtype, kernel=kernel)
    plan = B.mla_decode_plan(prob)
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty((T, w.num_heads, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, w.num_heads), dtype=torch.float32, device=dev)
    B.mla_decode_fwd(plan, dw.q, dw.cache, sparse_slots=slots, softmax_scale=w.softmax_scale,
                     q_scale=w.q_scale, kv_scale=w.kv_scale, workspace=ws, out=out, lse=lse)
    return out, lse


@pytest.mark.parametrize("kernel", [B.MLA_KERNEL_WARP_MMA, B.MLA_KERNEL_TCGEN05],
                         ids=["mma", "tcgen05"])
@pytest.mark.parametrize("world", [1, 2, 4])
def test_round_robin_shards_merge_on_gpu(world, kernel):
    w = I.build_dense(70 + world, seq_lens=[1, 3, 64, 200, 1000, 1537], num_heads=64,
                      block_size=64, with_sinks=True)
    dw = B.DeviceWorkload(w, plan=False)
    outs, lses = [], []
    for rank in range(world):
        o, l = _shard_decode(w, dw, world, rank, kernel)
        outs.append(o)
        lses.append(l)
    so = torch.stack(outs).contiguous()
    sl = torch.stack(lses).contiguous()
    B.mla_merge_lse(so, sl, sinks=dw.sinks, out=dw.out, lse=dw.lse)
    torch.cuda.synchronize()
    ref_o, ref_l = O.mla_decode(w.q, "bf16", 1.0, w.cache, "bf16", 1.0, w.block_table,
                                w.seq_lens, w.softmax_scale, sinks=w.sinks)
    # rows of 1 and 3 keys get the few-key bound, the others the workload bound
    assert_close(dw.out.float().cpu().numpy(), dw.lse.cpu().numpy(), ref_o, ref_l, "bf16",
                 f"dcp x{world}", keys=visible_keys(w))


def test_merge_lse_kernel_matches_oracle():
    rng = np.random.default_rng(0)
    W, T, H = 3, 5, 7
    so = rng.standard_normal((W, T, H, 512)).astype(np.float32)
    sl = (rng.standard_normal((W, T, H)) * 3).astype(np.float32)
    sl[1, 2, :] = -np.inf
    sl[:, 4, 0] = -np.inf
    so_bf = torch.from_numpy(so).to(torch.bfloat16)
    sinks = rng.standard_normal(H).astype(np.float32)
    for sk in (None, sinks):
        ref_o, ref_l = O.merge_lse_shards(so_bf.float().numpy(), sl, sinks=sk)
        dev = torch.device("cuda")
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
        B.mla_merge_lse(so_bf.to(dev), torch.from_numpy(sl).to(dev),
                        sinks=None if sk is None else torch.from_numpy(sk).to(dev),
                        out=out, lse=lse)
        torch.cuda.synchronize()
        assert_close(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, "bf16",
                     "merge_lse")
