"""fp64 CPU oracle for paged MLA decode.

TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. It shares no code
with the CUDA library and imports nothing from it.
"""
from .mla_oracle import (  # noqa: F401
    HEAD_DIM, KV_LORA_RANK, LOG2E, LN2,
    attend, concat_quant_q, decode_bf16, decode_e4m3fn, encode_e4m3fn, dense_slots, dequantize, index_convert,
    merge_lse_shards, merge_segments, mla_decode, partition_lengths, round_robin_positions,
    segment_bounds,
    segment_partials, tile_size_for_block, token_layout, visible_len, sparse_seqlen,
    fit_kpool_indices,
)
