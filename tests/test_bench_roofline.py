"""Host logic of the benchmark's roofline record: algorithmic bytes and flops
of a decode launch, the dtype's tensor peak, and the choice of bound."""
import bench
from paged_mla_decode_06_gb300 import inputs as I

PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


def test_algorithmic_units_count_each_key_once():
    w = I.build_dense(1, seq_lens=[100, 64], num_heads=8, block_size=64)
    # 164 keys x 1152 B + q (2 x 8 x 1152 B) + 3 block-table entries + 2 lengths
    assert bench._alg_bytes_decode(w) == 164 * 1152 + 2 * 8 * 1152 + 3 * 4 + 2 * 4
    assert bench._flops(w) == 164 * 8 * 2176.0
    # causally hidden keys carry no flops: a 3-token request of 10 keys sees 8 + 9 + 10
    m = I.build_dense(2, seq_lens=[10], num_heads=4, block_size=64, qlens=[3])
    assert bench._flops(m) == (8 + 9 + 10) * 4 * 2176.0


def test_e4m3_peak_is_twice_the_bf16_peak():
    assert bench.tensor_peak_tflops(PEAKS, "bf16") == 1900.0
    assert bench.tensor_peak_tflops(PEAKS, "fp8") == 3800.0


def test_bound_follows_bytes_against_flops():
    # 16 heads of e4m3: far more bytes than flops per unit time -> HBM
    few = I.build_dense(3, seq_lens=[4096] * 2, num_heads=16, block_size=64, dtype="fp8")
    r = bench.roofline_of(few, 10.0, PEAKS)
    assert r["bound"] == "hbm"
    assert abs(r["hbm_frac"] - r["hbm_gbs"] / PEAKS["hbm_gbs"]) < 1e-12
    # 128 heads x 4 tokens of bf16: 4 x 242 flop per byte -> tensor
    many = I.build_dense(4, seq_lens=[2048] * 2, num_heads=128, block_size=64, qlens=[4, 4])
    r = bench.roofline_of(many, 10.0, PEAKS)
    assert r["bound"] == "tensor"
    assert abs(r["tensor_frac"] - r["tensor_tflops"] / 1900.0) < 1e-12
