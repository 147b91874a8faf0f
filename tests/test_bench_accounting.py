"""The roofline accounting of bench.py against figures worked out by hand from the
method's cost model (the chunked-attention cost 2 L d^2 + 2 L C d per product kind of
"22580: от GPT-2 до Kimi K3", the chunked DeltaNet section) and the tensor sizes of the
workloads: these are the numbers the reported fractions divide by."""
import bench


def test_prefill_bytes_and_flops_per_token_head():
    # bf16, d = 128, one log alpha per key channel: q, k, g, v (4 x 256 B), beta (2 B),
    # o (256 B) per token-head; 6 d^2 + 10 C d flops
    b, f = bench.algorithmic_prefill(1, 0, 128, 128, 2)
    assert b == 1282 and f == 180_224
    # the state is read and written once per (sequence, head), in fp32
    b, _ = bench.algorithmic_prefill(0, 1, 128, 128, 2)
    assert b == 2 * 4 * 128 * 128
    # the gate layouts change only the g term
    assert bench.algorithmic_prefill(1, 0, 128, 128, 2, gate="scalar")[0] == 1282 - 254
    assert bench.algorithmic_prefill(1, 0, 128, 128, 2, gate="none")[0] == 1282 - 256


def test_workload_rooflines():
    hbm, tflops = 6774.9e9, 1868.9e12
    # 4 x 4096 tokens, 16 heads: 3.445e8 bytes, an HBM-bound 50.8 us
    b, f = bench.algorithmic_prefill(4 * 4096 * 16, 4 * 16, 128, 128, 2)
    assert abs(b - 3.445e8) / 3.445e8 < 1e-3
    assert abs(b / hbm - 50.85e-6) < 0.05e-6 and f / tflops < b / hbm
    # 1 x 65536 tokens, 32 heads: 2.693e9 bytes, 397.5 us
    b, f = bench.algorithmic_prefill(65536 * 32, 32, 128, 128, 2)
    assert abs(b - 2.693e9) / 2.693e9 < 1e-3 and abs(b / hbm - 397.5e-6) < 0.5e-6
    # one decode step, 256 x 32 sequence-heads: 1.084e9 bytes, 160.0 us
    d = bench.algorithmic_decode(256 * 32, 128, 128, 2)
    assert abs(d - 1.084e9) / 1.084e9 < 1e-3 and abs(d / hbm - 160.0e-6) < 0.1e-6


def test_aggregate_throughput_counts_every_rank():
    # 16384 tokens per rank in 0.25 ms on each of 4 ranks: 4 x 65.5 M tokens/s
    assert abs(bench.aggregate_throughput(16384, 4, 0.25) - 4 * 16384 / 0.25e-3) < 1e-3
