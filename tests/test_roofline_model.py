"""The roofline arithmetic the benchmark and the design notes use, pinned to
the figures the pages print (tests/golden/roofline_b200.txt), and the FLOP
convention of the workloads (4 B H N^2 d, halved for causal)."""
import attn_inputs as I
from conftest import read_golden_kv


def test_tile_costs_match_the_printed_figures():
    g = read_golden_kv("roofline_b200.txt")
    M = N = d = 128
    t_mma = 4 * M * N * d / g["mma_flops_per_clk"]
    t_exp = M * N / g["ex2_per_clk"]
    assert t_mma == t_exp == g["t_cycles_128cube"]


def test_exp_to_mma_ratio_is_128_over_d():
    g = read_golden_kv("roofline_b200.txt")
    for d in (32, 64, 128, 256):
        for M, N in ((128, 128), (64, 256), (256, 128)):
            ratio = (M * N / g["ex2_per_clk"]) / (4 * M * N * d / g["mma_flops_per_clk"])
            assert abs(ratio - 128 / d) < 1e-12
            ratio_b300 = (M * N / g["ex2_per_clk_b300"]) / (4 * M * N * d / g["mma_flops_per_clk"])
            assert abs(ratio_b300 - 64 / d) < 1e-12


def test_workload_flops_convention():
    # the tile cost summed over every (query, key) pair of a head: 4 N^2 d,
    # halved under the causal mask
    assert I.NONCAUSAL_D128.flops == 4 * 4 * 16 * 4096 ** 2 * 128
    assert I.CAUSAL_D128_WIDE.flops == 4 * 2 * 16 * 8192 ** 2 * 128 / 2
    assert I.CAUSAL_D64.flops == 4 * 8 * 16 * 4096 ** 2 * 64 / 2
    assert I.MXFP8_CAUSAL.flops == 4 * 2 * 16 * 16384 ** 2 * 128 / 2
    assert abs(I.NONCAUSAL_D128.flops - 5.50e11) / 5.50e11 < 1e-3
    assert abs(I.MXFP8_CAUSAL.flops - 2.20e12) / 2.20e12 < 1e-3
