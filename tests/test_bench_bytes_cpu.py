"""The algorithmic byte model behind bench.py's roofline numbers, on the CPU.

Each case is the one a committed ncu capture covers (profiles/traffic.txt),
with its routed-expert count as the capture's comment states it.  The
expected bytes are written out term by term from the definition: what a
launch must read and write at least (the routed experts' e4m3 weights and
valid bf16 block scales, its activation inputs once, its outputs once)."""
import os

import pytest

import bench
from block_fp8_mixture_route_gb300 import synthetic as syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# workload of each capture: (shape, T, routed experts D)
CASES = {
    "decode_small_T16": (syn.DECODE_SMALL, 16, 90),
    "wide_T16": (syn.DECODE_WIDE, 16, 109),
    "prefill_T4096": (syn.PREFILL, 4096, 128),
}

# term by term: weights, valid scales (2 B each), inputs, outputs
HAND = {
    ("decode_gemm1_kernel", "decode_small_T16"):
        90 * 2 * 512 * 2048 + 90 * 2 * (8 * 16) + 2 * 16 * 2048 + 4 * 128 * 512,
    ("decode_gemm2_kernel", "decode_small_T16"):
        90 * 2048 * 512 + 90 * 2 * (16 * 4) + 4 * 128 * 512 + 4 * 128 * 2048,
    ("prefill_gemm_kernel<1>", "wide_T16"):
        109 * 2 * 2048 * 7168 + 109 * 2 * (32 * 56) + 128 * 7168 + 128 * 2048 + 4 * 128 * (56 + 16),
    ("prefill_gemm_kernel<2>", "wide_T16"):
        109 * 7168 * 2048 + 109 * 2 * (56 * 16) + 128 * 2048 + 2 * 128 * 7168 + 4 * 128 * 16,
    ("prefill_gemm_kernel<1>", "prefill_T4096"):
        128 * 2 * 512 * 2048 + 128 * 2 * (8 * 16) + 32768 * 2048 + 32768 * 512 + 4 * 32768 * (16 + 4),
    ("prefill_gemm_kernel<2>", "prefill_T4096"):
        128 * 2048 * 512 + 128 * 2 * (16 * 4) + 32768 * 512 + 2 * 32768 * 2048 + 4 * 32768 * 4,
}


@pytest.mark.parametrize("kernel,case", sorted(HAND))
def test_kernel_bytes_by_hand(kernel, case):
    shape, T, D = CASES[case]
    assert bench.kernel_bytes(kernel, shape, T, D) == HAND[(kernel, case)]


def test_routed_bytes_per_expert():
    # gate/up and down weights plus their valid block scales
    assert bench.routed_per_expert(syn.DECODE_SMALL) == 2 * 512 * 2048 + 2048 * 512 + 2 * (8 * 16) + 2 * (16 * 4)
    assert bench.routed_per_expert(syn.DECODE_SMALL) == 3_146_112
    # the padded skewed layer: scale padding is not streamed bytes
    assert bench.routed_per_expert(syn.PADDED_SKEWED) == 3 * 2560 * 640 + 2 * (10 * 20) + 2 * (20 * 5)


def test_committed_traffic_lines_use_the_same_model():
    """Every line of profiles/traffic.txt carries the algorithmic bytes of
    its case as the model computes them, and DRAM bytes close to them (a
    capture far above the model would mean re-reads; far below, a wrong
    case)."""
    seen = 0
    for line in open(os.path.join(ROOT, "profiles", "traffic.txt")):
        f = line.split()
        if not f or line.startswith("#"):
            continue
        kernel, case, dram, alg, src = f[0], f[1], int(f[2]), int(f[3]), f[4]
        shape, T, D = CASES[case]
        assert alg == bench.kernel_bytes(kernel, shape, T, D), line
        assert alg == HAND[(kernel, case)], line
        assert 0.8 < dram / alg < 1.1, line
        assert os.path.exists(os.path.join(ROOT, "block_fp8_mixture_route_gb300", "csrc", src)), line
        seen += 1
    assert seen == len(HAND)
