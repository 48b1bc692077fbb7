"""Kernel-level parity on the GPU, bit-exact against the oracle: e4m3
widening, routing lists and activation quantisation codes/scales."""
import numpy as np
import pytest
import torch

from block_fp8_mixture_route_gb300 import api, synthetic as syn
from oracle import moe_oracle as mo

from helpers import bits

pytestmark = pytest.mark.gpu


def test_widen_all_codes_bit_exact(cuda_lib):
    codes = torch.arange(256, dtype=torch.uint8, device="cuda")
    got = api.moe_fp8_block_widen_e4m3(codes).cpu().numpy().astype(np.float64)
    ref = mo.e4m3_table()
    finite = np.array([b not in (0x7F, 0xFF) for b in range(256)])
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.signbit(got[finite]), np.signbit(ref[finite]))
    # odd length: the tail byte is widened too
    got3 = api.moe_fp8_block_widen_e4m3(codes[5:8]).cpu().numpy()
    assert np.array_equal(got3.astype(np.float64), ref[5:8])


def _route_case(ids: torch.Tensor, E: int):
    r = api.moe_fp8_block_route(ids.cuda(), E)
    torch.cuda.synchronize()
    ref = mo.route_lists(ids.cpu().numpy(), E)
    assert np.array_equal(r["counts"].cpu().numpy(), ref["counts"])
    assert np.array_equal(r["offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(r["perm"].cpu().numpy(), ref["perm"])
    assert np.array_equal(r["inv"].cpu().numpy(), ref["inv"])
    assert np.array_equal(r["glist"].cpu().numpy(), ref["glist"])
    assert int(r["n_distinct"].item()) == ref["D"]
    return ref


def test_route_hand_example(cuda_lib):
    ids = torch.tensor([[2, 0], [2, -1], [5, 2]], dtype=torch.int32)
    api.moe_fp8_block_device_status()
    _route_case(ids, 4)
    assert api.moe_fp8_block_device_status() & 1   # id 5 >= E flagged


@pytest.mark.parametrize("T,E,k,kind", [
    (4, 8, 2, "softmax"), (1, 128, 8, "softmax"), (16, 128, 8, "softmax"), (32, 256, 8, "hot"),
    (64, 256, 8, "softmax"), (1024, 128, 8, "zipf"), (4096, 128, 8, "softmax"), (16384, 128, 8, "zipf"),
    (3, 4096, 8, "softmax"), (777, 3000, 6, "softmax"),
])
def test_route_matches_oracle(cuda_lib, T, E, k, kind):
    ids, _ = syn.make_routing(T, E, k, seed=1, kind=kind)
    _route_case(ids, E)


def test_route_invalid_and_duplicate_ids(cuda_lib):
    g = torch.Generator().manual_seed(9)
    ids = torch.randint(-3, 70, (500, 8), generator=g, dtype=torch.int32)
    ids[0] = 5          # duplicates inside one token
    _route_case(ids, 64)


def test_route_empty(cuda_lib):
    ids = torch.zeros((0, 8), dtype=torch.int32)
    r = api.moe_fp8_block_route(ids.cuda(), 16)
    torch.cuda.synchronize()
    assert r["counts"].sum().item() == 0 and r["n_distinct"].item() == 0


@pytest.mark.parametrize("R,K", [(4, 256), (1024, 2048), (4096, 2048), (33, 7168), (16384, 2048)])
def test_act_quant_bit_exact(cuda_lib, R, K):
    x = syn.make_hidden(R, K, seed=3, device="cuda")
    codes, scales = api.moe_fp8_block_act_quant(x)
    torch.cuda.synchronize()
    rc, rs = mo.quantize_per_128(x.float().cpu().numpy())
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_act_quant_edge_groups(cuda_lib):
    x = torch.zeros(4, 384, dtype=torch.bfloat16)
    x[1, :128] = 3.0
    x[2, 128:256] = -0.5
    x[3] = torch.linspace(-1e4, 1e4, 384).to(torch.bfloat16)
    x[3, 300] = 2.0 ** -120          # tiny value in a group with a large amax
    xd = x.cuda()
    codes, scales = api.moe_fp8_block_act_quant(xd)
    rc, rs = mo.quantize_per_128(x.float().numpy())
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)
    # strided rows (row stride > K)
    big = torch.zeros(4, 512, dtype=torch.bfloat16, device="cuda")
    big[:, :384] = xd
    c2, s2 = api.moe_fp8_block_act_quant(big[:, :384])
    assert torch.equal(c2, codes) and torch.equal(s2, scales)
