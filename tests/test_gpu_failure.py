"""Failure detection on the GPU without a fault: a bounded pipeline wait runs
out, the kernel winds down and reports MOE_STATUS_TIMEOUT, and the context
stays usable.

The decode path's gate/up weight producer is told to skip one ring stage
(moe_options.debug_drop_stage): it neither copies the stage nor arrives on
the stage's barrier, so the consumers' wait for it can never complete.  The
wait limit is shortened to tens of microseconds for that call
(moe_options.debug_wait_timeout_us), so the kernels give up quickly: every
wait is bounded, the producer lets the copies it did issue land before its
CTA exits, and the decode kernels hold no tensor memory.  The host then reads
the status, and a normal forward on the same stream must still match the
oracle."""
import numpy as np
import pytest
import torch

from block_fp8_mixture_route_gb300 import _lib, api, synthetic as syn
from oracle import moe_oracle as mo

from helpers import TOL, check_per_token, oracle_args

pytestmark = pytest.mark.gpu


def _problem(T, step):
    shape = syn.DECODE_SMALL
    w13, w13s, w2, w2s = syn.make_weights(shape, 0, "cuda")
    ids, w = syn.make_routing(T, shape.E, shape.k, 0, "cuda", "softmax", step=step)
    return dict(hidden=syn.make_hidden(T, shape.H, 0, "cuda", step), topk_ids=ids, topk_weights=w, w13=w13,
                w13_scale=w13s, w2=w2, w2_scale=w2s)


@pytest.mark.parametrize("drop", [1, 3])
def test_dropped_stage_times_out_and_the_stream_recovers(cuda_lib, drop):
    prob = _problem(4, step=drop)
    s = torch.cuda.Stream()
    api.moe_fp8_block_device_status(stream=s)            # start from a clear status word
    out = torch.zeros(4, syn.DECODE_SMALL.H, dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(s):
        api.forward_problem(prob, out=out, stream=s, force_path="decode", debug_wait_timeout_us=50,
                            debug_drop_stage=drop)
    st = api.moe_fp8_block_device_status(stream=s)       # synchronises the stream: the kernels returned
    assert st & _lib.MOE_STATUS_TIMEOUT, st
    assert api.moe_fp8_block_device_status(stream=s) == 0   # reading clears it
    # the context and the workspace are usable: a normal forward on the same stream
    with torch.cuda.stream(s):
        good = api.forward_problem(prob, stream=s, force_path="decode")
    s.synchronize()
    assert api.moe_fp8_block_device_status(stream=s) == 0
    args, _ = oracle_args(prob)
    assert check_per_token(good.float().cpu().numpy(), mo.forward(*args)) < TOL


def test_short_limit_alone_changes_nothing(cuda_lib):
    """A shortened limit without a dropped stage: every wait completes long
    before 20 ms, so the forward is correct and the status stays clear."""
    prob = _problem(8, step=5)
    api.moe_fp8_block_device_status()
    out = api.forward_problem(prob, force_path="decode", debug_wait_timeout_us=20000)
    torch.cuda.synchronize()
    assert api.moe_fp8_block_device_status() == 0
    args, _ = oracle_args(prob)
    assert check_per_token(out.float().cpu().numpy(), mo.forward(*args)) < TOL
