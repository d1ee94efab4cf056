"""Failure detection on the GPU without a fault: a bounded wait that runs out.

attn_selftest_wait_timeout runs the kernels' own bounded-wait function on
mbarriers that nothing completes. The wait must give up after its limit,
record ATTN_ERR_TIMEOUT in the device status word (which attn_get_device_status
reports once and clears), make the block's other waiter return early through
the abort flag, and leave the context usable for the next attention call.
"""
import numpy as np
import pytest
import torch

import attn_inputs as I
from oracle.attention import attention_fwd
from parity import compare

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def attn():
    import online_softmax_fwd_gb300 as a
    a.lib()
    return a


def test_bounded_wait_times_out_and_the_context_survives(attn):
    lib = attn.lib()
    torch.cuda.synchronize()
    assert attn.device_status() == attn.Status.OK
    limit = 20_000_000                       # ~10 ms at the 2 GHz class SM clock
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    assert lib.attn_selftest_wait_timeout(limit, s.cuda_stream) == 0
    e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    assert attn.device_status() == attn.Status.TIMEOUT
    assert attn.device_status() == attn.Status.OK          # reported once, then cleared
    # about one limit (20M cycles: 9-20 ms at 1-2.2 GHz); the second waiter
    # (64x the limit, >= 0.58 s) must have left through the abort flag
    assert 20_000_000 / 2.2e9 * 1e3 <= ms < 150, ms
    # the context keeps working
    q, k, v = (I.to_bf16(x) for x in I.draw_fp32(1, 2, 300, 64, seed=9))
    o, lse = attn.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
    torch.cuda.synchronize()
    assert attn.device_status() == attn.Status.OK
    o_ref, lse_ref = attention_fwd(I.as_f64(q), I.as_f64(k), I.as_f64(v), True, 64 ** -0.5)
    compare(I.as_f64(o.cpu()), lse.cpu().double().numpy(), o_ref, lse_ref, "after a timeout")
