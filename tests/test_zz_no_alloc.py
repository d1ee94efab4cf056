"""attn_fwd_host_noalloc against attn_fwd_host with a caller workspace.

The no-allocation entry point is for callers that may not allocate device
memory themselves (a fixed memory budget set at start-up, or a host framework
whose allocator owns the device). Its staging buffers are one fixed array
inside the library, shared by every call on a device. Two calls in a row, on
different inputs, must each give bit-identical O and LSE, both on one stream
and on two streams with no host synchronisation between the calls (the
library orders them on the shared array itself)."""
import ctypes

import pytest
import torch

import attn_inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    import online_softmax_fwd_gb300 as a
    a.lib()
    return a


def pinned(x):
    return x.contiguous().pin_memory()


def launch_noalloc(attn, q, k, v, causal, stream):
    """One call on `stream`; returns the (pinned) outputs without waiting."""
    B, H, N, d = q.shape
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16).pin_memory()
    lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    st = attn.lib().attn_fwd_host_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                          B, H, N, d, int(causal), d ** -0.5, ctypes.c_void_p(stream.cuda_stream))
    assert st == 0
    return o, lse


def run_noalloc(attn, q, k, v, causal):
    s = torch.cuda.current_stream()
    out = launch_noalloc(attn, q, k, v, causal, s)
    s.synchronize()
    return out


@pytest.mark.parametrize("causal", [False, True])
def test_two_calls_in_a_row_match_the_workspace_entry_point(attn, causal):
    shapes = [(2, 3, 700, 128), (1, 5, 1300, 64)]
    inputs = [tuple(pinned(I.to_bf16(x)) for x in I.draw_fp32(*shp, seed=41 + i)) for i, shp in enumerate(shapes)]
    got = [run_noalloc(attn, *qkv, causal) for qkv in inputs]     # back to back
    for (q, k, v), (o, lse) in zip(inputs, got):
        o_ref, lse_ref = attn.attn_fwd_from_host(q, k, v, causal=causal)
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    assert attn.device_status() == attn.Status.OK


def test_calls_on_two_streams_do_not_race(attn):
    # both calls are issued before either finishes, on two non-blocking
    # streams: the second one's copies into the shared array must wait for the
    # first one's copies back
    shapes = [(2, 4, 1500, 128), (3, 2, 900, 64)]
    inputs = [tuple(pinned(I.to_bf16(x)) for x in I.draw_fp32(*shp, seed=61 + i)) for i, shp in enumerate(shapes)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    got = [launch_noalloc(attn, *qkv, causal, s) for qkv, s, causal in zip(inputs, streams, (True, False))]
    for s in streams:
        s.synchronize()
    for (q, k, v), (o, lse), causal in zip(inputs, got, (True, False)):
        o_ref, lse_ref = attn.attn_fwd_from_host(q, k, v, causal=causal)
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    assert attn.device_status() == attn.Status.OK
