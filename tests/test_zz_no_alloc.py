"""attn_fwd_host_noalloc (the chunk buffers in the library's fixed device
array, nothing allocated) against attn_fwd_host with a caller workspace: two
calls in a row, on different inputs, must each give bit-identical O and LSE."""
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


def run_noalloc(attn, q, k, v, causal):
    B, H, N, d = q.shape
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16).pin_memory()
    lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    s = torch.cuda.current_stream()
    st = attn.lib().attn_fwd_host_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                          B, H, N, d, int(causal), d ** -0.5, ctypes.c_void_p(s.cuda_stream))
    assert st == 0
    s.synchronize()
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_two_calls_in_a_row_match_the_workspace_entry_point(attn, causal):
    shapes = [(2, 3, 700, 128), (1, 5, 1300, 64)]
    inputs = [tuple(pinned(I.to_bf16(x)) for x in I.draw_fp32(*shp, seed=41 + i)) for i, shp in enumerate(shapes)]
    got = [run_noalloc(attn, *qkv, causal) for qkv in inputs]     # back to back
    for (q, k, v), (o, lse) in zip(inputs, got):
        o_ref, lse_ref = attn.attn_fwd_from_host(q, k, v, causal=causal)
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    assert attn.device_status() == attn.Status.OK
