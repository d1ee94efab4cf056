"""attn_fwd_host (host buffers, copies overlapped with the kernels) gives the
same bits as attn_fwd on device buffers."""
import pytest
import torch

import attn_inputs as I

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def attn():
    import online_softmax_fwd_gb300 as a
    a.lib()
    return a


@pytest.mark.parametrize("shape,causal", [((1, 2, 256, 64), False), ((2, 3, 1000, 128), True),
                                          ((1, 9, 300, 64), True), ((4, 16, 4096, 128), False)],
                         ids=lambda x: str(x))
def test_host_path_matches_device_path(attn, shape, causal):
    B, H, N, d = shape
    q, k, v = (I.to_bf16(x).pin_memory() for x in I.draw_fp32(B, H, N, d, seed=B * H + N))
    o_dev, lse_dev = attn.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal)
    torch.cuda.synchronize()
    ws = {}
    for _ in range(2):  # a second call reuses the workspace and the library's streams
        o_h, lse_h = attn.attn_fwd_from_host(q, k, v, causal=causal, workspace=ws)
        assert torch.equal(o_h, o_dev.cpu()) and torch.equal(lse_h, lse_dev.cpu())
    assert attn.device_status() == attn.Status.OK


def test_host_path_ordered_after_queued_work(attn):
    # the host call must start after work already queued on the caller's stream
    B, H, N, d = 1, 4, 512, 128
    q, k, v = (I.to_bf16(x).pin_memory() for x in I.draw_fp32(B, H, N, d, seed=1))
    big = torch.randn(4096, 4096, device=DEV)
    for _ in range(4):
        big = big @ big / 64.0      # keep the stream busy
    o_h, lse_h = attn.attn_fwd_from_host(q, k, v, causal=True)
    o_dev, lse_dev = attn.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_dev.cpu())
