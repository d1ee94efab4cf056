"""Parity of the CUDA path (through the C ABI) against the float64 oracle.

Small shapes are compared element by element: several 128-row tiles, ragged
tails, N = 1, both head dims, causal and not, every software-exp2 share, tau
0 and 8, and degenerate inputs. The three bf16 long-sequence workloads run at
full size in the launch configuration the benchmark times, checked on sampled
rows that the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import attn_inputs as I
from oracle.attention import attention_fwd, attention_rows
from parity import compare, compare_heads, method_reference, sample_rows

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
# the software exp2's largest relative error over the softmax range ("FlashAttention-4's
# Softmax Tricks", section "The emulated exp2": 8.77e-5 for degree 3), rounded up
EMU_REL_ERR = 1e-4


@pytest.fixture(scope="module")
def attn():
    import online_softmax_fwd_gb300 as a
    a.lib()
    return a


def run(attn, q, k, v, causal, scale, **kw):
    o, lse = attn.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=scale, **kw)
    torch.cuda.synchronize()
    assert attn.device_status() == attn.Status.OK
    return o.cpu(), lse.cpu()


def check_full(attn, q, k, v, causal, scale, what, **kw):
    """Every element against the exact oracle: 1e-2, except where the method
    at the kernel's precision (the recurrence with the kernel's tau, P rounded
    to bf16) is itself more than 1e-2 from the exact result; there the element
    is held to the method's tight bound (``parity.compare_heads``)."""
    o, lse = run(attn, q, k, v, causal, scale, **kw)
    qq, kk, vv = I.as_f64(q), I.as_f64(k), I.as_f64(v)
    o_ref, lse_ref = attention_fwd(qq, kk, vv, causal, scale)
    return compare_heads(I.as_f64(o), lse.double().numpy(), o_ref, lse_ref, qq, kk, vv, causal, scale,
                         kw.get("tau", 8.0), what, exp_rel_err=EMU_REL_ERR if kw.get("exp2_emu16") else 2.0 ** -21)


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_workload(attn, causal):
    w = I.TINY
    q, k, v = I.bf16_qkv(w)
    st = check_full(attn, q, k, v, causal, w.scale, f"{w.name} causal={causal}")
    assert st["o_over_1e-2"] == 0 and st["floor_exceptions"] == 0


SMALL = [(1, 1, 1, 64), (1, 1, 7, 128), (1, 2, 128, 64), (1, 1, 129, 128), (2, 3, 255, 64), (1, 2, 256, 128),
         (1, 2, 257, 64), (1, 1, 300, 128), (2, 2, 640, 64), (1, 2, 1000, 128), (1, 1, 1024, 64)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes(attn, shape, causal):
    B, H, N, d = shape
    q, k, v = (I.to_bf16(x) for x in I.draw_fp32(B, H, N, d, seed=N + d))
    check_full(attn, q, k, v, causal, d ** -0.5, f"{shape} causal={causal}")


@pytest.mark.parametrize("emu", [1, 2, 3, 4])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_software_exp2_shares(attn, emu, d, causal):
    q, k, v = (I.to_bf16(x) for x in I.draw_fp32(1, 3, 1000, d, seed=5))
    check_full(attn, q, k, v, causal, d ** -0.5, f"emu={emu} d={d}", exp2_emu16=emu)


@pytest.mark.parametrize("tau", [0.0, 4.0, 8.0, 16.0])
def test_rescale_thresholds(attn, tau):
    # Q, K ~ N(0, 2^2): the running max keeps growing along the keys. With
    # tau > 0 the method itself (float64, P rounded to bf16) is up to 0.018
    # from the exact result on the peaked rows; with tau = 0 it is within 1e-2.
    q, k, v = (I.to_bf16(x) for x in I.draw_fp32(1, 2, 1536, 128, qk_std=2.0, seed=9))
    st = check_full(attn, q, k, v, True, 128 ** -0.5, f"tau={tau}", tau=tau)
    if tau == 0.0:
        assert st["o_over_1e-2"] == 0 and st["method_floor_exceptions"] == 0


@pytest.mark.parametrize("causal", [False, True])
def test_peaked_rows_d64_large_scale(attn, causal):
    # Q, K ~ N(0, 2^2) at scale 0.37, d = 64: scaled scores with a standard
    # deviation near 12. Here the kernel's output can lie one bf16 step beyond
    # 1e-2 from the exact result where the method's own result does not (e.g.
    # 2.1875 against 2.1996 with the method at 2.2056, the kernel within the
    # method's bound); such an element is held to the method's bound.
    q, k, v = (I.to_bf16(x) for x in I.draw_fp32(1, 2, 1536, 64, qk_std=2.0, seed=9))
    check_full(attn, q, k, v, causal, 0.37, f"peaked d64 scale 0.37 causal={causal}")


def test_scores_rising_along_keys(attn):
    # a ramp along the key order makes the max grow block after block, so the
    # correction path fires many times
    q, k, v = I.draw_fp32(1, 2, 1024, 64, seed=13)
    q += 1.0
    k += np.linspace(0.0, 1.5, 1024, dtype=np.float32)[None, None, :, None]
    q, k, v = I.to_bf16(q), I.to_bf16(k), I.to_bf16(v)
    for causal in (False, True):
        check_full(attn, q, k, v, causal, 64 ** -0.5, f"ramp causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_average_values(attn, causal):
    _, k, v = (I.to_bf16(x) for x in I.draw_fp32(1, 2, 384, 64, seed=3))
    q = torch.zeros_like(k)
    o, lse = run(attn, q, k, v, causal, 0.125)
    vv = I.as_f64(v)
    n = np.arange(1, 385) if causal else np.full(384, 384)
    mean = np.cumsum(vv, axis=2) / n[None, None, :, None] if causal else np.broadcast_to(
        vv.mean(axis=2, keepdims=True), vv.shape)
    compare(I.as_f64(o), lse.double().numpy(), mean, np.broadcast_to(np.log(n), (1, 2, 384)), "zero q")


def test_large_scores(attn):
    # scaled scores with a standard deviation near 16: P spans the full range
    q, k, v = (I.to_bf16(x) for x in I.draw_fp32(1, 2, 512, 128, qk_std=4.0, seed=21))
    for causal in (False, True):
        check_full(attn, q, k, v, causal, 128 ** -0.5, f"large causal={causal}")


def test_non_default_scale(attn):
    q, k, v = (I.to_bf16(x) for x in I.draw_fp32(1, 2, 384, 64, seed=8))
    check_full(attn, q, k, v, True, 0.37, "scale 0.37")


def test_empty_problems(attn):
    for shape in ((0, 2, 128, 64), (1, 0, 128, 64), (1, 2, 0, 64)):
        q = torch.zeros(shape, dtype=torch.bfloat16, device=DEV)
        o, lse = attn.attn_fwd(q, q, q)
        assert o.shape == shape and lse.shape == shape[:3]
    assert attn.device_status() == attn.Status.OK


# The kernel is persistent: each CTA loops over work items (one pair of
# 128-row Q tiles of one head). Up to 8192 items go through a host-built work
# list; beyond that the CTAs take them in serpentine rounds. Every item must be
# computed exactly once either way: the outputs start as NaN and every row is
# compared with the oracle.
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(2, 40, 1000, 64), (1, 8193, 33, 128), (1, 4097, 260, 64)],
                         ids=["list_320_items", "rounds_8193_items", "rounds_8194_items"])
def test_every_work_item_once(attn, shape, causal):
    B, H, N, d = shape
    q, k, v = (I.to_bf16(x) for x in I.draw_fp32(B, H, N, d, seed=H + N))
    o = torch.full((B, H, N, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=DEV)
    attn.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=d ** -0.5, o=o, lse=lse)
    torch.cuda.synchronize()
    assert attn.device_status() == attn.Status.OK
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()
    qq, kk, vv = I.as_f64(q), I.as_f64(k), I.as_f64(v)
    o_ref, lse_ref = attention_fwd(qq, kk, vv, causal, d ** -0.5)
    compare_heads(I.as_f64(o.cpu()), lse.cpu().double().numpy(), o_ref, lse_ref, qq, kk, vv, causal, d ** -0.5,
                  8.0, f"{shape} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
def test_output_only_16_byte_aligned(attn, d):
    # O 16-byte but not 32-byte aligned: the epilogue falls back from 256-bit
    # to 128-bit stores; both must write the same rows
    B, H, N = 1, 2, 300
    q, k, v = (I.to_bf16(x) for x in I.draw_fp32(B, H, N, d, seed=d + 5))
    n = B * H * N * d
    buf = torch.full((n + 16,), float("nan"), dtype=torch.bfloat16, device=DEV)
    o = buf[8:8 + n].view(B, H, N, d)
    assert o.data_ptr() % 32 == 16
    lse = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    attn.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, scale=d ** -0.5, o=o, lse=lse)
    torch.cuda.synchronize()
    assert attn.device_status() == attn.Status.OK
    assert torch.isnan(buf[:8]).all() and torch.isnan(buf[8 + n:]).all()   # nothing written outside O
    qq, kk, vv = I.as_f64(q), I.as_f64(k), I.as_f64(v)
    o_ref, lse_ref = attention_fwd(qq, kk, vv, True, d ** -0.5)
    compare_heads(I.as_f64(o.cpu()), lse.cpu().double().numpy(), o_ref, lse_ref, qq, kk, vv, True, d ** -0.5, 8.0,
                  f"misaligned O d={d}")


def test_repeat_calls_are_identical(attn):
    q, k, v = (I.to_bf16(x).to(DEV) for x in I.draw_fp32(2, 2, 777, 128, seed=17))
    o1, l1 = attn.attn_fwd(q, k, v, causal=True)
    o2, l2 = attn.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("w", [I.NONCAUSAL_D128, I.CAUSAL_D128_WIDE, I.CAUSAL_D64], ids=lambda w: w.name)
def test_full_size_workloads_sampled(attn, w):
    q, k, v = I.bf16_qkv(w)
    o, lse = run(attn, q, k, v, w.causal, w.scale)
    assert torch.isfinite(lse).all()
    rng = np.random.default_rng(1)
    heads = {(0, 0), (w.B - 1, w.H - 1), (int(rng.integers(w.B)), int(rng.integers(w.H)))}
    for b, h in sorted(heads):
        rows = sample_rows(w.N, rng)
        o_ref, lse_ref = attention_rows(I.as_f64(q[b, h, rows]), I.as_f64(k[b, h]), I.as_f64(v[b, h]), rows,
                                        w.causal, w.scale)
        st = compare_heads(I.as_f64(o[b, h, rows])[None, None], lse[b, h, rows].double().numpy()[None, None],
                           o_ref[None, None], lse_ref[None, None], I.as_f64(q[b, h, rows])[None, None],
                           I.as_f64(k[b, h])[None, None], I.as_f64(v[b, h])[None, None], w.causal, w.scale, 8.0,
                           f"{w.name} b={b} h={h}", rows=rows)
        # the sampled rows of all three workloads have |O| < 4, so no element's
        # output-rounding floor exceeds 1e-2. On the unit-variance workloads every
        # element is within 1e-2; on the causal Q, K ~ N(0, 2^2) one the method
        # itself (tau = 8, P rounded to bf16) is 0.0113 from the exact result on one
        # sampled element, which is then held to the method's bound instead
        assert st["floor_exceptions"] == 0
        if w.qk_std == 1.0:
            assert st["o_over_1e-2"] == 0


@pytest.mark.parametrize("shape,causal", [((1, 1, (1 << 20) + 37, 64), True), ((1, 2, (1 << 18) + 5, 128), False)],
                         ids=["n1M_d64_causal", "n256K_d128"])
def test_long_sequences_sampled(attn, shape, causal):
    # a million keys per row (and a ragged tail): long key loops, many work
    # items per head, the last rows of the causal case see every key
    B, H, N, d = shape
    q, k, v = (I.to_bf16(x) for x in I.draw_fp32(B, H, N, d, seed=N % 1000))
    o, lse = run(attn, q, k, v, causal, d ** -0.5)
    assert torch.isfinite(lse).all()
    rng = np.random.default_rng(4)
    for b, h in {(0, 0), (B - 1, H - 1)}:
        rows = np.unique(np.concatenate([sample_rows(N, rng)[:24], [N - 1, N - 2, N // 2]]))
        o_ref, lse_ref = attention_rows(I.as_f64(q[b, h, rows]), I.as_f64(k[b, h]), I.as_f64(v[b, h]), rows,
                                        causal, d ** -0.5)
        compare_heads(I.as_f64(o[b, h, rows])[None, None], lse[b, h, rows].double().numpy()[None, None],
                      o_ref[None, None], lse_ref[None, None], I.as_f64(q[b, h, rows])[None, None],
                      I.as_f64(k[b, h])[None, None], I.as_f64(v[b, h])[None, None], causal, d ** -0.5, 8.0,
                      f"{shape} b={b} h={h}", rows=rows)


def test_exp_bound_workload_with_software_share(attn):
    w = I.CAUSAL_D64
    q, k, v = I.bf16_qkv(w)
    o, lse = run(attn, q, k, v, w.causal, w.scale, exp2_emu16=2)
    rng = np.random.default_rng(2)
    for b, h in ((0, 0), (w.B - 1, w.H - 1)):
        rows = sample_rows(w.N, rng)
        o_ref, lse_ref = attention_rows(I.as_f64(q[b, h, rows]), I.as_f64(k[b, h]), I.as_f64(v[b, h]), rows,
                                        w.causal, w.scale)
        compare_heads(I.as_f64(o[b, h, rows])[None, None], lse[b, h, rows].double().numpy()[None, None],
                      o_ref[None, None], lse_ref[None, None], I.as_f64(q[b, h, rows])[None, None],
                      I.as_f64(k[b, h])[None, None], I.as_f64(v[b, h])[None, None], w.causal, w.scale, 8.0,
                      "d64 emu2", rows=rows, exp_rel_err=EMU_REL_ERR)
