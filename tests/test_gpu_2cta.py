"""The CTA-pair forward (attn_fwd_2cta: tcgen05 cta_group::2, d = 128,
non-causal) against the float64 oracle, through the C ABI.

The same gate as the 1-CTA kernel (``parity.compare_heads``): small shapes with
ragged tails across 512-row work items (a pair's two 256-row tiles), every work
item computed once on the list-scheduled and the serpentine paths (outputs
start as NaN), the non-causal d = 128 benchmark workload at full size on
sampled rows, and agreement with attn_fwd.
"""
import numpy as np
import pytest
import torch

import attn_inputs as I
from oracle.attention import attention_fwd, attention_rows
from parity import compare_heads, sample_rows

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def attn():
    import online_softmax_fwd_gb300 as a
    a.lib()
    return a


def run2(attn, q, k, v, scale, o=None, lse=None):
    o, lse = attn.attn_fwd_2cta(q.to(DEV), k.to(DEV), v.to(DEV), scale=scale, o=o, lse=lse)
    torch.cuda.synchronize()
    assert attn.device_status() == attn.Status.OK
    return o, lse


SHAPES = [(1, 1, 1, 128), (1, 2, 7, 128), (1, 2, 128, 128), (1, 1, 300, 128), (2, 3, 511, 128), (1, 2, 512, 128),
          (1, 2, 513, 128), (1, 1, 1000, 128), (2, 2, 2048, 128)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes(attn, shape):
    B, H, N, d = shape
    q, k, v = (I.to_bf16(x) for x in I.draw_fp32(B, H, N, d, seed=N + 7))
    o, lse = run2(attn, q, k, v, d ** -0.5)
    qq, kk, vv = I.as_f64(q), I.as_f64(k), I.as_f64(v)
    o_ref, lse_ref = attention_fwd(qq, kk, vv, False, d ** -0.5)
    compare_heads(I.as_f64(o.cpu()), lse.cpu().double().numpy(), o_ref, lse_ref, qq, kk, vv, False, d ** -0.5, 8.0,
                  f"2cta {shape}")


def test_peaked_rows_and_other_scale(attn):
    # Q, K ~ N(0, 2^2): the running max moves and the correction path runs
    q, k, v = (I.to_bf16(x) for x in I.draw_fp32(1, 2, 1536, 128, qk_std=2.0, seed=9))
    for scale in (128 ** -0.5, 0.37):
        o, lse = run2(attn, q, k, v, scale)
        qq, kk, vv = I.as_f64(q), I.as_f64(k), I.as_f64(v)
        o_ref, lse_ref = attention_fwd(qq, kk, vv, False, scale)
        compare_heads(I.as_f64(o.cpu()), lse.cpu().double().numpy(), o_ref, lse_ref, qq, kk, vv, False, scale, 8.0,
                      f"2cta peaked scale={scale}")


@pytest.mark.parametrize("shape", [(3, 40, 1000, 128), (1, 8193, 33, 128)], ids=["list_240_items", "rounds_8193_items"])
def test_every_work_item_once(attn, shape):
    B, H, N, d = shape
    q, k, v = (I.to_bf16(x) for x in I.draw_fp32(B, H, N, d, seed=H + N))
    o = torch.full((B, H, N, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=DEV)
    run2(attn, q, k, v, d ** -0.5, o=o, lse=lse)
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()
    qq, kk, vv = I.as_f64(q), I.as_f64(k), I.as_f64(v)
    o_ref, lse_ref = attention_fwd(qq, kk, vv, False, d ** -0.5)
    compare_heads(I.as_f64(o.cpu()), lse.cpu().double().numpy(), o_ref, lse_ref, qq, kk, vv, False, d ** -0.5, 8.0,
                  f"2cta {shape}")


def test_agrees_with_one_cta_kernel(attn):
    q, k, v = (I.to_bf16(x).to(DEV) for x in I.draw_fp32(2, 3, 1300, 128, seed=3))
    o1, l1 = attn.attn_fwd(q, k, v)
    o2, l2 = attn.attn_fwd_2cta(q, k, v)
    o3, l3 = attn.attn_fwd_2cta(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(o2, o3) and torch.equal(l2, l3)          # repeatable
    d = (o1.float() - o2.float()).abs()
    print(f"2cta vs 1-CTA: identical {torch.equal(o1, o2)}, max |diff| {d.max().item():.3g}, "
          f"pairs resident {torch.cuda.get_device_properties(0).multi_processor_count // 2} at most, "
          f"lse max |diff| {(l1 - l2).abs().max().item():.3g}")
    # the same products over the same K steps in the same order, the pair's B
    # halves only staged in two shared memories: the results are identical
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_full_size_workload_sampled(attn):
    w = I.NONCAUSAL_D128
    q, k, v = I.bf16_qkv(w)
    o, lse = (t.cpu() for t in run2(attn, q, k, v, w.scale))
    assert torch.isfinite(lse).all()
    rng = np.random.default_rng(1)
    heads = {(0, 0), (w.B - 1, w.H - 1), (int(rng.integers(w.B)), int(rng.integers(w.H)))}
    for b, h in sorted(heads):
        rows = sample_rows(w.N, rng)
        o_ref, lse_ref = attention_rows(I.as_f64(q[b, h, rows]), I.as_f64(k[b, h]), I.as_f64(v[b, h]), rows,
                                        False, w.scale)
        st = compare_heads(I.as_f64(o[b, h, rows])[None, None], lse[b, h, rows].double().numpy()[None, None],
                           o_ref[None, None], lse_ref[None, None], I.as_f64(q[b, h, rows])[None, None],
                           I.as_f64(k[b, h])[None, None], I.as_f64(v[b, h])[None, None], False, w.scale, 8.0,
                           f"2cta {w.name} b={b} h={h}", rows=rows)
        assert st["o_over_1e-2"] == 0


def test_bit_identical_to_one_cta_kernel_many_shapes_and_repeats(attn):
    # CTA 1 hands P to CTA 0 with a relaxed remote arrive (its data is TMEM,
    # ordered by the tcgen05 fences): a missed ordering would show up as a
    # product reading stale P, i.e. an output that differs from the one-CTA
    # kernel's. Many shapes (ragged tails, several items per pair, peaked
    # rows), each run three times.
    rng = np.random.default_rng(11)
    shapes = [(1, 1, 200, 128), (2, 3, 777, 128), (1, 24, 1536, 128), (4, 8, 1024, 128), (1, 150, 512, 128),
              (2, 16, 2048, 128)]
    for i, (B, H, N, d) in enumerate(shapes):
        qk_std = 2.0 if i % 2 else 1.0
        q, k, v = (I.to_bf16(x).to(DEV) for x in I.draw_fp32(B, H, N, d, qk_std=qk_std, seed=int(rng.integers(1000))))
        o1, l1 = attn.attn_fwd(q, k, v)
        for _ in range(3):
            o2, l2 = attn.attn_fwd_2cta(q, k, v)
            torch.cuda.synchronize()
            assert torch.equal(o1, o2) and torch.equal(l1, l2), f"{(B, H, N, d)}: 2-CTA output differs"
    assert attn.device_status() == attn.Status.OK
