"""Parity of the backward pass (attn_bwd, through the C ABI) against the
float64 oracle. The forward's O and LSE that the backward consumes come from
the oracle too (O rounded to bf16, LSE to fp32), so both sides start from the
same inputs.

Two references, both float64 from the oracle:
  * the exact gradient. The kernel rounds P to bf16 before dV = P^T dO and
    dS = P (dP - D), and dS to bf16 before dK and dQ, each a relative error of
    at most 2^-8; an output element then moves by at most 2^-7 times the same
    product over absolute values (A = |P|^T |dO| for dV, s |dS|^T |Q| for dK,
    s |dS| |K| for dQ), and the bf16 output adds half an ulp. Allowed, with a
    factor two: |x - x_ref| <= 2^-6 A + ulp_bf16(x_ref) + 1e-4.
  * the same method with P and dS rounded to bf16 where the kernel rounds them
    (the oracle's p_cast / ds_cast). What is left is the output's rounding
    (half an ulp, 0.29 ulp r.m.s.), fp32 accumulation and the rare P or dS
    value whose fp32 and float64 forms round to different bf16 neighbours (one
    bf16 step, 2^-8 of one term). Allowed: |x - x_emu| <= ulp_bf16(x_emu) +
    2^-7 A + 1e-5 elementwise and, over each output, an r.m.s. error at most
    the r.m.s. of ulp_bf16(x_emu) -- a missing or doubled block of terms moves
    the r.m.s. by far more than that.
"""
import numpy as np
import pytest
import torch

import attn_inputs as I
from oracle.attention import attention_fwd
from oracle.backward import attention_bwd_abs_head, attention_bwd_head
from parity import bf16_ulp, sample_rows

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def attn():
    import online_softmax_fwd_gb300 as a
    a.lib()
    return a


def inputs(B, H, N, d, causal, scale, qk_std=1.0, seed=0):
    q, k, v = (I.to_bf16(x) for x in I.draw_fp32(B, H, N, d, qk_std=qk_std, seed=seed))
    do = I.to_bf16(I.draw_grad(B, H, N, d, seed=seed + 1))
    o_ref, lse_ref = attention_fwd(I.as_f64(q), I.as_f64(k), I.as_f64(v), causal, scale)
    o = torch.from_numpy(o_ref).to(torch.bfloat16)
    lse = torch.from_numpy(lse_ref).to(torch.float32)
    return q, k, v, o, do, lse


def run(attn, q, k, v, o, do, lse, causal, scale):
    dq, dk, dv = attn.attn_bwd(*(t.to(DEV) for t in (q, k, v, o, do, lse)), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert attn.device_status() == attn.Status.OK
    return I.as_f64(dq), I.as_f64(dk), I.as_f64(dv)


def check(got, ref, absref, what):
    err = np.abs(got - ref)
    bound = 2.0 ** -6 * absref + bf16_ulp(ref) + 1e-4
    assert np.isfinite(got).all(), f"{what}: non-finite"
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements beyond the bound; max err {err.max():.4g}, "
                           f"worst ratio {(err / bound).max():.3g}")
    return float(err.max())


def to_bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).double().numpy()


def check_emulated(got, emu, absref, what):
    err = np.abs(got - emu)
    ulp = bf16_ulp(emu)
    bound = ulp + 2.0 ** -7 * absref + 1e-5
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements beyond the bound (bf16 method); max err "
                           f"{err.max():.4g}, worst ratio {(err / bound).max():.3g}")
    rms, rms_ulp = np.sqrt((err ** 2).mean()), np.sqrt((ulp ** 2).mean())
    assert rms <= rms_ulp, f"{what}: r.m.s. error {rms:.3g} above the r.m.s. ulp {rms_ulp:.3g} (bf16 method)"


def check_head(got, args, causal, scale, what, rows=None):
    """got = (dq, dk, dv) of one head; args = (q, k, v, o, do, lse) float64 of that head."""
    ref = attention_bwd_head(*args, causal, scale)
    emu = attention_bwd_head(*args, causal, scale, p_cast=to_bf16, ds_cast=to_bf16)
    absref = attention_bwd_abs_head(*args, causal, scale)
    for name, g, r, m, a in zip(("dQ", "dK", "dV"), got, ref, emu, absref):
        if rows is not None:
            g, r, m, a = g[rows], r[rows], m[rows], a[rows]
        check(g, r, a, f"{what} {name}")
        check_emulated(g, m, a, f"{what} {name}")


SHAPES = [(1, 1, 1, 64), (1, 2, 128, 64), (1, 1, 129, 128), (1, 2, 256, 128), (2, 1, 300, 64), (1, 1, 384, 128),
          (1, 2, 1000, 128), (1, 1, 1024, 64)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes(attn, shape, causal):
    B, H, N, d = shape
    scale = d ** -0.5
    q, k, v, o, do, lse = inputs(B, H, N, d, causal, scale, seed=N + d)
    got = run(attn, q, k, v, o, do, lse, causal, scale)
    f64 = [I.as_f64(t) if t.dtype == torch.bfloat16 else t.double().numpy() for t in (q, k, v, o, do, lse)]
    for b in range(B):
        for h in range(H):
            check_head([g[b, h] for g in got], [x[b, h] for x in f64], causal, scale, f"{shape} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_peaked_rows(attn, causal):
    # Q, K ~ N(0, 2^2): P has a few dominant keys per row
    B, H, N, d = 1, 2, 512, 128
    scale = d ** -0.5
    q, k, v, o, do, lse = inputs(B, H, N, d, causal, scale, qk_std=2.0, seed=11)
    got = run(attn, q, k, v, o, do, lse, causal, scale)
    f64 = [I.as_f64(t) if t.dtype == torch.bfloat16 else t.double().numpy() for t in (q, k, v, o, do, lse)]
    for h in range(H):
        check_head([g[0, h] for g in got], [x[0, h] for x in f64], causal, scale, f"peaked causal={causal} h={h}")


def test_long_sequence_sampled(attn):
    # N = 4096 at d = 128 (32 key tiles, 32 query tiles per CTA), checked on sampled rows
    B, H, N, d = 1, 2, 4096, 128
    scale = d ** -0.5
    for causal in (False, True):
        q, k, v, o, do, lse = inputs(B, H, N, d, causal, scale, seed=5)
        got = run(attn, q, k, v, o, do, lse, causal, scale)
        f64 = [I.as_f64(t) if t.dtype == torch.bfloat16 else t.double().numpy() for t in (q, k, v, o, do, lse)]
        rows = sample_rows(N, np.random.default_rng(7))
        for h in range(H):
            check_head([g[0, h] for g in got], [x[0, h] for x in f64], causal, scale,
                       f"N=4096 causal={causal} h={h}", rows=rows)


def test_repeated_calls_identical_dk_dv(attn):
    # dK and dV are plain sums inside one CTA: bit-identical from call to call
    B, H, N, d = 1, 2, 640, 64
    q, k, v, o, do, lse = inputs(B, H, N, d, True, d ** -0.5, seed=2)
    a = run(attn, q, k, v, o, do, lse, True, d ** -0.5)
    b = run(attn, q, k, v, o, do, lse, True, d ** -0.5)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])


@pytest.mark.parametrize("name", ["bwd_bf16_b4h16n4096d128", "bwd_bf16_causal_b2h16n8192d128_qk2"])
def test_full_workload_sampled(attn, name):
    # the benchmark's workload at full size and in its launch configuration
    # (O and LSE from attn_fwd, as there), sampled rows of the first and the
    # last head against both oracles
    w = I.WORKLOADS[name]
    q, k, v = I.bf16_qkv(w)
    do = I.to_bf16(I.draw_grad(w.B, w.H, w.N, w.d, seed=w.seed + 1))
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    o, lse = attn.attn_fwd(qd, kd, vd, causal=w.causal, scale=w.scale)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, o, dod, lse, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert attn.device_status() == attn.Status.OK
    got = [I.as_f64(x.cpu()) for x in (dq, dk, dv)]
    f64 = [I.as_f64(x) for x in (q, k, v)] + [I.as_f64(o.cpu()), I.as_f64(do), lse.double().cpu().numpy()]
    rows = sample_rows(w.N, np.random.default_rng(9))
    for b, h in ((0, 0), (w.B - 1, w.H - 1)):
        check_head([g[b, h] for g in got], [x[b, h] for x in f64], w.causal, w.scale, f"{name} head ({b},{h})",
                   rows=rows)
