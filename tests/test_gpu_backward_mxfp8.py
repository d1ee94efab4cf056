"""Parity of the MXFP8 backward pass (attn_bwd_mxfp8, through the C ABI)
against the float64 oracle of the same method (oracle.backward's
attention_bwd_mxfp8: Q, K, V, dO in 32 x 32 blocks, P in E4M3 with the
constant 2^-8 scale for dV, dS in 32 x 32 blocks for dK and dQ). Both sides get
the same fp32 inputs (each quantises them itself, by the same rule) and the
same O (bf16) and LSE (fp32), from the float64 forward of the dequantised Q,
K, V.

What the oracle leaves to the kernel: the bf16 rounding of the outputs (half an
ulp, 0.29 ulp r.m.s.), fp32 accumulation, and the rare P or dS whose fp32 and
float64 values round to neighbouring E4M3 codes (one E4M3 step, 2^-3 of the
term) or, rarer still, a block whose fp32 and float64 maxima fall on either
side of a scale boundary. Allowed, for every element: ulp_bf16(x_emu) + 2^-2 T +
1e-5, T the output's largest single term (s |dS_ij| |K_jd| for dQ, s |dS_ij|
|Q_id| for dK, |P_ij| |dO_id| for dV, in E4M3) -- up to two terms a whole E4M3
step off; no element beyond 2^-3 times the sum of its absolute terms; and over
each output an r.m.s. error at most the r.m.s. of ulp_bf16(x_emu). A dropped,
doubled or mis-scaled block of terms moves the r.m.s. far past that. Each check
prints how many elements exceed the per-element bound (none may).
"""
import numpy as np
import pytest
import torch

import attn_inputs as I
from oracle.attention import attention_fwd
from oracle.backward import attention_bwd_mxfp8_head
from oracle.mxfp8 import p_to_mxfp8_constant, quantize_blocks
from parity import bf16_ulp, sample_rows

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def attn():
    import online_softmax_fwd_gb300 as a
    a.lib()
    return a


def inputs(B, H, N, causal, scale, qk_std=1.0, seed=0):
    """fp32 Q, K, V, dO and the bf16 O / fp32 LSE of the float64 forward of
    the dequantised Q, K, V."""
    q, k, v = I.draw_fp32(B, H, N, 128, qk_std=qk_std, seed=seed)
    do = I.draw_grad(B, H, N, 128, seed=seed + 1)
    qd, kd, vd = (quantize_blocks(x.astype(np.float64))[2] for x in (q, k, v))
    o_ref, lse_ref = attention_fwd(qd, kd, vd, causal, scale)
    o = torch.from_numpy(o_ref).to(torch.bfloat16)
    lse = torch.from_numpy(lse_ref).to(torch.float32)
    return q, k, v, do, o, lse


def run(attn, q, k, v, do, o, lse, causal, scale):
    t = [torch.from_numpy(np.ascontiguousarray(x)).to(DEV) for x in (q, k, v, do)]
    q8, q_sf = attn.mxfp8_quantize(t[0], role=2)
    k8, k_sf = attn.mxfp8_quantize(t[1], role=2)
    v8, v_sf = attn.mxfp8_quantize(t[2], role=0)
    do8, do_sf = attn.mxfp8_quantize(t[3], role=2)
    dq, dk, dv = attn.attn_bwd_mxfp8(q8, q_sf, k8, k_sf, v8, v_sf, o.to(DEV), do8, do_sf, lse.to(DEV),
                                     causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert attn.device_status() == attn.Status.OK
    return I.as_f64(dq), I.as_f64(dk), I.as_f64(dv)


def _max_products(a, b, rows):
    """For each row r in rows: max over j of a[r, j] * b[j, :] (a, b >= 0)."""
    out = np.empty((len(rows), b.shape[1]))
    for c0 in range(0, len(rows), 32):
        out[c0:c0 + 32] = (a[rows[c0:c0 + 32]][:, :, None] * b[None]).max(axis=1)
    return out


def largest_terms(q, k, v, o, do, lse, causal, scale, rows):
    """Per output element of the given rows, the largest absolute single term
    of its sum (the E4M3 values the method multiplies), and the sum of the
    absolute terms."""
    qd, kd, vd, dod = (quantize_blocks(x)[2] for x in (q, k, v, do))
    n = q.shape[0]
    p = np.exp(scale * qd @ kd.T - lse[:, None])
    if causal:
        p = np.where(np.tril(np.ones((n, n), dtype=bool)), p, 0.0)
    ds = quantize_blocks(p * (dod @ vd.T - (dod * o).sum(axis=1)[:, None]))[2]
    p8 = p_to_mxfp8_constant(p)
    aq, ak, av = np.abs(ds), np.abs(ds.T), np.abs(p8.T)
    tq = scale * _max_products(aq, np.abs(kd), rows)
    tk = scale * _max_products(ak, np.abs(qd), rows)
    tv = _max_products(av, np.abs(dod), rows)
    sq, sk, sv = scale * aq[rows] @ np.abs(kd), scale * ak[rows] @ np.abs(qd), av[rows] @ np.abs(dod)
    return (tq, tk, tv), (sq, sk, sv)


def check(got, emu, term, total, what):
    err = np.abs(got - emu)
    ulp = bf16_ulp(emu)
    assert np.isfinite(got).all(), f"{what}: non-finite"
    bound = ulp + 2.0 ** -2 * term + 1e-5
    over = err > bound
    print(f"bwd mxfp8 {what}: {int(over.sum())} of {err.size} beyond the bound, worst ratio "
          f"{(err / bound).max():.3g}, max err {err.max():.4g}")
    assert not over.any(), (f"{what}: {int(over.sum())} of {err.size} elements beyond the bound; "
                            f"max err {err.max():.4g}, worst ratio {(err / bound).max():.3g}")
    loose = ulp + 2.0 ** -3 * total + 1e-5
    assert not (err > loose).any(), f"{what}: an element beyond 2^-3 of its absolute terms ({err.max():.4g})"
    rms, rms_ulp = np.sqrt((err ** 2).mean()), np.sqrt((ulp ** 2).mean())
    assert rms <= rms_ulp, f"{what}: r.m.s. error {rms:.3g} above the r.m.s. ulp {rms_ulp:.3g}"


def check_head(got, args, causal, scale, what, rows=None):
    """got = (dq, dk, dv) of one head; args = (q, k, v, o, do, lse) float64 of that head."""
    emu = attention_bwd_mxfp8_head(*args, causal, scale)
    if rows is None:
        rows = np.arange(args[0].shape[0])
    terms, totals = largest_terms(*args, causal, scale, rows)
    for name, g, m, t, s in zip(("dQ", "dK", "dV"), got, emu, terms, totals):
        check(g[rows], m[rows], t, s, f"{what} {name}")


def f64_args(q, k, v, do, o, lse, b, h):
    return [np.asarray(q[b, h], np.float64), np.asarray(k[b, h], np.float64), np.asarray(v[b, h], np.float64),
            I.as_f64(o)[b, h], np.asarray(do[b, h], np.float64), lse.double().numpy()[b, h]]


SHAPES = [(1, 1, 1), (1, 2, 128), (1, 1, 129), (1, 2, 300), (2, 1, 512), (1, 1, 1000)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes(attn, shape, causal):
    B, H, N = shape
    scale = 128 ** -0.5
    q, k, v, do, o, lse = inputs(B, H, N, causal, scale, seed=N + 3)
    got = run(attn, q, k, v, do, o, lse, causal, scale)
    for b in range(B):
        for h in range(H):
            check_head([g[b, h] for g in got], f64_args(q, k, v, do, o, lse, b, h), causal, scale,
                       f"{shape} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_peaked_rows(attn, causal):
    # Q, K ~ N(0, 2^2): a few dominant keys per row, dS spread over many binades
    B, H, N = 1, 2, 512
    scale = 128 ** -0.5
    q, k, v, do, o, lse = inputs(B, H, N, causal, scale, qk_std=2.0, seed=11)
    got = run(attn, q, k, v, do, o, lse, causal, scale)
    for h in range(H):
        check_head([g[0, h] for g in got], f64_args(q, k, v, do, o, lse, 0, h), causal, scale,
                   f"peaked causal={causal} h={h}")


def test_quantizer_role_two_is_both_layouts(attn):
    # role 2 writes the codes of role 0 (= role 1) and both atom arrays
    x = torch.from_numpy(I.draw_fp32(1, 3, 300, 128, seed=4)[0]).to(DEV)
    c2, s2 = attn.mxfp8_quantize(x, role=2)
    c0, s0 = attn.mxfp8_quantize(x, role=0)
    c1, s1 = attn.mxfp8_quantize(x, role=1)
    torch.cuda.synchronize()
    n = s0.numel()
    assert torch.equal(c2, c0) and torch.equal(c0, c1)
    assert torch.equal(s2[:n], s0) and torch.equal(s2[n:], s1)


def test_long_sequence_sampled(attn):
    # N = 4096 (32 key tiles, up to 32 query tiles per CTA), sampled rows
    B, H, N = 1, 2, 4096
    scale = 128 ** -0.5
    for causal in (False, True):
        q, k, v, do, o, lse = inputs(B, H, N, causal, scale, seed=5)
        got = run(attn, q, k, v, do, o, lse, causal, scale)
        rows = sample_rows(N, np.random.default_rng(7))
        for h in range(H):
            check_head([g[0, h] for g in got], f64_args(q, k, v, do, o, lse, 0, h), causal, scale,
                       f"N=4096 causal={causal} h={h}", rows=rows)


def test_repeated_calls_identical_dk_dv(attn):
    # dK and dV are sums inside one CTA: bit-identical from call to call
    B, H, N = 1, 2, 640
    q, k, v, do, o, lse = inputs(B, H, N, True, 128 ** -0.5, seed=2)
    a = run(attn, q, k, v, do, o, lse, True, 128 ** -0.5)
    b = run(attn, q, k, v, do, o, lse, True, 128 ** -0.5)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])


@pytest.mark.parametrize("name", ["bwd_mxfp8_b4h16n4096d128", "bwd_mxfp8_causal_b2h16n16384d128"])
def test_full_workload_sampled(attn, name):
    # the benchmark's workload at full size and in its launch configuration
    # (O and LSE from the MXFP8 forward, as there), checked on sampled rows of
    # the first and the last head against the row-sampled oracle
    from oracle.backward import attention_bwd_mxfp8_rows
    w = I.WORKLOADS[name]
    xq, xk, xv = I.draw_fp32(w.B, w.H, w.N, w.d, w.qk_std, w.v_std, w.seed)
    xdo = I.draw_grad(w.B, w.H, w.N, w.d, seed=w.seed + 1)
    t = [torch.from_numpy(x).to(DEV) for x in (xq, xk, xv, xdo)]
    fq, fq_sf = attn.mxfp8_quantize(t[0], role=0)
    fk, fk_sf = attn.mxfp8_quantize(t[1], role=0)
    fv, fv_sf = attn.mxfp8_quantize(t[2], role=1)
    o, lse = attn.attn_fwd_mxfp8(fq, fq_sf, fk, fk_sf, fv, fv_sf, causal=w.causal, scale=w.scale)
    del fq, fq_sf, fk, fk_sf, fv, fv_sf
    q8, q_sf = attn.mxfp8_quantize(t[0], role=2)
    k8, k_sf = attn.mxfp8_quantize(t[1], role=2)
    v8, v_sf = attn.mxfp8_quantize(t[2], role=0)
    do8, do_sf = attn.mxfp8_quantize(t[3], role=2)
    dq, dk, dv = attn.attn_bwd_mxfp8(q8, q_sf, k8, k_sf, v8, v_sf, o, do8, do_sf, lse, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert attn.device_status() == attn.Status.OK
    o_h, lse_h = I.as_f64(o.cpu()), lse.double().cpu().numpy()
    rows = sample_rows(w.N, np.random.default_rng(9))
    for b, h in ((0, 0), (w.B - 1, w.H - 1)):
        args = (xq[b, h].astype(np.float64), xk[b, h].astype(np.float64), xv[b, h].astype(np.float64), o_h[b, h],
                xdo[b, h].astype(np.float64), lse_h[b, h])
        ref = attention_bwd_mxfp8_rows(*args, w.causal, w.scale, rows, rows)
        qd, kd, dod = (quantize_blocks(x)[2] for x in (args[0], args[1], args[4]))
        all_r = np.arange(len(rows))
        for what, got, want, a, m, s in (
                ("dQ", dq, ref["dq"], np.abs(ref["ds_rows"]), np.abs(kd), w.scale),
                ("dK", dk, ref["dk"], np.abs(ref["ds_cols"]), np.abs(qd), w.scale),
                ("dV", dv, ref["dv"], np.abs(ref["p_cols"]), np.abs(dod), 1.0)):
            g = I.as_f64(got[b, h].cpu())[rows]
            check(g, want, s * _max_products(a, m, all_r), s * (a @ m), f"{name} head ({b},{h}) {what}")
