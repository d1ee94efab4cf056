"""attn_combine (the merge of attention results over disjoint key sets)
against the float64 oracle, through the C ABI.

The merge itself is checked against ``oracle.attention.combine_partials`` on
the same bf16 partial outputs (its only roundings are the fp32 sums and the
bf16 output: within one bf16 step), including rows without keys, 1 to 40 parts
and both head dims; one part is returned bit for bit. Then a sequence split as
a context-parallel ring would do it, emulated on one GPU: the sequence is cut
into equal chunks, each (query chunk, key chunk) pair is an attn_fwd call
(causal on the diagonal chunk, skipped above it), and the merged rows are held
to the same gate as attn_fwd against the exact oracle over the whole sequence.
"""
import numpy as np
import pytest
import torch

import attn_inputs as I
from oracle.attention import attention_fwd, attention_rows, combine_partials
from parity import bf16_ulp, compare, sample_rows

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def attn():
    import online_softmax_fwd_gb300 as a
    a.lib()
    return a


@pytest.mark.parametrize("parts", [1, 2, 3, 33, 40])
@pytest.mark.parametrize("d", [64, 128])
def test_merge_matches_oracle(attn, parts, d):
    rng = np.random.default_rng(parts * 7 + d)
    B, H, N = 2, 3, 77
    o_parts = I.to_bf16(rng.standard_normal((parts, B, H, N, d)).astype(np.float32))
    lse = (rng.standard_normal((parts, B, H, N)) * 3.0).astype(np.float32)
    if parts > 1:
        lse[rng.random((parts, B, H, N)) < 0.2] = -np.inf      # parts without keys for some rows
        lse[:, 0, 0, 5] = -np.inf                             # a row without any key
        o_parts[0][torch.from_numpy(~np.isfinite(lse[0]))] = float("nan")  # a part without keys may hold anything
    o, l = attn.attn_combine(o_parts.to(DEV), torch.from_numpy(lse).to(DEV))
    torch.cuda.synchronize()
    assert attn.device_status() == attn.Status.OK
    o, l = I.as_f64(o.cpu()), l.cpu().double().numpy()
    op = I.as_f64(o_parts)
    op[~np.isfinite(lse)] = 0.0                                # (the oracle multiplies by the zero weight)
    o_ref, l_ref = combine_partials(op, lse.astype(np.float64))
    if parts == 1:
        assert np.array_equal(o, I.as_f64(o_parts)[0]) and np.array_equal(l, lse[0].astype(np.float64))
        return
    empty = ~np.isfinite(l_ref)
    assert np.array_equal(empty, ~np.isfinite(l)) and np.all(o[empty] == 0)
    err = np.abs(o - o_ref)
    # one bf16 rounding of the result, plus the fp32 weights (MUFU exp2) and
    # sums of at most 40 terms relative to the terms' size A = sum w |O_p| / l
    m = np.where(np.isfinite(lse.max(0)), lse.max(0), 0.0)
    w = np.exp(lse.astype(np.float64) - m)
    with np.errstate(invalid="ignore", divide="ignore"):
        big_a = np.where(empty[..., None], 0.0, (w[..., None] * np.abs(op)).sum(0) / w.sum(0)[..., None])
    bound = bf16_ulp(np.abs(o_ref)) + 2.0 ** -18 * big_a
    assert np.all(err <= bound), float((err / bound).max())
    assert np.max(np.abs(l[~empty] - l_ref[~empty])) <= 2e-5
    print(f"merge parts={parts} d={d}: max |dO| {err.max():.3g}, max |dLSE| {np.abs(l[~empty] - l_ref[~empty]).max():.3g}")


def ring(attn, q, k, v, chunks, causal, scale):
    """Attention over the whole sequence from (query chunk, key chunk) calls of
    attn_fwd merged by attn_combine, as a ring of `chunks` ranks would compute it."""
    B, H, N, d = q.shape
    c = N // chunks
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    for i in range(chunks):
        qi = q[:, :, i * c:(i + 1) * c].contiguous()
        js = range(i + 1) if causal else range(chunks)
        o_parts = torch.empty((len(js), B, H, c, d), dtype=torch.bfloat16, device=q.device)
        l_parts = torch.empty((len(js), B, H, c), dtype=torch.float32, device=q.device)
        for n, j in enumerate(js):
            kj = k[:, :, j * c:(j + 1) * c].contiguous()
            vj = v[:, :, j * c:(j + 1) * c].contiguous()
            attn.attn_fwd(qi, kj, vj, causal=causal and j == i, scale=scale, o=o_parts[n], lse=l_parts[n])
        oi, li = attn.attn_combine(o_parts, l_parts)
        o[:, :, i * c:(i + 1) * c] = oi
        lse[:, :, i * c:(i + 1) * c] = li
    torch.cuda.synchronize()
    assert attn.device_status() == attn.Status.OK
    return o, lse


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("shape,chunks", [((2, 3, 1536, 64), 3), ((1, 2, 1200, 128), 4), ((1, 2, 512, 128), 1)],
                         ids=["n1536_3chunks", "n1200_4chunks_ragged_tiles", "one_chunk"])
def test_sequence_split_matches_whole_sequence(attn, shape, chunks, causal):
    B, H, N, d = shape
    q, k, v = (I.to_bf16(x).to(DEV) for x in I.draw_fp32(B, H, N, d, seed=N + chunks))
    o, lse = ring(attn, q, k, v, chunks, causal, d ** -0.5)
    qq, kk, vv = (I.as_f64(t.cpu()) for t in (q, k, v))
    o_ref, lse_ref = attention_fwd(qq, kk, vv, causal, d ** -0.5)
    st = compare(I.as_f64(o.cpu()), lse.cpu().double().numpy(), o_ref, lse_ref,
                 f"ring {shape} chunks={chunks} causal={causal}")
    assert st["o_over_1e-2"] == 0
    if chunks == 1:  # one chunk is attn_fwd itself (the merge of one part is the identity)
        o1, l1 = attn.attn_fwd(q, k, v, causal=causal)
        assert torch.equal(o1, o) and torch.equal(l1, lse)


def test_sequence_split_of_the_benchmark_workload(attn):
    # B4 H16 N4096 d128 as four ranks of 1024 rows: sixteen attn_fwd calls and
    # four merges, checked on sampled rows of three heads
    w = I.NONCAUSAL_D128
    q, k, v = I.bf16_qkv(w)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o, lse = ring(attn, qd, kd, vd, 4, False, w.scale)
    o_whole, lse_whole = attn.attn_fwd(qd, kd, vd)
    torch.cuda.synchronize()
    d_o = (o.float() - o_whole.float()).abs().max().item()
    d_l = (lse - lse_whole).abs().max().item()
    print(f"ring of 4 vs one call: max |dO| {d_o:.3g}, max |dLSE| {d_l:.3g}")
    assert d_l <= 1e-3
    o, lse = o.cpu(), lse.cpu()
    rng = np.random.default_rng(4)
    for b, h in sorted({(0, 0), (w.B - 1, w.H - 1), (int(rng.integers(w.B)), int(rng.integers(w.H)))}):
        rows = sample_rows(w.N, rng)
        o_ref, lse_ref = attention_rows(I.as_f64(q[b, h, rows]), I.as_f64(k[b, h]), I.as_f64(v[b, h]), rows,
                                        False, w.scale)
        st = compare(I.as_f64(o[b, h, rows]), lse[b, h, rows].double().numpy(), o_ref, lse_ref,
                     f"ring of 4 {w.name} b={b} h={h}")
        assert st["o_over_1e-2"] == 0
