"""The kernel's rescale decisions, checked one by one against the lagging-max
rule ("FlashAttention-4's Softmax Tricks", section "Conditional rescaling, and
when it's exact"): per row and 128-key block, keep the stale max iff the block
raises it by at most tau (log2 units of the scaled score), else move it; a
warp rescales O when any of its 32 rows moved (block > 0).

attn_fwd_rescale_log writes the decisions of the same kernel as attn_fwd
(bit 0: the row moved its max, bit 1: its warp rescaled O), and
attn_fwd_mxfp8_rescale_log those of the MXFP8 kernel (checked against the
recurrence on the dequantised inputs). The oracle's
blockwise recurrence gives the row decisions in float64 (``fired``) and the
reference max of every block. A decision whose growth lies within the fp32
error of the scores of tau can go either way in fp32; such a decision and the
rest of its row are left out (and counted). Integer scores are exact in fp32,
so there nothing is left out, and a block that only ties the running max at
tau = 0 (growth exactly tau) must not move it.
"""
import math

import numpy as np
import pytest
import torch

import attn_inputs as I
from oracle.attention import blockwise_attention

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
LOG2E = 1.0 / math.log(2.0)


@pytest.fixture(scope="module")
def attn():
    import online_softmax_fwd_gb300 as a
    a.lib()
    return a


def expected_decisions(q, k, causal, scale, tau, exact=False):
    """Row decisions of the oracle for one head, which (row, block) entries
    the kernel streams, and which of them are left out as too close to tau."""
    n = q.shape[0]
    nb = (n + 127) // 128
    v = np.zeros((n, 1))
    _, _, fired, m_used = blockwise_attention(q, k, v, causal, scale, block=128, tau=tau, max_history=True)
    fired = np.zeros((n, nb), dtype=bool) if fired.shape[1] == 0 else np.pad(
        fired, ((0, 0), (0, nb - fired.shape[1])))
    m_used = np.pad(m_used, ((0, 0), (0, nb - m_used.shape[1])), constant_values=-np.inf)
    streamed = np.ones((n, nb), dtype=bool)
    if causal:
        streamed = np.arange(nb)[None, :] <= (np.arange(n) // 128)[:, None]
    s = q @ k.T
    allowed = np.ones_like(s, dtype=bool)
    if causal:
        allowed = np.arange(n)[None, :] <= np.arange(n)[:, None]
    sl2 = scale * LOG2E
    a_row = np.where(allowed, np.abs(q) @ np.abs(k).T, 0.0).max(axis=1)
    left_out = np.zeros((n, nb), dtype=bool)
    if not exact:
        m_prev = np.full(n, -np.inf)
        gone = np.zeros(n, dtype=bool)
        for jb in range(nb):
            j0, j1 = jb * 128, min(n, jb * 128 + 128)
            bmax = np.where(allowed[:, j0:j1], s[:, j0:j1], -np.inf).max(axis=1)
            live = np.isfinite(m_prev) & np.isfinite(bmax)
            g = np.where(live, (bmax - np.where(live, m_prev, 0.0)) * sl2, np.inf)
            # fp32 scores err by a few ulps of sum |q_c k_c|; the growth's own rounding
            margin = 2.0 ** -18 * sl2 * a_row + 2.0 ** -20 * np.abs(np.where(np.isfinite(g), g, 0.0))
            gone |= live & (np.abs(g - tau) <= margin)
            left_out[:, jb] = gone
            m_prev = np.where(np.isfinite(m_used[:, jb]), m_used[:, jb], m_prev)
    return fired, streamed, left_out


def check_head(log, q, k, causal, scale, tau, what, exact=False):
    n = q.shape[0]
    fired, streamed, left_out = expected_decisions(q, k, causal, scale, tau, exact)
    moved = (log & 1).astype(bool)
    warp = (log & 2).astype(bool)
    use = streamed & ~left_out
    # row decisions
    bad = use & (moved != fired)
    assert not bad.any(), f"{what}: {int(bad.sum())} row decisions differ, first at {np.argwhere(bad)[:5].tolist()}"
    # nothing written outside the blocks the row's tile streams (the log starts at 0)
    assert not (log[~streamed] != 0).any(), f"{what}: bytes written past the streamed blocks"
    # every streamed block of a row starts with a move at block 0
    assert moved[:, 0].all(), f"{what}: block 0 must move the max from -inf"
    # warp decisions: any of the 32 rows of the group, block > 0 (own decisions, and the oracle's)
    groups = (n + 31) // 32
    pad = groups * 32 - n
    mv = np.pad(moved, ((0, pad), (0, 0))).reshape(groups, 32, -1)
    fr = np.pad(fired & streamed, ((0, pad), (0, 0))).reshape(groups, 32, -1)
    lo = np.pad(left_out & streamed, ((0, pad), (0, 0))).reshape(groups, 32, -1).any(axis=1)
    wg = np.pad(warp, ((0, pad), (0, 0))).reshape(groups, 32, -1)
    st = np.pad(streamed, ((0, pad), (0, 0))).reshape(groups, 32, -1)
    any_own = mv.any(axis=1)
    any_ref = fr.any(axis=1)
    for g in range(groups):
        rows = slice(g * 32, min(n, g * 32 + 32))
        w_rows = wg[g][: rows.stop - rows.start]
        s_rows = st[g][: rows.stop - rows.start]
        # every row of the group logs the same warp decision on a streamed block
        for j in range(1, mv.shape[2]):
            if not s_rows[:, j].any():
                continue
            col = w_rows[s_rows[:, j], j]
            assert (col == col[0]).all(), f"{what}: warp decision not uniform, group {g} block {j}"
            assert col[0] == any_own[g, j], f"{what}: warp decision != any of its rows, group {g} block {j}"
            if not lo[g, j]:
                assert col[0] == any_ref[g, j], f"{what}: warp decision != oracle's any, group {g} block {j}"
        assert not w_rows[:, 0].any(), f"{what}: no O correction at block 0"
    return {"decisions": int(use.sum()), "left_out": int((streamed & left_out).sum()),
            "row_moves": int((moved & use)[:, 1:].sum()), "warp_rescales": int(any_own[:, 1:].sum())}


def run_log(attn, q, k, v, causal, scale, tau):
    o, lse, log = attn.attn_fwd_rescale_log(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=scale, tau=tau)
    torch.cuda.synchronize()
    assert attn.device_status() == attn.Status.OK
    # the logging variant computes the same O and LSE as the product kernel
    o2, lse2 = attn.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=scale, tau=tau)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    return log.cpu().numpy()


def ramp_inputs():
    q, k, v = I.draw_fp32(1, 2, 1024, 64, seed=13)
    q += 1.0
    k += np.linspace(0.0, 1.5, 1024, dtype=np.float32)[None, None, :, None]
    return I.to_bf16(q), I.to_bf16(k), I.to_bf16(v), 64 ** -0.5


def peaked_inputs():
    q, k, v = (I.to_bf16(x) for x in I.draw_fp32(1, 2, 1536, 128, qk_std=2.0, seed=9))
    return q, k, v, 128 ** -0.5


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("tau", [0.0, 8.0])
@pytest.mark.parametrize("inputs", ["ramp", "qk_std2"])
def test_rescale_decisions_match_the_rule(attn, inputs, tau, causal):
    q, k, v, scale = ramp_inputs() if inputs == "ramp" else peaked_inputs()
    log = run_log(attn, q, k, v, causal, scale, tau)
    totals = {"decisions": 0, "left_out": 0, "row_moves": 0, "warp_rescales": 0}
    for h in range(q.shape[1]):
        st = check_head(log[0, h], I.as_f64(q[0, h]), I.as_f64(k[0, h]), causal, scale, tau,
                        f"{inputs} tau={tau} causal={causal} h={h}")
        totals = {kk: totals[kk] + st[kk] for kk in totals}
    print(f"rescale log {inputs} tau={tau} causal={causal}: {totals}")
    assert totals["left_out"] <= 0.01 * totals["decisions"]
    assert totals["row_moves"] > 0          # the inputs do exercise the rule


def test_a_tie_at_tau_zero_does_not_move_the_max(attn):
    # small-integer Q and K: every score is an integer, exact in fp32, and many
    # later blocks tie the running max exactly (growth == tau == 0)
    rng = np.random.default_rng(7)
    n, d = 1024, 64
    q = rng.integers(-2, 3, size=(1, 2, n, d)).astype(np.float32)
    k = rng.integers(-2, 3, size=(1, 2, n, d)).astype(np.float32)
    v = rng.standard_normal((1, 2, n, d)).astype(np.float32)
    q, k, v = I.to_bf16(q), I.to_bf16(k), I.to_bf16(v)
    scale = 0.125
    log = run_log(attn, q, k, v, False, scale, 0.0)
    ties = 0
    for h in range(2):
        qq, kk = I.as_f64(q[0, h]), I.as_f64(k[0, h])
        check_head(log[0, h], qq, kk, False, scale, 0.0, f"integer h={h}", exact=True)
        s = qq @ kk.T
        bm = np.stack([s[:, j:j + 128].max(axis=1) for j in range(0, n, 128)], axis=1)
        run = np.maximum.accumulate(bm, axis=1)
        ties += int((bm[:, 1:] == run[:, :-1]).sum())
    assert ties > 100   # the case is exercised


# The MXFP8 kernel: the same rule on the scores of the quantised inputs. The
# oracle's decisions come from the float64 recurrence on the dequantised Q
# and K (the values the block-scaled products multiply).
def mx_run_log(attn, xq, xk, xv, causal, scale, tau):
    import ctypes
    from test_gpu_mxfp8 import quantize_gpu
    q8, q_sf = quantize_gpu(attn, xq, 0)
    k8, k_sf = quantize_gpu(attn, xk, 0)
    v8, v_sf = quantize_gpu(attn, xv, 1)
    B, H, N, d = xq.shape
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    log = torch.zeros((B, H, N, (N + 127) // 128), dtype=torch.uint8, device=DEV)
    st = attn.lib().attn_fwd_mxfp8_rescale_log(*(t.data_ptr() for t in (q8, q_sf, k8, k_sf, v8, v_sf, o, lse, log)),
                                               log.numel(), B, H, N, d, int(causal), scale, tau, None)
    assert st == 0
    torch.cuda.synchronize()
    assert attn.device_status() == attn.Status.OK
    # O and LSE as the product kernel's (attn_fwd_mxfp8_ex with the same tau)
    o2, lse2 = attn.attn_fwd_mxfp8(q8, q_sf, k8, k_sf, v8, v_sf, causal=causal, scale=scale, tau=tau)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    return log.cpu().numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("tau", [0.0, 8.0])
@pytest.mark.parametrize("inputs", ["ramp", "qk_std2"])
def test_mxfp8_rescale_decisions_match_the_rule(attn, inputs, tau, causal):
    from oracle.mxfp8 import quantize_blocks
    if inputs == "ramp":
        xq, xk, xv = I.draw_fp32(1, 2, 1024, 128, seed=13)
        xq += 1.0
        xk += np.linspace(0.0, 1.5, 1024, dtype=np.float32)[None, None, :, None]
    else:
        xq, xk, xv = I.draw_fp32(1, 2, 1536, 128, qk_std=2.0, seed=9)
    scale = 128 ** -0.5
    log = mx_run_log(attn, xq, xk, xv, causal, scale, tau)
    totals = {"decisions": 0, "left_out": 0, "row_moves": 0, "warp_rescales": 0}
    for h in range(xq.shape[1]):
        qd = quantize_blocks(xq[0, h].astype(np.float64))[2]
        kd = quantize_blocks(xk[0, h].astype(np.float64))[2]
        st = check_head(log[0, h], qd, kd, causal, scale, tau, f"mxfp8 {inputs} tau={tau} causal={causal} h={h}")
        totals = {kk: totals[kk] + st[kk] for kk in totals}
    print(f"mxfp8 rescale log {inputs} tau={tau} causal={causal}: {totals}")
    assert totals["left_out"] <= 0.01 * totals["decisions"]
    assert totals["row_moves"] > 0
