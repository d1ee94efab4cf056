"""The C ABI library loads, exports every function include/attn.h declares, and
rejects bad arguments on the host (no GPU needed: rejected calls never reach
CUDA)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "attn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(attn_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    import online_softmax_fwd_gb300 as attn
    return attn.lib()


def test_header_declares_entry_points():
    names = declared_functions()
    for want in ("attn_fwd", "attn_fwd_ex", "attn_exp2_emulated", "attn_get_device_status",
                 "attn_status_string", "attn_version"):
        assert want in names


def test_library_exports_every_declared_function(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    raw = ctypes.CDLL(lib._name)
    for name in declared_functions():
        getattr(raw, name)  # raises AttributeError if the symbol is missing


def test_version_and_strings(lib):
    assert lib.attn_version() >= 100
    assert lib.attn_status_string(0) == b"ATTN_OK"
    assert lib.attn_status_string(5) == b"ATTN_ERR_TIMEOUT"
    assert lib.attn_status_string(99) == b"ATTN_ERR_UNKNOWN"


# fake, never dereferenced device addresses
A = 0x10000
GOOD = dict(q=A, k=A * 2, v=A * 3, o=A * 4, lse=A * 5, B=1, H=2, N=256, d=64, causal=0, scale=0.125)


def call(lib, **over):
    a = dict(GOOD, **over)
    return lib.attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["d"],
                        a["causal"], a["scale"], None)


def call_ex(lib, tau=8.0, emu=0, **over):
    a = dict(GOOD, **over)
    return lib.attn_fwd_ex(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["d"],
                           a["causal"], a["scale"], tau, emu, None)


@pytest.mark.parametrize("over,code", [
    (dict(d=96), 2), (dict(d=256), 2), (dict(d=0), 1), (dict(d=-64), 1),
    (dict(B=-1), 1), (dict(H=-3), 1), (dict(N=-1), 1), (dict(N=(1 << 24) + 1), 2),
    (dict(causal=2), 1), (dict(scale=0.0), 1), (dict(scale=-0.1), 1), (dict(scale=float("inf")), 1),
    (dict(scale=float("nan")), 1), (dict(q=0), 1), (dict(lse=0), 1),
    (dict(q=A + 8), 3), (dict(o=A + 2), 3), (dict(lse=A + 2), 3),
])
def test_rejects_bad_arguments(lib, over, code):
    assert call(lib, **over) == code


@pytest.mark.parametrize("over", [dict(B=0), dict(H=0), dict(N=0), dict(B=0, q=0, k=0, v=0, o=0, lse=0)])
def test_empty_problem_is_a_no_op(lib, over):
    assert call(lib, **over) == 0


@pytest.mark.parametrize("tau,emu,code", [(-1.0, 0, 1), (17.0, 0, 1), (float("nan"), 0, 1),
                                          (8.0, -1, 1), (8.0, 5, 2), (8.0, 16, 2), (8.0, 17, 1)])
def test_ex_rejects_bad_tunables(lib, tau, emu, code):
    assert call_ex(lib, tau=tau, emu=emu) == code


def test_exp2_entry_rejects_bad_arguments(lib):
    assert lib.attn_exp2_emulated(A, A, -1, None) == 1
    assert lib.attn_exp2_emulated(A, A, 0, None) == 0
    assert lib.attn_exp2_emulated(0, A, 10, None) == 1
    assert lib.attn_exp2_emulated(A + 2, A, 10, None) == 3


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import online_softmax_fwd_gb300._binding as b
    monkeypatch.setattr(b, "_lib", None)
    monkeypatch.setattr(b, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU or PyTorch fallback"):
        b.lib()


def test_host_entry_rejects_bad_arguments(lib):
    H = A  # fake host addresses, never dereferenced on these paths
    args = lambda ws, nbytes, d=64, causal=0, scale=0.125, B=1: (H, H, H, H, H, B, 2, 256, d, causal, scale, ws, nbytes,
                                                                 None)
    need = lib.attn_fwd_host_workspace_bytes(1, 2, 256, 64)
    assert need > 0 and lib.attn_fwd_host_workspace_bytes(1, 2, 256, 96) == 0
    assert lib.attn_fwd_host(*args(0, need)) == 1             # no workspace
    assert lib.attn_fwd_host(*args(A * 7, need - 1)) == 1     # too small
    assert lib.attn_fwd_host(*args(A * 7 + 16, need)) == 3    # not 256-byte aligned
    assert lib.attn_fwd_host(*args(A * 7, need, d=96)) == 2
    assert lib.attn_fwd_host(*args(A * 7, need, causal=3)) == 1
    assert lib.attn_fwd_host(*args(A * 7, need, scale=-1.0)) == 1
    assert lib.attn_fwd_host(*args(A * 7, need, B=0)) == 0    # nothing to do


def test_mxfp8_ex_rejects_bad_p_scaling(lib):
    a = dict(GOOD, d=128)
    args = lambda tau, ps: (a["q"], a["q"], a["k"], a["k"], a["v"], a["v"], a["o"], a["lse"], a["B"], a["H"],
                            a["N"], 128, 1, a["scale"], tau, 0, ps, None)
    assert lib.attn_fwd_mxfp8_ex(*args(0.0, 3)) == 1          # unknown mode
    assert lib.attn_fwd_mxfp8_ex(*args(0.0, -1)) == 1
    assert lib.attn_fwd_mxfp8_ex(*args(0.9, 1)) == 1          # 2^0.9 * 256 > 448
    assert lib.attn_fwd_mxfp8_ex(*args(8.0, 1)) == 1
    assert lib.attn_fwd_mxfp8_ex(*args(7.81, 2)) == 1         # 2^7.81 * 256 > 57344 (E5M2)
    assert lib.attn_fwd_mxfp8_ex(*args(16.0, 2)) == 1
    zero = lambda tau, ps: args(tau, ps)[:9] + (0,) + args(tau, ps)[10:]   # H = 0: valid, nothing to do
    assert lib.attn_fwd_mxfp8_ex(*zero(0.8, 1)) == 0
    assert lib.attn_fwd_mxfp8_ex(*zero(8.0, 0)) == 0
    assert lib.attn_fwd_mxfp8_ex(*zero(7.8, 2)) == 0


def test_selftest_rejects_bad_limits(lib):
    assert lib.attn_selftest_wait_timeout(999, None) == 1
    assert lib.attn_selftest_wait_timeout(10 ** 10 + 1, None) == 1


def test_host_noalloc_limits_and_validation(lib):
    H = A  # fake host addresses, never dereferenced on these paths
    cap = lib.attn_fwd_host_noalloc_max_workspace()
    assert cap == 128 << 20
    call = lambda B, Hh, N, d, causal=0, scale=0.125: lib.attn_fwd_host_noalloc(H, H, H, H, H, B, Hh, N, d, causal,
                                                                                 scale, None)
    assert lib.attn_fwd_host_workspace_bytes(1, 64, 65536, 128) > cap
    assert call(1, 64, 65536, 128) == 2     # needs more than the fixed array: rejected before any work
    assert call(1, 2, 256, 96) == 2         # unsupported head dim, as attn_fwd_host
    assert call(1, -2, 256, 64) == 1
    assert call(0, 2, 256, 64) == 0         # nothing to do


def test_bwd_rejects_bad_arguments(lib):
    A = 1 << 20  # fake, 256-byte aligned addresses: rejected calls never dereference them
    B, H, N, d = 1, 2, 300, 128
    need = lib.attn_bwd_workspace_bytes(B, H, N, d)
    # fp32 dQ accumulator and two fp32 row vectors (LSE log2 e, D), N padded to 128
    assert need == (B * H * 384 * d * 4 + 255) // 256 * 256 + 2 * ((B * H * 384 * 4 + 255) // 256 * 256)
    assert lib.attn_bwd_workspace_bytes(B, H, N, 96) == 0
    assert lib.attn_bwd_workspace_bytes(0, H, N, d) == 0

    def args(ws=A * 9, ws_bytes=need, d_=d, causal=1, scale=0.1, b=B, q=A, lse=A * 6, h=H):
        return (q, A * 2, A * 3, A * 4, A * 5, lse, A * 7, A * 8, A * 10, b, h, N, d_, causal, scale, ws, ws_bytes,
                None)

    assert lib.attn_bwd(*args(d_=96)) == 2
    assert lib.attn_bwd(*args(d_=0)) == 1
    assert lib.attn_bwd(*args(causal=2)) == 1
    assert lib.attn_bwd(*args(scale=0.0)) == 1
    assert lib.attn_bwd(*args(scale=float("nan"))) == 1
    assert lib.attn_bwd(*args(ws_bytes=need - 1)) == 1
    assert lib.attn_bwd(*args(ws=0)) == 1
    assert lib.attn_bwd(*args(q=A + 8)) == 3
    assert lib.attn_bwd(*args(lse=A * 6 + 2)) == 3
    assert lib.attn_bwd(*args(ws=A * 9 + 16)) == 3
    assert lib.attn_bwd(*args(b=300, h=300)) == 2   # B*H above the preparation kernel's grid limit
    assert lib.attn_bwd(*args(b=0)) == 0     # nothing to do


def test_bwd_mxfp8_rejects_bad_arguments(lib):
    A = 1 << 20  # fake, 256-byte aligned addresses: rejected calls never dereference them
    B, H, N, d = 1, 2, 300, 128
    need = lib.attn_bwd_workspace_bytes(B, H, N, d)

    def args(ws=A * 14, ws_bytes=need, d_=d, causal=0, scale=0.1, b=B, q_sf=A * 2, do8=A * 8, lse=A * 10, h=H):
        # q8, q_sf, k8, k_sf, v8, v_sf, o, do8, do_sf, lse, dq, dk, dv
        return (A, q_sf, A * 3, A * 4, A * 5, A * 6, A * 7, do8, A * 9, lse, A * 11, A * 12, A * 13, b, h, N, d_,
                causal, scale, ws, ws_bytes, None)

    assert lib.attn_bwd_mxfp8(*args(d_=64)) == 2     # MXFP8 is d = 128 only
    assert lib.attn_bwd_mxfp8(*args(d_=0)) == 1
    assert lib.attn_bwd_mxfp8(*args(causal=3)) == 1
    assert lib.attn_bwd_mxfp8(*args(scale=-1.0)) == 1
    assert lib.attn_bwd_mxfp8(*args(ws_bytes=need - 1)) == 1
    assert lib.attn_bwd_mxfp8(*args(q_sf=0)) == 1
    assert lib.attn_bwd_mxfp8(*args(q_sf=A * 2 + 4)) == 3
    assert lib.attn_bwd_mxfp8(*args(do8=A * 8 + 8)) == 3
    assert lib.attn_bwd_mxfp8(*args(lse=A * 10 + 1)) == 3
    assert lib.attn_bwd_mxfp8(*args(ws=A * 14 + 64)) == 3
    assert lib.attn_bwd_mxfp8(*args(b=300, h=300)) == 2   # B*H above the quantiser's grid limit
    assert lib.attn_bwd_mxfp8(*args(b=0)) == 0            # nothing to do


def test_quantize_roles(lib):
    A = 1 << 20
    q = lambda role, d=128: lib.attn_mxfp8_quantize(A, A * 2, A * 3, 1, 2, 256, d, role, None)
    assert q(3) == 1 and q(-1) == 1
    assert q(0, d=64) == 2
    assert lib.attn_mxfp8_quantize(A, A * 2, A * 3, 0, 2, 256, 128, 2, None) == 0   # role 2 accepted; empty


def test_rescale_log_rejects_bad_arguments(lib):
    A = 1 << 20
    need = 1 * 2 * 256 * 2              # B H N ceil(N / 128)
    f = lambda log=A * 6, tau=8.0, b=1, d=64, nbytes=need: lib.attn_fwd_rescale_log(
        A, A * 2, A * 3, A * 4, A * 5, log, nbytes, b, 2, 256, d, 0, 0.125, tau, None)
    assert f(log=0) == 1                # the log is required
    assert f(nbytes=need - 1) == 1      # and must hold one byte per (head, row, key block)
    assert f(tau=-1.0) == 1 and f(tau=17.0) == 1
    assert f(d=96) == 2
    assert f(log=0, b=0) == 0           # empty problem: nothing to do, nothing checked


def test_2cta_accepts_only_d128_non_causal(lib):
    A = 1 << 20
    f = lambda d=128, causal=0, b=1, scale=0.1: lib.attn_fwd_2cta(A, A * 2, A * 3, A * 4, A * 5, b, 2, 300, d, causal,
                                                                  scale, None)
    assert f(causal=1) == 2 and f(d=64) == 2 and f(d=96) == 2
    assert f(scale=0.0) == 1 and f(causal=2) == 1
    assert f(b=0) == 0


def test_mxfp8_unroll_kv_rejects_bad_arguments(lib):
    A = 1 << 20
    f = lambda d=128, causal=0, b=1, scale=0.1, q_sf=A * 2: lib.attn_fwd_mxfp8_unroll_kv(
        A, q_sf, A * 3, A * 4, A * 5, A * 6, A * 7, A * 8, b, 2, 300, d, causal, scale, None)
    assert f(d=64) == 2 and f(causal=2) == 1 and f(scale=-1.0) == 1
    assert f(q_sf=A * 2 + 4) == 3
    assert f(b=0) == 0


def test_mxfp8_rescale_log_rejects_bad_arguments(lib):
    A = 1 << 20
    need = 1 * 2 * 256 * 2
    f = lambda log=A * 9, tau=0.0, b=1, d=128, nbytes=need: lib.attn_fwd_mxfp8_rescale_log(
        A, A * 2, A * 3, A * 4, A * 5, A * 6, A * 7, A * 8, log, nbytes, b, 2, 256, d, 0, 0.1, tau, None)
    assert f(log=0) == 1
    assert f(nbytes=need - 1) == 1
    assert f(tau=-1.0) == 1 and f(tau=17.0) == 1
    assert f(d=64) == 2
    assert f(log=0, b=0) == 0


def test_combine_rejects_bad_arguments(lib):
    A = 1 << 20
    f = lambda parts=3, d=128, b=1, o_parts=A, lse_parts=A * 2, o=A * 3, lse=A * 4: lib.attn_combine(
        o_parts, lse_parts, parts, o, lse, b, 2, 300, d, None)
    assert f(parts=0) == 1 and f(parts=1025) == 1 and f(parts=-2) == 1
    assert f(d=96) == 2 and f(d=0) == 1
    assert f(o_parts=0) == 1 and f(lse=0) == 1
    assert f(o_parts=A + 8) == 3 and f(o=A * 3 + 2) == 3 and f(lse_parts=A * 2 + 1) == 3
    assert f(b=-1) == 1
    assert f(b=0, o_parts=0, lse=0) == 0   # empty problem: nothing to do, pointers unchecked
