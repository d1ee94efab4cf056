"""The kernels' software exp2, run on the GPU, equals the oracle's scalar C
model bit for bit (4M inputs on the softmax range, plus a wide sweep and
special values), and its accuracy reproduces the printed degree-3 row."""
import numpy as np
import pytest
import torch

from attn_inputs import uniform_fp32
from conftest import read_golden_kv
from oracle import cmodel, exp2_model

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    import online_softmax_fwd_gb300 as a
    a.lib()
    return a


def gpu_exp2(attn, x: np.ndarray) -> np.ndarray:
    y = attn.exp2_emulated(torch.from_numpy(x).to("cuda"))
    torch.cuda.synchronize()
    return y.cpu().numpy()


def test_bit_exact_on_softmax_range(attn):
    g = read_golden_kv("sw_exp2_accuracy.txt")
    x = uniform_fp32(int(g["inputs"]), g["domain_lo"], g["domain_hi"], seed=0)
    y = gpu_exp2(attn, x)
    ref = cmodel.exp2_emulated(x)
    assert np.array_equal(y.view(np.int32), ref.view(np.int32))
    acc = exp2_model.accuracy(x, y)
    assert acc["max_rel"] == pytest.approx(g["max_rel"], abs=5e-8)
    assert 100 * acc["bf16_within_1ulp"] == g["bf16_within_1ulp_pct"]


def test_bit_exact_wide_sweep(attn):
    x = uniform_fp32(1 << 20, -140.0, 40.0, seed=1)
    assert np.array_equal(gpu_exp2(attn, x).view(np.int32), cmodel.exp2_emulated(x).view(np.int32))


def test_bit_exact_special_values(attn):
    x = np.array([-np.inf, -1e30, -200.0, -127.0, -126.5, -126.0, -1e-40, -0.0, 0.0, 1e-40, 1e-30,
                  0.5, 1.0, 7.999999, 8.0, 100.0, 127.0, 127.9], dtype=np.float32)
    assert np.array_equal(gpu_exp2(attn, x).view(np.int32), cmodel.exp2_emulated(x).view(np.int32))
