"""Tensor-core operand forms of the backward kernel, on single tiles."""
import pytest
import torch

import deterministic_attn_backward_gb300 as dab


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
def test_mma_operand_forms(d):
    g = torch.Generator().manual_seed(100 + d)
    x = torch.randn(128, d, generator=g).bfloat16()
    y = torch.randn(128, d, generator=g).bfloat16()
    z = torch.randn(128, 128, generator=g).bfloat16()
    pm = torch.randn(128, 128, generator=g).bfloat16()
    outs = dab.selftest_mma(d, *(t.cuda() for t in (x, y, z, pm)))
    X, Y, Z, P = (t.double() for t in (x, y, z, pm))
    want = [X @ Y.T, P @ Y, Z @ Y, (X.T @ Z) if d == 128 else (Z.T @ X)]
    for n, (got, w) in enumerate(zip(outs, want)):
        err = (got.cpu().double() - w).abs().max().item() / w.abs().max().item()
        assert err < 1e-5, f"form {n}: rel err {err:.3e}"


@pytest.mark.gpu
def test_mma_peak_is_a_plausible_tensor_rate():
    """The build's own tcgen05 throughput measurement: positive, completes
    without a device error, and below the nominal dense bf16 rate of the chip
    at its highest clock (8192 flops per clock per SM)."""
    r = dab.mma_peak(iters=20000)
    sms = r["grid"]
    ceiling = sms * 8192 * 2.2e9 / 1e12   # TFLOP/s at 2.2 GHz, above any clock the part runs
    assert 0.3 * ceiling < r["tflops"] < ceiling, r
