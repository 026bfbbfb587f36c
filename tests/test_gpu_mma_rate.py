"""The tensor-core rate probe does the work it is timed for: CTA 0's
accumulator after `iters` iterations equals the product of its documented
operand pattern (exact small integers in fp32), and the FLOP count it reports
matches one CTA per SM."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

E2M1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6])


@pytest.fixture(scope="module")
def mx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mxfp4_precision_attention_gb300 as m

    m.load()
    return m


@pytest.mark.parametrize("n", [128, 256])
@pytest.mark.parametrize("iters", [1, 255, 256, 257, 1000])
def test_probe_accumulator_and_flops(mx, iters, n):
    out = torch.full((128, n), float("nan"), dtype=torch.float32, device="cuda")
    flops = mx.mxattn_mxf4_mma_rate(iters, n=n, out=out)
    mx.mxattn_check()
    a = E2M1[(7 * np.arange(128) + 1) % 16]
    b = E2M1[(11 * np.arange(n) + 5) % 16]
    want = 128.0 * iters * np.outer(a, b)
    got = out.cpu().numpy().astype(np.float64)
    assert np.array_equal(got, want), f"{(got != want).sum()} accumulator entries differ"
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert flops == sms * iters * 2 * (2 * 128 * n * 64)


@pytest.mark.parametrize("n", [128, 256])
def test_probe_rate_is_plausible(mx, n):
    """A few ms of back-to-back MMAs run at a rate between 5 % and 150 % of the
    nominal 13.5 PFLOP/s dense FP4: the probe is neither idle nor skipping work."""
    iters = 20000
    mx.mxattn_mxf4_mma_rate(iters, n=n)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    flops = mx.mxattn_mxf4_mma_rate(iters, n=n)
    e1.record()
    mx.mxattn_check()
    tflops = flops / (e0.elapsed_time(e1) * 1e-3) / 1e12
    assert 0.05 * 13500 < tflops < 1.5 * 13500, tflops
