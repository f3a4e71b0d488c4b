"""The arithmetic-peak microbenchmarks run through the C ABI and report positive rates of the
right order (short loops; the rates printed by peaks.py come from longer ones)."""
import pytest

pytestmark = pytest.mark.gpu


def test_every_peak_kernel_runs_and_reports_a_rate():
    from _gpu import torch_cuda
    torch = torch_cuda()
    from matrix_dense_linear_spd_gb300 import peaks
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    res = {k: peaks.measure(k, sms, 2.0, 2, torch)["tflops"] for k in peaks.KINDS}
    assert all(v > 0 for v in res.values()), res
    assert res["tf32"] > 10 * res["ffma"]              # tensor cores well above the FP32 pipe
    assert res["ffma"] > 10 * res["dfma"]              # FP64 is a small fraction of FP32 on GB300
    assert res["bf16"] > res["tf32"]
