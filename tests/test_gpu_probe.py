"""The tensor-core rate probe (the MXFP4 MMA rate the prefill scorer is measured against) runs
through the C ABI without a timeout and reports a consistent FLOP count."""
import pytest
import torch

import fp4_sparse_attention_mxfp4_gb300 as fx

pytestmark = pytest.mark.gpu


def test_mxf4_probe_runs_and_reports_a_plausible_rate():
    """The tensor-core rate probe completes without a timeout and its FLOP count is consistent
    with its launch (a rate above zero and below twice the nominal dense FP4 figure)."""
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fx.idx_fp4_mxf4_probe(64, status)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    fx.idx_fp4_mxf4_probe(1024, status)
    b.record()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    flops = fx.idx_fp4_mxf4_probe_flops(1024)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert flops == sms * 8 * 1024 * 2 * (2 * 128 * 128 * 64)
    tflops = flops / (a.elapsed_time(b) / 1e3) / 1e12
    assert 0 < tflops < 2 * 13500
