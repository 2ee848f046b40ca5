"""Failure reporting on the GPU without a fault: a bounded device wait on a
flag that nothing sets runs out, reports SP_ERR_DEVICE_TIMEOUT through the
device error word, and leaves the context usable."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_timeout(cuda_dev, lib):
    from prefill_only_shared_gb300 import sp
    flag = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    limit_ns = 50_000_000
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    sp.sp_wait_flag(flag, 1, limit_ns)
    end.record()
    with pytest.raises(sp.SpError) as e:
        sp.sp_check_device_error()
    assert e.value.status == 5
    waited_ms = start.elapsed_time(end)
    assert 50.0 <= waited_ms < 1000.0, waited_ms
    sp.sp_check_device_error()  # the word was cleared
    # the context still works: a set flag ends the wait at once, no error
    flag.fill_(1)
    start.record()
    sp.sp_wait_flag(flag, 1, limit_ns)
    end.record()
    sp.sp_check_device_error()
    assert start.elapsed_time(end) < 10.0
    x = torch.arange(1000, device=cuda_dev, dtype=torch.float32)
    assert x.sum().item() == 499500.0


def test_wait_limit_is_clamped(cuda_dev, lib):
    """A limit above the library's ceiling still ends (clamped to 2 s); a
    limit of 0 becomes 1 us."""
    from prefill_only_shared_gb300 import sp
    flag = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    sp.sp_wait_flag(flag, 7, 0)
    with pytest.raises(sp.SpError) as e:
        sp.sp_check_device_error()
    assert e.value.status == 5
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    sp.sp_wait_flag(flag, 7, 60_000_000_000)
    end.record()
    with pytest.raises(sp.SpError) as e:
        sp.sp_check_device_error()
    assert e.value.status == 5
    assert 1900.0 <= start.elapsed_time(end) < 4000.0


def test_wait_flag_argument_errors(cuda_dev, lib):
    from prefill_only_shared_gb300 import sp
    flag = torch.zeros(4, dtype=torch.int32, device=cuda_dev)
    with pytest.raises(sp.SpError) as e:
        sp.sp_wait_flag(flag, 1, -5)
    assert e.value.status == 1
