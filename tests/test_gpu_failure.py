"""Failure detection without a GPU fault: a bounded wait that nothing
completes reports BD_ERR_TIMEOUT through the workspace status word, the
device stays usable, and host-side argument errors never launch anything."""
import pytest
import torch

from tests.gpu_util import load_bd

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    bd = load_bd()
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert bd.bitdelta_check_bounded_wait(ws.data_ptr(), 64, 0, stream) == bd.BD_OK
    assert bd.device_status(ws) == bd.BD_ERR_TIMEOUT
    diag = ws[8:12].view(torch.int32).item()
    assert diag == 99
    # the status word was cleared by the read, and the device still works
    assert bd.device_status(ws) == bd.BD_OK
    assert bd.bitdelta_check_bounded_wait(ws.data_ptr(), 64, 1, stream) == bd.BD_OK
    assert bd.device_status(ws) == bd.BD_OK
    x = torch.ones(1024, device="cuda")
    assert float(x.sum().item()) == 1024.0


def test_status_accumulates_until_read():
    bd = load_bd()
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(3):
        assert bd.bitdelta_check_bounded_wait(ws.data_ptr(), 16, 0, stream) == bd.BD_OK
    assert bd.device_status(ws) == bd.BD_ERR_TIMEOUT
    assert bd.device_status(ws) == bd.BD_OK
