"""The bounded waits give up and the kernel returns.

Every mbarrier wait in the library's kernels gives up after a time limit,
sets PKV_DEVERR_TIMEOUT in the error word and lets its kernel leave in
order.  pkv_check_bounded_wait runs that wait routine in a small kernel with
the attention kernels' roles (tensor-memory owner, producer, consumers)
whose barriers nothing arrives at, with a 1 ms limit: each wait must give
up, the error bit must be set, the tensor memory must be freed and the
kernel must return, leaving the context usable for the attention calls
that follow.
"""
import ctypes

import pytest
import torch

import paged_kv_cache_84_gb300 as pkv
from workloads import config_spec, make_batch
from _helpers import DeviceStep, assert_close, cpu_copy, oracle_full, oracle_write

pytestmark = pytest.mark.gpu


def _check(err, report, limit_us):
    fn = pkv.load().pkv_check_bounded_wait
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint32, ctypes.c_void_p]
    return fn(err.data_ptr(), report.data_ptr(), limit_us, torch.cuda.current_stream().cuda_stream)


def test_waits_give_up_after_their_limit_and_the_context_stays_usable():
    for limit_us in (1000, 3000):                   # twice: the first run freed its tensor memory
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        report = torch.zeros(2, dtype=torch.int32, device="cuda")
        assert _check(err, report, limit_us) == 0
        torch.cuda.synchronize()
        assert int(err.item()) == pkv.DEVERR_TIMEOUT
        gave_up, us = (int(x) for x in report.tolist())
        assert gave_up == 0b1101                    # producer warp 0, consumer warps 2 and 3
        assert limit_us <= us < limit_us + 200000
    b = make_batch(config_spec(2), device="cpu")
    ref = cpu_copy(b)
    oracle_write(ref)
    dev = DeviceStep(b)
    dev.combined()
    assert_close(dev.out, oracle_full(ref), "attention after the timed-out check kernel")
    assert pkv.read_device_error(dev.ws) == 0


def test_check_rejects_bad_arguments():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    report = torch.zeros(2, dtype=torch.int32, device="cuda")
    assert _check(err, report, 0) == 1
    assert _check(err, report, 200000) == 1
