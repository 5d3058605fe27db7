"""The bounded-wait failure path on the GPU, without a fault.

Every wait of the library's kernels on an mbarrier gives up after a limit:
the CTA unwinds and FLARE_ERR_TIMEOUT is recorded in the device status word
that flare_device_status reads and clears. flare_check_bounded_wait runs that
path in isolation (a kernel waiting on a barrier nothing arrives on, with a
short limit); these tests check that the timeout is reported, that it is
reported once, and that the next mixer call on the same context is correct."""
import numpy as np
import pytest
import torch

import oracle
from latent_query_split_gb300 import flare
from parity import assert_L_close, assert_close

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_then_context_stays_usable(cuda_device):
    flare.flare_device_status()            # start from a clear status word
    st = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    flare.flare_check_bounded_wait(2000)   # gives up after 2 ms
    b.record(st)
    with pytest.raises(flare.FlareError) as e:
        flare.flare_device_status()
    assert e.value.status == flare.FLARE_ERR_TIMEOUT
    assert a.elapsed_time(b) >= 2.0        # it did wait for its limit
    flare.flare_device_status()            # read once, then cleared

    # the next call on the same context runs and is correct
    g = torch.Generator().manual_seed(5)
    B, H, M, N, D = 1, 2, 128, 3000, 64
    off = [0, 1000, 3000]
    Q = (torch.randn((H, M, D), generator=g) * 0.5).bfloat16().cuda()
    K = torch.randn((B, N, H, D), generator=g).bfloat16().cuda()
    V = torch.randn((B, N, H, D), generator=g).bfloat16().cuda()
    Y, Z, L = flare.flare_fwd(Q, K, V, None, off)
    flare.flare_device_status()
    Zo, Lo, Yo = oracle.flare_fwd(Q, K, V, None)
    assert_close("Z", Z, Zo, "bf16")
    assert_L_close("L", L, Lo)
    assert_close("Y", Y, Yo, "bf16")


def test_timeouts_do_not_accumulate(cuda_device):
    flare.flare_device_status()
    for _ in range(3):
        flare.flare_check_bounded_wait(100)
    with pytest.raises(flare.FlareError) as e:
        flare.flare_device_status()
    assert e.value.status == flare.FLARE_ERR_TIMEOUT
    flare.flare_device_status()
