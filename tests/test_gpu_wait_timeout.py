"""The bounded in-kernel wait of the asynchronous-copy kernels: on a barrier
that completes it returns with the status word untouched; on a barrier that
nothing completes it gives up after its cycle limit with GAI4_ERR_TIMEOUT
(no fault, no trap, no hang), and the context stays usable afterwards."""
import time

import numpy as np
import pytest
import torch

import gemm_affine_int4_gb300 as g4
import oracle
import synth
from gpu_util import to_dev, to_host_f64
from tolerance import assert_within

pytestmark = pytest.mark.gpu


def test_wait_on_completed_barrier_leaves_status():
    st = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    assert g4.gai4_check_bounded_wait(True, 2_000_000, st) == 12345


@pytest.mark.parametrize("limit", [1, 100_000, 4_000_000])
def test_wait_on_barrier_nobody_completes_times_out(limit):
    t0 = time.perf_counter()
    assert g4.gai4_check_bounded_wait(False, limit) == g4.GAI4_ERR_TIMEOUT
    # 4e6 cycles is about 2 ms at the SM clock: the wait ended by its limit
    assert time.perf_counter() - t0 < 5.0
    # the library's own status word was not touched
    assert g4.gai4_last_device_status() == g4.GAI4_OK


def test_context_usable_after_timeout():
    assert g4.gai4_check_bounded_wait(False, 1_000_000) == g4.GAI4_ERR_TIMEOUT
    bits, gs, dt = 4, 64, "bf16"
    N, K = 384, 2048
    W = synth.affine_weights(N, K, 41)
    packed, s, b = oracle.quantize(W, bits, gs, dt)
    x = synth.activations(1, K, dt, 42)
    out = g4.gai4_qmv(to_dev(packed), to_dev(s, dt), to_dev(b, dt), to_dev(x.reshape(-1), dt), bits=bits,
                      group_size=gs)
    ref, absdot = oracle.qmm(packed, s, b, x[0], bits, gs, dt)
    assert_within(to_host_f64(out, dt), ref, absdot, dt, "qmv after a timed-out wait")
    assert g4.gai4_last_device_status() == g4.GAI4_OK
    assert g4.gai4_check_bounded_wait(True, 1_000_000) == 0
