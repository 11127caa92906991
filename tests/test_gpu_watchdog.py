"""Failure detection without a GPU fault: a wait that nothing satisfies gives up,
the host reads the timeout, and the CUDA context stays usable."""
import math
import time

import numpy as np
import pytest

from attention_fa2_forward_02_gb300 import binding, synth
from oracle import attention as A
from tests import gpu_util as G
from tests.tolerance import check_16bit

pytestmark = pytest.mark.gpu

OK, TIMEOUT = 0, 5


def test_bounded_wait_reports_timeout_and_context_survives():
    torch = G.require_gpu()
    lib = binding.library()
    torch.cuda.synchronize()
    assert lib.fa2_device_status(None) == OK  # nothing pending from earlier work
    t0 = time.perf_counter()
    assert lib.fa2_watchdog_selftest(None) == OK
    assert lib.fa2_device_status(None) == TIMEOUT  # synchronises, reads and clears the word
    assert time.perf_counter() - t0 >= 0.5  # the wait really waited for its limit
    assert lib.fa2_device_status(None) == OK  # cleared
    # the context still runs the real kernels correctly
    q, k, v = G.inputs("watchdog/after", 1, 200, 300, 64, "bf16")
    qd, kd, vd = (G.to_device(x, "bf16") for x in (q, k, v))
    o = G.empty((1, 200, 64), "bf16")
    lse = torch.empty((1, 200), dtype=torch.float32, device="cuda")
    binding.fa2_forward(qd, kd, vd, o, lse, 1 / math.sqrt(64))
    binding.fa2_device_status()
    ref, _ = A.forward(*(synth.widen(x, "bf16") for x in (q, k, v)), 1 / math.sqrt(64))
    check_16bit(G.to_f64(o), ref, "O after a watchdog timeout")
    assert np.all(np.isfinite(G.to_f64(lse)))
