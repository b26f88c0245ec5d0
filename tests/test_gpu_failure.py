"""Failure detection on the GPU without a fault: a kernel waits on a barrier
that nothing completes, gives up after a short limit, records the timeout in
the device status word and returns; the host reads MMDIT_ERR_TIMEOUT, the
word is cleared, and the context keeps working."""
import numpy as np
import pytest
import torch

from diffusion_transformer_image_mmdit_gb300 import api
from tests.gpu_common import f32, host, need_gpu

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    need_gpu()
    assert api.sync_status() == 0
    api.selftest_wait_timeout(20000)  # 20 ms limit
    assert api.sync_status() == -6  # MMDIT_ERR_TIMEOUT
    assert api.sync_status() == 0  # cleared on read
    x = f32(np.arange(8, dtype=np.float32))
    v = f32(np.ones(8, dtype=np.float32))
    api.euler_step(x, v, 1.0, 0.5)
    assert np.array_equal(host(x), np.arange(8) - 0.5)
    assert api.sync_status() == 0
