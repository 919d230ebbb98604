"""A device-side wait that runs out reports ZFFN_ERR_TIMEOUT and the context
stays usable (no trap, no hang)."""
import numpy as np
import pytest
import torch

from quantized_ffn_gb300 import synth, zffn
from tests.gpu_util import dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    assert zffn.get_device_error() == zffn.OK
    zffn.selftest_wait_timeout(2_000_000)          # about a millisecond of SM clocks
    assert zffn.get_device_error() == zffn.ERR_TIMEOUT
    assert zffn.get_device_error() == zffn.OK      # reading clears the word
    # the context still works
    w = np.random.default_rng(0).standard_normal((4, 256)).astype(np.float32)
    b = zffn.q4k_quantize(dev(w))
    torch.cuda.synchronize()
    assert b.shape == (4, 144)
