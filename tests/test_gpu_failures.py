"""Failure detection without a GPU fault: a bounded device wait gives up, the
error is reported through te_get_last_error(), and the context stays usable."""
import pytest
import torch

import nvfp4_precision_transformer_gb300 as te
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def test_device_wait_timeout_is_reported_and_context_survives():
    assert te.te_get_last_error() == 0
    te.te_selftest_wait_timeout()
    assert te.te_get_last_error() == 7          # TE_ERR_TIMEOUT
    assert te.te_get_last_error() == 0          # reading clears it
    x = torch.full((32, 64), -3.0, dtype=torch.bfloat16, device=G.DEV)
    a, _ = G.amax(x)
    assert a == 3.0


def test_rejected_calls_enqueue_nothing():
    before = te.te_launch_count()
    x = torch.zeros(24, 32, dtype=torch.bfloat16, device=G.DEV)
    with pytest.raises(te.TEError):
        G.fp8(x, te.E4M3, scale=1.0)
    assert te.te_launch_count() == before
