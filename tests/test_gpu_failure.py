"""Failure detection on the GPU without a fault: a bounded device wait that runs out sets the
device error word, kda_device_status reports KDA_ERR_TIMEOUT once (and clears the word), and
the context stays usable.  The wait is on an mbarrier that nothing arrives on (see
kda_selftest_timeout); nothing traps, faults or spins without a limit."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def test_timeout_is_reported_once_and_context_survives():
    import torch
    from serving_kda_chunkwise_gb300 import inputs, kda
    kda.device_status()  # start clean
    kda.selftest_timeout(50000)  # 50 ms
    with pytest.raises(kda.KdaError) as ei:
        kda.device_status()
    assert ei.value.status == kda.KDA_ERR_TIMEOUT
    kda.device_status()  # the word was cleared: no error now
    # the context is still usable: a small forward runs and is finite
    sp = inputs.forward_spec(seed=5, H=2, dk=128, dv=128, dtype="bf16", B=1, T=200)
    d = sp.to_device("cuda")
    o, S = kda.fwd_chunked(d["q"], d["k"], d["v"], d["beta"], d["z"], d["A_log"], sp.g_min)
    kda.device_status()
    assert torch.isfinite(o.float()).all() and torch.isfinite(S).all()
