"""The pipelined host-buffer forward (copies of one piece overlapping the compute of its
neighbours) returns exactly what one device-resident call returns: pieces end at multiples
of 64 tokens and carry the fp32 state, or hold whole sequences."""
import numpy as np
import pytest

from serving_kda_chunkwise_gb300 import inputs

pytestmark = pytest.mark.gpu


def _host(t):
    return t.cpu().pin_memory()


@pytest.mark.parametrize("T,segments,dtype,d,with_state", [
    (4096 + 37, 3, "bf16", 128, True), (1024, 8, "bf16", 128, False), (64, 4, "bf16", 128, True),
    (1000, 4, "f32", 64, True)])
def test_single_sequence_pieces_match_one_call(T, segments, dtype, d, with_state):
    import torch
    from serving_kda_chunkwise_gb300 import kda
    sp = inputs.forward_spec(seed=31, B=1, T=T, H=3, dk=d, dv=d, dtype=dtype,
                             with_state=with_state)
    dev = sp.to_device("cuda")
    o_ref, S_ref = kda.fwd_chunked(dev["q"], dev["k"], dev["v"], dev["beta"], dev["z"],
                                   dev["A_log"], sp.g_min, S0=dev["S0"], cu_seqlens=dev["cu"])
    torch.cuda.synchronize()
    h = {k: _host(dev[k]) for k in ("q", "k", "v", "beta", "z")}
    o, S = kda.fwd_chunked_host(h["q"], h["k"], h["v"], h["beta"], h["z"], dev["A_log"].cpu(),
                                sp.g_min, S0=None if dev["S0"] is None else _host(dev["S0"]),
                                segments=segments)
    assert torch.equal(o, o_ref.cpu())
    assert torch.equal(S, S_ref.cpu())


def test_varlen_groups_match_one_call():
    import torch
    from serving_kda_chunkwise_gb300 import kda
    sp = inputs.forward_spec(seed=32, H=2, dk=128, dv=128, dtype="bf16",
                             lengths=[100, 64, 1, 300, 0, 129, 77], with_state=True)
    d = sp.to_device("cuda")
    o_ref, S_ref = kda.fwd_chunked(d["q"], d["k"], d["v"], d["beta"], d["z"], d["A_log"],
                                   sp.g_min, S0=d["S0"], cu_seqlens=d["cu"])
    torch.cuda.synchronize()
    h = {k: _host(d[k]) for k in ("q", "k", "v", "beta", "z")}
    o, S = kda.fwd_chunked_host(h["q"], h["k"], h["v"], h["beta"], h["z"], d["A_log"].cpu(),
                                sp.g_min, S0=None if d["S0"] is None else _host(d["S0"]),
                                cu_seqlens=d["cu"].cpu(), segments=3)
    assert torch.equal(o, o_ref.cpu())
    assert torch.equal(S, S_ref.cpu())
