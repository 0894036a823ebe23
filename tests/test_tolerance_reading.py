"""Pins the reading of the bf16 tolerance ("2e-2 absolute after per-head normalisation").

The exact result, rounded once to bf16, must pass any sensible reading of a bf16 output
tolerance.  On the seeded B=2, T=4096, H=16, d=128 workload the outputs are heavy-tailed
(max|o| / rms(o) ~ 20 per head), so the plain reading max|o_bf16 - o| / rms > 2e-2 for the
exact answer itself; the reading used by the parity tests allows on top of 2e-2 of rms only
the output's own rounding, at most half a bf16 ulp (<= 2^-8 |o|), and so accepts the
rounded exact answer with zero excess, while still rejecting a 5% error on the largest
output or a 5%-of-rms error on a typical one.
"""
import numpy as np

import oracle
from serving_kda_chunkwise_gb300 import inputs
from kda_testutil import BF16_NORM_TOL, BF16_RMS_TOL, bf16_norm_err, bf16_rms_err, plain_norm_err


def test_bf16_rounding_of_exact_result():
    inp = inputs.workload("fwd_bf16_B2_T4096_H16_d128")
    o, _ = oracle.recurrent(inp.q.values, inp.k.values, inp.v.values, inp.beta.values,
                            inp.z.values, inp.A_log, inp.g_min, S0=inp.S0,
                            cu_seqlens=inp.cu_seqlens, want_state=False)
    o_b = inputs.bf16_bits_to_f32(inputs.f32_to_bf16_bits(o.astype(np.float32))).astype(
        np.float64)
    plain = max(plain_norm_err(o_b[a:b, h], o[a:b, h])
                for a, b in zip(inp.cu_seqlens[:-1], inp.cu_seqlens[1:]) for h in range(inp.H))
    ours = max(bf16_norm_err(o_b[a:b, h], o[a:b, h])
               for a, b in zip(inp.cu_seqlens[:-1], inp.cu_seqlens[1:]) for h in range(inp.H))
    assert plain > BF16_NORM_TOL       # the plain reading rejects the exact answer
    assert ours < 1e-6                 # ours accepts it
    a, b = inp.cu_seqlens[0], inp.cu_seqlens[1]
    ref = o[a:b, 0]
    rms = np.sqrt(np.mean(ref ** 2))
    big = np.unravel_index(np.argmax(np.abs(ref)), ref.shape)
    bad = o_b[a:b, 0].copy()
    bad[big] *= 1.05                                   # 5% off on the largest output
    assert bf16_norm_err(bad, ref) > BF16_NORM_TOL
    typical = np.unravel_index(np.argmin(np.abs(np.abs(ref) - rms)), ref.shape)
    bad = o_b[a:b, 0].copy()
    bad[typical] += 0.05 * rms                         # 5%-of-rms off on a typical output
    assert bf16_norm_err(bad, ref) > BF16_NORM_TOL
    bad = o_b[a:b, 0] * 1.02                           # a systematic 2% scale error
    assert bf16_rms_err(bad, ref) > BF16_RMS_TOL
