"""The element-wise O bound the stress parity cases use (tests/parity_util.py,
``o_bound_elementwise``), checked on the CPU against an emulation of the forward
kernel's arithmetic: fp32 scores, base-2 exponentials with a per-row maximum,
P rounded to the 16-bit input type before P.V, fp32 sums, O rounded at the end.

Two pins: the bound holds for that arithmetic on Q, K ~ N(0, 4^2) inputs (large
row maxima, nearly one-hot rows), and it is tight enough to reject a plausible
mistake, P rounded to bf16 while the inputs (and the bound) are fp16."""
import math

import numpy as np
import torch

import oracle
from exact_io_aware_22_gb300 import inputs
from tests.parity_util import allowed_keys, o_bound_elementwise


def _emulate(q, k, v, causal, scale, p_dtype):
    t = torch.float16 if p_dtype == "fp16" else torch.bfloat16
    _, nh, N, d = q.shape
    ok = torch.from_numpy(allowed_keys(N, causal))
    c = torch.tensor(scale * 1.4426950408889634, dtype=torch.float32)
    out = np.empty_like(q)
    for h in range(nh):
        q32, k32, v32 = (torch.from_numpy(a[0, h]).float() for a in (q, k, v))
        s = torch.where(ok, q32 @ k32.T, torch.tensor(-math.inf))
        m = s.max(dim=1, keepdim=True).values * c
        p = torch.exp2(s * c - m)
        acc = p.to(t).float() @ v32
        out[0, h] = (acc / p.sum(dim=1, keepdim=True)).to(t).double().numpy()
    return out


def _case(dtype, N, d, causal, seed, p_dtype):
    B, H = 1, 2
    x = inputs.make_inputs(B, H, N, d, dtype, seed=seed, qk_std=4.0)
    q, k, v = (x[n].double().reshape(1, B * H, N, d).numpy() for n in ("q", "k", "v"))
    scale = 1.0 / math.sqrt(d)
    o_ref, l_ref = oracle.fwd(q, k, v, causal, scale)
    got = _emulate(q, k, v, causal, scale, p_dtype)
    bound = o_bound_elementwise(q, k, v, o_ref, l_ref, causal, scale, dtype)
    return float(np.max(np.abs(got - o_ref) / (1.25 * bound + 1e-6)))


def test_bound_holds_for_kernel_arithmetic():
    for dtype in ("fp16", "bf16"):
        for N, d, causal, seed in ((640, 128, True, 3), (383, 64, False, 4), (500, 32, True, 0)):
            r = _case(dtype, N, d, causal, seed, dtype)
            assert r <= 1.0, (dtype, N, d, causal, r)


def test_bound_rejects_coarser_p():
    for N, d, seed in ((640, 128, 3), (500, 32, 0)):
        assert _case("fp16", N, d, True, seed, "bf16") > 1.0, (N, d)
