"""Shared GPU-vs-oracle comparison for the parity tests.

Tolerances (max over every compared element):
  O:            max|err| <= 2e-3 (fp16), 1.6e-2 (bf16)   for N(0,1) inputs
  L:            max|err| <= 1e-4 (fp32 output)
  dQ, dK, dV:   max|err| / max|ref| <= 1e-2 (fp16), 3e-2 (bf16)
Two cases fall outside what those bounds were stated for:
  * Q, K ~ N(0, 4^2) (the stress inputs): rows are nearly one-hot, so |O| reaches
    max|V| (about 4.5) and the 16-bit rounding of P and of O grows with it.  The O
    bound is then multiplied by max(1, max|O_ref|).
  * N = 1: one key gives P = 1 and dS = dP - D = 0, so the reference dQ and dK are
    identically zero and the relative error is undefined.  Where max|ref| is below
    1e-6 of the size of a single term scale * |dP| * |k| (exact cancellation), the
    error is measured relative to that term size instead.
The oracle runs in fp64 on the 16-bit input values upcast exactly; the inputs
come from the shared seeded generator, never from the CUDA path.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from exact_io_aware_22_gb300 import inputs

TOL_O = {"fp16": 2e-3, "bf16": 1.6e-2}
TOL_L = 1e-4
TOL_G = {"fp16": 1e-2, "bf16": 3e-2}


def gpu_fwd_bwd(x: dict, causal: bool, scale: float, device="cuda", window: int = 0):
    import exact_io_aware_22_gb300 as fa
    q, k, v, do = (x[n].to(device) for n in ("q", "k", "v", "do"))
    o, lse = fa.fwd(q, k, v, causal=causal, scale=scale, window=window)
    dq, dk, dv = fa.bwd(q, k, v, o, lse, do, causal=causal, scale=scale, window=window)
    torch.cuda.synchronize()
    assert fa.device_status() == 0, "a kernel reported a bounded-wait timeout"
    return {n: t.float().cpu() for n, t in
            (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}


def _sel(t: torch.Tensor, heads):
    B, H = t.shape[:2]
    flat = t.reshape(B * H, *t.shape[2:])
    if heads is None:
        return flat.unsqueeze(0)
    return flat[list(heads)].unsqueeze(0)


def compare(B, H, N, d, dtype, causal, qk_std=1.0, heads=None, seed=0, scale=None, Hkv=None,
            window=0):
    """Run the CUDA path on the whole problem and the oracle on ``heads`` (flat b*H+h
    indices; None = all).  Returns the error report; asserts the tolerances.

    With ``Hkv`` (K/V heads shared by groups of H/Hkv query heads) ``heads`` lists
    flat K/V head indices b*Hkv+j, and each is compared with all its query heads.
    ``window`` > 0: causal sliding window of that many keys."""
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    x = inputs.make_inputs(B, H, N, d, dtype, seed=seed, qk_std=qk_std, Hkv=Hkv)
    g = gpu_fwd_bwd(x, causal, scale, window=window)
    if Hkv is None:
        q, k, v, do = (_sel(x[n].double(), heads).numpy() for n in ("q", "k", "v", "do"))
        o_ref, l_ref = oracle.fwd(q, k, v, causal, scale, window)
        dq_ref, dk_ref, dv_ref, _ = oracle.bwd(q, k, v, do, causal, scale, window)
        qheads = kvheads = heads
    else:
        grp = H // Hkv
        kvheads = heads
        qheads = None if heads is None else [j * grp + t for j in heads for t in range(grp)]
        q, do = (_sel(x[n].double(), qheads).numpy() for n in ("q", "do"))
        k, v = (_sel(x[n].double(), kvheads).numpy() for n in ("k", "v"))
        if heads is not None:   # the selected groups as one batch of len(heads) K/V heads
            q, do = (t.reshape(1, len(heads) * grp, N, d) for t in (q, do))
        o_ref, l_ref = oracle.fwd_gqa(q, k, v, causal, scale, window)
        dq_ref, dk_ref, dv_ref, _ = oracle.bwd_gqa(q, k, v, do, causal, scale, window)
    rep = {}
    # size of one dS_ij * k_j term: scale * max|dP| * max|k|, with |dP| <= |dO| |v|
    term = scale * float(np.max(np.linalg.norm(do, axis=-1)) * np.max(np.linalg.norm(v, axis=-1))
                         * max(np.max(np.abs(k)), np.max(np.abs(q))))
    for name, ref in (("o", o_ref), ("lse", l_ref), ("dq", dq_ref), ("dk", dk_ref), ("dv", dv_ref)):
        got = _sel(g[name], kvheads if name in ("dk", "dv") else qheads).double().numpy()
        got = got.reshape(ref.shape)
        assert np.isfinite(got).all(), f"{name}: non-finite values"
        err = float(np.max(np.abs(got - ref)))
        if name in ("dq", "dk", "dv"):
            mref = float(np.max(np.abs(ref)))
            err /= mref if mref >= 1e-6 * term else term
        rep[name] = err
    o_scale = 1.0 if qk_std == 1.0 else max(1.0, float(np.max(np.abs(o_ref))))
    rep["o_bound"] = TOL_O[dtype] * o_scale
    assert rep["o"] <= rep["o_bound"], rep
    assert rep["lse"] <= TOL_L, rep
    for n in ("dq", "dk", "dv"):
        assert rep[n] <= TOL_G[dtype], rep
    return rep


def compare_varlen(lens, H, d, dtype, causal, Hkv=None, window=0, seed=0, scale=None):
    """Packed variable-length sequences through fwd_varlen / bwd_varlen against the
    oracle, every sequence and head compared; same tolerances as ``compare``."""
    import exact_io_aware_22_gb300 as fa
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    x = inputs.make_packed_inputs(lens, H, d, dtype, seed=seed, Hkv=Hkv)
    cu = x["cu_seqlens"]
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    cug = cu.cuda()
    max_len = max(max(lens), 1)
    o, lse = fa.fwd_varlen(q, k, v, cug, max_len, causal=causal, scale=scale, window=window)
    dq, dk, dv = fa.bwd_varlen(q, k, v, o, lse, do, cug, max_len, causal=causal, scale=scale,
                               window=window)
    torch.cuda.synchronize()
    assert fa.device_status() == 0, "a kernel reported a bounded-wait timeout"
    xd = {n: x[n].double().numpy() for n in ("q", "k", "v", "do")}
    cun = cu.numpy()
    o_ref, l_ref = oracle.fwd_varlen(xd["q"], xd["k"], xd["v"], cun, causal, scale, window)
    dq_ref, dk_ref, dv_ref, _ = oracle.bwd_varlen(xd["q"], xd["k"], xd["v"], xd["do"], cun, causal,
                                                  scale, window)
    rep = {}
    for name, got, ref in (("o", o, o_ref), ("lse", lse, l_ref), ("dq", dq, dq_ref),
                           ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
        g = got.double().cpu().numpy()
        assert np.isfinite(g).all(), f"{name}: non-finite values"
        err = float(np.max(np.abs(g - ref)))
        if name in ("dq", "dk", "dv"):
            err /= max(float(np.max(np.abs(ref))), 1e-30)
        rep[name] = err
    assert rep["o"] <= TOL_O[dtype], rep
    assert rep["lse"] <= TOL_L, rep
    for n in ("dq", "dk", "dv"):
        assert rep[n] <= TOL_G[dtype], rep
    return rep
