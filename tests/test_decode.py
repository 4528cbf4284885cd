"""Split-KV decoding on the GPU against the oracle's decode (one key tile over the
whole cache: the safe softmax), through the C ABI.

Tolerances are the forward's: O max|err| <= 2e-3 (fp16) / 1.6e-2 (bf16) for N(0,1)
inputs, L max|err| <= 1e-4.  Cache rows at and past each sequence's length are
filled with NaN: any read of them into a result shows up as a non-finite value."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_22_gb300 import inputs
from tests.parity_util import TOL_L, TOL_O

pytestmark = pytest.mark.gpu


def run_decode(B, H, Hkv, Nmax, d, lens, dtype, seed=0, rows=None, scale=None):
    """GPU decode of the whole batch; the oracle on batch entries ``rows`` (None = all)."""
    import exact_io_aware_22_gb300 as fa
    x = inputs.make_decode_inputs(B, H, Hkv, Nmax, d, lens, dtype, seed=seed, fill=float("nan"))
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    q, kc, vc, cl = (x[n].cuda() for n in ("q", "k_cache", "v_cache", "cache_seqlens"))
    o, lse = fa.decode(q, kc, vc, cl, scale=scale)
    torch.cuda.synchronize()
    assert fa.device_status() == 0, "a kernel reported a bounded-wait timeout"
    o, lse = o.double().cpu().numpy(), lse.double().cpu().numpy()
    sel = list(range(B)) if rows is None else list(rows)
    xq = x["q"].double().numpy()[sel]
    xk = x["k_cache"].double().numpy()[sel]
    xv = x["v_cache"].double().numpy()[sel]
    o_ref, l_ref = oracle.decode(xq, xk, xv, x["cache_seqlens"].numpy()[sel], scale)
    o, lse = o[sel], lse[sel]
    assert np.isfinite(o).all(), "non-finite O: a row past a sequence's length was read"
    empty = l_ref == -np.inf
    assert (lse[empty] == -np.inf).all() and (o[empty] == 0).all()
    assert np.isfinite(lse[~empty]).all()
    rep = {"o": float(np.max(np.abs(o - o_ref), initial=0.0)),
           "lse": float(np.max(np.abs(lse[~empty] - l_ref[~empty]), initial=0.0))}
    assert rep["o"] <= TOL_O[dtype], rep
    assert rep["lse"] <= TOL_L, rep
    return rep


# (B, H, Hkv, Nmax, d, dtype, lens)
CASES = [
    (4, 32, 8, 1000, 128, "bf16", (1000, 1, 517, 64)),        # GQA 4: R = 4
    (3, 16, 2, 777, 128, "fp16", (0, 777, 300)),              # empty cache, GQA 8
    (2, 16, 1, 2000, 128, "bf16", (1999, 1234)),              # MQA: G = 16, two row groups
    (2, 8, 8, 513, 128, "fp16", (513, 17)),                   # MHA: R = 1
    (2, 6, 2, 300, 64, "bf16", (300, 129)),                   # G = 3: R = 1
    (3, 12, 2, 1500, 64, "fp16", (1, 33, 1500)),              # G = 6: R = 2
    (2, 8, 2, 640, 32, "bf16", (640, 255)),
    (1, 4, 4, 5000, 32, "fp16", (4097,)),
    (2, 4, 1, 16, 128, "bf16", (16, 15)),                     # shorter than one ring stage
    (5, 8, 4, 64, 64, "fp16", (0, 0, 0, 0, 0)),               # every cache empty
]


@pytest.mark.parametrize("case", CASES, ids=[str(c[:6]) + str(c[6][:3]) for c in CASES])
def test_decode(case):
    B, H, Hkv, Nmax, d, dt, lens = case
    print(case[:6], run_decode(B, H, Hkv, Nmax, d, lens, dt, seed=len(lens) + Nmax))


def test_decode_non_default_scale():
    print(run_decode(2, 8, 2, 700, 128, (700, 333), "bf16", seed=3, scale=0.3))


def test_decode_lengths_past_the_cache_are_clamped():
    import exact_io_aware_22_gb300 as fa
    x = inputs.make_decode_inputs(2, 4, 2, 100, 64, (100, 100), "bf16", seed=4)
    q, kc, vc = (x[n].cuda() for n in ("q", "k_cache", "v_cache"))
    o1, l1 = fa.decode(q, kc, vc, torch.tensor([100, 100], dtype=torch.int32, device="cuda"))
    o2, l2 = fa.decode(q, kc, vc, torch.tensor([5000, 100], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_full_size_sampled():
    # 16 sequences x 32 query heads over 8 K/V heads, caches of up to 32768 keys of
    # d = 128, bf16, lengths uniform in [Nmax/2, Nmax]; batch entries 0, 7, 15 compared
    # with every head
    B, H, Hkv, Nmax, d = 16, 32, 8, 32768, 128
    lens = tuple(int(n) for n in np.random.default_rng(2027).integers(Nmax // 2, Nmax + 1, B))
    print(run_decode(B, H, Hkv, Nmax, d, lens, "bf16", seed=1, rows=(0, 7, 15)))


def test_decode_caller_workspace_matches_library_allocation():
    import exact_io_aware_22_gb300 as fa
    B, H, Hkv, Nmax, d = 3, 16, 4, 900, 128
    x = inputs.make_decode_inputs(B, H, Hkv, Nmax, d, (900, 450, 3), "bf16", seed=6)
    q, kc, vc, cl = (x[n].cuda() for n in ("q", "k_cache", "v_cache", "cache_seqlens"))
    ws = torch.empty(fa.decode_workspace_size(B, H, Hkv, Nmax, d), dtype=torch.uint8,
                     device="cuda")
    o1, l1 = fa.decode(q, kc, vc, cl)
    o2, l2 = fa.decode(q, kc, vc, cl, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def run_decode_fp8(B, H, Hkv, Nmax, lens, dtype, seed=0, rows=None):
    """E4M3 caches: the oracle's decode of the dequantized caches (codes times their
    descale factors).  Only the cache is in 8 bits: the scores are exact products summed
    in fp32 and P is rounded to f16 for the tensor-core P.V product (half the 16-bit
    input's rounding or less), so the 16-bit decode tolerances hold."""
    import exact_io_aware_22_gb300 as fa
    d = 128
    x = inputs.make_decode_fp8_inputs(B, H, Hkv, Nmax, d, lens, dtype, seed=seed, fill_code=0x7F)
    scale = 1.0 / math.sqrt(d)
    q, k8, v8, cl = (x[n].cuda() for n in ("q", "k8", "v8", "cache_seqlens"))
    o, lse = fa.decode_fp8(q, k8, v8, cl, x["k_scale"], x["v_scale"], scale=scale)
    torch.cuda.synchronize()
    assert fa.device_status() == 0, "a kernel reported a bounded-wait timeout"
    o, lse = o.double().cpu().numpy(), lse.double().cpu().numpy()
    sel = list(range(B)) if rows is None else list(rows)
    kd = oracle.e4m3_values(x["k8"].numpy()[sel]) * x["k_scale"]
    vd = oracle.e4m3_values(x["v8"].numpy()[sel]) * x["v_scale"]
    o_ref, l_ref = oracle.decode(x["q"].double().numpy()[sel], kd, vd,
                                 x["cache_seqlens"].numpy()[sel], scale)
    o, lse = o[sel], lse[sel]
    assert np.isfinite(o).all(), "non-finite O: a row past a sequence's length was read"
    empty = l_ref == -np.inf
    assert (lse[empty] == -np.inf).all() and (o[empty] == 0).all()
    rep = {"o": float(np.max(np.abs(o - o_ref), initial=0.0)),
           "lse": float(np.max(np.abs(lse[~empty] - l_ref[~empty]), initial=0.0))}
    assert rep["o"] <= TOL_O[dtype], rep
    assert rep["lse"] <= TOL_L, rep
    return rep


FP8_CASES = [
    (4, 32, 8, 1000, "bf16", (1000, 1, 517, 64)),
    (3, 16, 2, 777, "fp16", (0, 777, 300)),
    (2, 16, 1, 2000, "bf16", (1999, 1234)),
    (2, 8, 8, 513, "fp16", (513, 17)),
    (2, 12, 2, 300, "bf16", (300, 31)),
    (2, 4, 1, 16, "bf16", (16, 15)),                          # shorter than one ring stage
    (5, 8, 4, 64, "fp16", (0, 0, 0, 0, 0)),                   # every cache empty
    (3, 24, 8, 2049, "fp16", (2049, 2048, 33)),               # G = 3, a 32-key stage plus one
]


@pytest.mark.parametrize("case", FP8_CASES, ids=[str(c[:5]) for c in FP8_CASES])
def test_decode_fp8_cache(case):
    B, H, Hkv, Nmax, dt, lens = case
    print(case[:5], run_decode_fp8(B, H, Hkv, Nmax, lens, dt, seed=Nmax))


def test_decode_fp8_full_size_sampled():
    B, H, Hkv, Nmax = 16, 32, 8, 32768
    lens = tuple(int(n) for n in np.random.default_rng(2027).integers(Nmax // 2, Nmax + 1, B))
    print(run_decode_fp8(B, H, Hkv, Nmax, lens, "bf16", seed=1, rows=(0, 7, 15)))
