"""Attention forward on 8-bit E4M3 inputs against the oracle, through the C ABI.

The oracle is the exact attention (fp64) of the values the codes stand for.  The
kernel rounds P to E4M3 before the P V product, so the tolerance comes from that
rounding (round to nearest even, 3 mantissa bits):
  * a probability p >= 2^-6 in the kernel's running-max scale is a normal E4M3
    value and is off by at most 2^-4 p; a smaller one is off by at most 2^-10
    (half the subnormal spacing 2^-9).  The kernel's running max never exceeds the
    row's true maximum, so in the true-maximum scale p_j = exp(s_j - max s) each
    term is off by at most 2^-4 p_j + 2^-10 [p_j < 2^-6];
  * l sums the unrounded p, so O_ic is off by at most
        E_ic = sum_j (2^-4 p_j + 2^-10 [p_j < 2^-6]) |v_jc| / l  (+ bf16 rounding of O)
    and the test checks every element against 1.25 E_ic + 2^-8 |O_ic| + 1e-6;
  * the rounding errors have mean 0 and are at most the bounds above, so the root
    mean square error over a head is at most the root of the mean of
    sum_j (bound_j)^2 / 3 |v_jc|^2 / l^2; the test checks it, which a systematic
    error anywhere would exceed;
  * L carries no P rounding: S is an fp32 sum of 128 exact products, so
    |dL| <= scale q_scale k_scale 128 2^-24 max_j sum_k |q_k k_jk|, plus 1e-5 for
    the exp2/log2 steps.
Inputs come from the shared generator (CPU torch rounding to E4M3), never from the
GPU quantiser, which is tested on its own bit for bit against torch."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_22_gb300 import inputs

pytestmark = pytest.mark.gpu


def _bounds(q, k, v, causal, scale_eff, rows):
    """Per-element bound E (rows x d), its RMS prediction, and the L bound, for one
    head: q (N, d), k, v (N, d) dequantized fp64; rows: the query rows checked."""
    N = k.shape[0]
    s = (q[rows] @ k.T) * scale_eff
    if causal:
        s = np.where(np.arange(N)[None, :] <= np.asarray(rows)[:, None], s, -np.inf)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    l = p.sum(axis=1, keepdims=True)
    bj = 2.0 ** -4 * p + 2.0 ** -10 * ((p < 2.0 ** -6) & (p > 0))
    av = np.abs(v)
    E = (bj @ av) / l
    var = ((bj ** 2) / 3.0 @ (v ** 2)) / l ** 2
    acc = (np.abs(q[rows]) @ np.abs(k).T) * scale_eff
    if causal:
        acc = np.where(np.arange(N)[None, :] <= np.asarray(rows)[:, None], acc, 0.0)
    lb = 1e-5 + 128 * 2.0 ** -24 * acc.max(axis=1)
    return E, var, lb


def run_fp8(B, H, Hkv, N, causal, heads=None, seed=0, scale=None, chunk=1024):
    import exact_io_aware_22_gb300 as fa
    d = 128
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    x = inputs.make_fp8_inputs(B, H, N, d, seed=seed, Hkv=Hkv)
    qs, ks, vs = x["q_scale"], x["k_scale"], x["v_scale"]
    q8, k8, vt8 = (x[n].cuda() for n in ("q8", "k8", "vt8"))
    o, lse = fa.fwd_fp8(q8, k8, vt8, qs, ks, vs, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.device_status() == 0, "a kernel reported a bounded-wait timeout"
    o = o.double().cpu().numpy().reshape(B * H, N, d)
    lse = lse.double().cpu().numpy().reshape(B * H, N)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    g = H // Hkv
    qd = oracle.e4m3_values(x["q8"].numpy()).reshape(B * H, N, d) * qs
    kd = oracle.e4m3_values(x["k8"].numpy()).reshape(B * Hkv, N, d) * ks
    vd = oracle.e4m3_values(x["v8"].numpy()).reshape(B * Hkv, N, d) * vs
    rep = {"o_max_over_bound": 0.0, "rms_over_pred": 0.0, "l_max_over_bound": 0.0, "o_max": 0.0}
    for hf in (range(B * H) if heads is None else heads):
        hk = (hf // H) * Hkv + (hf % H) // g
        o_ref, l_ref = oracle.fwd_fp8(x["q8"].numpy().reshape(B * H, N, d)[hf][None, None],
                                      x["k8"].numpy().reshape(B * Hkv, N, d)[hk][None, None],
                                      x["v8"].numpy().reshape(B * Hkv, N, d)[hk][None, None],
                                      qs, ks, vs, causal, scale)
        o_ref, l_ref = o_ref[0, 0], l_ref[0, 0]
        err = np.abs(o[hf] - o_ref)
        sq, var_sum = 0.0, 0.0
        for r0 in range(0, N, chunk):
            rows = np.arange(r0, min(N, r0 + chunk))
            E, var, lb = _bounds(qd[hf], kd[hk], vd[hk], causal, scale, rows)
            tol = 1.25 * E + 2.0 ** -8 * np.abs(o_ref[rows]) + 1e-6
            rep["o_max_over_bound"] = max(rep["o_max_over_bound"], float(np.max(err[rows] / tol)))
            rep["l_max_over_bound"] = max(rep["l_max_over_bound"],
                                          float(np.max(np.abs(lse[hf, rows] - l_ref[rows]) / lb)))
            sq += float(np.sum(err[rows] ** 2))
            var_sum += float(np.sum(var)) + float(np.sum((2.0 ** -9 * o_ref[rows]) ** 2))
        rep["rms_over_pred"] = max(rep["rms_over_pred"], math.sqrt(sq / var_sum))
        rep["o_max"] = max(rep["o_max"], float(err.max()))
    assert rep["o_max_over_bound"] <= 1.0, rep
    assert rep["rms_over_pred"] <= 1.0, rep
    assert rep["l_max_over_bound"] <= 1.0, rep
    return rep


# (B, H, Hkv, N, causal)
CASES = [
    (1, 2, 2, 256, True),
    (1, 2, 2, 256, False),
    (2, 4, 2, 384, True),          # GQA, ragged query-tile pairs
    (1, 4, 1, 1008, False),        # MQA, N off the 128-key tile
    (1, 2, 2, 16, True),           # one partial tile
    (1, 2, 1, 2064, True),
]


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_fwd_fp8(case):
    B, H, Hkv, N, causal = case
    print(case, run_fp8(B, H, Hkv, N, causal, seed=N))


def test_fwd_fp8_full_size_sampled():
    # 1 x 32 heads x 8192 x 128 causal (the FP8 bench workload); heads 0, 16, 31 in full
    print(run_fp8(1, 32, 32, 8192, True, heads=(0, 16, 31), seed=5))


def test_fwd_fp8_non_default_scale():
    print(run_fp8(1, 2, 2, 512, True, seed=9, scale=0.05))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("transpose", [False, True])
def test_quantize_matches_torch(dtype, transpose):
    import exact_io_aware_22_gb300 as fa
    g = torch.Generator().manual_seed(3)
    x = (torch.randn((3, 2, 100, 72), generator=g) * 3).to(inputs.DTYPES[dtype])
    inv = 448.0 / float(x.float().abs().max())
    got = fa.quantize_fp8(x.cuda(), inv, transpose=transpose).cpu()
    ref = (x.float() * torch.tensor(inv, dtype=torch.float32)).to(torch.float8_e4m3fn)
    ref = ref.view(torch.uint8)
    if transpose:
        ref = ref.transpose(-1, -2).contiguous()
    assert torch.equal(got, ref)


def test_quantize_saturates():
    import exact_io_aware_22_gb300 as fa
    x = torch.tensor([[1000.0, -1000.0, 448.0, 0.0]], dtype=torch.bfloat16)
    got = fa.quantize_fp8(x.cuda(), 1.0).cpu()
    assert got.tolist() == [[0x7E, 0xFE, 0x7E, 0x00]]
