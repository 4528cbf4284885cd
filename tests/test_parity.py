"""CUDA path vs the fp64 oracle, through the C ABI, on the GPU.

The workload configurations (sizes the oracle finishes in seconds: every head)
and the full-size long-context ones (sampled heads, each compared in full:
heads are independent), plus ragged and degenerate sizes."""
import pytest

from tests.parity_util import compare, compare_varlen

pytestmark = pytest.mark.gpu


# (B, H, N, d, dtype, causal, qk_std, heads)
WORKLOAD_CASES = {
    "tiny_full_d64_fp16": (1, 1, 128, 64, "fp16", False, 1.0, None),
    "ragged_causal_d32_fp16": (4, 8, 1000, 32, "fp16", True, 1.0, None),
    "ragged_causal_d32_fp16_stress": (4, 8, 1000, 32, "fp16", True, 4.0, None),
    "gpt2m_causal_d64_fp16": (8, 16, 1024, 64, "fp16", True, 1.0, None),
    "n4k_full_d128_bf16": (2, 16, 4096, 128, "bf16", False, 1.0, (0, 8, 31)),
    "n4k_causal_d128_bf16": (2, 16, 4096, 128, "bf16", True, 1.0, (0, 8, 31)),
    "n8k_causal_d128_bf16": (1, 32, 8192, 128, "bf16", True, 1.0, (0, 16, 31)),
    "n16k_causal_d128_bf16": (1, 32, 16384, 128, "bf16", True, 1.0, (0, 16, 31)),
}


@pytest.mark.parametrize("name", list(WORKLOAD_CASES))
def test_workload(name):
    B, H, N, d, dt, causal, std, heads = WORKLOAD_CASES[name]
    rep = compare(B, H, N, d, dt, causal, qk_std=std, heads=heads)
    print(name, rep)


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 2, 127, 129, 257, 383])
def test_ragged_and_degenerate(N, d, dtype, causal):
    compare(1, 2, N, d, dtype, causal, seed=N)


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_multi_batch_head(d, causal):
    compare(2, 3, 300, d, "bf16", causal, seed=7)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_stress_row_maxima(dtype):
    # Q, K ~ N(0, 4^2): large row maxima exercise the running-max update
    compare(2, 2, 640, 128, dtype, True, qk_std=4.0, seed=3)
    compare(2, 2, 640, 64, dtype, False, qk_std=4.0, seed=4)


def test_non_default_scale():
    compare(1, 2, 256, 64, "fp16", True, scale=0.05, seed=5)
    compare(1, 2, 256, 64, "bf16", False, scale=0.4, seed=6)


# Grouped-query / multi-query attention: (B, H, Hkv, N, d, dtype, causal)
GQA_CASES = [
    (2, 8, 2, 300, 128, "bf16", True),
    (1, 8, 1, 257, 128, "fp16", False),     # MQA
    (2, 6, 3, 200, 64, "fp16", True),
    (1, 4, 2, 129, 32, "bf16", True),
    (1, 4, 2, 1, 64, "fp16", True),         # one key
    (1, 16, 4, 2048, 128, "bf16", True),
]


@pytest.mark.parametrize("case", GQA_CASES, ids=[str(c) for c in GQA_CASES])
def test_gqa(case):
    B, H, Hkv, N, d, dt, causal = case
    print(case, compare(B, H, N, d, dt, causal, seed=11, Hkv=Hkv))


def test_gqa_full_size_sampled():
    # 1 x 32 query heads x 8 K/V heads x 8192 x 128, bf16 causal; K/V heads 0 and 7, each
    # with its four query heads, compared in full
    print(compare(1, 32, 8192, 128, "bf16", True, heads=(0, 7), Hkv=8))


# Causal sliding window of W keys: (B, H, Hkv, N, d, dtype, W)
WINDOW_CASES = [
    (1, 2, 2, 300, 128, "bf16", 1),          # every row sees only itself
    (1, 2, 2, 300, 128, "bf16", 64),
    (1, 2, 2, 256, 128, "fp16", 128),        # window of exactly one tile
    (1, 2, 2, 257, 128, "fp16", 127),
    (2, 2, 2, 1000, 64, "fp16", 200),
    (1, 2, 2, 383, 32, "bf16", 100),
    (1, 4, 2, 517, 128, "bf16", 129),        # with shared K/V heads
    (1, 2, 2, 700, 128, "bf16", 333),
    (1, 2, 2, 300, 64, "bf16", 5000),        # window longer than N: plain causal
    (1, 8, 2, 2048, 64, "bf16", 300),        # d = 64 with shared K/V heads, many tiles
]


@pytest.mark.parametrize("case", WINDOW_CASES, ids=[str(c) for c in WINDOW_CASES])
def test_sliding_window(case):
    B, H, Hkv, N, d, dt, W = case
    print(case, compare(B, H, N, d, dt, True, seed=13, Hkv=None if Hkv == H else Hkv, window=W))


def test_sliding_window_full_size_sampled():
    # 1 x 32 query heads x 8 K/V heads x 16384 x 128, bf16, window 4096; K/V heads 0 and 7
    # compared in full with their query heads
    print(compare(1, 32, 16384, 128, "bf16", True, heads=(0, 7), Hkv=8, window=4096))


# Packed variable-length batches: (lengths, H, Hkv, d, dtype, causal, window)
VARLEN_CASES = [
    ((1, 127, 128, 129, 500, 37), 2, 2, 128, "bf16", True, 0),
    ((300, 0, 64, 257), 4, 2, 128, "fp16", True, 0),        # an empty sequence, shared K/V
    ((200, 383, 1), 2, 2, 128, "bf16", False, 0),
    ((700, 90, 333), 4, 1, 128, "bf16", True, 100),          # MQA with a window
    ((129, 64, 255), 2, 2, 64, "fp16", True, 0),
    ((96, 400), 3, 1, 64, "bf16", False, 0),
    ((33, 250, 130), 2, 2, 32, "fp16", True, 50),
    ((1000,), 2, 2, 128, "bf16", True, 0),                   # one sequence
]


@pytest.mark.parametrize("case", VARLEN_CASES, ids=[str(c) for c in VARLEN_CASES])
def test_varlen(case):
    lens, H, Hkv, d, dt, causal, W = case
    print(case, compare_varlen(lens, H, d, dt, causal, Hkv=Hkv, window=W, seed=17))


def test_varlen_many_sequences():
    # 32 sequences from 1 to 2000 tokens, 8 query heads over 2 K/V heads, d = 128
    import numpy as np
    lens = tuple(int(x) for x in np.random.default_rng(5).integers(1, 2000, 32))
    print(compare_varlen(lens, 8, 128, "bf16", True, Hkv=2, seed=19))


def test_varlen_full_size_sampled():
    """The packed workload the bench times (64 sequences of 256..8192 tokens drawn with
    seed 2026, 270,160 tokens, 32 query heads over 8 K/V heads, d = 128 bf16, causal),
    run whole; sampled against the oracle: the longest sequence with K/V head 0 and
    its four query heads, the shortest with K/V head 7.  Sequences and K/V heads are
    independent, so each sample is a dense GQA problem of its own, compared in full."""
    import math
    import numpy as np
    import torch
    import exact_io_aware_22_gb300 as fa
    import oracle
    from exact_io_aware_22_gb300 import inputs
    from tests.parity_util import TOL_G, TOL_L, TOL_O
    lens = [int(x) for x in np.random.default_rng(2026).integers(256, 8193, 64)]
    H, Hkv, d = 32, 8, 128
    grp = H // Hkv
    scale = 1.0 / math.sqrt(d)
    x = inputs.make_packed_inputs(lens, H, d, "bf16", seed=0, Hkv=Hkv)
    cu = x["cu_seqlens"]
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    cug = cu.cuda()
    o, lse = fa.fwd_varlen(q, k, v, cug, max(lens), causal=True, scale=scale)
    dq, dk, dv = fa.bwd_varlen(q, k, v, o, lse, do, cug, max(lens), causal=True, scale=scale)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    got_all = {"o": o.cpu(), "lse": lse.cpu(), "dq": dq.cpu(), "dk": dk.cpu(), "dv": dv.cpu()}
    for s_idx, g in ((int(np.argmax(lens)), 0), (int(np.argmin(lens)), Hkv - 1)):
        a, b = int(cu[s_idx]), int(cu[s_idx + 1])
        qh = slice(g * grp, (g + 1) * grp)
        # (rows, heads, d) -> (1, heads, rows, d) in fp64
        sel = lambda t, hs: t[a:b, hs].double().permute(1, 0, 2).unsqueeze(0).numpy()
        qs, dos = sel(x["q"], qh), sel(x["do"], qh)
        ks, vs = sel(x["k"], slice(g, g + 1)), sel(x["v"], slice(g, g + 1))
        o_ref, l_ref = oracle.fwd_gqa(qs, ks, vs, True, scale)
        dq_ref, dk_ref, dv_ref, _ = oracle.bwd_gqa(qs, ks, vs, dos, True, scale)
        got = {"o": sel(got_all["o"], qh), "lse": got_all["lse"][qh, a:b].double().numpy(),
               "dq": sel(got_all["dq"], qh), "dk": sel(got_all["dk"], slice(g, g + 1)),
               "dv": sel(got_all["dv"], slice(g, g + 1))}
        rep = {}
        for name, ref in (("o", o_ref), ("lse", l_ref), ("dq", dq_ref), ("dk", dk_ref),
                          ("dv", dv_ref)):
            gv = got[name].reshape(ref.shape)
            assert np.isfinite(gv).all(), name
            err = float(np.max(np.abs(gv - ref)))
            if name in ("dq", "dk", "dv"):
                err /= float(np.max(np.abs(ref)))
            rep[name] = err
        print("sequence", s_idx, "length", b - a, "K/V head", g, rep)
        assert rep["o"] <= TOL_O["bf16"] and rep["lse"] <= TOL_L, rep
        for n in ("dq", "dk", "dv"):
            assert rep[n] <= TOL_G["bf16"], rep


def test_d64_full_size_sampled():
    # 1 x 16 x 8192 x 64 bf16 causal (the d = 64 backward on many query tiles per key
    # block); heads 0 and 15 compared in full
    print(compare(1, 16, 8192, 64, "bf16", True, heads=(0, 15)))


def test_d32_full_size_sampled():
    # 2 x 8 x 4096 x 32 fp16 causal with shared K/V heads (4 query heads per K/V head);
    # K/V heads 0 and 3 compared in full with their query heads
    print(compare(2, 8, 4096, 32, "fp16", True, heads=(0, 3), Hkv=2))
