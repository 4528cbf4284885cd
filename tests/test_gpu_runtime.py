"""GPU runtime behaviour of the C ABI: output guards, determinism, workspace
handling, streams, and the bounded-wait failure detection (no fault)."""
import math

import pytest
import torch

from exact_io_aware_22_gb300 import inputs

pytestmark = pytest.mark.gpu


def _fa():
    import exact_io_aware_22_gb300 as fa
    return fa


@pytest.mark.parametrize("N", [1, 129, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_nan_prefill_and_canaries(N, causal):
    """Outputs pre-filled with NaN are completely overwritten; memory past the end
    of every output is untouched."""
    fa = _fa()
    B, H, d = 1, 2, 64
    x = inputs.make_inputs(B, H, N, d, "bf16", seed=1)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    n = B * H * N * d
    pad = 4096
    canary = -12345.0

    def guarded(count, dtype):
        buf = torch.full((count + pad,), float("nan"), dtype=dtype, device="cuda")
        buf[count:] = canary
        return buf

    ob, lb = guarded(n, torch.bfloat16), guarded(B * H * N, torch.float32)
    o, lse = ob[:n].view(B, H, N, d), lb[:B * H * N].view(B, H, N)
    fa.fwd(q, k, v, causal=causal, out=o, lse=lse)
    gb = [guarded(n, torch.bfloat16) for _ in range(3)]
    dq, dk, dv = (g[:n].view(B, H, N, d) for g in gb)
    fa.bwd(q, k, v, o, lse, do, causal=causal, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    for buf, count in [(ob, n), (lb, B * H * N)] + [(g, n) for g in gb]:
        assert torch.isfinite(buf[:count].float()).all()
        stored = torch.tensor(canary, dtype=buf.dtype).float().item()   # canary as the dtype holds it
        assert (buf[count:].float() == stored).all()


@pytest.mark.parametrize("B,H,N,d", [(2, 4, 777, 128), (4, 16, 1500, 64), (8, 8, 1000, 32),
                                     (4, 8, 1000, 32)])
def test_deterministic(B, H, N, d):
    """Twice the same inputs, bit-identical results.  At d <= 64 the kernels are
    persistent and take tiles in whatever order the hardware hands them out; every
    tile still writes its outputs alone, with no atomics, so the order cannot show."""
    fa = _fa()
    x = inputs.make_inputs(B, H, N, d, "bf16", seed=2)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    outs = []
    for _ in range(2):
        o, lse = fa.fwd(q, k, v, causal=True)
        dq, dk, dv = fa.bwd(q, k, v, o, lse, do, causal=True)
        outs.append([t.clone() for t in (o, lse, dq, dk, dv)])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_explicit_workspace_and_side_stream():
    fa = _fa()
    B, H, N, d = 2, 2, 500, 32
    x = inputs.make_inputs(B, H, N, d, "fp16", seed=3)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.fwd(q, k, v, causal=True)
    ref = fa.bwd(q, k, v, o, lse, do, causal=True)
    ws = torch.empty(fa.bwd_workspace_size(B, H, N, d, True), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o2, lse2 = fa.fwd(q, k, v, causal=True)
        got = fa.bwd(q, k, v, o2, lse2, do, causal=True, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    for a, b in zip(ref, got):
        assert torch.equal(a, b)


def test_bounded_wait_reports_timeout_and_context_survives():
    fa = _fa()
    assert fa.device_status() == 0
    assert fa.selftest_timeout(2_000_000) == 5          # FA_ERR_TIMEOUT, no fault
    assert fa.device_status() == 0                       # read clears the word
    x = inputs.make_inputs(1, 1, 256, 64, "fp16", seed=4)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = fa.fwd(q, k, v, causal=False)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all() and fa.device_status() == 0


def test_errors_raise_before_launch():
    fa = _fa()
    q = torch.zeros(1, 1, 64, 48, dtype=torch.float16, device="cuda")
    with pytest.raises(fa.FAError, match="UNSUPPORTED"):
        fa.fwd(q, q.clone(), q.clone())
    q = torch.zeros(1, 1, 64, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(fa.FAError, match="INVALID"):
        fa.fwd(q, q.clone(), q.clone(), scale=-1.0)


def test_gqa_entry_points_with_equal_heads_match_mha():
    """fa_fwd_gqa / fa_bwd_gqa with Hkv == H compute what fa_fwd / fa_bwd compute, bit
    for bit (the same kernels run with groups of one)."""
    import ctypes
    import exact_io_aware_22_gb300 as fa
    from exact_io_aware_22_gb300 import inputs
    B, H, N, d = 2, 4, 383, 128
    x = inputs.make_inputs(B, H, N, d, "bf16", seed=21)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.fwd(q, k, v, causal=True)
    dq, dk, dv = fa.bwd(q, k, v, o, lse, do, causal=True)
    lib = fa.load_library()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    o2, lse2 = torch.empty_like(o), torch.empty_like(lse)
    scale = 1.0 / d ** 0.5
    assert lib.fa_fwd_gqa(p(q), p(k), p(v), p(o2), p(lse2), B, H, H, N, d, 1, scale, 1, stream) == 0
    dq2, dk2, dv2 = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    assert lib.fa_bwd_gqa(p(q), p(k), p(v), p(o), p(do), p(lse), p(dq2), p(dk2), p(dv2), None, 0,
                          B, H, H, N, d, 1, scale, 1, stream) == 0
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    for a, b in ((o, o2), (lse, lse2), (dq, dq2), (dk, dk2), (dv, dv2)):
        assert torch.equal(a, b)


def _guarded(count, dtype, pad=4096, canary=-12345.0):
    buf = torch.full((count + pad,), float("nan"), dtype=dtype, device="cuda")
    buf[count:] = canary
    return buf


def _check_guard(buf, count, canary=-12345.0):
    stored = torch.tensor(canary, dtype=buf.dtype).float().item()
    head, tail = buf[:count].float(), buf[count:].float()
    return bool(torch.isfinite(head).all()) and bool((tail == stored).all())


@pytest.mark.parametrize("fp8_cache", [False, True])
def test_decode_outputs_guarded_and_deterministic(fp8_cache):
    """Split-KV decoding overwrites every O and L element (pre-filled with NaN; an empty
    cache gives O = 0, L = -inf), writes nothing past them, and repeats bit for bit."""
    fa = _fa()
    B, H, Hkv, Nmax, d = 3, 16, 4, 1500, 128
    lens = (1500, 0, 333)
    if fp8_cache:
        x = inputs.make_decode_fp8_inputs(B, H, Hkv, Nmax, d, lens, "bf16", seed=8)
        kc, vc = x["k8"].cuda(), x["v8"].cuda()
    else:
        x = inputs.make_decode_inputs(B, H, Hkv, Nmax, d, lens, "bf16", seed=8)
        kc, vc = x["k_cache"].cuda(), x["v_cache"].cuda()
    q, cl = x["q"].cuda(), x["cache_seqlens"].cuda()

    def run():
        ob, lb = _guarded(B * H * d, torch.bfloat16), _guarded(B * H, torch.float32)
        o, lse = ob[:B * H * d].view(B, H, d), lb[:B * H].view(B, H)
        if fp8_cache:
            fa.decode_fp8(q, kc, vc, cl, x["k_scale"], x["v_scale"], out=o, lse=lse)
        else:
            fa.decode(q, kc, vc, cl, out=o, lse=lse)
        torch.cuda.synchronize()
        return ob, lb, o.clone(), lse.clone()

    ob, lb, o1, l1 = run()
    assert fa.device_status() == 0
    assert _check_guard(ob, B * H * d)
    assert bool((lb[B * H:] == -12345.0).all())
    assert bool(torch.isfinite(lb[:B * H].view(B, H)[[0, 2]]).all())
    assert bool((lb[:B * H].view(B, H)[1] == -float("inf")).all())
    _, _, o2, l2 = run()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_fwd_fp8_outputs_guarded_and_deterministic():
    """The FP8 forward overwrites every O and L element, writes nothing past them, and
    repeats bit for bit."""
    fa = _fa()
    B, H, N, d = 1, 4, 400, 128
    x = inputs.make_fp8_inputs(B, H, N - N % 16, d, seed=9, Hkv=2)
    N = N - N % 16
    q8, k8, vt8 = (x[n].cuda() for n in ("q8", "k8", "vt8"))

    def run():
        ob, lb = _guarded(B * H * N * d, torch.bfloat16), _guarded(B * H * N, torch.float32)
        o, lse = ob[:B * H * N * d].view(B, H, N, d), lb[:B * H * N].view(B, H, N)
        fa.fwd_fp8(q8, k8, vt8, x["q_scale"], x["k_scale"], x["v_scale"], causal=True, out=o,
                   lse=lse)
        torch.cuda.synchronize()
        return ob, lb, o.clone(), lse.clone()

    ob, lb, o1, l1 = run()
    assert fa.device_status() == 0
    assert _check_guard(ob, B * H * N * d) and _check_guard(lb, B * H * N)
    _, _, o2, l2 = run()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("B,H,N,d,dtype", [(8, 16, 1024, 64, "fp16"), (2, 8, 2048, 128, "bf16"),
                                           (4, 8, 1000, 32, "fp16")])
def test_cuda_graph_replay_matches_eager(B, H, N, d, dtype):
    """Every call is asynchronous on the caller's stream with no host synchronisation, so
    a whole step (forward, backward with a caller workspace) can be captured into a CUDA
    graph; its replay gives the eager results bit for bit.  (Lazy set-up, such as shared
    memory opt-in, happens on the eager calls before the capture.)"""
    fa = _fa()
    x = inputs.make_inputs(B, H, N, d, dtype, seed=9)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.bwd_workspace_size(B, H, N, d, True), dtype=torch.uint8, device="cuda")

    def step():
        fa.fwd(q, k, v, causal=True, out=o, lse=lse)
        fa.bwd(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv, workspace=ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    ref = [t.clone() for t in (o, lse, dq, dk, dv)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for t in (o, lse, dq, dk, dv):
        t.fill_(float("nan"))
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(ref, (o, lse, dq, dk, dv)):
            assert torch.equal(a, b)
    assert fa.device_status() == 0


@pytest.mark.parametrize("B,H,N,d,dtype", [(4, 16, 1000, 64, "fp16"), (8, 8, 777, 32, "bf16"),
                                           (1, 8, 2048, 128, "bf16"), (4, 8, 1000, 32, "fp16")])
def test_back_to_back_steps_share_o_lse_workspace(B, H, N, d, dtype):
    """Steps launched back to back, with no host synchronisation or other kernel between
    them, as a training loop runs them.  Every kernel is a dependent launch: it may start
    while the kernel before it drains, and waits (griddepcontrol.wait) before touching
    global memory.  The steps share O, L and the workspace, which the next step's forward
    and backward overwrite, but each writes dQ, dK and dV of its own; every step's
    gradients must equal those of the same inputs run alone.  The inputs alternate
    between two sets, so a step that read the next step's O, L or D would show it."""
    fa = _fa()
    sets = []
    for seed in (11, 12):
        x = inputs.make_inputs(B, H, N, d, dtype, seed=seed)
        sets.append([x[n].cuda() for n in ("q", "k", "v", "do")])
    ref = []
    for q, k, v, do in sets:
        o, lse = fa.fwd(q, k, v, causal=True)
        ref.append([t.clone() for t in fa.bwd(q, k, v, o, lse, do, causal=True)])
        torch.cuda.synchronize()
    q0 = sets[0][0]
    o = torch.empty_like(q0)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(fa.bwd_workspace_size(B, H, N, d, True), dtype=torch.uint8, device="cuda")
    steps = 6
    grads = [[torch.empty_like(q0) for _ in range(3)] for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        q, k, v, do = sets[i % 2]
        dq, dk, dv = grads[i]
        fa.fwd(q, k, v, causal=True, out=o, lse=lse)
        fa.bwd(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv, workspace=ws)
    torch.cuda.synchronize()
    for i in range(steps):
        for a, b in zip(ref[i % 2], grads[i]):
            assert torch.equal(a, b), f"step {i}"
    assert fa.device_status() == 0


@pytest.mark.parametrize("B,H,N,d", [(4, 16, 1000, 64), (1, 8, 2048, 128)])
def test_traced_step_matches_untraced(B, H, N, d):
    """The per-kernel CUDA-event trace records an event between every two kernels, which
    makes each kernel wait for the previous one to finish before it starts; without it
    the kernels overlap as dependent launches.  Both orderings give the same bits."""
    fa = _fa()
    x = inputs.make_inputs(B, H, N, d, "bf16", seed=13)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    outs = []
    for traced in (False, True):
        fa.trace_enable(traced)
        try:
            o, lse = fa.fwd(q, k, v, causal=True)
            dq, dk, dv = fa.bwd(q, k, v, o, lse, do, causal=True)
            torch.cuda.synchronize()
        finally:
            fa.trace_enable(False)
        outs.append([t.clone() for t in (o, lse, dq, dk, dv)])
    for a, b in zip(*outs):
        assert torch.equal(a, b)
