"""Pins that tie the fp64 oracle to facts other than itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with a closed form, an invariant, a library special case,
finite differences or a size printed on the pages.  ``tests/test_oracle.py``
runs them on the real oracle; ``tests/test_oracle_mutations.py`` runs them on
copies of the oracle with one planted mistake each and expects a failure.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    if a.size == 0:
        return
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin), f"{what}: finiteness differs"
    err = float(np.max(np.abs(a[fin] - b[fin]))) if fin.any() else 0.0
    assert err <= tol, f"{what}: max abs err {err:.3e} > {tol:.1e}"
    assert np.array_equal(a[~fin], b[~fin]), f"{what}: non-finite values differ"


def pin_rows_sum_to_one(orc):
    """With V = I (d = N), O equals P itself: rows sum to 1, entries >= 0, and under the
    causal mask the strict upper triangle is exactly 0 (docs page, 'Tiling softmax is exact
    algebra'; FlashAttention note, causal masking)."""
    rng = np.random.default_rng(1)
    N = 37
    q = _rand(rng, 1, 2, N, N)
    k = _rand(rng, 1, 2, N, N)
    v = np.broadcast_to(np.eye(N), (1, 2, N, N)).copy()
    for causal in (False, True):
        P, _ = orc.fwd(q, k, v, causal, 1.0 / math.sqrt(N))
        _close(P.sum(-1), np.ones((1, 2, N)), 1e-12, "row sums of P")
        assert (P >= 0).all(), "P has negative entries"
        if causal:
            upper = np.triu(np.ones((N, N), dtype=bool), 1)
            assert (P[..., upper] == 0).all(), "causal P leaks above the diagonal"
        else:
            assert (P > 0).all(), "full P has zero entries"


def pin_constant_keys(orc):
    """All keys equal: P is uniform over the allowed keys.  Full: O_i = mean(V) and
    L_i = scale q_i.k + ln N.  Causal: O_i = mean(V_0..V_i), L_i = scale q_i.k + ln(i+1).
    The gradient w.r.t. Q vanishes and dV_j collects dO_i / (#allowed keys of row i)."""
    rng = np.random.default_rng(2)
    B, H, N, d = 2, 3, 29, 8
    scale = 0.37
    q = _rand(rng, B, H, N, d)
    kv = _rand(rng, B, H, 1, d)
    k = np.repeat(kv, N, axis=2)
    v = _rand(rng, B, H, N, d)
    do = _rand(rng, B, H, N, d)
    qk = scale * np.einsum("bhnd,bhd->bhn", q, kv[:, :, 0])
    for causal in (False, True):
        o, lse = orc.fwd(q, k, v, causal, scale)
        if causal:
            cnt = np.arange(1, N + 1, dtype=np.float64)
            o_ref = np.cumsum(v, axis=2) / cnt[None, None, :, None]
            l_ref = qk + np.log(cnt)[None, None, :]
            dv_ref = np.cumsum((do / cnt[None, None, :, None])[:, :, ::-1], axis=2)[:, :, ::-1]
        else:
            o_ref = np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape)
            l_ref = qk + math.log(N)
            dv_ref = np.broadcast_to(do.mean(axis=2, keepdims=True), o.shape)
        _close(o, o_ref, 1e-12, f"O with constant K (causal={causal})")
        _close(lse, l_ref, 1e-12, f"L with constant K (causal={causal})")
        dq, dk, dv, _ = orc.bwd(q, k, v, do, causal, scale)
        _close(dq, np.zeros_like(dq), 1e-12, "dQ with constant K")
        _close(dv, dv_ref, 1e-12, "dV with constant K")


def pin_causal_first_row(orc):
    """Causal row 0 sees only key 0: O_0 = V_0 and L_0 = scale q_0.k_0."""
    rng = np.random.default_rng(3)
    B, H, N, d = 1, 4, 17, 16
    scale = 0.25
    q, k, v = _rand(rng, B, H, N, d), _rand(rng, B, H, N, d), _rand(rng, B, H, N, d)
    o, lse = orc.fwd(q, k, v, True, scale)
    _close(o[:, :, 0], v[:, :, 0], 1e-13, "causal O_0")
    _close(lse[:, :, 0], scale * np.sum(q[:, :, 0] * k[:, :, 0], -1), 1e-13, "causal L_0")


def pin_online_matches_safe(orc):
    """The per-tile online update (docs page Fig. 3) equals the safe softmax for any tile
    size, including sizes that do not divide N and T = 1, in base e and in base 2."""
    rng = np.random.default_rng(4)
    B, H, N, d = 1, 2, 50, 12
    scale = 1.0 / math.sqrt(d)
    q, k, v = 3 * _rand(rng, B, H, N, d), 3 * _rand(rng, B, H, N, d), _rand(rng, B, H, N, d)
    for causal in (False, True):
        o_ref, l_ref = orc.fwd(q, k, v, causal, scale)
        for T in (1, 3, 7, 16, 49, 50, 64):
            for base2 in (False, True):
                o, lse = orc.fwd_online(q, k, v, causal, scale, T, base2)
                _close(o, o_ref, 1e-12, f"online O (T={T}, base2={base2}, causal={causal})")
                _close(lse, l_ref, 1e-12, f"online L (T={T}, base2={base2}, causal={causal})")


def pin_L_is_logsumexp(orc):
    """L is the natural-log logsumexp of the scaled, masked scores (scipy's logsumexp on
    scores formed by a numpy matmul)."""
    from scipy.special import logsumexp
    rng = np.random.default_rng(5)
    B, H, N, d = 2, 2, 33, 20
    scale = 0.4
    q, k, v = 2 * _rand(rng, B, H, N, d), 2 * _rand(rng, B, H, N, d), _rand(rng, B, H, N, d)
    s = scale * np.einsum("bhid,bhjd->bhij", q, k)
    for causal in (False, True):
        sm = s.copy()
        if causal:
            sm[..., np.triu(np.ones((N, N), dtype=bool), 1)] = -np.inf
        _, lse = orc.fwd(q, k, v, causal, scale)
        _close(lse, logsumexp(sm, axis=-1), 1e-12, f"L vs logsumexp (causal={causal})")


def pin_merge(orc):
    """Two partial results merge into the whole (tutorial page, 'Softmax in pieces'): any
    split point, any order, associatively; an empty partial is the identity."""
    rng = np.random.default_rng(6)
    N, d = 41, 9
    scale = 0.5
    qi = 2 * _rand(rng, d)
    k, v = 2 * _rand(rng, N, d), _rand(rng, N, d)
    i = N - 1
    for base2 in (False, True):
        whole = orc.row_partial(qi, k, v, i, 0, N, False, scale, 5, base2)
        for a in (1, 13, 40):
            p1 = orc.row_partial(qi, k, v, i, 0, a, False, scale, 4, base2)
            p2 = orc.row_partial(qi, k, v, i, a, N, False, scale, 6, base2)
            for m in (orc.merge(p1, p2, base2), orc.merge(p2, p1, base2)):
                assert abs(m[0] - whole[0]) <= 1e-12, "merged max differs"
                assert abs(m[1] / whole[1] - 1) <= 1e-12, "merged sum differs"
                _close(m[2] / m[1], whole[2] / whole[1], 1e-12, "merged output differs")
        p1 = orc.row_partial(qi, k, v, i, 0, 10, False, scale, 3, base2)
        p2 = orc.row_partial(qi, k, v, i, 10, 30, False, scale, 3, base2)
        p3 = orc.row_partial(qi, k, v, i, 30, N, False, scale, 3, base2)
        left = orc.merge(orc.merge(p1, p2, base2), p3, base2)
        right = orc.merge(p1, orc.merge(p2, p3, base2), base2)
        perm = orc.merge(orc.merge(p3, p1, base2), p2, base2)
        for m in (left, right, perm):
            assert abs(m[0] - whole[0]) <= 1e-12
            assert abs(m[1] / whole[1] - 1) <= 1e-12
            _close(m[2] / m[1], whole[2] / whole[1], 1e-12, "3-way merge output")
        empty = (-math.inf, 0.0, np.zeros(d))
        m = orc.merge(empty, whole, base2)
        assert m[0] == whole[0] and m[1] == whole[1]
        _close(m[2], whole[2], 0.0, "merge with the empty partial")
        m = orc.merge(empty, empty, base2)
        assert m[0] == -math.inf and m[1] == 0.0 and not np.isnan(m[2]).any()
    # the finished row equals the forward's row (base e: L = m + ln l)
    whole = orc.row_partial(qi, k, v, i, 0, N, False, scale, 5, False)
    q = np.zeros((1, 1, N, d))
    q[0, 0, i] = qi
    o, lse = orc.fwd(q, k[None, None], v[None, None], False, scale)
    _close(whole[2] / whole[1], o[0, 0, i], 1e-12, "finished partial vs forward")
    assert abs(whole[0] + math.log(whole[1]) - lse[0, 0, i]) <= 1e-12


def _loss(orc, q, k, v, do, causal, scale):
    o, _ = orc.fwd(q, k, v, causal, scale)
    return float(np.sum(o * do))


def pin_finite_differences(orc):
    """Central differences of loss = sum(O o dO) match dQ, dK, dV (relative error < 1e-6)
    on tiny shapes; D equals rowsum(dO o O)."""
    rng = np.random.default_rng(7)
    h = 1e-6
    for N in (1, 2, 5, 7):
        for d in (1, 3, 4):
            for causal in (False, True):
                scale = 0.9
                q, k, v, do = (_rand(rng, 1, 1, N, d) for _ in range(4))
                dq, dk, dv, D = orc.bwd(q, k, v, do, causal, scale)
                o, _ = orc.fwd(q, k, v, causal, scale)
                _close(D, np.sum(o * do, -1), 1e-13, "D = rowsum(dO o O)")
                for name, x, g in (("dQ", q, dq), ("dK", k, dk), ("dV", v, dv)):
                    fd = np.zeros_like(x)
                    for idx in np.ndindex(x.shape):
                        xp, xm = x.copy(), x.copy()
                        xp[idx] += h
                        xm[idx] -= h
                        args_p = {"q": q, "k": k, "v": v}
                        args_m = dict(args_p)
                        key = name[1].lower()
                        args_p[key], args_m[key] = xp, xm
                        fd[idx] = (_loss(orc, args_p["q"], args_p["k"], args_p["v"], do, causal,
                                         scale)
                                   - _loss(orc, args_m["q"], args_m["k"], args_m["v"], do, causal,
                                           scale)) / (2 * h)
                    ref = max(float(np.max(np.abs(fd))), 1e-3)
                    err = float(np.max(np.abs(fd - g))) / ref
                    assert err < 1e-6, f"finite differences {name} N={N} d={d} causal={causal}: {err:.2e}"


def pin_gradient_invariants(orc):
    """Rows of dS sum to 0, so the dK rows sum to 0; rows of P sum to 1, so the dV rows sum
    to the dO rows."""
    rng = np.random.default_rng(8)
    B, H, N, d = 2, 2, 45, 16
    q, k, v, do = (_rand(rng, B, H, N, d) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv, _ = orc.bwd(q, k, v, do, causal, 0.3)
        _close(dk.sum(axis=2), np.zeros((B, H, d)), 1e-11, "sum_j dK_j")
        _close(dv.sum(axis=2), do.sum(axis=2), 1e-11, "sum_j dV_j")


def pin_torch_sdpa(orc, shapes=((1, 1, 128, 64, False), (2, 3, 100, 32, True),
                                (4, 8, 1000, 32, True))):
    """Library special case: torch's scaled_dot_product_attention in fp64 on the CPU, with
    autograd for the gradients."""
    import torch
    rng = np.random.default_rng(9)
    for B, H, N, d, causal in shapes:
        scale = 1.0 / math.sqrt(d)
        q, k, v, do = (_rand(rng, B, H, N, d) for _ in range(4))
        tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
        to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal,
                                                              scale=scale)
        to.backward(torch.tensor(do, dtype=torch.float64))
        o, _ = orc.fwd(q, k, v, causal, scale)
        dq, dk, dv, _ = orc.bwd(q, k, v, do, causal, scale)
        _close(o, to.detach().numpy(), 1e-10, f"O vs SDPA {B, H, N, d, causal}")
        _close(dq, tq.grad.numpy(), 1e-10, f"dQ vs SDPA {B, H, N, d, causal}")
        _close(dk, tk.grad.numpy(), 1e-10, f"dK vs SDPA {B, H, N, d, causal}")
        _close(dv, tv.grad.numpy(), 1e-10, f"dV vs SDPA {B, H, N, d, causal}")


def pin_gqa(orc, shapes=((1, 4, 2, 37, 8, False), (2, 6, 2, 45, 16, True),
                         (1, 4, 1, 33, 8, True), (1, 3, 3, 20, 8, True))):
    """Grouped-query / multi-query attention.  Library special case: torch's
    scaled_dot_product_attention with enable_gqa (query head h reads K/V head
    h // (H/Hkv)) in fp64 with autograd.  Then central finite differences of
    sum(O o dO) on tiny shapes, where a shared K/V head's gradient must be the sum
    over its query heads."""
    import torch
    rng = np.random.default_rng(10)
    for B, H, Hkv, N, d, causal in shapes:
        scale = 1.0 / math.sqrt(d)
        q, do = _rand(rng, B, H, N, d), _rand(rng, B, H, N, d)
        k, v = _rand(rng, B, Hkv, N, d), _rand(rng, B, Hkv, N, d)
        tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
        to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal,
                                                              scale=scale, enable_gqa=True)
        to.backward(torch.tensor(do, dtype=torch.float64))
        o, _ = orc.fwd_gqa(q, k, v, causal, scale)
        dq, dk, dv, _ = orc.bwd_gqa(q, k, v, do, causal, scale)
        tag = f"{B, H, Hkv, N, d, causal}"
        _close(o, to.detach().numpy(), 1e-10, f"GQA O vs SDPA {tag}")
        _close(dq, tq.grad.numpy(), 1e-10, f"GQA dQ vs SDPA {tag}")
        _close(dk, tk.grad.numpy(), 1e-10, f"GQA dK vs SDPA {tag}")
        _close(dv, tv.grad.numpy(), 1e-10, f"GQA dV vs SDPA {tag}")
    h = 1e-6
    for Hkv in (1, 2):
        for causal in (False, True):
            q, do = _rand(rng, 1, 4, 3, 2), _rand(rng, 1, 4, 3, 2)
            k, v = _rand(rng, 1, Hkv, 3, 2), _rand(rng, 1, Hkv, 3, 2)
            dq, dk, dv, _ = orc.bwd_gqa(q, k, v, do, causal, 0.8)

            def loss(qq, kk, vv):
                return float(np.sum(orc.fwd_gqa(qq, kk, vv, causal, 0.8)[0] * do))
            for name, x, g in (("dK", k, dk), ("dV", v, dv), ("dQ", q, dq)):
                fd = np.zeros_like(x)
                for idx in np.ndindex(x.shape):
                    xp, xm = x.copy(), x.copy()
                    xp[idx] += h
                    xm[idx] -= h
                    ap = {"q": q, "k": k, "v": v}
                    am = dict(ap)
                    ap[name[1].lower()], am[name[1].lower()] = xp, xm
                    fd[idx] = (loss(ap["q"], ap["k"], ap["v"]) - loss(am["q"], am["k"], am["v"])) / (2 * h)
                err = float(np.max(np.abs(fd - g))) / max(float(np.max(np.abs(fd))), 1e-3)
                assert err < 1e-6, f"GQA finite differences {name} Hkv={Hkv} causal={causal}: {err:.2e}"


def pin_window(orc, shapes=((1, 2, 70, 16, 5), (2, 1, 130, 8, 17), (1, 2, 64, 8, 64),
                            (1, 1, 40, 4, 2))):
    """Causal sliding window of W keys.  W = 1: every row sees only its own key, so
    O = V, L_i = scale q_i.k_i, dV = dO and dQ = dK = 0.  W >= N: plain causal.
    Library special case: torch's scaled_dot_product_attention with the band mask
    j <= i < j + W in fp64, with autograd for the gradients."""
    import torch
    rng = np.random.default_rng(11)
    q, k, v, do = (_rand(rng, 1, 2, 33, 8) for _ in range(4))
    o, lse = orc.fwd(q, k, v, True, 0.7, window=1)
    dq, dk, dv, _ = orc.bwd(q, k, v, do, True, 0.7, window=1)
    _close(o, v, 1e-12, "W=1: O = V")
    _close(lse, 0.7 * np.sum(q * k, -1), 1e-12, "W=1: L = scale q.k")
    _close(dv, do, 1e-12, "W=1: dV = dO")
    _close(dq, np.zeros_like(dq), 1e-12, "W=1: dQ = 0")
    _close(dk, np.zeros_like(dk), 1e-12, "W=1: dK = 0")
    for W in (33, 40):
        ow, lw = orc.fwd(q, k, v, True, 0.7, window=W)
        oc, lc = orc.fwd(q, k, v, True, 0.7)
        _close(ow, oc, 1e-13, f"W={W} >= N: O as causal")
        _close(lw, lc, 1e-13, f"W={W} >= N: L as causal")
    for B, H, N, d, W in shapes:
        scale = 1.0 / math.sqrt(d)
        q, k, v, do = (_rand(rng, B, H, N, d) for _ in range(4))
        i = np.arange(N)[:, None]
        j = np.arange(N)[None, :]
        band = torch.tensor((j <= i) & (i - j < W))
        tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
        to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=band,
                                                              scale=scale)
        to.backward(torch.tensor(do, dtype=torch.float64))
        o, _ = orc.fwd(q, k, v, True, scale, window=W)
        dq, dk, dv, _ = orc.bwd(q, k, v, do, True, scale, window=W)
        tag = f"{B, H, N, d} W={W}"
        _close(o, to.detach().numpy(), 1e-10, f"window O vs SDPA {tag}")
        _close(dq, tq.grad.numpy(), 1e-10, f"window dQ vs SDPA {tag}")
        _close(dk, tk.grad.numpy(), 1e-10, f"window dK vs SDPA {tag}")
        _close(dv, tv.grad.numpy(), 1e-10, f"window dV vs SDPA {tag}")


def pin_varlen(orc):
    """Variable-length batches.  Library special case: the packed sequence as one
    attention problem under a block-diagonal mask (each token sees only its own
    sequence's keys; causal or a sliding window inside the block), torch's
    scaled_dot_product_attention in fp64 with autograd; shared K/V heads through
    enable_gqa.  Empty sequences contribute nothing."""
    import torch
    rng = np.random.default_rng(12)
    for lens, H, Hkv, d, causal, W in (((5, 17, 1, 40), 2, 2, 8, True, 0),
                                       ((33, 0, 20), 4, 2, 8, False, 0),
                                       ((64, 70, 3), 2, 1, 16, True, 9)):
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        T = int(cu[-1])
        q, do = _rand(rng, T, H, d), _rand(rng, T, H, d)
        k, v = _rand(rng, T, Hkv, d), _rand(rng, T, Hkv, d)
        seg = np.repeat(np.arange(len(lens)), lens)
        i, j = np.arange(T)[:, None], np.arange(T)[None, :]
        allow = seg[:, None] == seg[None, :]
        if causal:
            allow &= j <= i
        if W:
            allow &= i - j < W
        scale = 1.0 / math.sqrt(d)
        tq, tk, tv = (torch.tensor(x.transpose(1, 0, 2)[None], dtype=torch.float64,
                                   requires_grad=True) for x in (q, k, v))
        to = torch.nn.functional.scaled_dot_product_attention(
            tq, tk, tv, attn_mask=torch.tensor(allow), scale=scale, enable_gqa=Hkv != H)
        to.backward(torch.tensor(do.transpose(1, 0, 2)[None], dtype=torch.float64))
        o, lse = orc.fwd_varlen(q, k, v, cu, causal, scale, W)
        dq, dk, dv, _ = orc.bwd_varlen(q, k, v, do, cu, causal, scale, W)
        tag = f"lens={lens} H={H} Hkv={Hkv} causal={causal} W={W}"
        back = lambda t: t.detach().numpy()[0].transpose(1, 0, 2)
        _close(o, back(to), 1e-10, f"varlen O vs SDPA {tag}")
        _close(dq, back(tq.grad), 1e-10, f"varlen dQ vs SDPA {tag}")
        _close(dk, back(tk.grad), 1e-10, f"varlen dK vs SDPA {tag}")
        _close(dv, back(tv.grad), 1e-10, f"varlen dV vs SDPA {tag}")
        # L of every token: the logsumexp of its allowed scaled scores
        s_ = np.einsum("ihc,jhc->hij", q, np.repeat(k, H // Hkv, axis=1)) * scale
        s_ = np.where(allow[None], s_, -np.inf)
        mx = s_.max(-1, keepdims=True)
        _close(lse, (mx + np.log(np.exp(s_ - mx).sum(-1, keepdims=True)))[..., 0], 1e-11,
               f"varlen L {tag}")


def pin_decode(orc):
    """Split-KV decoding: the new query of sequence b against its first n_b cached keys is
    the last row of the causal forward over those n_b rows (query n_b - 1 sees keys
    0 .. n_b - 1), with K/V heads shared as in GQA; an empty cache gives O = 0, L = -inf.
    The split/merge algebra itself is pinned by pin_merge."""
    rng = np.random.default_rng(13)
    B, H, Hkv, Nmax, d = 3, 4, 2, 50, 8
    kc, vc = _rand(rng, B, Hkv, Nmax, d), _rand(rng, B, Hkv, Nmax, d)
    q = _rand(rng, B, H, d)
    lens = (37, 0, 50)
    o, lse = orc.decode(q, kc, vc, lens, 0.4)
    for b, n in enumerate(lens):
        if n == 0:
            _close(o[b], np.zeros((H, d)), 0.0, "empty cache: O = 0")
            assert np.all(lse[b] == -np.inf), "empty cache: L = -inf"
            continue
        qq = np.zeros((1, H, n, d))
        qq[0, :, n - 1] = q[b]
        of, lf = orc.fwd_gqa(qq, kc[b:b + 1, :, :n], vc[b:b + 1, :, :n], True, 0.4)
        _close(o[b], of[0, :, n - 1], 1e-12, f"decode O = last causal row (n={n})")
        _close(lse[b], lf[0, :, n - 1], 1e-12, f"decode L = last causal row (n={n})")


def pin_page_sizes(iomodel):
    """Sizes the pages print (tests/golden/page_sizes.json) from the byte model."""
    with open(os.path.join(GOLDEN, "page_sizes.json")) as f:
        cases = json.load(f)["cases"]
    c0, c1, c2, c3 = cases
    assert iomodel.score_matrix_bytes(c0["B"], c0["H"], c0["N"], c0["elem_bytes"]) == c0["bytes"]
    assert c0["bytes"] == 128 * 2**20
    e = iomodel.score_entries(c1["N"])
    assert abs(e / c1["entries_approx"] - 1) <= c1["rel_tol"]
    assert iomodel.tile_bytes(c2["block_m"], c2["block_n"], c2["elem_bytes"]) == c2["bytes"]
    assert c2["bytes"] == 32 * 2**10
    r = iomodel.tiled_hbm_ratio(c3["d"], c3["sram_bytes"])
    assert abs(r / c3["ratio_approx"] - 1) <= c3["rel_tol"]


def pin_fp8(orc):
    """8-bit E4M3 inputs.  The code table against torch's float8_e4m3fn decoding
    (library) over all 256 codes, plus closed forms of the format (1.0, the largest
    finite value 448, the smallest normal 2^-6 and subnormal 2^-9, NaN patterns).
    Attention on the codes: torch SDPA (fp64, enable_gqa) on the decoded values;
    the descale factors enter as q_scale k_scale times the softmax scale (powers of
    two: exact) and v_scale multiplies O and leaves L."""
    import torch
    codes = np.arange(256, dtype=np.uint8)
    got = orc.e4m3_values(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2, "E4M3 NaN codes"
    assert np.array_equal(got[~nan], ref[~nan]), "E4M3 code table vs torch"
    for c, val in ((0x38, 1.0), (0x7E, 448.0), (0x08, 2.0 ** -6), (0x01, 2.0 ** -9),
                   (0xB8, -1.0), (0x00, 0.0), (0x44, 3.0)):
        assert orc.e4m3_values([c])[0] == val, f"E4M3 code {c:#x} = {val}"
    rng = np.random.default_rng(14)
    for B, H, Hkv, N, d, causal in ((1, 4, 2, 40, 16, True), (2, 2, 1, 33, 8, False)):
        q8, k8, v8 = (rng.integers(0, 256, (B, hh, N, d)).astype(np.uint8) for hh in (H, Hkv, Hkv))
        for a in (q8, k8, v8):
            a[(a & 0x7F) == 0x7F] = 0x3C          # no NaN codes in the inputs
        q8 &= 0xBF                                # |q| < 2: keep the scores moderate
        k8 &= 0xBF
        scale = 0.3
        o, lse = orc.fwd_fp8(q8, k8, v8, 1.0, 1.0, 1.0, causal, scale)
        tq, tk, tv = (torch.tensor(orc.e4m3_values(x)) for x in (q8, k8, v8))
        to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal,
                                                              scale=scale, enable_gqa=True)
        _close(o, to.numpy(), 1e-10, f"FP8 O vs SDPA on the decoded values {B, H, Hkv, N, d}")
        o2, l2 = orc.fwd_fp8(q8, k8, v8, 2.0, 0.25, 1.0, causal, 2.0 * scale)
        _close(o2, o, 1e-12, "FP8: q_scale k_scale fold into the softmax scale (O)")
        _close(l2, lse, 1e-12, "FP8: q_scale k_scale fold into the softmax scale (L)")
        o3, l3 = orc.fwd_fp8(q8, k8, v8, 1.0, 1.0, 0.125, causal, scale)
        _close(o3, 0.125 * o, 1e-12, "FP8: v_scale multiplies O")
        _close(l3, lse, 1e-12, "FP8: v_scale leaves L")


ORACLE_PINS = [pin_rows_sum_to_one, pin_constant_keys, pin_causal_first_row,
               pin_online_matches_safe, pin_L_is_logsumexp, pin_merge, pin_finite_differences,
               pin_gradient_invariants, pin_torch_sdpa, pin_gqa, pin_window, pin_varlen,
               pin_decode, pin_fp8]
