"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
and reference legs import this package.  The product path (the CUDA library
and its Python binding) never imports, links or calls it, and it imports
nothing from the product package.

Contents
  * ``fwd``/``bwd``: the plain definition of attention and its gradients,
    written in C (``fa_oracle.c``), fp64, one query row at a time, OpenMP over
    (batch, head).  Definitions follow the "flash-attn-triton" docs page,
    section "The argument" (S = QK^T/sqrt(d), row softmax, P V), with causal
    masking lower-triangular (FlashAttention note, "Key Mechanisms").
  * ``fwd_gqa``/``bwd_gqa``: grouped-query / multi-query attention (the docs
    page lists MQA/GQA as "not yet", "Scope"; FlashAttention-2 added them, note
    "Versions and Evolution"): K and V have Hkv heads, each shared by H/Hkv
    consecutive query heads.  Defined as the plain attention of every query head
    with its group's K/V head; the gradient of a shared head is the sum over the
    query heads that read it (chain rule).
  * ``fwd_varlen``/``bwd_varlen``: variable-length batches (docs page "Scope":
    not yet): sequences of different lengths packed one after another, Q/O/dO
    (total, H, d), K/V (total, Hkv, d), L (H, total), sequence b holding tokens
    cu_seqlens[b] .. cu_seqlens[b+1]-1.  Defined as attention of every sequence
    on its own, no token seeing another sequence's keys.
  * ``decode``: one new query per sequence against a key/value cache of
    cache_seqlens[b] rows (split-KV decoding, with the two-partial merge of the
    tutorial page, "Softmax in pieces"): the plain safe softmax of the row over
    all cached keys, K/V heads shared as in GQA.
  * ``window`` (fwd, bwd and the GQA pair): a causal sliding window of W keys,
    query i seeing keys i - W < j <= i (docs page "Scope" lists sliding windows
    as not yet supported and fixes no convention; this is the plain reading).
  * ``e4m3_values``/``fwd_fp8``: attention on 8-bit E4M3 inputs (the FP8 of
    the note's FlashAttention-3 entry, "Versions and Evolution") with per-tensor
    descale factors, defined as the exact attention of the values the codes
    stand for; the codes are decoded from the format's definition.
  * ``fwd_online``/``row_partial``/``merge``: the separate naive online-softmax
    oracle of the docs page's Fig. 3 and the two-partial merge of the tutorial
    page ("Softmax in pieces").
  * ``iomodel``: byte and FLOP counts of the pages' arithmetic (footprint
    calculator, Fig. 2; HBM access counts, Table 2).

Inputs are numpy arrays convertible to fp64 (callers pass the 16-bit values
upcast exactly).  Nothing here rounds to 16 bits.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libfa_oracle.so")


def build(force: bool = False, src: str = _SRC, out: str = _SO) -> str:
    """Compile the C oracle with gcc (fp64, no fast-math, OpenMP)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC",
               "-shared", src, "-o", tmp, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, out)
    return out


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


class Oracle:
    """ctypes view of one compiled copy of ``fa_oracle.c``."""

    def __init__(self, so_path: str):
        lib = ctypes.CDLL(so_path)
        dp = ctypes.POINTER(ctypes.c_double)
        i, dbl = ctypes.c_int, ctypes.c_double
        lib.oracle_fwd.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, dbl, i]
        lib.oracle_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, i, i, i, i, i, dbl, i]
        lib.oracle_fwd_online.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, dbl, i, i]
        lib.oracle_row_partial.argtypes = [dp, dp, dp, i, i, i, i, i, dbl, i, i, dp, dp]
        lib.oracle_row_partial.restype = dbl
        lib.oracle_merge.argtypes = [dbl, dbl, dp, dbl, dbl, dp, i, i, dp, dp]
        lib.oracle_merge.restype = dbl
        lib.oracle_num_threads.restype = ctypes.c_int
        self.lib = lib

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    @staticmethod
    def _window(causal: bool, window: int) -> int:
        if window < 0 or (window > 0 and not causal):
            raise ValueError("a sliding window is a causal band of window >= 1 keys")
        return int(window)

    def fwd(self, q, k, v, causal: bool, scale: float, window: int = 0):
        """O, L for (B,H,N,d) inputs.  L is the natural-log logsumexp of scaled scores.
        window > 0 (causal only): query i sees keys i - window < j <= i."""
        window = self._window(causal, window)
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, N, d = q.shape
        o = np.empty_like(q)
        lse = np.empty((B, H, N), dtype=np.float64)
        self.lib.oracle_fwd(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, N, d, int(causal),
                            float(scale), window)
        return o, lse

    def bwd(self, q, k, v, do, causal: bool, scale: float, window: int = 0):
        """dQ, dK, dV and D = rowsum(dO o O) from the plain definition."""
        window = self._window(causal, window)
        q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
        B, H, N, d = q.shape
        dq, dk, dv = np.empty_like(q), np.empty_like(q), np.empty_like(q)
        D = np.empty((B, H, N), dtype=np.float64)
        self.lib.oracle_bwd(_p(q), _p(k), _p(v), _p(do), _p(dq), _p(dk), _p(dv), _p(D),
                            B, H, N, d, int(causal), float(scale), window)
        return dq, dk, dv, D

    @staticmethod
    def _group(q, k) -> int:
        H, Hkv = q.shape[1], k.shape[1]
        if Hkv < 1 or H % Hkv:
            raise ValueError("H must be a multiple of the K/V head count")
        return H // Hkv

    def fwd_gqa(self, q, k, v, causal: bool, scale: float, window: int = 0):
        """O, L with K, V of shape (B, Hkv, N, d): query head h uses K/V head h // (H/Hkv)."""
        g = self._group(q, k)
        return self.fwd(q, np.repeat(_f64(k), g, axis=1), np.repeat(_f64(v), g, axis=1), causal,
                        scale, window)

    def bwd_gqa(self, q, k, v, do, causal: bool, scale: float, window: int = 0):
        """dQ (B, H, N, d); dK, dV (B, Hkv, N, d), each the sum over the group's query
        heads of the per-head gradient; D = rowsum(dO o O)."""
        g = self._group(q, k)
        B, Hkv, N, d = k.shape
        dq, dk, dv, D = self.bwd(q, np.repeat(_f64(k), g, axis=1), np.repeat(_f64(v), g, axis=1),
                                 do, causal, scale, window)
        return (dq, dk.reshape(B, Hkv, g, N, d).sum(axis=2), dv.reshape(B, Hkv, g, N, d).sum(axis=2),
                D)

    def fwd_varlen(self, q, k, v, cu_seqlens, causal: bool, scale: float, window: int = 0):
        """O (total, H, d), L (H, total) for packed sequences (K, V: (total, Hkv, d))."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        total, H, d = q.shape
        o = np.zeros_like(q)
        lse = np.full((H, total), -np.inf)
        for b in range(len(cu_seqlens) - 1):
            a, e = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
            if e == a:
                continue
            qs, ks, vs = (x[a:e].transpose(1, 0, 2)[None] for x in (q, k, v))
            ob, lb = self.fwd_gqa(qs, ks, vs, causal, scale, window)
            o[a:e] = ob[0].transpose(1, 0, 2)
            lse[:, a:e] = lb[0]
        return o, lse

    def bwd_varlen(self, q, k, v, do, cu_seqlens, causal: bool, scale: float, window: int = 0):
        """dQ (total, H, d), dK, dV (total, Hkv, d) and D (H, total) for packed sequences."""
        q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
        total, H, d = q.shape
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        D = np.zeros((H, total))
        for b in range(len(cu_seqlens) - 1):
            a, e = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
            if e == a:
                continue
            qs, ks, vs, dos = (x[a:e].transpose(1, 0, 2)[None] for x in (q, k, v, do))
            gq, gk, gv, Db = self.bwd_gqa(qs, ks, vs, dos, causal, scale, window)
            dq[a:e], dk[a:e], dv[a:e] = (g[0].transpose(1, 0, 2) for g in (gq, gk, gv))
            D[:, a:e] = Db[0]
        return dq, dk, dv, D

    def decode(self, q, kc, vc, cache_seqlens, scale: float):
        """O (B, H, d), L (B, H) of one query row per (batch, head) against the first
        cache_seqlens[b] rows of the caches kc, vc (B, Hkv, Nmax, d); an empty cache gives
        O = 0, L = -inf.  One key tile spanning the whole cache: the safe softmax."""
        q, kc, vc = _f64(q), _f64(kc), _f64(vc)
        B, H, d = q.shape
        g = H // kc.shape[1]
        o = np.zeros((B, H, d))
        lse = np.full((B, H), -np.inf)
        for b in range(B):
            n = int(cache_seqlens[b])
            if n == 0:
                continue
            for h in range(H):
                m, l, acc = self.row_partial(q[b, h], kc[b, h // g, :n], vc[b, h // g, :n], 0, 0,
                                             n, False, scale, n)
                o[b, h] = acc / l
                lse[b, h] = m + np.log(l)
        return o, lse

    @staticmethod
    def e4m3_values(codes) -> np.ndarray:
        """fp64 values of 8-bit E4M3 codes: sign bit 7, exponent bits 6..3 with bias 7,
        mantissa bits 2..0; exponent field 0 holds the subnormals (m/8) 2^-6; the
        pattern with every exponent and mantissa bit set is NaN, and there is no
        infinity (the E4M3 variant of the OCP 8-bit floating-point formats)."""
        c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
        sign = np.where(c & 0x80, -1.0, 1.0)
        e = (c >> 3) & 0xF
        m = (c & 0x7).astype(np.float64)
        mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
        return np.where((e == 15) & (m == 7), np.nan, sign * mag)

    def fwd_fp8(self, q8, k8, v8, q_scale: float, k_scale: float, v_scale: float, causal: bool,
                scale: float):
        """O, L of attention on 8-bit E4M3 inputs with per-tensor descale factors: the
        exact attention of q_scale Q, k_scale K, v_scale V, the values the codes stand
        for (q8 (B, H, N, d); k8, v8 (B, Hkv, N, d), shared as in GQA).  FP8 is the
        precision the note's FlashAttention-3 entry adds ("Versions and Evolution")."""
        q = self.e4m3_values(q8) * q_scale
        k = self.e4m3_values(k8) * k_scale
        v = self.e4m3_values(v8) * v_scale
        return self.fwd_gqa(q, k, v, causal, scale)

    def fwd_online(self, q, k, v, causal: bool, scale: float, tile: int, base2: bool = False):
        """O, L by the per-tile online update (docs page Fig. 3), key tiles of ``tile``."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, N, d = q.shape
        o = np.empty_like(q)
        lse = np.empty((B, H, N), dtype=np.float64)
        self.lib.oracle_fwd_online(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, N, d,
                                   int(causal), float(scale), int(tile), int(base2))
        return o, lse

    def row_partial(self, qi, k, v, i: int, j0: int, j1: int, causal: bool, scale: float,
                    tile: int, base2: bool = False):
        """(m, l, acc) of query row i over keys [j0, j1) of one head (k, v: (N, d))."""
        qi, k, v = _f64(qi), _f64(k), _f64(v)
        d = k.shape[1]
        acc = np.empty(d, dtype=np.float64)
        l = ctypes.c_double()
        m = self.lib.oracle_row_partial(_p(qi), _p(k), _p(v), d, i, j0, j1, int(causal),
                                        float(scale), int(tile), int(base2), ctypes.byref(l),
                                        _p(acc))
        return m, l.value, acc

    def merge(self, p1, p2, base2: bool = False):
        """Merge two partial states (m, l, acc) of one row."""
        m1, l1, a1 = p1
        m2, l2, a2 = p2
        a1, a2 = _f64(a1), _f64(a2)
        out = np.empty_like(a1)
        l = ctypes.c_double()
        m = self.lib.oracle_merge(float(m1), float(l1), _p(a1), float(m2), float(l2), _p(a2),
                                  a1.shape[0], int(base2), ctypes.byref(l), _p(out))
        return m, l.value, out


_default = None


def get() -> Oracle:
    """The oracle compiled from this directory's ``fa_oracle.c``."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def num_threads() -> int:
    return get().num_threads()


def fwd(q, k, v, causal: bool, scale: float, window: int = 0):
    return get().fwd(q, k, v, causal, scale, window)


def bwd(q, k, v, do, causal: bool, scale: float, window: int = 0):
    return get().bwd(q, k, v, do, causal, scale, window)


def fwd_gqa(q, k, v, causal: bool, scale: float, window: int = 0):
    return get().fwd_gqa(q, k, v, causal, scale, window)


def bwd_gqa(q, k, v, do, causal: bool, scale: float, window: int = 0):
    return get().bwd_gqa(q, k, v, do, causal, scale, window)


def fwd_varlen(q, k, v, cu_seqlens, causal: bool, scale: float, window: int = 0):
    return get().fwd_varlen(q, k, v, cu_seqlens, causal, scale, window)


def bwd_varlen(q, k, v, do, cu_seqlens, causal: bool, scale: float, window: int = 0):
    return get().bwd_varlen(q, k, v, do, cu_seqlens, causal, scale, window)


def decode(q, kc, vc, cache_seqlens, scale: float):
    return get().decode(q, kc, vc, cache_seqlens, scale)


def e4m3_values(codes):
    return Oracle.e4m3_values(codes)


def fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal: bool, scale: float):
    return get().fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal, scale)


def fwd_online(q, k, v, causal: bool, scale: float, tile: int, base2: bool = False):
    return get().fwd_online(q, k, v, causal, scale, tile, base2)


def row_partial(qi, k, v, i, j0, j1, causal, scale, tile, base2=False):
    return get().row_partial(qi, k, v, i, j0, j1, causal, scale, tile, base2)


def merge(p1, p2, base2: bool = False):
    return get().merge(p1, p2, base2)
