"""Seeded synthetic inputs for exact attention.

This module holds no attention arithmetic: it only draws random tensors, so
that the CUDA path and the CPU oracle can be fed the very same values.

Recipe: one CPU ``torch.Generator`` seeded per workload; draws in the fixed
order Q, K, V, dO, each i.i.d. N(0, 1) in fp32 of shape (B, H, N, d); Q and K
are then multiplied by ``qk_std`` (4 for the large-row-maximum stress case);
finally every tensor is rounded to the 16-bit dtype.  The oracle consumes the
rounded values upcast exactly to fp64.  With ``Hkv`` (grouped-query attention)
K and V are drawn with Hkv heads instead of H, in the same order.  Decoding
inputs draw one query row per (batch, head) and then the K and V caches.  FP8
inputs are the fp32 draws divided by a per-tensor scale and rounded to E4M3.
"""
from __future__ import annotations

import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


def make_inputs(B: int, H: int, N: int, d: int, dtype: str = "bf16", seed: int = 0,
                qk_std: float = 1.0, Hkv: int | None = None):
    """Return dict(q, k, v, do) of CPU tensors in ``dtype``: q and do (B, H, N, d),
    k and v (B, Hkv, N, d) (Hkv defaults to H)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    shape = (B, H, N, d)
    kv_shape = (B, H if Hkv is None else Hkv, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(kv_shape, generator=g, dtype=torch.float32)
    v = torch.randn(kv_shape, generator=g, dtype=torch.float32)
    do = torch.randn(shape, generator=g, dtype=torch.float32)
    if qk_std != 1.0:
        q = q * qk_std
        k = k * qk_std
    t = DTYPES[dtype]
    return {"q": q.to(t), "k": k.to(t), "v": v.to(t), "do": do.to(t)}


def make_packed_inputs(lens, H: int, d: int, dtype: str = "bf16", seed: int = 0,
                       Hkv: int | None = None):
    """Packed variable-length sequences: dict(q, k, v, do) of CPU tensors, q and do
    (total, H, d), k and v (total, Hkv, d), drawn in that order like make_inputs, plus
    cu_seqlens (int32, len(lens) + 1 offsets)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    total = int(sum(lens))
    kvh = H if Hkv is None else Hkv
    q = torch.randn((total, H, d), generator=g, dtype=torch.float32)
    k = torch.randn((total, kvh, d), generator=g, dtype=torch.float32)
    v = torch.randn((total, kvh, d), generator=g, dtype=torch.float32)
    do = torch.randn((total, H, d), generator=g, dtype=torch.float32)
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(list(lens), dtype=torch.int64), 0).to(torch.int32)
    t = DTYPES[dtype]
    return {"q": q.to(t), "k": k.to(t), "v": v.to(t), "do": do.to(t), "cu_seqlens": cu}


def make_decode_inputs(B: int, H: int, Hkv: int, Nmax: int, d: int, lens, dtype: str = "bf16",
                       seed: int = 0, fill: float | None = None):
    """One query row per (batch, head) and K/V caches: dict(q (B, H, d), k_cache, v_cache
    (B, Hkv, Nmax, d)) of CPU tensors in ``dtype``, drawn in that order i.i.d. N(0, 1),
    plus cache_seqlens (int32, the B values of ``lens``).  With ``fill`` every cache row
    at or past its sequence's length is overwritten with that value (e.g. NaN), rows
    that no result may depend on."""
    if len(lens) != B:
        raise ValueError("lens must hold B lengths")
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn((B, H, d), generator=g, dtype=torch.float32)
    k = torch.randn((B, Hkv, Nmax, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, Hkv, Nmax, d), generator=g, dtype=torch.float32)
    t = DTYPES[dtype]
    q, k, v = q.to(t), k.to(t), v.to(t)
    if fill is not None:
        for b, n in enumerate(lens):
            k[b, :, int(n):] = fill
            v[b, :, int(n):] = fill
    return {"q": q, "k_cache": k, "v_cache": v,
            "cache_seqlens": torch.tensor([int(n) for n in lens], dtype=torch.int32)}


def make_decode_fp8_inputs(B: int, H: int, Hkv: int, Nmax: int, d: int, lens,
                           dtype: str = "bf16", seed: int = 0, fill_code: int | None = None):
    """Decoding inputs with E4M3 caches: q drawn and rounded as in make_decode_inputs, then
    K and V caches drawn in fp32 N(0, 1), each divided by its scale amax / 448 and rounded
    to E4M3 by torch's float8_e4m3fn conversion.  Returns dict(q, k8, v8 (uint8 codes,
    (B, Hkv, Nmax, d)), cache_seqlens, k_scale, v_scale).  With ``fill_code`` every cache
    row at or past its sequence's length holds that code (0x7F: NaN)."""
    if len(lens) != B:
        raise ValueError("lens must hold B lengths")
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn((B, H, d), generator=g, dtype=torch.float32).to(DTYPES[dtype])
    out = {"q": q}
    for name in ("k", "v"):
        x = torch.randn((B, Hkv, Nmax, d), generator=g, dtype=torch.float32)
        sc = torch.tensor(float(x.abs().max()) / 448.0, dtype=torch.float32)
        codes = (x / sc).to(torch.float8_e4m3fn).view(torch.uint8).clone()
        if fill_code is not None:
            for b, n in enumerate(lens):
                codes[b, :, int(n):] = int(fill_code)
        out[name + "8"] = codes
        out[name + "_scale"] = float(sc)
    out["cache_seqlens"] = torch.tensor([int(n) for n in lens], dtype=torch.int32)
    return out


def make_fp8_inputs(B: int, H: int, N: int, d: int, seed: int = 0, Hkv: int | None = None):
    """8-bit E4M3 inputs with per-tensor scales: Q, K, V drawn like make_inputs (fp32
    N(0, 1), in that order), each divided by its scale amax / 448 (so the largest
    magnitude lands on the largest finite E4M3 value) and rounded to E4M3 by torch's
    float8_e4m3fn conversion (round to nearest even).  Returns dict(q8, k8, v8, vt8)
    of uint8 code tensors -- q8 (B, H, N, d), k8 and v8 (B, Hkv, N, d), vt8 = v8 with
    the last two axes swapped (B, Hkv, d, N) -- and the scales q_scale, k_scale,
    v_scale (Python floats, exact fp32 values)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    kvh = H if Hkv is None else Hkv
    out = {}
    for name, heads in (("q", H), ("k", kvh), ("v", kvh)):
        x = torch.randn((B, heads, N, d), generator=g, dtype=torch.float32)
        sc = torch.tensor(float(x.abs().max()) / 448.0, dtype=torch.float32)
        out[name + "8"] = (x / sc).to(torch.float8_e4m3fn).view(torch.uint8)
        out[name + "_scale"] = float(sc)
    out["vt8"] = out["v8"].transpose(-1, -2).contiguous()
    return out


# Workloads: (name, B, H, N, d, dtype, causal, qk_std)
WORKLOADS = {
    "tiny_full_d64_fp16": (1, 1, 128, 64, "fp16", False, 1.0),
    "ragged_causal_d32_fp16": (4, 8, 1000, 32, "fp16", True, 1.0),
    "ragged_causal_d32_fp16_stress": (4, 8, 1000, 32, "fp16", True, 4.0),
    "gpt2m_causal_d64_fp16": (8, 16, 1024, 64, "fp16", True, 1.0),
    "n4k_full_d128_bf16": (2, 16, 4096, 128, "bf16", False, 1.0),
    "n4k_causal_d128_bf16": (2, 16, 4096, 128, "bf16", True, 1.0),
    "n8k_causal_d128_bf16": (1, 32, 8192, 128, "bf16", True, 1.0),
    "n16k_causal_d128_bf16": (1, 32, 16384, 128, "bf16", True, 1.0),
}
