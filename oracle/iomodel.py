"""Byte and FLOP arithmetic of attention -- TEST INFRASTRUCTURE ONLY.

Plain counts of tensor sizes, as the "flash-attn-triton" docs page does in its
footprint calculator (Fig. 2: score matrix B*H*N*N against the linear Q, K, V,
O and L) and its HBM-access table (Table 2: Theta(N^2 + N d) for ordinary
attention, Theta(N^2 d^2 / M) for the tiled kernel); the tutorial page
("What is FlashAttention?") counts the entries of one head's score table.
FLOPs follow the usual matmul count: 2*N*N*d for each of QK^T and PV per head,
the backward five such products (2.5x), and causal masking halving both.
"""
from __future__ import annotations


def score_entries(N: int) -> int:
    """Entries of one head's N x N score table."""
    return N * N


def score_matrix_bytes(B: int, H: int, N: int, elem_bytes: int = 2) -> int:
    """Bytes of the whole B*H*N*N score matrix at ``elem_bytes`` per entry."""
    return B * H * N * N * elem_bytes


def linear_footprint_bytes(B: int, H: int, N: int, d: int, elem_bytes: int = 2) -> int:
    """Q, K, V, O in the input dtype plus L in fp32: everything the tiled kernel keeps."""
    return 4 * B * H * N * d * elem_bytes + 4 * B * H * N


def tile_bytes(block_m: int, block_n: int, elem_bytes: int = 2) -> int:
    """One BLOCK_M x BLOCK_N score tile held on chip."""
    return block_m * block_n * elem_bytes


def tiled_hbm_ratio(d: int, sram_bytes: int) -> float:
    """The d^2 / M factor by which tiling shrinks the N^2 term of HBM accesses."""
    return d * d / sram_bytes


def standard_hbm_bytes_fwd(B: int, H: int, N: int, d: int, elem_bytes: int = 2) -> int:
    """Ordinary attention forward, counted plainly: read Q, K; write S; read S; write P;
    read P, V; write O."""
    n = B * H * N * d * elem_bytes
    s = score_matrix_bytes(B, H, N, elem_bytes)
    return 2 * n + s + s + s + s + n + n


def attention_flops(B: int, H: int, N: int, d: int, causal: bool) -> tuple[float, float]:
    """(forward, backward) FLOPs: 4*B*H*N^2*d forward, 2.5x that backward, both halved
    when causal (the halving convention of the benchmark, not N(N+1)/2)."""
    f = 4.0 * B * H * N * N * d
    if causal:
        f *= 0.5
    return f, 2.5 * f


def fwd_algorithmic_bytes(B: int, H: int, N: int, d: int, elem_bytes: int = 2) -> int:
    """Forward reads Q, K, V once and writes O and L once."""
    return 4 * B * H * N * d * elem_bytes + 4 * B * H * N


def bwd_algorithmic_bytes(B: int, H: int, N: int, d: int, elem_bytes: int = 2) -> int:
    """Backward reads Q, K, V, O, dO, L and writes dQ, dK, dV (D round trip included)."""
    return 8 * B * H * N * d * elem_bytes + 3 * 4 * B * H * N
