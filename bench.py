"""Benchmark of the fused attention forward pass (filled in below)."""


def attention_flops(B, Hq, Nq, Nk, d, causal):
    """Algorithmic FLOPs: Q K^T and P V, 2 flops per multiply-add, 4*d per
    score; the causal mask halves the count."""
    f = 4.0 * B * Hq * Nq * Nk * d
    return f / 2 if causal else f
