"""Helpers for the GPU parity tests (tolerances from the accuracy target:
max-abs 2e-2 against the float64 oracle for bf16 KV, 6e-2 for fp8 KV)."""
import numpy as np
import torch

TOL_BF16 = 2e-2
TOL_FP8 = 6e-2


def max_abs(gpu: torch.Tensor, ref: torch.Tensor) -> float:
    d = (gpu.detach().double().cpu() - ref).abs()
    assert not torch.isnan(d).any(), "NaN in compared rows"
    return d.max().item() if d.numel() else 0.0


def sample_tokens(q_lens, per_chunk=6, seed=0):
    """All decode tokens plus first/last/random tokens of every longer chunk."""
    rng = np.random.default_rng(seed)
    toks, off = [], 0
    for ql in q_lens:
        if ql <= 4:
            toks.extend(range(off, off + ql))
        elif ql > 0:
            pick = {off, off + ql - 1, *rng.integers(off, off + ql, size=per_chunk - 2).tolist()}
            toks.extend(sorted(pick))
        off += ql
    return toks


def gpu(t):
    return t.to("cuda", non_blocking=False)
