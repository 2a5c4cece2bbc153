"""Shared test helpers: the GEMM tolerance and comparisons."""
from __future__ import annotations

import numpy as np
import torch

import oracle.fp8q_oracle as O

# max |gpu - oracle| <= REL * ||a_i|| * ||b_j|| + 1 ulp of the output dtype at
# the oracle value (a_i, b_j: dequantized row of A and column of B).
REL = 1e-4


def ulp(x: np.ndarray, out: str) -> np.ndarray:
    """Spacing of the output format at |x| (normal range)."""
    mant = 7 if out == "bf16" else 23
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(ax)) - mant)


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.numpy()


def assert_gemm_close(gpu: np.ndarray, ref: np.ndarray, na: np.ndarray, nb: np.ndarray,
                      out: str) -> float:
    """Element-wise bound; returns the worst |err| / bound (must be <= 1)."""
    gpu = np.asarray(gpu, np.float64)
    bound = REL * np.outer(na, nb) + ulp(ref, out)
    err = np.abs(gpu - ref)
    ratio = err / bound
    worst = float(ratio.max()) if ratio.size else 0.0
    if worst > 1.0:
        i, j = np.unravel_index(np.argmax(ratio), ratio.shape)
        raise AssertionError(f"GEMM mismatch at ({i},{j}): gpu={gpu[i, j]!r} oracle={ref[i, j]!r}"
                             f" err={err[i, j]:.3e} bound={bound[i, j]:.3e}"
                             f" ({int((ratio > 1).sum())} of {ratio.size} outside)")
    assert np.isfinite(gpu).all()
    return worst


def check_gemm_sampled(d_gpu, qa, sa, qb, sb, rows, col_blocks, out, scale_b="128x128"):
    """Oracle on rows x (128-column blocks) of a large GEMM; qa/qb/sa/sb numpy."""
    cols = np.concatenate([np.arange(c * 128, (c + 1) * 128) for c in col_blocks])
    if scale_b == "128x128":
        sb_sel = sb[:, col_blocks]
    else:
        sb_sel = sb[:, cols]
    qa_r, sa_r = qa[rows], sa[:, rows]
    qb_c = qb[cols]
    ref = O.gemm_blockscaled(qa_r, sa_r, qb_c, sb_sel, scale_b)
    na, nb = O.row_col_norms(qa_r, sa_r, qb_c, sb_sel, scale_b)
    gpu = d_gpu[np.ix_(rows, cols)]
    return assert_gemm_close(gpu, ref, na, nb, out)


def bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a).view(np.uint32)
