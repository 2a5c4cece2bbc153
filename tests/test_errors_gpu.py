"""Device-side failure detection without a GPU fault: a pipeline wait that
nothing will satisfy gives up after its limit, the kernel stops cleanly and
reports FP8Q_ERR_TIMEOUT, and the context stays usable. Malformed grouped
offsets are clamped and reported."""
import os

import numpy as np
import pytest
import torch

import oracle.fp8q_oracle as O
from fp8_block_scaled_17_b300 import workloads as W
from tests.helpers import assert_gemm_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F(cuda_device):
    from fp8_block_scaled_17_b300 import fp8q
    return fp8q


def _problem(F):
    a = W.bf16_normal((256, 512), 1.0, seed=40).cuda()
    w = W.bf16_normal((512, 512), 0.02, seed=41).cuda()
    qa, sa = F.quant_act_1x128(a)
    qb, sb = F.quant_w_128x128(w)
    return qa, sa, qb, sb


def test_injected_timeout_is_reported_and_recoverable(F, monkeypatch):
    qa, sa, qb, sb = _problem(F)
    assert F.get_status() == F.OK
    monkeypatch.setenv("FP8Q_DEBUG_INJECT_TIMEOUT", "1")
    F.gemm_blockscaled(qa, sa, qb, sb, out_dtype=torch.float32)
    assert F.get_status() == F.ERR_TIMEOUT
    assert F.get_status() == F.OK  # reading clears it
    monkeypatch.delenv("FP8Q_DEBUG_INJECT_TIMEOUT")
    d = F.gemm_blockscaled(qa, sa, qb, sb, out_dtype=torch.float32)
    assert F.get_status() == F.OK
    qa_n, sa_n, qb_n, sb_n = (t.cpu().numpy() for t in (qa, sa, qb, sb))
    ref = O.gemm_blockscaled(qa_n, sa_n, qb_n, sb_n)
    na, nb = O.row_col_norms(qa_n, sa_n, qb_n, sb_n)
    assert_gemm_close(to_np(d), ref, na, nb, "f32")


def test_malformed_offsets_are_clamped_and_reported(F):
    qa, sa, qb, sb = _problem(F)
    qb3 = qb.unsqueeze(0).expand(3, -1, -1).contiguous()
    sb3 = sb.unsqueeze(0).expand(3, -1, -1).contiguous()
    bad = torch.tensor([0, 200, 100, 9999], dtype=torch.int32, device="cuda")
    d = torch.zeros((256, 512), dtype=torch.float32, device="cuda")
    F.grouped_gemm(qa, sa, bad, qb3, sb3, d=d)
    assert F.get_status() == F.ERR_INVALID_ARG
    # clamped to [0, 200, 200, 256]: rows 0..199 expert 0, rows 200..255 expert 2
    qa_n, sa_n, qb_n, sb_n = (t.cpu().numpy() for t in (qa, sa, qb, sb))
    ref = O.gemm_blockscaled(qa_n, sa_n, qb_n, sb_n)
    na, nb = O.row_col_norms(qa_n, sa_n, qb_n, sb_n)
    assert_gemm_close(to_np(d), ref, na, nb, "f32")
