"""The microscaling GEMM (FP8Q_MX_BLOCK_SCALE: tcgen05 kind::mxf8f6f4 with
UE8M0 scales) vs the CPU oracle. With power-of-two 1x128 / 128x128 scales it
computes the same D as the promoted GEMM, so it is held to the same bound:
max|gpu - oracle| <= 1e-4 * ||a_i|| * ||b_j|| + 1 ulp of the output format."""
import numpy as np
import pytest
import torch

import oracle.fp8q_oracle as O
from fp8_block_scaled_17_b300 import workloads as W
from tests.helpers import assert_gemm_close, check_gemm_sampled, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F(cuda_device):
    from fp8_block_scaled_17_b300 import fp8q
    return fp8q


def _pow2_problem(F, M, N, K, seed, outlier_frac=0.001, outlier_scale=100.0):
    a = W.bf16_normal((M, K), 1.0, seed, outlier_frac, outlier_scale).cuda()
    w = W.bf16_normal((K, N), 0.02, seed + 1).cuda()
    qa, sa = F.quant_act_1x128(a, True)
    qb, sb = F.quant_w_128x128(w, True)
    return qa, sa, qb, sb


def _check(d, qa, sa, qb, sb, out, scale_b="128x128"):
    qa, sa, qb, sb = (x.cpu().numpy() for x in (qa, sa, qb, sb))
    ref = O.gemm_blockscaled(qa, sa, qb, sb, scale_b)
    na, nb = O.row_col_norms(qa, sa, qb, sb, scale_b)
    return assert_gemm_close(to_np(d), ref, na, nb, out)


@pytest.mark.parametrize("M,N,K,out", [
    (256, 256, 512, "f32"),     # whole tiles, K = one scale group of four K-blocks
    (300, 384, 640, "bf16"),    # ragged M, a 128-column last N tile, KB = 5 (partial group)
    (1, 128, 128, "f32"),       # one row, one K-block
    (129, 640, 1152, "f32"),    # 9 K-blocks: three groups, the last with one K-block
    (517, 1280, 2048, "bf16"),
])
def test_mx_against_oracle(F, M, N, K, out):
    qa, sa, qb, sb = _pow2_problem(F, M, N, K, seed=M + N + K)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    d = F.gemm_blockscaled(qa, sa, qb, sb, out_dtype=dt, mx=True)
    assert F.get_status() == F.OK
    _check(d, qa, sa, qb, sb, out)


def test_mx_strided_and_16b_aligned_output(F):
    """D with a row pitch that is 16- but not 32-byte aligned (the 16-byte
    store path), written inside a larger buffer whose other columns stay put."""
    qa, sa, qb, sb = _pow2_problem(F, 200, 256, 384, seed=5)
    big = torch.full((200, 264), -7.0, dtype=torch.float32, device="cuda")
    d = big[:, :256]
    F.gemm_blockscaled(qa, sa, qb, sb, d=d, mx=True)
    assert F.get_status() == F.OK
    assert (big[:, 256:] == -7.0).all()
    _check(d, qa, sa, qb, sb, "f32")


def test_mx_scale_b_1x128(F):
    """Wgrad-shaped call: both operands 1x128 along K with power-of-two scales
    (X requantized to 128x1, dY quantized along tokens)."""
    x = W.bf16_normal((512, 256), 1.0, seed=21)
    dy = W.bf16_normal((512, 384), 1e-3, seed=22)
    qx, sx = F.quant_act_1x128(x.cuda(), True)
    qa, sa = F.requant_1x128_to_128x1(qx, sx, True)                    # [256][512]
    qb, sb = F.quant_act_1x128(dy.cuda(), True, transposed_input=True)  # [384][512]
    d = F.gemm_blockscaled(qa, sa, qb, sb, out_dtype=torch.float32, scale_b_1x128=True,
                           mx=True)
    assert F.get_status() == F.OK
    _check(d, qa, sa, qb, sb, "f32", "1x128")


def test_mx_per_column_scales_distinct(F):
    """Every B column and every A row gets its own power-of-two scale (1x128
    mode, scales drawn over 2^-20 .. 2^20): a scale read from the wrong TMEM
    lane, column or byte changes the result by a power of two."""
    M, N, K = 256, 512, 1024
    g = np.random.default_rng(3)
    qa = torch.from_numpy(g.integers(0, 256, (M, K), dtype=np.uint8))
    qb = torch.from_numpy(g.integers(0, 256, (N, K), dtype=np.uint8))
    qa[(qa & 0x7F) == 0x7F] = 0x38   # no NaN codes
    qb[(qb & 0x7F) == 0x7F] = 0x38
    sa = torch.from_numpy(np.exp2(g.integers(-20, 21, (K // 128, M))).astype(np.float32))
    sb = torch.from_numpy(np.exp2(g.integers(-20, 21, (K // 128, N))).astype(np.float32))
    qa, qb, sa, sb = qa.cuda(), qb.cuda(), sa.cuda(), sb.cuda()
    d = F.gemm_blockscaled(qa, sa, qb, sb, out_dtype=torch.float32, scale_b_1x128=True, mx=True)
    assert F.get_status() == F.OK
    _check(d, qa, sa, qb, sb, "f32", "1x128")


def test_mx_matches_promoted(F):
    """Same codes and power-of-two scales through both kernels: both meet the
    bound against the oracle, and their difference is within twice it."""
    qa, sa, qb, sb = _pow2_problem(F, 384, 768, 2048, seed=9)
    d_p = F.gemm_blockscaled(qa, sa, qb, sb, out_dtype=torch.float32)
    d_x = F.gemm_blockscaled(qa, sa, qb, sb, out_dtype=torch.float32, mx=True)
    assert F.get_status() == F.OK
    w_p = _check(d_p, qa, sa, qb, sb, "f32")
    w_x = _check(d_x, qa, sa, qb, sb, "f32")
    print(f"worst error / bound: promoted {w_p:.3e}, block-scaled MMA {w_x:.3e}")


@pytest.mark.parametrize("sizes,out", [([3, 0, 1, 130, 0, 257], "f32"),
                                       ([128, 128, 1, 300], "bf16")])
def test_mx_grouped(F, sizes, out):
    E, K, N = len(sizes), 640, 384
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    Mtot = int(offs[-1])
    x = W.bf16_normal((Mtot, K), 1.0, seed=sum(sizes), outlier_frac=0.002,
                      outlier_scale=100.0).cuda()
    qa, sa = F.quant_act_1x128(x, True)
    qb = torch.empty((E, N, K), dtype=torch.uint8, device="cuda")
    sb = torch.empty((E, K // 128, N // 128), dtype=torch.float32, device="cuda")
    for e in range(E):
        F.quant_w_128x128(W.bf16_normal((K, N), 0.02, seed=40 + e).cuda(), True, q=qb[e],
                          sb=sb[e])
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    d = F.grouped_gemm(qa, sa, torch.from_numpy(offs).cuda(), qb, sb, out_dtype=dt, mx=True)
    assert F.get_status() == F.OK
    qa_n, sa_n, qb_n, sb_n = (t.cpu().numpy() for t in (qa, sa, qb, sb))
    ref = O.grouped_gemm_blockscaled(qa_n, sa_n, offs, qb_n, sb_n)
    dn = to_np(d)
    for e in range(E):
        r0, r1 = offs[e], offs[e + 1]
        if r1 > r0:
            na, nb = O.row_col_norms(qa_n[r0:r1], sa_n[:, r0:r1], qb_n[e], sb_n[e])
            assert_gemm_close(dn[r0:r1], ref[r0:r1], na, nb, out)


def test_mx_reports_scales_that_are_not_powers_of_two(F):
    """Plain (non-power-of-two) scales have no UE8M0 form: the call is
    reported as FP8Q_ERR_INVALID_ARG by get_status; power-of-two ones are not."""
    a = W.bf16_normal((128, 256), 1.0, seed=1).cuda()
    w = W.bf16_normal((256, 256), 0.02, seed=2).cuda()
    qa, sa = F.quant_act_1x128(a)       # plain scales
    qb, sb = F.quant_w_128x128(w, True)
    assert F.get_status() == F.OK
    F.gemm_blockscaled(qa, sa, qb, sb, mx=True)
    assert F.get_status() == F.ERR_INVALID_ARG
    qa2, sa2 = F.quant_act_1x128(a, True)
    F.gemm_blockscaled(qa2, sa2, qb, sb, mx=True)
    assert F.get_status() == F.OK


def test_mx_partial_last_wave_reproducible(F):
    """151 tiles of 128 x 256 on a 148-SM grid: every output against the
    oracle, bitwise reproducible across calls."""
    props = torch.cuda.get_device_properties(0)
    M = 128 * (props.multi_processor_count + 3)
    qa, sa, qb, sb = _pow2_problem(F, M, 256, 1024, seed=77)
    d1 = F.gemm_blockscaled(qa, sa, qb, sb, out_dtype=torch.float32, mx=True)
    d2 = F.gemm_blockscaled(qa, sa, qb, sb, out_dtype=torch.float32, mx=True)
    assert F.get_status() == F.OK
    assert torch.equal(d1, d2)
    _check(d1, qa, sa, qb, sb, "f32")


def _sample_rows(M, n, seed):
    g = np.random.default_rng(seed)
    return np.unique(np.concatenate([g.choice(M, n, replace=False), [0, 127, 128, M - 1]]))


def test_mx_dense_forward_full_sampled(F):
    """The dense forward workload [8192][7168] x [7168][7168] -> bf16 with
    power-of-two scales, as bench.py's block-scaled-MMA workload times it:
    sampled rows x 128-column blocks against the oracle."""
    p = W.DENSE_FWD
    a, w = p.make()
    qa, sa = F.quant_act_1x128(a.cuda(), True)
    qb, sb = F.quant_w_128x128(w.cuda(), True)
    d = F.gemm_blockscaled(qa, sa, qb, sb, out_dtype=torch.bfloat16, mx=True)
    assert F.get_status() == F.OK
    check_gemm_sampled(to_np(d), qa.cpu().numpy(), sa.cpu().numpy(), qb.cpu().numpy(),
                       sb.cpu().numpy(), _sample_rows(p.M, 40, 3), [0, 28, 55], "bf16")


@pytest.mark.parametrize("K", [4096, 16384])
def test_mx_long_k_accuracy(F, K):
    """Accumulation over long K at M = N = 4096 (the K-sweep operands, all
    scales 2^-6): the block-scaled MMA against the exact result, next to the
    promoted kernel; both must meet the bound on the sampled rows."""
    M = N = 4096
    qa, sa = F.quant_act_1x128(W.ksweep_operand(M, K, 1).cuda(), True)
    qb, sb = F.quant_act_1x128(W.ksweep_operand(N, K, 2).cuda(), True)
    d_x = to_np(F.gemm_blockscaled(qa, sa, qb, sb, out_dtype=torch.float32, scale_b_1x128=True,
                                   mx=True))
    d_p = to_np(F.gemm_blockscaled(qa, sa, qb, sb, out_dtype=torch.float32, scale_b_1x128=True))
    assert F.get_status() == F.OK
    rows = _sample_rows(M, 60, K)
    qa_n, sa_n, qb_n, sb_n = qa.cpu().numpy(), sa.cpu().numpy(), qb.cpu().numpy(), sb.cpu().numpy()
    ref = O.gemm_blockscaled(qa_n[rows], sa_n[:, rows], qb_n, sb_n, "1x128")
    na, nb = O.row_col_norms(qa_n[rows], sa_n[:, rows], qb_n, sb_n, "1x128")
    norm = np.outer(na, nb)
    for name, d in (("promoted", d_p), ("block-scaled MMA", d_x)):
        err = np.abs(d[rows] - ref)
        print(f"K={K} {name}: max|C-R|/max|R| = {O.max_relative_error(d[rows], ref):.3e}, "
              f"max|C-R|/(|a_i||b_j|) = {(err / norm).max():.3e}")
        assert_gemm_close(d[rows], ref, na, nb, "f32")


def test_mx_injected_timeout_is_reported_and_recoverable(F, monkeypatch):
    """A wait that nothing satisfies (FP8Q_DEBUG_INJECT_TIMEOUT) gives up after
    its limit; every role of the block-scaled MMA kernel stops, the call is
    reported as FP8Q_ERR_TIMEOUT, and the next call is correct."""
    qa, sa, qb, sb = _pow2_problem(F, 256, 512, 512, seed=40)
    assert F.get_status() == F.OK
    monkeypatch.setenv("FP8Q_DEBUG_INJECT_TIMEOUT", "1")
    F.gemm_blockscaled(qa, sa, qb, sb, out_dtype=torch.float32, mx=True)
    assert F.get_status() == F.ERR_TIMEOUT
    assert F.get_status() == F.OK  # reading clears it
    monkeypatch.delenv("FP8Q_DEBUG_INJECT_TIMEOUT")
    d = F.gemm_blockscaled(qa, sa, qb, sb, out_dtype=torch.float32, mx=True)
    assert F.get_status() == F.OK
    _check(d, qa, sa, qb, sb, "f32")
