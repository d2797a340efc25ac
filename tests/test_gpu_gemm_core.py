"""The tcgen05 GEMM core alone, for each operand layout the loss uses.

C = A_op B_op^T with bf16 inputs and fp32 accumulation is compared with a
float64 CPU product of the same bf16 values.  Sizes span several tiles in
every dimension and end in ragged tails (M, N, K not multiples of the
128 x BN x 64 single-CTA tile or of the 256 x 256 x 64 CTA-pair tile).
"""
import numpy as np
import pytest
import torch

import chunked_top_kl_gemm_b300 as kd
from tests.gpu_util import ensure_lib

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bn", [0, 192, 256])
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 384, 192), (136, 264, 72),
                                   (392, 520, 328)])
def test_gemm_layouts(a_mn, b_mn, bn, M, N, K):
    ensure_lib()
    g = torch.Generator().manual_seed(M * 7 + N * 3 + K + 2 * a_mn + b_mn)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)
    Ad = (A.t().contiguous() if a_mn else A).cuda()
    Bd = (B.t().contiguous() if b_mn else B).cuda()
    C = kd.kd_gemm_bf16_test(Ad, Bd, bool(a_mn), bool(b_mn), bn).cpu().double().numpy()
    ref = A.double().numpy() @ B.double().numpy().T
    err = np.abs(C - ref).max() / np.abs(ref).max()
    assert err < 1e-5, err


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(256, 256, 64), (512, 768, 448), (136, 264, 72),
                                   (392, 520, 328), (1000, 2880, 200), (2880, 600, 136)])
def test_gemm_layouts_cta_pair(a_mn, b_mn, M, N, K):
    """The 2-CTA MMA form: a 256 x 256 tile per CTA pair, ragged last tiles
    multiplied at their valid width (rounded to 32 columns)."""
    ensure_lib()
    g = torch.Generator().manual_seed(M * 5 + N * 11 + K + 2 * a_mn + b_mn)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)
    Ad = (A.t().contiguous() if a_mn else A).cuda()
    Bd = (B.t().contiguous() if b_mn else B).cuda()
    C = kd.kd_gemm_bf16_test(Ad, Bd, bool(a_mn), bool(b_mn), 0, pair=True).cpu().double().numpy()
    ref = A.double().numpy() @ B.double().numpy().T
    err = np.abs(C - ref).max() / np.abs(ref).max()
    assert err < 1e-5, err


@pytest.mark.parametrize("M,N,K", [(256, 256, 64), (136, 264, 72), (392, 520, 136),
                                   (1000, 2880, 200), (512, 768, 2880)])
def test_gemm_cta_pair_two_kblocks_per_stage(M, N, K):
    """The FWD / DZ ring: two 64-deep k-blocks per stage, odd k-block counts
    included (the stage's second k-block is then loaded but not multiplied)."""
    ensure_lib()
    g = torch.Generator().manual_seed(M + 3 * N + 7 * K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)
    C = kd.kd_gemm_bf16_test(A.cuda(), B.cuda(), False, False, 0, pair=2).cpu().double().numpy()
    ref = A.double().numpy() @ B.double().numpy().T
    err = np.abs(C - ref).max() / np.abs(ref).max()
    assert err < 1e-5, err


def test_gemm_cta_pair_is_deterministic_and_matches_single_cta():
    ensure_lib()
    g = torch.Generator().manual_seed(3)
    A = torch.randn(640, 320, generator=g).to(torch.bfloat16).cuda()
    B = torch.randn(776, 320, generator=g).to(torch.bfloat16).cuda()
    c1 = kd.kd_gemm_bf16_test(A, B, False, False, 256)
    c2 = kd.kd_gemm_bf16_test(A, B, False, False, 0, pair=True)
    c3 = kd.kd_gemm_bf16_test(A, B, False, False, 0, pair=True)
    assert torch.equal(c2, c3)
    assert torch.allclose(c1, c2, rtol=0, atol=1e-5 * float(c1.abs().max()))
