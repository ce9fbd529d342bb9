"""Tensor-core operand layouts on the device: one tcgen05 product per layout
combination the chunked kernels use, against a plain fp64 matrix product."""
import numpy as np
import pytest
import torch

from linear_attention_05_gb300 import binding as B
from util import rel_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("a_mn,b_mn,N,K", [
    (0, 0, 64, 128),   # [Kt;Qt] x Kh^T, S^T x ... (K-major A and B)
    (0, 0, 64, 64),    # W^T x P^T
    (1, 0, 64, 64),    # Kt^T / V^T x T'^T (MN-major A)
    (0, 1, 128, 64),   # W^T x Kd (MN-major B)
    (0, 1, 128, 128),  # S^T x Phi'^T
    (0, 1, 64, 128),   # S^T x Q'^T
    (1, 1, 192, 64),
])
def test_umma_layout(a_mn, b_mn, N, K):
    g = torch.Generator(device="cuda").manual_seed(1000 + 16 * N + K + 2 * a_mn + b_mn)
    A = torch.randn((128, K), generator=g, device="cuda").to(torch.bfloat16)
    Bm = torch.randn((K, N), generator=g, device="cuda").to(torch.bfloat16)
    D = torch.full((128, N), float("nan"), device="cuda")
    assert B.kda_selftest_umma(A, Bm, D, a_mn, b_mn) == B.KDA_OK
    ref = A.double().cpu().numpy() @ Bm.double().cpu().numpy()
    assert rel_err(D.cpu().numpy(), ref) < 1e-5
