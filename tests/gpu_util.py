"""Helpers shared by the GPU tests: upload operands, run through the C ABI,
download results.  Device memory comes from torch; every step of the GEMM
runs in the library's kernels."""
import numpy as np
import torch

from bit_tensor_gemm_gb300 import lbgemm as L

DEV = torch.device("cuda:0")


def to_dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).to(DEV)
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def gemm(bits, A, B, K, variant=-1, stream=None):
    M, N = A.shape[0], B.shape[0]
    dA, dB = to_dev(A), to_dev(B)
    dC = torch.full((M, N), -7, dtype=torch.int32, device=DEV)
    if variant < 0:
        L.lbgemm_run(bits, M, N, K, dA, dB, dC, stream)
    else:
        L.lbgemm_run_variant(bits, M, N, K, dA, dB, dC, variant, stream)
    L.lbgemm_device_status(stream)
    return dC.cpu().numpy()


def fused(A, B, K, tile_n):
    """lbgemm_run_fused: the larger operand converted from int8 in the kernel."""
    M, N = A.shape[0], B.shape[0]
    dA, dB = to_dev(A), to_dev(B)
    dC = torch.full((M, N), -7, dtype=torch.int32, device=DEV)
    L.lbgemm_run_fused(M, N, K, dA, dB, dC, tile_n)
    L.lbgemm_device_status()
    return dC.cpu().numpy()


def warpmma(A, B, K):
    """lbgemm_run_warpmma: the warp-level fp16 MMA kernel (small side <= 32)."""
    M, N = A.shape[0], B.shape[0]
    dA, dB = to_dev(A), to_dev(B)
    dC = torch.full((M, N), -7, dtype=torch.int32, device=DEV)
    L.lbgemm_run_warpmma(M, N, K, dA, dB, dC)
    L.lbgemm_device_status()
    return dC.cpu().numpy()


def linear(X, sx, W, sw, variant=-1):
    M, K = X.shape
    N = W.shape[0]
    dY = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    args = (M, N, K, to_dev(X), to_dev(sx), to_dev(W), to_dev(sw), dY)
    if variant < 0:
        L.lbgemm_linear(*args)
    else:
        L.lbgemm_linear_variant(*args, variant)
    L.lbgemm_device_status()
    return dY.float().cpu().numpy().astype(np.float64)


def sample_positions(M, N, count, seed):
    g = np.random.default_rng(seed)
    rows = np.concatenate([g.integers(0, M, count), [0, M - 1, M - 1, 0]])
    cols = np.concatenate([g.integers(0, N, count), [0, N - 1, 0, N - 1]])
    return rows, cols


def encoded(bits, A, B, K, variant=-1):
    """lbgemm_encode of both operands, then lbgemm_run_encoded (the GEMM
    kernel alone on the re-encoded operands)."""
    M, N = A.shape[0], B.shape[0]
    dA, dB = to_dev(A), to_dev(B)
    eA = torch.empty(L.lbgemm_encoded_size(bits, M, K), dtype=torch.uint8, device=DEV)
    eB = torch.empty(L.lbgemm_encoded_size(bits, N, K), dtype=torch.uint8, device=DEV)
    L.lbgemm_encode(bits, M, K, dA, eA)
    L.lbgemm_encode(bits, N, K, dB, eB)
    dC = torch.full((M, N), -7, dtype=torch.int32, device=DEV)
    L.lbgemm_run_encoded(bits, M, N, K, eA, eB, dC, variant)
    L.lbgemm_device_status()
    return dC.cpu().numpy()
