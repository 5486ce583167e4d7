"""Shared helpers for the GPU parity tests (device transfer of generator outputs)."""
import numpy as np
import pytest
import torch


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def dev_u16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to("cuda")


def dev_u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def sample_rows(M: int, bm: int, n_random: int, seed: int) -> np.ndarray:
    """Rows at tile boundaries and edges plus random ones (sorted, unique)."""
    rows = {0, M - 1, min(bm - 1, M - 1), min(bm, M - 1), M // 2, max(M - bm, 0)}
    rng = np.random.default_rng(seed)
    rows.update(int(r) for r in rng.integers(0, M, n_random))
    return np.array(sorted(rows), dtype=np.int64)
