import os
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads")


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def np_i32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.int64)


def oracle_args(case):
    """Numpy views of a workloads.PagedCase for the oracle."""
    return dict(
        q_bits=bits(case.q),
        k_pool_bits=bits(case.k_pool),
        v_pool_bits=bits(case.v_pool),
        block_table=np_i32(case.block_table),
        seq_lens=case.seq_lens_host,
        cu_seqlens_q=np_i32(case.cu_seqlens_q),
        num_q_heads=case.num_q_heads,
        num_kv_heads=case.num_kv_heads,
        page_size=case.page_size,
        scale=case.softmax_scale,
    )


@pytest.fixture(scope="session")
def cuda_device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")
