"""The allocation-free decode entry point, called through the C ABI.

Some callers cannot allocate device memory (allocator or memory-pool
callbacks, plugins inside a framework that owns every device allocation), so
they cannot hand attn_decode_paged a workspace.  attn_decode_paged_noalloc
keeps that scratch in a fixed device array inside the library.  Both calls run
the same kernels with the same split, so their results must be bit-identical;
the result is also checked against the fp64 oracle.  This file is collected
last on purpose: its calls share that array, and it must pass both alone in a
fresh process and after every other test.
"""

import ctypes

import pytest
import torch

import oracle
import workloads
from tests.conftest import assert_attention_close, compact_for_oracle

pytestmark = pytest.mark.gpu

PA_ERR_SCRATCH_LIMIT = -9


def _lib():
    pa = pytest.importorskip("paged_kv_decode_17_gb300")
    return pa, pa.load_library(build_if_missing=True)


def _noalloc(lib, g, out, lse, status):
    return lib.attn_decode_paged_noalloc(
        out.data_ptr(), lse.data_ptr(), g.q.data_ptr(), g.k_pool.data_ptr(), g.v_pool.data_ptr(), g.num_pages,
        g.block_table.data_ptr(), g.max_pages_per_seq, g.seq_lens.data_ptr(), g.batch, max(1, g.max_seq_len),
        g.page_size, g.num_q_heads, g.num_kv_heads, g.head_dim, ctypes.c_float(g.softmax_scale),
        status.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("make", [
    lambda dev: workloads.tiny_decode(seed=3, device=dev),
    lambda dev: workloads.make_paged_case("ragged", [3000, 1, 700, 12000, 45], [1] * 5, 32, 8, 128, seed=5,
                                          device=dev),
    lambda dev: workloads.make_paged_case("d64", [4096] * 8, [1] * 8, 16, 2, 64, seed=6, device=dev),
])
def test_noalloc_matches_workspace_entry_point_twice(cuda_device, make):
    pa, lib = _lib()
    g = make(cuda_device)
    ref, ref_lse = pa.attn_decode_paged(g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens, g.softmax_scale,
                                        max_seq_len=max(1, g.max_seq_len), return_lse=True)
    want_out, want_lse = oracle.paged_attention(**compact_for_oracle(g, list(range(g.batch)))[0])
    for _ in range(2):  # the second call sees what the first left in the shared array
        out = torch.full_like(g.q, float("nan"))
        lse = torch.full((g.batch, g.num_q_heads), float("nan"), device=cuda_device)
        status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
        assert _noalloc(lib, g, out, lse, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        # same kernels, same split, same merge order: bit-identical to the workspace entry point
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), \
            "allocation-free output differs from attn_decode_paged"
        assert torch.equal(lse, ref_lse), "allocation-free lse differs from attn_decode_paged"
        assert_attention_close(out, want_out, lse, want_lse, what="attn_decode_paged_noalloc")


def test_noalloc_rejects_problems_beyond_its_scratch(cuda_device):
    pa, lib = _lib()
    g = workloads.make_paged_case("big", [16] * 2048, [1] * 2048, 8, 8, 128, seed=7, device=cuda_device)
    out = torch.empty_like(g.q)
    lse = torch.empty((g.batch, g.num_q_heads), device=cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    assert _noalloc(lib, g, out, lse, status) == PA_ERR_SCRATCH_LIMIT
    assert "scratch" in lib.pa_status_string(PA_ERR_SCRATCH_LIMIT).decode()
