"""The calls that take their scratch space as a workspace argument can be
captured in a CUDA graph: they neither synchronise with the host nor
allocate.  A captured decode step (the newest K/V rows written back by the
same kernel) and a captured mixed prefill + decode call, on both prefill
paths, replay to the same bits as the eager calls, and a replay after the
inputs change in place follows the new inputs."""

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


def _pa():
    return pytest.importorskip("paged_kv_decode_17_gb300")


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def _capture(fn):
    """Run fn once eagerly on a side stream (the library's one-time set-up), then
    capture it in a graph."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def test_decode_append_step_replays_in_a_graph(cuda_device):
    pa = _pa()
    case = workloads.make_paged_case("graph_decode", [700, 33, 1500, 4096], [1] * 4, 8, 2, 128, seed=131,
                                     device=cuda_device)
    B, Hq, D = case.q.shape
    Hkv = case.num_kv_heads
    gen = torch.Generator(device="cpu").manual_seed(132)
    k_new = torch.randn(B, Hkv, D, generator=gen).to(torch.bfloat16).to(cuda_device)
    v_new = torch.randn(B, Hkv, D, generator=gen).to(torch.bfloat16).to(cuda_device)
    ws = pa.Workspace(pa.decode_workspace_bytes(B, Hq, Hkv, D), cuda_device)
    out = torch.empty_like(case.q)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=cuda_device)
    status = pa.new_status(cuda_device)

    def step():
        pa.attn_decode_paged(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, case.softmax_scale,
                             max_seq_len=case.max_seq_len, out=out, lse=lse, workspace=ws, status=status,
                             k_new=k_new, v_new=v_new)

    g = _capture(step)
    want, want_lse = out.clone(), lse.clone()
    out.fill_(float("nan"))
    lse.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    pa.check_status(status, "captured decode step")
    assert torch.equal(_bits(out), _bits(want)) and torch.equal(_bits(lse), _bits(want_lse))

    # new query rows, written in place: the replay reads them
    case.q.copy_(torch.randn(case.q.shape, generator=gen).to(torch.bfloat16))
    g.replay()
    torch.cuda.synchronize()
    got, got_lse = out.clone(), lse.clone()
    assert not torch.equal(_bits(got), _bits(want))
    step()
    torch.cuda.synchronize()
    assert torch.equal(_bits(got), _bits(out)) and torch.equal(_bits(got_lse), _bits(lse))


@pytest.mark.parametrize("path", ["fused", "separate"])
def test_mixed_prefill_call_replays_in_a_graph(cuda_device, monkeypatch, path):
    pa = _pa()
    monkeypatch.setenv("PAGEDATTN_PREFILL_PATH", path)
    # prefill chunks next to one-row decode entries, with cached tokens before the chunks
    case = workloads.make_paged_case("graph_mixed", [900, 1, 77, 3000, 256], [256, 1, 1, 1, 256], 32, 8, 128,
                                     seed=133, device=cuda_device)
    B = case.batch
    ws = pa.Workspace(pa.prefill_workspace_bytes(B, case.total_q, case.num_q_heads, case.num_kv_heads,
                                                 case.head_dim), cuda_device)
    out = torch.empty_like(case.q)
    lse = torch.empty(case.total_q, case.num_q_heads, dtype=torch.float32, device=cuda_device)
    status = pa.new_status(cuda_device)

    def call():
        pa.attn_prefill_varlen_causal(case.q, case.k_pool, case.v_pool, case.block_table, case.cu_seqlens_q,
                                      case.seq_lens, case.softmax_scale, max_q_len=case.max_q_len,
                                      max_seq_len=case.max_seq_len, out=out, lse=lse, workspace=ws,
                                      status=status)

    g = _capture(call)
    want, want_lse = out.clone(), lse.clone()
    for _ in range(3):  # replays back to back reuse the workspace's plan area
        out.fill_(float("nan"))
        g.replay()
    torch.cuda.synchronize()
    pa.check_status(status, "captured prefill call")
    assert torch.equal(_bits(out), _bits(want)) and torch.equal(_bits(lse), _bits(want_lse))

    gen = torch.Generator(device="cpu").manual_seed(134)
    case.q.copy_(torch.randn(case.q.shape, generator=gen).to(torch.bfloat16))
    g.replay()
    torch.cuda.synchronize()
    got = out.clone()
    call()
    torch.cuda.synchronize()
    assert torch.equal(_bits(got), _bits(out))
