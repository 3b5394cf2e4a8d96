"""CUDA-graph capture of the C-ABI calls: a launch captured on a stream that
has already run the op (so its stream-K workspace exists) replays to the same
bits as the eager launch, and the masked variant replays correctly too.  The
per-stream workspaces (stream-K scratch, scale images of row-major activation
scales) are not allocated during a capture, and one that a later, larger call
on the stream grows keeps the buffer an earlier capture points at.  A call on
another stream may allocate its workspaces while a graph is being captured in
torch's default (global) capture mode without breaking that capture."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_gb300 as fb
import synth

from _parity import SENTINEL, all_rows, compare

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bits(d):
    return d.view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1, d.shape[-1])


def test_contiguous_graph_replay_matches_eager(gg):
    # 80 units on 76 pairs: the stream-K tail is part of the captured launch
    p = synth.make_problem("contiguous", 2, 2560, 512, [1024, 1000], seed=701, device=DEV)
    s = torch.cuda.Stream()
    d_eager = torch.zeros((p.rows, p.N), dtype=torch.bfloat16, device=DEV)
    d_graph = torch.zeros_like(d_eager)
    with torch.cuda.stream(s):
        fb.gemm_grouped_contiguous(p.a, p.sa_mk_view(), p.b, p.sb, d_eager, p.grouped_layout)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fb.gemm_grouped_contiguous(p.a, p.sa_mk_view(), p.b, p.sb, d_graph, p.grouped_layout)
    for _ in range(3):
        d_graph.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(_bits(d_graph), _bits(d_eager))
    assert fb.device_error() == 0
    valid, untouched = all_rows(p)
    compare(p, _bits(d_eager), valid, [])


def test_masked_graph_replay(gg):
    p = synth.make_problem("masked", 3, 512, 512, [0, 77, 256], seed=702, M_max=256, device=DEV)
    d = torch.full((p.G, p.M_max, p.N), 0x7FA5, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fb.gemm_grouped_masked(p.a, p.sa_mk_view(), p.b, p.sb, d, p.masked_m)
    s.synchronize()
    with torch.cuda.graph(g, stream=s):
        fb.gemm_grouped_masked(p.a, p.sa_mk_view(), p.b, p.sb, d, p.masked_m)
    d.view(torch.int16).fill_(0x7FA5)
    g.replay()
    torch.cuda.synchronize()
    assert fb.device_error() == 0
    valid, untouched = all_rows(p)
    compare(p, _bits(d), valid, untouched)


def test_capture_on_a_fresh_stream_matches_eager(gg):
    """Nothing allocated on the stream yet (the first stream of torch's
    high-priority pool, which no other test uses): the captured call runs without
    the stream-K split and without scale images.  The split changes the order of
    the fp32 sums, so the replay is held to the oracle, not to the eager bits."""
    p = synth.make_problem("contiguous", 2, 2560, 512, [1024, 1000], seed=703, device=DEV)
    d_graph = torch.full((p.rows, p.N), SENTINEL, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    s = torch.cuda.Stream(priority=-1)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fb.gemm_grouped_contiguous(p.a, p.sa_mk_view(), p.b, p.sb, d_graph, p.grouped_layout)
    g.replay()
    torch.cuda.synchronize()
    assert fb.device_error() == 0
    valid, untouched = all_rows(p)
    compare(p, _bits(d_graph), valid, untouched)


def test_graph_replays_after_the_workspace_grew(gg):
    small = synth.make_problem("contiguous", 2, 512, 512, [200, 150], seed=704, device=DEV)
    large = synth.make_problem("contiguous", 4, 1024, 2048, [1024, 900, 700, 1024], seed=705,
                               device=DEV)
    s = torch.cuda.Stream(priority=-1)  # a stream no earlier call made large workspaces for
    d_small = torch.zeros((small.rows, small.N), dtype=torch.bfloat16, device=DEV)
    d_graph = torch.zeros_like(d_small)
    d_large = torch.full((large.rows, large.N), SENTINEL, dtype=torch.int16,
                         device=DEV).view(torch.bfloat16)
    with torch.cuda.stream(s):
        fb.gemm_grouped_contiguous(small.a, small.sa_mk_view(), small.b, small.sb, d_small,
                                   small.grouped_layout)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fb.gemm_grouped_contiguous(small.a, small.sa_mk_view(), small.b, small.sb, d_graph,
                                   small.grouped_layout)
    with torch.cuda.stream(s):  # needs larger scale images: the workspace grows
        fb.gemm_grouped_contiguous(large.a, large.sa_mk_view(), large.b, large.sb, d_large,
                                   large.grouped_layout)
    s.synchronize()
    for _ in range(2):
        d_graph.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(_bits(d_graph), _bits(d_small))
    assert fb.device_error() == 0
    valid, untouched = all_rows(large)
    compare(large, _bits(d_large), valid, untouched)


def test_first_call_on_a_stream_while_another_stream_captures(gg):
    p = synth.make_problem("contiguous", 2, 512, 512, [200, 150], seed=706, device=DEV)

    def sentinel():
        return torch.full((p.rows, p.N), SENTINEL, dtype=torch.int16, device=DEV).view(torch.bfloat16)

    def call(d, stream=None):
        fb.gemm_grouped_contiguous(p.a, p.sa_mk_view(), p.b, p.sb, d, p.grouped_layout, stream=stream)

    d_ref, d_graph, d_other = sentinel(), sentinel(), sentinel()
    call(d_ref)  # 4 units: no stream-K split, so every stream gives the same bits
    torch.cuda.synchronize()
    s_cap = torch.cuda.Stream(priority=-1)
    s_new = torch.cuda.Stream(priority=-1)  # no call has run on it yet
    with torch.cuda.stream(s_cap):
        call(d_graph)  # the capturing stream's workspaces exist before the capture
    s_cap.synchronize()
    d_graph.view(torch.int16).fill_(SENTINEL)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s_cap):  # capture_error_mode="global"
        call(d_graph)
        call(d_other, stream=s_new)  # eager, allocates s_new's workspaces
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert fb.device_error() == 0
    assert np.array_equal(_bits(d_graph), _bits(d_ref))
    assert np.array_equal(_bits(d_other), _bits(d_ref))
