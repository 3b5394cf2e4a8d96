"""CUDA-graph capture of the C-ABI calls: a launch captured on a stream that
has already run the op (so its stream-K workspace exists) replays to the same
bits as the eager launch, and the masked variant replays correctly too."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_gb300 as fb
import synth

from _parity import all_rows, compare

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
