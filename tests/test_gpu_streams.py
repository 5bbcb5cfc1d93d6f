"""Concurrent calls on several streams, and capture into a CUDA graph, against the oracle.

The library's calls are stream-ordered and allocate nothing when given a workspace, so
they may run at the same time on different streams (each with its own workspace) and be
captured into CUDA graphs.  Covered: two persistent LayerNorm launches (cooperative, every
SM) on two streams at once beside the cluster kernels of GroupNorm and LayerNorm, the
row kernel, the (N, C) GroupNorm (vector and team-per-group kernels) and RMSNorm; a graph
replaying every non-cooperative path several times; and a graph replaying the cooperative
persistent kernel (LayerNorm fp32 and bf16, the NCHW GroupNorm form) on caller workspaces.
"""
import numpy as np
import pytest
import torch

import normgen
import oracle
from gpu_util import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ng():
    import memory_bound_normalization_norm_gb300 as m
    return m


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def ln_case(rows, L, seed):
    x = normgen.normal(rows * L, seed=seed, tensor_id=0)
    g = normgen.normal(L, 1.0, 0.1, seed=seed, tensor_id=1)
    b = normgen.normal(L, 0.0, 0.1, seed=seed, tensor_id=2)
    return x, g, b, oracle.layer_norm(x, g, b, rows, L)


def gn_case(N, C, S, G, seed):
    x = normgen.normal(N * C * S, seed=seed, tensor_id=0)
    g = normgen.normal(C, 1.0, 0.1, seed=seed, tensor_id=1)
    b = normgen.normal(C, 0.0, 0.1, seed=seed, tensor_id=2)
    return x, g, b, oracle.group_lrelu_x2_nchw(x, g, b, N, C, S, G)


def test_concurrent_streams(ng):
    jobs = []
    # two persistent LayerNorms, each with its own workspace
    for seed in (1, 2):
        rows, L = 3, 1 << 20
        x, g, b, want = ln_case(rows, L, seed)
        nb = ng.norm_layer_workspace_bytes(rows, L)
        ws = torch.zeros(nb // 4 + 64, device="cuda")
        xd, gd, bd = dev(x), dev(g), dev(b)
        yd = torch.empty_like(xd)
        jobs.append((lambda xd=xd, gd=gd, bd=bd, yd=yd, ws=ws, nb=nb, rows=rows, L=L, s=None:
                     ng.norm_layer_fwd(xd, gd, bd, yd, rows, L, 1e-5, ws, nb, s), yd, want, f"LN persistent {seed}"))
    # LayerNorm rows on the cluster kernel and on the row kernel
    for rows, L, seed in ((40, 65536, 3), (500, 4096, 4)):
        x, g, b, want = ln_case(rows, L, seed)
        xd, gd, bd = dev(x), dev(g), dev(b)
        yd = torch.empty_like(xd)
        jobs.append((lambda xd=xd, gd=gd, bd=bd, yd=yd, rows=rows, L=L, s=None:
                     ng.norm_layer_fwd(xd, gd, bd, yd, rows, L, 1e-5, stream=s), yd, want, f"LN {rows}x{L}"))
    # GroupNorm over NCHW (cluster kernel) and (N, C)
    x, g, b, want = gn_case(4, 256, 4096, 16, 5)
    xd, gd, bd = dev(x), dev(g), dev(b)
    yd = torch.empty_like(xd)
    jobs.append((lambda xd=xd, gd=gd, bd=bd, yd=yd, s=None:
                 ng.norm_group_lrelu_x2_nchw_fwd(xd, gd, bd, yd, 4, 256, 4096, 16, 1e-5, 0.01, stream=s),
                 yd, want, "GN NCHW"))
    x2 = normgen.normal(512 * 8192, seed=6, tensor_id=0)
    g2 = normgen.normal(8192, 1.0, 0.1, seed=6, tensor_id=1)
    b2 = normgen.normal(8192, 0.0, 0.1, seed=6, tensor_id=2)
    xd2, gd2, bd2 = dev(x2), dev(g2), dev(b2)
    yd2 = torch.empty_like(xd2)
    jobs.append((lambda s=None: ng.norm_group_lrelu_x2_fwd(xd2, gd2, bd2, yd2, 512, 8192, 512, 1e-5, 0.01, stream=s),
                 yd2, oracle.group_lrelu_x2(x2, g2, b2, 512, 8192, 512), "GN (N, C)"))
    # GroupNorm with groups of 48 channels: the team-per-group kernel
    x5 = normgen.normal(1000 * 1536, seed=8, tensor_id=0)
    g5 = normgen.normal(1536, 1.0, 0.1, seed=8, tensor_id=1)
    b5 = normgen.normal(1536, 0.0, 0.1, seed=8, tensor_id=2)
    xd5, gd5, bd5 = dev(x5), dev(g5), dev(b5)
    yd5 = torch.empty_like(xd5)
    jobs.append((lambda s=None: ng.norm_group_lrelu_x2_fwd(xd5, gd5, bd5, yd5, 1000, 1536, 32, 1e-5, 0.01, stream=s),
                 yd5, oracle.group_lrelu_x2(x5, g5, b5, 1000, 1536, 32), "GN groups of 48"))
    # RMSNorm
    x3 = normgen.normal(4 * 64 * 65536, seed=7, tensor_id=0)
    xd3 = dev(x3)
    yd3 = torch.empty_like(xd3)
    jobs.append((lambda s=None: ng.norm_rms_channel_fwd(xd3, yd3, 4, 64, 65536, 1e-5, stream=s), yd3,
                 oracle.rms_channel(x3, 4, 64, 65536), "RMS"))

    streams = [torch.cuda.Stream() for _ in jobs]
    torch.cuda.synchronize()
    for _ in range(3):
        for (call, y, _, _), st in zip(jobs, streams):
            y.fill_(float("nan"))
        torch.cuda.synchronize()
        for (call, _, _, _), st in zip(jobs, streams):
            call(s=st.cuda_stream)
        torch.cuda.synchronize()
        assert ng.norm_last_error() == 0
        for call, y, want, what in jobs:
            assert_parity(y.cpu().numpy(), want, f"{what} on its own stream")


def test_graph_capture_and_replay(ng):
    rows, L = 64, 65536
    x1, g1, b1, w1 = ln_case(rows, L, 11)
    rows2, L2 = 1000, 2048
    x2, g2, b2, w2 = ln_case(rows2, L2, 12)
    x3, g3, b3, w3 = gn_case(2, 128, 4096, 8, 13)
    x4 = normgen.normal(2 * 64 * 1024, seed=14, tensor_id=0)
    w4 = oracle.rms_channel(x4, 2, 64, 1024)
    x5 = normgen.normal(300 * 960, seed=15, tensor_id=0)
    g5 = normgen.normal(960, 1.0, 0.1, seed=15, tensor_id=1)
    b5 = normgen.normal(960, 0.0, 0.1, seed=15, tensor_id=2)
    w5 = oracle.group_lrelu_x2(x5, g5, b5, 300, 960, 32)
    d1 = [dev(a) for a in (x1, g1, b1)]
    d2 = [dev(a) for a in (x2, g2, b2)]
    d3 = [dev(a) for a in (x3, g3, b3)]
    d4 = dev(x4)
    d5 = [dev(a) for a in (x5, g5, b5)]
    y1, y2, y3, y4, y5 = (torch.empty_like(t) for t in (d1[0], d2[0], d3[0], d4, d5[0]))
    s = torch.cuda.Stream()

    def step():
        ng.norm_layer_fwd(d1[0], d1[1], d1[2], y1, rows, L, 1e-5, stream=s.cuda_stream)
        ng.norm_layer_fwd(d2[0], d2[1], d2[2], y2, rows2, L2, 1e-5, stream=s.cuda_stream)
        ng.norm_group_lrelu_x2_nchw_fwd(d3[0], d3[1], d3[2], y3, 2, 128, 4096, 8, 1e-5, 0.01, stream=s.cuda_stream)
        ng.norm_rms_channel_fwd(d4, y4, 2, 64, 1024, 1e-5, stream=s.cuda_stream)
        # groups of 30 channels: the team kernel's 2-element form
        ng.norm_group_lrelu_x2_fwd(d5[0], d5[1], d5[2], y5, 300, 960, 32, 1e-5, 0.01, stream=s.cuda_stream)

    with torch.cuda.stream(s):
        step()  # first calls outside the capture: per-device setup happens here
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    for y in (y1, y2, y3, y4, y5):
        y.fill_(float("nan"))
    torch.cuda.synchronize()
    for _ in range(5):
        graph.replay()
    torch.cuda.synchronize()
    assert ng.norm_last_error() == 0
    for y, want, what in ((y1, w1, "LN cluster kernel"), (y2, w2, "LN row kernel"), (y3, w3, "GN NCHW"),
                          (y4, w4, "RMS"), (y5, w5, "GN team kernel")):
        assert_parity(y.cpu().numpy(), want, f"{what} replayed from a graph")


def test_graph_capture_of_persistent_kernels(ng):
    """The cooperative persistent kernel captured into a graph and replayed: LayerNorm fp32 and
    bf16 and the NCHW GroupNorm form, each on a caller workspace (the kernel advances the
    workspace's row base itself, so replays need no host step), plus bf16 RMSNorm pairs."""
    rows, L = 3, 1 << 20
    x1, g1, b1, w1 = ln_case(rows, L, 21)
    nb1 = ng.norm_layer_workspace_bytes(rows, L)
    ws1 = torch.zeros(nb1 // 4 + 64, device="cuda")
    N, C, S, G = 2, 8, 36000, 2
    x2, g2, b2, w2 = gn_case(N, C, S, G, 22)
    nb2 = ng.norm_group_lrelu_x2_nchw_workspace_bytes(N, C, S, G)
    ws2 = torch.zeros(nb2 // 4 + 64, device="cuda")
    rows3, L3 = 2, 262144
    x3 = normgen.round_bf16(normgen.normal(rows3 * L3, seed=23, tensor_id=0))
    g3 = normgen.round_bf16(normgen.normal(L3, 1.0, 0.1, seed=23, tensor_id=1))
    b3 = normgen.round_bf16(normgen.normal(L3, 0.0, 0.1, seed=23, tensor_id=2))
    w3 = oracle.layer_norm(x3, g3, b3, rows3, L3, f64=True)
    nb3 = ng.norm_layer_workspace_bytes(rows3, L3)
    ws3 = torch.zeros(nb3 // 4 + 64, device="cuda")
    x4 = normgen.round_bf16(normgen.normal(2 * 64 * 1024, seed=24, tensor_id=0))
    w4 = oracle.rms_channel(x4, 2, 64, 1024, f64=True)
    d1 = [dev(a) for a in (x1, g1, b1)]
    d2 = [dev(a) for a in (x2, g2, b2)]
    d3 = [dev(a).to(torch.bfloat16) for a in (x3, g3, b3)]
    d4 = dev(x4).to(torch.bfloat16)
    y1, y2, y3, y4 = (torch.empty_like(t) for t in (d1[0], d2[0], d3[0], d4))
    s = torch.cuda.Stream()
    ng.norm_set_option(ng.NORM_OPT_GN_PATH, 6)
    try:
        def step():
            ng.norm_layer_fwd(d1[0], d1[1], d1[2], y1, rows, L, 1e-5, ws1, nb1, stream=s.cuda_stream)
            ng.norm_group_lrelu_x2_nchw_fwd(d2[0], d2[1], d2[2], y2, N, C, S, G, 1e-5, 0.01, ws2, nb2,
                                            stream=s.cuda_stream)
            ng.norm_layer_fwd_bf16(d3[0], d3[1], d3[2], y3, rows3, L3, 1e-5, ws3, nb3, stream=s.cuda_stream)
            ng.norm_rms_channel_fwd_bf16(d4, y4, 2, 64, 1024, 1e-5, stream=s.cuda_stream)

        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            step()  # first calls outside the capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            step()
    finally:
        ng.norm_set_option(ng.NORM_OPT_GN_PATH, 0)
    for y in (y1, y2, y3, y4):
        y.fill_(float("nan"))
    torch.cuda.synchronize()
    for _ in range(5):
        graph.replay()
    torch.cuda.synchronize()
    assert ng.norm_last_error() == 0
    from gpu_util import assert_bf16_parity
    assert_parity(y1.cpu().numpy(), w1, "persistent LN replayed from a graph")
    assert_parity(y2.cpu().numpy(), w2, "persistent GN NCHW replayed from a graph")
    assert_bf16_parity(y3.float().cpu().numpy(), w3, "persistent LN bf16 replayed from a graph")
    assert_bf16_parity(y4.float().cpu().numpy(), w4, "RMS bf16 pairs replayed from a graph")
