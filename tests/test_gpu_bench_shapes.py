"""Every workload bench.py times, at the shape, inputs and call it times, against the
float64 oracle element by element.

The inputs come from bench.py's own generator recipe (seed 0; x, gamma, beta as
the workload states; bfloat16 workloads rounded to nearest even on the host, so
the oracle sees the values the GPU reads) and the call from bench.py's own
call builder (same entry point, workspace and arguments), made twice in a row
on the same workspace as the timed steps make it.  Every output element is
compared with the oracle: within 1e-4 (1 + |y_ref|) for fp32, plus the bfloat16
rounding of the result (2^-8 |y_ref|) for bf16.

The two RMSNorm (112, 64, 512, 512) workloads (1.88e9 elements) are generated,
uploaded and compared one batch entry (64 MiB of fp32) at a time, so no host
copy of the whole tensor is needed; every entry is compared.
"""
import pytest
import torch

import bench
import normgen
import oracle
from gpu_util import TOL, assert_bf16_parity, assert_parity, bf16_values

pytestmark = pytest.mark.gpu

BIG_RMS = [n for n, c in bench.CONFIGS.items() if c["op"] == "rms" and c["B"] > 8]
OTHERS = [n for n in sorted(bench.CONFIGS) if n not in BIG_RMS]


@pytest.fixture(scope="module")
def ng():
    import memory_bound_normalization_norm_gb300 as m
    return m


def _workspace(ng, cfg):
    dev = torch.device("cuda")
    if cfg["op"] == "ln":
        nb = ng.norm_layer_workspace_bytes(cfg["rows"], cfg["L"])
    elif cfg["op"] == "gn_nchw":
        nb = ng.norm_group_lrelu_x2_nchw_workspace_bytes(cfg["N"], cfg["C"], cfg["S"], cfg["G"])
    else:
        return None, 0
    return torch.zeros((nb + 3) // 4 + 64, dtype=torch.float32, device=dev), nb


def _oracle(cfg, x, g, b):
    f64 = bool(cfg.get("bf16"))
    op = cfg["op"]
    if op == "linear_gn":  # g = (W, bias), b = (gamma, beta)
        return oracle.linear_group_lrelu_x2(x, g[0], g[1], b[0], b[1], cfg["M"], cfg["K"], cfg["N"], cfg["G"],
                                            1e-5, 0.01)
    if op == "ln":
        return oracle.layer_norm(x, g, b, cfg["rows"], cfg["L"], 1e-5, f64=f64)
    if op == "gn":
        return oracle.group_lrelu_x2(x, g, b, cfg["N"], cfg["C"], cfg["G"], 1e-5, 0.01, f64=f64)
    if op == "gn_nchw":
        return oracle.group_lrelu_x2_nchw(x, g, b, cfg["N"], cfg["C"], cfg["S"], cfg["G"], 1e-5, 0.01, f64=f64)
    return oracle.rms_channel(x, cfg["B"], cfg["C"], cfg["S"], 1e-5, f64=f64)


def _check(cfg, got_dev, want, what):
    if cfg.get("bf16"):
        assert_bf16_parity(bf16_values(got_dev), want, what)
    else:
        assert_parity(got_dev.cpu().numpy(), want, what, TOL)


@pytest.mark.parametrize("name", OTHERS)
def test_bench_workload(ng, name):
    cfg = bench.CONFIGS[name]
    dev = torch.device("cuda")
    x, g, b = bench.host_inputs(cfg)
    if cfg["op"] == "linear_gn":
        xd, gd, bd, yd = bench.linear_gn_device(cfg, x, g, b, dev)
    else:
        xd, gd, bd = (None if a is None else bench.device_tensor(a, cfg, dev) for a in (x, g, b))
        yd = torch.empty_like(xd)
    ws, ws_bytes = _workspace(ng, cfg)
    stream = torch.cuda.current_stream().cuda_stream
    call, _ = bench.make_call(ng, cfg, xd, gd, bd, yd, ws, ws_bytes, stream)
    want = _oracle(cfg, x, g, b)
    for k in range(2):
        yd.fill_(float("nan"))
        call()
        assert ng.norm_last_error() == ng.NORM_OK
        _check(cfg, yd, want, f"{name} call {k + 1}")


@pytest.mark.slow
@pytest.mark.parametrize("name", BIG_RMS)
def test_bench_rms_full_size_every_element(ng, name):
    """(112, 64, 512, 512): every batch entry, element by element, streamed one entry at a time."""
    cfg = bench.CONFIGS[name]
    B, C, S = cfg["B"], cfg["C"], cfg["S"]
    per = C * S
    bf16 = bool(cfg.get("bf16"))
    dt = torch.bfloat16 if bf16 else torch.float32
    xd = torch.empty(B * per, dtype=dt, device="cuda")

    def entry(bi):  # the workload's x restricted to batch entry bi (same stream indices)
        v = normgen.normal(per, cfg["x"][0], cfg["x"][1], seed=0, tensor_id=normgen.TENSOR_X, start=bi * per)
        return normgen.round_bf16(v) if bf16 else v

    for bi in range(B):
        xd[bi * per:(bi + 1) * per].copy_(bench.device_tensor(entry(bi), cfg, torch.device("cpu")))
    yd = torch.empty_like(xd)
    call, _ = bench.make_call(ng, cfg, xd, None, None, yd, None, 0, torch.cuda.current_stream().cuda_stream)
    call()
    assert ng.norm_last_error() == ng.NORM_OK
    del xd
    for bi in range(B):
        want = oracle.rms_channel(entry(bi), 1, C, S, 1e-5, f64=bf16)
        _check(cfg, yd[bi * per:(bi + 1) * per], want, f"{name} batch entry {bi}")
