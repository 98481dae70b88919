"""Overlapped launches on the decode path.

The activation quantiser and the decode-size GEMM are launched with
programmatic stream serialisation: each may start while the kernel ahead of it
on the stream is still running, and waits for that kernel before it reads an
activation or writes anything (the decode GEMM fetches its first weight tiles
before the wait).  A chain of dependent steps, each reading what the one
before wrote, must give what the oracle gives on the chain's own intermediate
values, bit for bit where the oracle is exact, and exactly what the same calls
give with the overlap switched off (test hook 13) and from a CUDA graph.
Buffers start filled with a pattern no step would write, so a read that ran
ahead of its producer shows up as a wrong value."""
import numpy as np
import pytest
import torch

import fp8_w8a8_rollout_gb300 as fp8rl
import oracle
from fp8_w8a8_rollout_gb300 import synth

pytestmark = pytest.mark.gpu

RTOL, ATOL_RMS = 1e-2, 1e-3
# a decode step's projections, each one's output the next one's input
CHAIN = [(4096, 4096), (12288, 4096), (4096, 12288), (6144, 4096), (4096, 6144)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fp8rl.load_library(build_if_missing=True)
    yield
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_RESET, 0)


@pytest.fixture
def pdl_off():
    yield lambda off: fp8rl.fp8rl_debug_set(fp8rl.DEBUG_PDL, 1 if off else 0)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_PDL, 0)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_DECODE, 0)


def within(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    bad = int(np.count_nonzero(np.abs(got - ref) > RTOL * np.abs(ref) + ATOL_RMS * rms))
    assert bad == 0, f"{bad}/{ref.size} outside tolerance"


@pytest.fixture(scope="module", params=[fp8rl.SCALE_FP32, fp8rl.SCALE_UE8M0], ids=["fp32", "ue8m0"])
def weights(request):
    """Oracle-quantised weights of the chain, uploaded once per format."""
    fmt = request.param
    out = []
    for i, (n, k) in enumerate(CHAIN):
        wq, sw = oracle.quant_weight_blockwise(synth.bf16_bits(synth.weight_bf16(n, k, 40 + i, "pdl-w")), fmt)
        out.append((n, k, wq, sw, torch.from_numpy(wq).cuda(), torch.from_numpy(np.ascontiguousarray(sw)).cuda()))
    return fmt, out


def make_buffers(m, fmt, layers):
    sdt = torch.float32 if fmt == fp8rl.SCALE_FP32 else torch.uint8
    bufs = []
    for n, k, *_ in layers:
        bufs.append((torch.empty((m, k), dtype=torch.uint8, device="cuda"),
                     torch.empty((k // 128, m), dtype=sdt, device="cuda"),
                     torch.empty((m, n), dtype=torch.bfloat16, device="cuda")))
    return bufs


def poison(bufs):
    for q, s, y in bufs:
        q.fill_(0x7E)          # +448: never the code of these activations' maxima
        s.fill_(3) if s.dtype == torch.uint8 else s.fill_(-1.0)
        y.fill_(float("nan"))


def run_chain(x0, fmt, layers, bufs):
    """Every call on the current stream (the capturing one inside a graph)."""
    m = x0.shape[0]
    x = x0
    for (n, k, _, _, dwq, dsw), (q, s, y) in zip(layers, bufs):
        fp8rl.fp8rl_quant_act_group(x, m, k, k, q, k, s, fmt)
        fp8rl.fp8rl_gemm_blockscaled(q, s, dwq, dsw, y, m, n, k, fmt)
        x = y


def host(bufs):
    return [(q.cpu().numpy(), s.cpu().numpy(), y.view(torch.int16).cpu().numpy()) for q, s, y in bufs]


@pytest.mark.parametrize("m", [16, 1, 7, 40, 128])
def test_chain_matches_oracle_on_its_own_intermediates(m, weights, pdl_off):
    fmt, layers = weights
    pdl_off(False)
    if m > 32:  # the decode kernel's 64- and 128-column forms (test hook)
        fp8rl.fp8rl_debug_set(fp8rl.DEBUG_DECODE, 1)
    x0 = synth.activation_bf16(m, CHAIN[0][1], 50 + m, "pdl-x", device="cuda")
    bufs = make_buffers(m, fmt, layers)
    poison(bufs)
    run_chain(x0, fmt, layers, bufs)
    assert fp8rl.fp8rl_sync_status() == 0
    got = host(bufs)
    x_bits = synth.bf16_bits(x0.cpu())
    for (n, k, wq, sw, _, _), (q, s, ybits) in zip(layers, got):
        rq, rs = oracle.quant_act_group(x_bits, fmt)
        assert np.array_equal(q, rq), "codes differ from the oracle's on the step's own input"
        assert np.array_equal(s.view(np.uint8), np.ascontiguousarray(rs).view(np.uint8)), "scales differ"
        y = ybits.astype(np.uint16).astype(np.uint32) << 16
        within(y.view(np.float32), oracle.gemm_blockscaled(q, s, wq, sw, fmt))
        x_bits = ybits.astype(np.uint16)


def test_chain_is_identical_with_overlap_off_and_from_a_graph(weights, pdl_off):
    fmt, layers = weights
    m = 16
    x0 = synth.activation_bf16(m, CHAIN[0][1], 77, "pdl-x2", device="cuda")
    results = []
    for off in (False, True):
        pdl_off(off)
        bufs = make_buffers(m, fmt, layers)
        poison(bufs)
        run_chain(x0, fmt, layers, bufs)
        assert fp8rl.fp8rl_sync_status() == 0
        results.append(host(bufs))
    pdl_off(False)
    bufs = make_buffers(m, fmt, layers)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run_chain(x0, fmt, layers, bufs)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run_chain(x0, fmt, layers, bufs)
    for _ in range(3):
        poison(bufs)
        g.replay()
        torch.cuda.synchronize()
        results.append(host(bufs))
    assert fp8rl.fp8rl_sync_status() == 0
    for other in results[1:]:
        for a, b in zip(results[0], other):
            for u, v in zip(a, b):
                assert np.array_equal(u, v)


def test_weight_sync_right_before_a_decode_gemm(pdl_off):
    """The weight quantiser does not let its successor start early, so a
    decode GEMM enqueued right behind it (overlapped launch on) reads the new
    weights, never the ones the buffer held before."""
    pdl_off(False)
    fmt = fp8rl.SCALE_FP32
    m, n, k = 16, 6144, 4096
    x = synth.activation_bf16(m, k, 5, "pdl-sync-x")
    xq, sx = oracle.quant_act_group(synth.bf16_bits(x), fmt)
    dxq, dsx = torch.from_numpy(xq).cuda(), torch.from_numpy(np.ascontiguousarray(sx)).cuda()
    wq = torch.empty((n, k), dtype=torch.uint8, device="cuda")
    sw = torch.empty((n // 128, k // 128), dtype=torch.float32, device="cuda")
    y = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    for i in range(3):
        w = synth.weight_bf16(n, k, 60 + i, "pdl-sync-w")
        dw = w.cuda()
        torch.cuda.synchronize()
        wq.fill_(0x7E)
        sw.fill_(1.0e6)
        fp8rl.fp8rl_quant_weight_blockwise(dw, n, k, k, wq, k, sw, fmt)
        fp8rl.fp8rl_gemm_blockscaled(dxq, dsx, wq, sw, y, m, n, k, fmt)
        assert fp8rl.fp8rl_sync_status() == 0
        rwq, rsw = oracle.quant_weight_blockwise(synth.bf16_bits(w), fmt)
        within(y.float().cpu().numpy(), oracle.gemm_blockscaled(xq, sx, rwq, rsw, fmt))
