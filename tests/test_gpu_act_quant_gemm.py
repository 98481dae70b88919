"""fp8rl_gemm_act_quant: the 1x128 activation quantisation and the
block-scaled GEMM in one call, one kernel at up to 16 rows (the decode GEMM
quantises each 128-wide chunk of X as it streams the weights).

Its codes and scales must be bit for bit those of fp8rl_quant_act_group on the
same X (and so the oracle's), and Y bit for bit that of fp8rl_gemm_blockscaled
on those codes, hence within R11 of the oracle.  Shapes above the fused range,
and X rows the fused kernel cannot fetch (a row stride that is not a multiple
of 8 elements), take the two-kernel path and must agree the same way."""
import numpy as np
import pytest
import torch

import fp8_w8a8_rollout_gb300 as fp8rl
import oracle
from fp8_w8a8_rollout_gb300 import synth

pytestmark = pytest.mark.gpu

FMTS = [fp8rl.SCALE_FP32, fp8rl.SCALE_UE8M0]
RTOL, ATOL_RMS = 1e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fp8rl.load_library(build_if_missing=True)
    yield
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_RESET, 0)


@pytest.fixture
def hooks():
    yield
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_RESET, 0)


def within(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    bad = int(np.count_nonzero(np.abs(got - ref) > RTOL * np.abs(ref) + ATOL_RMS * rms))
    assert bad == 0, f"{bad}/{ref.size} outside tolerance"


def weights(n, k, fmt, seed):
    wq, sw = oracle.quant_weight_blockwise(synth.bf16_bits(synth.weight_bf16(n, k, seed, "aqg-w")), fmt)
    return wq, sw, torch.from_numpy(wq).cuda(), torch.from_numpy(np.ascontiguousarray(sw)).cuda()


def bits(t):
    return t.contiguous().view(torch.uint8).cpu().numpy()


def check(x, wq, sw, dwq, dsw, fmt):
    """One fused call against the two calls and the oracle."""
    y, xq, sx = fp8rl.gemm_act_quant(x, dwq, dsw, fmt)
    assert fp8rl.fp8rl_sync_status() == 0
    xq2, sx2 = fp8rl.quant_act(x.contiguous(), fmt)
    y2 = fp8rl.gemm(xq2, sx2, dwq, dsw, fmt)
    assert fp8rl.fp8rl_sync_status() == 0
    assert np.array_equal(bits(xq), bits(xq2)), "codes differ from fp8rl_quant_act_group's"
    assert np.array_equal(bits(sx), bits(sx2)), "scales differ from fp8rl_quant_act_group's"
    assert np.array_equal(bits(y), bits(y2)), "Y differs from fp8rl_gemm_blockscaled's on the same codes"
    rxq, rsx = oracle.quant_act_group(synth.bf16_bits(x.cpu()), fmt)
    assert np.array_equal(xq.cpu().numpy(), rxq)
    assert np.array_equal(bits(sx), np.ascontiguousarray(rsx).view(np.uint8).reshape(bits(sx).shape))
    within(y.float().cpu().numpy(), oracle.gemm_blockscaled(rxq, rsx, wq, sw, fmt))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m,n,k", [(1, 128, 128), (7, 256, 640), (16, 6144, 4096), (16, 4096, 12288),
                                   (20, 384, 1280), (32, 4096, 4096), (32, 24576, 4096),
                                   (33, 256, 512), (100, 512, 384)])
def test_matches_two_calls_and_oracle(m, n, k, fmt):
    wq, sw, dwq, dsw = weights(n, k, fmt, n + k)
    x = synth.activation_bf16(m, k, m + 1, "aqg-x", n, device="cuda")
    check(x, wq, sw, dwq, dsw, fmt)


@pytest.mark.parametrize("splits", [2, 3, 8])
def test_forced_splits(splits, hooks):
    fmt = fp8rl.SCALE_FP32
    m, n, k = 16, 384, 2048
    wq, sw, dwq, dsw = weights(n, k, fmt, 7)
    x = synth.activation_bf16(m, k, 8, "aqg-xs", device="cuda")
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_SPLITS, splits)
    check(x, wq, sw, dwq, dsw, fmt)


@pytest.mark.parametrize("pad", [64, 3])
def test_strided_activations(pad):
    """X as a column slice of a wider tensor: a row stride that is a multiple
    of 8 elements stays fused, one that is not takes the two-kernel path."""
    fmt = fp8rl.SCALE_FP32
    m, n, k = 16, 512, 1024
    wq, sw, dwq, dsw = weights(n, k, fmt, 9)
    wide = synth.activation_bf16(m, k + pad, 10, "aqg-xw", device="cuda")
    x = wide[:, :k]
    assert x.stride(0) == k + pad
    check(x, wq, sw, dwq, dsw, fmt)


def test_chain_from_poisoned_buffers():
    """Five projections, each fused call reading the bf16 output of the one
    before (overlapped launches): codes bit-exact against the oracle on the
    chain's own intermediate values, outputs within R11."""
    fmt = fp8rl.SCALE_FP32
    chain = [(4096, 4096), (12288, 4096), (4096, 12288), (6144, 4096), (4096, 6144)]
    ws = [weights(n, k, fmt, 30 + i) for i, (n, k) in enumerate(chain)]
    m = 16
    x0 = synth.activation_bf16(m, chain[0][1], 11, "aqg-chain", device="cuda")
    ys, xqs, sxs = [], [], []
    for n, k in chain:
        ys.append(torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda"))
        xqs.append(torch.full((m, k), 0x7E, dtype=torch.uint8, device="cuda"))
        sxs.append(torch.full((k // 128, m), -1.0, dtype=torch.float32, device="cuda"))
    x = x0
    for (n, k), (_, _, dwq, dsw), y, xq, sx in zip(chain, ws, ys, xqs, sxs):
        fp8rl.fp8rl_gemm_act_quant(x, x.stride(0), dwq, dsw, y, m, n, k, fmt, xq, sx)
        x = y
    assert fp8rl.fp8rl_sync_status() == 0
    xb = synth.bf16_bits(x0.cpu())
    for (n, k), (wq, sw, _, _), y, xq, sx in zip(chain, ws, ys, xqs, sxs):
        rxq, rsx = oracle.quant_act_group(xb, fmt)
        assert np.array_equal(xq.cpu().numpy(), rxq)
        assert np.array_equal(sx.cpu().numpy(), rsx)
        within(y.float().cpu().numpy(), oracle.gemm_blockscaled(rxq, rsx, wq, sw, fmt))
        xb = synth.bf16_bits(y.cpu())


def test_n_zero_quantises_only():
    m, k = 8, 256
    x = synth.activation_bf16(m, k, 12, "aqg-n0", device="cuda")
    xq = torch.empty((m, k), dtype=torch.uint8, device="cuda")
    sx = torch.empty((k // 128, m), dtype=torch.float32, device="cuda")
    fp8rl.fp8rl_gemm_act_quant(x, k, None, None, None, m, 0, k, fp8rl.SCALE_FP32, xq, sx)
    assert fp8rl.fp8rl_sync_status() == 0
    rxq, rsx = oracle.quant_act_group(synth.bf16_bits(x.cpu()), fp8rl.SCALE_FP32)
    assert np.array_equal(xq.cpu().numpy(), rxq)
    assert np.array_equal(sx.cpu().numpy(), rsx)


@pytest.mark.parametrize("skip", [0, 5])
def test_wait_runs_out_and_is_reported(skip, hooks):
    """A chunk that never arrives (the producer skips it): the quantiser and
    MMA waits run out, TIMEOUT is reported, the next call is correct."""
    fmt = fp8rl.SCALE_FP32
    m, n, k = 16, 256, 2048
    wq, sw, dwq, dsw = weights(n, k, fmt, 13)
    x = synth.activation_bf16(m, k, 14, "aqg-fault", device="cuda")
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_SPLITS, 1)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_TIMEOUT_NS, 50_000_000)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_FAULT_SKIP_KB, skip)
    fp8rl.gemm_act_quant(x, dwq, dsw, fmt)
    assert fp8rl.fp8rl_sync_status() == 6
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_FAULT_SKIP_KB, -1)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_TIMEOUT_NS, 2_000_000_000)
    assert fp8rl.fp8rl_sync_status() == 0
    check(x, wq, sw, dwq, dsw, fmt)
