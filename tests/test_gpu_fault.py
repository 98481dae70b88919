"""Failure detection without a GPU fault: a device-side wait that can never
complete (the producer is told to skip one K chunk, so nothing ever arrives on
that stage's barrier) must run out after its limit, leave the kernel through
the normal teardown, and be reported as FP8RL_ERR_TIMEOUT on the host; the
context must stay usable for the next call."""
import numpy as np
import pytest
import torch

import fp8_w8a8_rollout_gb300 as fp8rl
import oracle
from fp8_w8a8_rollout_gb300 import synth

pytestmark = pytest.mark.gpu

TIMEOUT = 6


@pytest.fixture(autouse=True)
def _reset():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fp8rl.load_library(build_if_missing=True)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_RESET, 0)
    yield
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_RESET, 0)


def operands(m, n, k, seed):
    x = synth.activation_bf16(m, k, seed, "fault-x")
    w = synth.weight_bf16(n, k, seed, "fault-w")
    xq, sx = oracle.quant_act_group(synth.bf16_bits(x))
    wq, sw = oracle.quant_weight_blockwise(synth.bf16_bits(w))
    return xq, sx, wq, sw


def dev(*a):
    return [torch.from_numpy(np.ascontiguousarray(v)).cuda() for v in a]


@pytest.mark.parametrize("bn", [128, 256])
def test_wait_runs_out_and_is_reported(bn):
    m, n, k = 256, 512, 512
    xq, sx, wq, sw = operands(m, n, k, 1)
    dx, dsx, dw, dsw = dev(xq, sx, wq, sw)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_GEMM_BN, bn)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_TIMEOUT_NS, 50_000_000)   # 50 ms
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_FAULT_SKIP_KB, 1)         # chunk 1 never arrives
    fp8rl.gemm(dx, dsx, dw, dsw)
    assert fp8rl.fp8rl_sync_status() == TIMEOUT
    # the word is cleared by the read, and the context still works
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_RESET, 0)
    assert fp8rl.fp8rl_sync_status() == 0
    y = fp8rl.gemm(dx, dsx, dw, dsw)
    assert fp8rl.fp8rl_sync_status() == 0
    ref = oracle.gemm_blockscaled(xq, sx, wq, sw)
    got = y.float().cpu().numpy()
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert np.all(np.abs(got - ref) <= 1e-2 * np.abs(ref) + 1e-3 * rms)


@pytest.mark.parametrize("skip", [0, 1, 5])
def test_pair_wait_runs_out_and_is_reported(skip):
    """Tensor-core pairs (UE8M0): a chunk that never arrives stops the even CTA's MMA
    thread and, through the missing commits, the odd CTA's roles; both leave
    through the teardown (the even CTA lets both CTAs' copies land), TIMEOUT is
    reported and the next call on the same context is correct."""
    m, n, k = 512, 512, 1024
    fmt = fp8rl.SCALE_UE8M0
    x = synth.activation_bf16(m, k, 4, "fault-x")
    w = synth.weight_bf16(n, k, 4, "fault-w")
    xq, sx = oracle.quant_act_group(synth.bf16_bits(x), fmt)
    wq, sw = oracle.quant_weight_blockwise(synth.bf16_bits(w), fmt)
    dx, dsx, dw, dsw = dev(xq, sx, wq, sw)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_MX, 2)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_PAIR, 1)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_TIMEOUT_NS, 50_000_000)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_FAULT_SKIP_KB, skip)
    fp8rl.gemm(dx, dsx, dw, dsw, fmt)
    assert fp8rl.fp8rl_sync_status() == TIMEOUT
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_FAULT_SKIP_KB, -1)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_TIMEOUT_NS, 2_000_000_000)
    assert fp8rl.fp8rl_sync_status() == 0
    y = fp8rl.gemm(dx, dsx, dw, dsw, fmt)
    assert fp8rl.fp8rl_sync_status() == 0
    ref = oracle.gemm_blockscaled(xq, sx, wq, sw, fmt)
    got = y.float().cpu().numpy()
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert np.all(np.abs(got - ref) <= 1e-2 * np.abs(ref) + 1e-3 * rms)


def test_grouped_wait_runs_out_and_is_reported():
    counts = [100, 0, 300]
    offsets = synth.routing_with_counts(counts)
    rows, n, k = int(offsets[-1]), 256, 384
    x = synth.normal_bf16((rows, k), 1.0, 2, "fault-gx")
    xq, sx = oracle.quant_act_group(synth.bf16_bits(x))
    ws = synth.moe_expert_weights(n, k, 3, 2, 0, "fault")
    wq, sw = oracle.quant_weight_blockwise(synth.bf16_bits(ws.reshape(-1, k)))
    dx, dsx, dw, dsw, doff = dev(xq, sx, wq.reshape(3, n, k), sw.reshape(3, n // 128, k // 128), offsets)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_TIMEOUT_NS, 50_000_000)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_FAULT_SKIP_KB, 2)
    fp8rl.grouped_gemm(dx, dsx, dw, dsw, doff)
    assert fp8rl.fp8rl_sync_status() == TIMEOUT
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_RESET, 0)
    fp8rl.grouped_gemm(dx, dsx, dw, dsw, doff)
    assert fp8rl.fp8rl_sync_status() == 0


def test_debug_hook_rejects_bad_values():
    with pytest.raises(fp8rl.Fp8rlError):
        fp8rl.fp8rl_debug_set(fp8rl.DEBUG_GEMM_BN, 96)
    with pytest.raises(fp8rl.Fp8rlError):
        fp8rl.fp8rl_debug_set(fp8rl.DEBUG_TIMEOUT_NS, 0)
    with pytest.raises(fp8rl.Fp8rlError):
        fp8rl.fp8rl_debug_set(99, 0)


def test_split_k_cluster_wait_runs_out_and_is_reported():
    m, n, k = 16, 256, 1024
    xq, sx, wq, sw = operands(m, n, k, 3)
    dx, dsx, dw, dsw = dev(xq, sx, wq, sw)
    fp8rl.fp8rl_debug_set(6, 4)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_TIMEOUT_NS, 50_000_000)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_FAULT_SKIP_KB, 1)
    fp8rl.gemm(dx, dsx, dw, dsw)
    assert fp8rl.fp8rl_sync_status() == TIMEOUT
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_RESET, 0)
    y = fp8rl.gemm(dx, dsx, dw, dsw)
    assert fp8rl.fp8rl_sync_status() == 0
    ref = oracle.gemm_blockscaled(xq, sx, wq, sw)
    got = y.float().cpu().numpy()
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert np.all(np.abs(got - ref) <= 1e-2 * np.abs(ref) + 1e-3 * rms)


def test_stream_k_owner_wait_runs_out_and_workspace_recovers():
    """One tile of ten K chunks over three stream-K CTAs ([0,3) owner, [3,6),
    [6,10)).  Only the last CTA has a fourth chunk, and it is the one skipped:
    that CTA's MMA wait runs out and it publishes nothing, so the owner's wait
    for its flag runs out as well.  The workspace needs no clean-up: the next
    call with it is correct."""
    m, n, k = 64, 256, 1280
    xq, sx, wq, sw = operands(m, n, k, 5)
    dx, dsx, dw, dsw = dev(xq, sx, wq, sw)
    ws = fp8rl.gemm_workspace()
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_STREAMK, 2)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_STREAMK_GRID, 3)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_GEMM_BN, 256)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_TIMEOUT_NS, 50_000_000)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_FAULT_SKIP_KB, 3)
    fp8rl.gemm(dx, dsx, dw, dsw, workspace=ws)
    assert fp8rl.fp8rl_sync_status() == TIMEOUT
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_FAULT_SKIP_KB, -1)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_TIMEOUT_NS, 2_000_000_000)
    y = fp8rl.gemm(dx, dsx, dw, dsw, workspace=ws)
    assert fp8rl.fp8rl_sync_status() == 0
    ref = oracle.gemm_blockscaled(xq, sx, wq, sw)
    got = y.float().cpu().numpy()
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert np.all(np.abs(got - ref) <= 1e-2 * np.abs(ref) + 1e-3 * rms)


def test_fused_epilogue_wait_runs_out_and_is_reported():
    """The fused gate-up epilogue exchanges row maxima behind a barrier of all
    epilogue warps; a wait that runs out must still end the kernel (every
    warp leaves together) and be reported, and the next call must work."""
    m, inter, k = 300, 256, 512
    x = synth.activation_bf16(m, k, 6, "fault-fx")
    w = synth.weight_bf16(2 * inter, k, 6, "fault-fw")
    xq, sx = oracle.quant_act_group(synth.bf16_bits(x))
    wq, sw = oracle.quant_weight_blockwise(synth.bf16_bits(w[torch.from_numpy(oracle.interleave_gate_up_rows(2 * inter))]))
    dx, dsx, dw, dsw = dev(xq, sx, wq, sw)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_TIMEOUT_NS, 50_000_000)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_FAULT_SKIP_KB, 1)  # each CTA's second K chunk never arrives
    fp8rl.gemm_swiglu_quant(dx, dsx, dw, dsw)
    assert fp8rl.fp8rl_sync_status() == TIMEOUT
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_RESET, 0)
    hq, hs = fp8rl.gemm_swiglu_quant(dx, dsx, dw, dsw)
    assert fp8rl.fp8rl_sync_status() == 0
    h_ref, hq_ref, hs_ref = oracle.gemm_swiglu_quant(xq, sx, wq, sw)
    assert np.all(np.abs(hs.cpu().numpy() - hs_ref) <= 1e-4 * hs_ref)


@pytest.mark.parametrize("skip,m", [(0, 16), (7, 16), (3, 96)])
def test_decode_wait_runs_out_and_is_reported(skip, m):
    """The decode-size GEMM launched behind the activation quantiser with
    overlapped launches: a chunk among the weight stages fetched before the
    wait for the quantiser (0) or one of the later ones (7) never arrives; the
    MMA's wait runs out, TIMEOUT is reported, and the next call is correct."""
    n, k = 256, 4096
    x = synth.activation_bf16(m, k, 8, "fault-dx", device="cuda")
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_DECODE, 1)
    w = synth.weight_bf16(n, k, 8, "fault-dw")
    wq, sw = oracle.quant_weight_blockwise(synth.bf16_bits(w))
    dw, dsw = dev(wq, sw)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_SPLITS, 1)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_TIMEOUT_NS, 50_000_000)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_FAULT_SKIP_KB, skip)
    xq, sx = fp8rl.quant_act(x)
    fp8rl.gemm(xq, sx, dw, dsw)
    assert fp8rl.fp8rl_sync_status() == TIMEOUT
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_FAULT_SKIP_KB, -1)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_TIMEOUT_NS, 2_000_000_000)
    assert fp8rl.fp8rl_sync_status() == 0
    xq, sx = fp8rl.quant_act(x)
    y = fp8rl.gemm(xq, sx, dw, dsw)
    assert fp8rl.fp8rl_sync_status() == 0
    rxq, rsx = oracle.quant_act_group(synth.bf16_bits(x.cpu()))
    assert np.array_equal(xq.cpu().numpy(), rxq)
    ref = oracle.gemm_blockscaled(rxq, rsx, wq, sw)
    got = y.float().cpu().numpy()
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert np.all(np.abs(got - ref) <= 1e-2 * np.abs(ref) + 1e-3 * rms)
