"""GPU parity of the fused gate-up path (block-scaled GEMM -> SiLU(gate) * up
in fp32 -> 1x128 E4M3 quantisation) against the oracle, through the C ABI.

Operands are quantised by the oracle on the host.  The GPU's h is an fp32
accumulation and the oracle's is fp64, so codes are compared through what
they must satisfy rather than bit for bit:
  * scales: fp32 within 1e-4 relative of the oracle's (the group maxima
    differ only by accumulation rounding); UE8M0 equal, or one power of two
    apart where the oracle's amax / 448 lies within 1e-4 of a power of two;
  * codes: dec(q) * s_gpu within half an E4M3 step (at s_gpu) of the oracle's
    h, plus TOL_REL |h| + TOL_RMS rms(h) for the accumulation difference;
  * fp32 scales: each group's largest |code| is 0x7E (448), as it must be for
    the GPU's own maximum.
A chained check feeds the GPU's quantised h to the down projection and
compares with the oracle's chain (codes may differ by one step near a
rounding boundary, so its tolerance is twice the GEMM tests')."""
import numpy as np
import pytest
import torch

import fp8_w8a8_rollout_gb300 as fp8rl
import oracle
from fp8_w8a8_rollout_gb300 import synth

pytestmark = pytest.mark.gpu

FMTS = [fp8rl.SCALE_FP32, fp8rl.SCALE_UE8M0]
TOL_REL, TOL_RMS = 2e-3, 2e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fp8rl.load_library(build_if_missing=True)
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_RESET, 0)
    yield
    fp8rl.fp8rl_debug_set(fp8rl.DEBUG_RESET, 0)


def to_dev(*arrs):
    return [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in arrs]


def operands(m, inter, k, fmt, seed, experts=None):
    x = synth.activation_bf16(m, k, seed, "fused-x", m, inter, k)
    order = oracle.interleave_gate_up_rows(2 * inter)
    xq, sx = oracle.quant_act_group(synth.bf16_bits(x), fmt)
    if experts is None:
        w = synth.weight_bf16(2 * inter, k, seed + 1, "fused-w", inter, k)
        wq, sw = oracle.quant_weight_blockwise(synth.bf16_bits(w[torch.from_numpy(order)]), fmt)
    else:
        ws = synth.moe_expert_weights(2 * inter, k, experts, seed + 1, 0, "fused")
        wq = np.empty((experts, 2 * inter, k), np.uint8)
        sw = np.empty((experts, 2 * inter // 128, k // 128), np.float32 if fmt == 0 else np.uint8)
        for e in range(experts):
            wq[e], sw[e] = oracle.quant_weight_blockwise(synth.bf16_bits(ws[e][torch.from_numpy(order)]), fmt)
    return xq, sx, wq, sw


def check_codes(hq, hs, h_ref, fmt, rows=None):
    """hq [r, inter] uint8, hs [inter/128, r] against the oracle's fp64 h [r, inter]."""
    table = oracle.e4m3_decode_table()
    inter = h_ref.shape[1]
    groups = inter // 128
    hs = hs.astype(np.float64) if fmt == 0 else np.ldexp(1.0, hs.astype(np.int64) - 127)
    amax_ref = np.abs(h_ref).reshape(h_ref.shape[0], groups, 128).max(axis=2).T  # [groups, r]
    if fmt == 0:
        s_ref = np.where(amax_ref == 0, 1.0, amax_ref / 448.0)
        assert np.all(np.abs(hs - s_ref) <= 1e-4 * s_ref), "fp32 scales differ"
    else:
        e_ref = np.where(amax_ref == 0, 0, np.ceil(np.log2(np.maximum(amax_ref, 1e-300) / 448.0)))
        e_gpu = np.log2(hs)
        near = np.abs(np.log2(np.maximum(amax_ref, 1e-300) / 448.0) - np.round(np.log2(np.maximum(amax_ref, 1e-300) / 448.0))) < 1e-4
        assert np.all((e_gpu == e_ref) | (near & (np.abs(e_gpu - e_ref) == 1))), "UE8M0 scales differ"
    srep = np.repeat(hs.T, 128, axis=1)  # [r, inter]
    deq = table[hq] * srep
    rms = float(np.sqrt(np.mean(h_ref ** 2))) if h_ref.size else 0.0
    tol = TOL_REL * np.abs(h_ref) + TOL_RMS * rms
    v = (np.abs(h_ref) + tol) / srep
    with np.errstate(divide="ignore"):
        step = np.where(v < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(v, 1e-300))) - 3))
    bound = 0.5 * step * srep + tol
    bad = np.abs(deq - h_ref) > bound
    assert not bad.any(), f"{int(bad.sum())}/{bad.size} codes outside the bound"
    if fmt == 0:
        gmax = (hq & 0x7F).reshape(hq.shape[0], groups, 128).max(axis=2)
        nonzero = amax_ref.T > 0
        assert np.all(gmax[nonzero] == 0x7E), "a group maximum is not 448"


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m,inter,k", [(1, 128, 128), (100, 256, 640), (300, 384, 256), (129, 128, 1024)])
def test_fused_dense_small_full(m, inter, k, fmt):
    xq, sx, wq, sw = operands(m, inter, k, fmt, 51)
    h_ref, _, _ = oracle.gemm_swiglu_quant(xq, sx, wq, sw, fmt, fmt)
    hq, hs = fp8rl.gemm_swiglu_quant(*to_dev(xq, sx, wq, sw), fmt)
    assert fp8rl.fp8rl_sync_status() == 0
    check_codes(hq.cpu().numpy(), hs.cpu().numpy(), h_ref, fmt)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("counts", [[3, 0, 200, 129], [128, 128], [0, 0, 5]])
def test_fused_grouped_small_full(counts, fmt):
    offsets = synth.routing_with_counts(counts)
    rows, inter, k = int(offsets[-1]), 256, 384
    xq, sx, wq, sw = operands(rows, inter, k, fmt, 52, experts=len(counts))
    h_ref, _, _ = oracle.gemm_swiglu_quant(xq, sx, wq, sw, fmt, fmt, offsets=offsets)
    dx, dsx, dw, dsw, doff = to_dev(xq, sx, wq, sw, offsets)
    hq, hs = fp8rl.grouped_gemm_swiglu_quant(dx, dsx, dw, dsw, doff, fmt)
    assert fp8rl.fp8rl_sync_status() == 0
    check_codes(hq.cpu().numpy(), hs.cpu().numpy(), h_ref, fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_fused_then_down_projection(fmt):
    """gate-up (fused) -> down on the GPU against the oracle's chain."""
    m, inter, k = 200, 512, 384
    xq, sx, wq, sw = operands(m, inter, k, fmt, 53)
    wd = synth.weight_bf16(k, inter, 54, "fused-down")
    wdq, wds = oracle.quant_weight_blockwise(synth.bf16_bits(wd), fmt)
    _, hq_ref, hs_ref = oracle.gemm_swiglu_quant(xq, sx, wq, sw, fmt, fmt)
    y_ref = oracle.gemm_blockscaled(hq_ref, hs_ref, wdq, wds, fmt)
    hq, hs = fp8rl.gemm_swiglu_quant(*to_dev(xq, sx, wq, sw), fmt)
    dwq, dws = to_dev(wdq, wds)
    y = fp8rl.gemm(hq, hs, dwq, dws, fmt)
    assert fp8rl.fp8rl_sync_status() == 0
    got = y.float().cpu().numpy()
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    err = np.abs(got - y_ref)
    assert np.all(err <= 2e-2 * np.abs(y_ref) + 2e-3 * rms)


def sampled_rows_reference(xq, sx, wq, sw, rows, fmt, offsets=None):
    """The oracle's h for whole rows `rows` only (GEMM at sampled positions)."""
    n2 = wq.shape[-2]
    rr = np.repeat(rows, n2)
    cc = np.tile(np.arange(n2), len(rows))
    if offsets is None:
        y = oracle.gemm_blockscaled_at(xq, sx, wq, sw, rr, cc, fmt)
    else:
        y = oracle.grouped_gemm_blockscaled_at(xq, sx, wq, sw, offsets, rr, cc, fmt)
    y = y.reshape(len(rows), n2)
    order = oracle.interleave_gate_up_rows(n2)
    plain = np.empty_like(y)
    plain[:, order] = y
    inter = n2 // 2
    return oracle.swiglu(plain[:, :inter], plain[:, inter:])


@pytest.mark.parametrize("m", [1024, 8192])
def test_fused_qwen3_8b_mlp_sampled_rows(m):
    """Full-size launch (inter 12288, k 4096); the oracle evaluates 4 whole rows."""
    inter, k, fmt = 12288, 4096, fp8rl.SCALE_FP32
    x = synth.activation_bf16(m, k, 55, "fused-q", m)
    w = synth.weight_bf16(2 * inter, k, 56, "fused-q")
    order = torch.from_numpy(oracle.interleave_gate_up_rows(2 * inter))
    xq, sx = oracle.quant_act_group(synth.bf16_bits(x))
    wq, sw = oracle.quant_weight_blockwise(synth.bf16_bits(w[order]))
    hq, hs = fp8rl.gemm_swiglu_quant(*to_dev(xq, sx, wq, sw), fmt)
    assert fp8rl.fp8rl_sync_status() == 0
    rows = np.unique(np.array([0, m - 1, 777 % m, (m * 5) // 7]))
    h_ref = sampled_rows_reference(xq, sx, wq, sw, rows, fmt)
    check_codes(hq.cpu().numpy()[rows], hs.cpu().numpy()[:, rows], h_ref, fmt)


def test_fused_moe_qwen3_30b_a3b_sampled_rows():
    """128 experts, inter 768, k 2048, T = 4096 top-8 routing (32768 rows)."""
    fmt = fp8rl.SCALE_FP32
    r = synth.moe_routing(4096, synth.MOE_EXPERTS, synth.MOE_TOPK, 0, 0)
    offsets = oracle.moe_dispatch_plan(r.topk, synth.MOE_EXPERTS)[0]
    rows_total, inter, k = int(offsets[-1]), synth.MOE_INTER, synth.MOE_HIDDEN
    x = synth.normal_bf16((rows_total, k), 1.0, 57, "fused-moe-x")
    xq, sx = oracle.quant_act_group(synth.bf16_bits(x))
    dev = torch.device("cuda")
    wg = synth.moe_expert_weights(inter, k, synth.MOE_EXPERTS, 58, 0, "gate", device=dev)
    wu = synth.moe_expert_weights(inter, k, synth.MOE_EXPERTS, 58, 0, "up", device=dev)
    wq, sw = fp8rl.quant_gate_up_interleaved(wg, wu)  # the GPU quantiser, bit-exact by its own tests
    wq_h, sw_h = wq.cpu().numpy(), sw.cpu().numpy()
    # the same layout from the oracle's quantiser, for the reference
    order = torch.from_numpy(oracle.interleave_gate_up_rows(2 * inter))
    wcat = torch.cat([wg, wu], dim=1).cpu()
    for e in (0, 77, 127):
        q_ref, s_ref = oracle.quant_weight_blockwise(synth.bf16_bits(wcat[e][order]))
        assert np.array_equal(wq_h[e], q_ref) and np.array_equal(sw_h[e], s_ref)
    dx, dsx, doff = to_dev(xq, sx, offsets)
    hq, hs = fp8rl.grouped_gemm_swiglu_quant(dx, dsx, wq, sw, doff, fmt)
    assert fp8rl.fp8rl_sync_status() == 0
    rows = np.unique(np.array([0, rows_total - 1, int(offsets[64]), int(offsets[100]) + 3]))
    ref = [oracle.quant_weight_blockwise(synth.bf16_bits(wcat[e][order])) for e in range(128)]
    wq_ref = np.stack([q for q, _ in ref])
    sw_ref = np.stack([sc for _, sc in ref])
    h_ref = sampled_rows_reference(xq, sx, wq_ref, sw_ref, rows, fmt, offsets=offsets)
    check_codes(hq.cpu().numpy()[rows], hs.cpu().numpy()[:, rows], h_ref, fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_quant_gate_up_interleaved_matches_oracle_layout(fmt):
    gate = synth.weight_bf16(256, 384, 59, "il-gate")
    up = synth.weight_bf16(256, 384, 60, "il-up")
    q, s = fp8rl.quant_gate_up_interleaved(gate.cuda(), up.cuda(), fmt)
    assert fp8rl.fp8rl_sync_status() == 0
    order = torch.from_numpy(oracle.interleave_gate_up_rows(512))
    q_ref, s_ref = oracle.quant_weight_blockwise(synth.bf16_bits(torch.cat([gate, up])[order]), fmt)
    assert np.array_equal(q.cpu().numpy(), q_ref) and np.array_equal(s.cpu().numpy(), s_ref)
