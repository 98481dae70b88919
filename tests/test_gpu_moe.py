"""GPU parity of the MoE dispatch plan, the gathered 1x128 quantisation and
the weighted combine against the oracle, through the C ABI.

The plan is integer work: bit-exact.  Dispatch codes and scales are the
quantiser's bytes: bit-exact.  The combine is fp32 fused multiply-adds over at
most k = 32 slots and one bf16 rounding, against the fp64 oracle; the bound
used: |gpu - ref| <= 2^-8 |ref| + 2^-18 sum_j |g_j y_j| (the bf16 unit
roundoff, 8 significant bits, plus k * 2^-24 of the magnitude sum for the fp32
chain, k <= 32, with a factor 2 of margin)."""
import numpy as np
import pytest
import torch

import fp8_w8a8_rollout_gb300 as fp8rl
import oracle
from fp8_w8a8_rollout_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fp8rl.load_library(build_if_missing=True)


def random_topk(tokens, k, experts, drop, seed, skew=False):
    rng = np.random.default_rng(seed)
    if skew:  # nearly every pair on one expert: one huge segment, many empty ones
        idx = np.where(rng.random((tokens, k)) < 0.9, 3 % experts, rng.integers(0, experts, (tokens, k)))
    elif k <= experts:
        idx = np.stack([rng.permutation(experts)[:k] for _ in range(tokens)]) if tokens else \
            np.zeros((0, k), np.int64)
    else:
        idx = rng.integers(0, experts, (tokens, k))
    idx = idx.astype(np.int32)
    if drop:
        idx[rng.random((tokens, k)) < drop] = -1
        idx[rng.random((tokens, k)) < drop / 4] = experts + 7
    return idx


def gpu_plan(idx, experts):
    t = torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).cuda()
    off, rop, tor = fp8rl.moe_plan(t, experts)
    assert fp8rl.fp8rl_sync_status() == 0
    return off.cpu().numpy(), rop.cpu().numpy(), tor.cpu().numpy()


@pytest.mark.parametrize("tokens,k,experts,drop,skew", [
    (4096, 8, 128, 0.0, False),     # Qwen3-30B-A3B-shaped routing, T = 4096
    (37, 3, 5, 0.2, False),
    (1, 1, 1, 0.0, False),
    (0, 8, 4, 0.0, False),
    (20000, 8, 128, 0.05, False),   # many tiles, a dropped tail
    (65536, 8, 128, 0.0, False),    # tiles widened beyond 1024 pairs
    (300, 2, 8192, 0.0, False),     # the largest expert count
    (64, 32, 7, 0.1, False),        # the largest k (more slots than experts)
    (5000, 4, 16, 0.0, True),       # skewed: one expert takes ~90 %
    (1024, 8, 256, 0.02, False),    # the largest plan done by one CTA
    (1025, 8, 256, 0.0, False),     # one token more: the tiled kernels
])
def test_plan_bit_exact(tokens, k, experts, drop, skew):
    idx = random_topk(tokens, k, experts, drop, tokens + k + experts, skew)
    ref = oracle.moe_dispatch_plan(idx, experts)
    got = gpu_plan(idx, experts)
    for g, r, name in zip(got, ref, ("offsets", "row_of_pair", "token_of_row")):
        assert np.array_equal(g, r), name


def test_plan_of_replayed_router_indices_and_determinism():
    r = synth.moe_routing(4096, 128, 8, seed=0)
    a = gpu_plan(r.topk, 128)
    b = gpu_plan(r.topk, 128)
    ref = oracle.moe_dispatch_plan(r.topk, 128)
    for x, y, z in zip(a, b, ref):
        assert np.array_equal(x, z) and np.array_equal(x, y)


@pytest.mark.parametrize("tokens,hidden,k,experts,fmt,qpad", [
    (256, 2048, 8, 16, fp8rl.SCALE_FP32, 0),
    (256, 2048, 8, 16, fp8rl.SCALE_UE8M0, 0),
    (97, 300, 3, 7, fp8rl.SCALE_FP32, 0),    # ragged K: partial last group
    (64, 2048, 4, 8, fp8rl.SCALE_FP32, 8),   # code rows 8-byte but not 16-byte aligned
    (50, 4608, 2, 5, fp8rl.SCALE_UE8M0, 0),  # more than one 2048-column pass, a partial round
    (4096, 2048, 8, 128, fp8rl.SCALE_FP32, 0),  # the MoE layer's full gate-up input
    (4096, 768, 8, 128, fp8rl.SCALE_FP32, 0),   # the down input width
])
def test_dispatch_quant_bit_exact(tokens, hidden, k, experts, fmt, qpad):
    idx = random_topk(tokens, k, experts, 0.05, tokens + hidden)
    x = synth.normal_bf16((tokens, hidden), 1.0, 9, "gpu-dispatch", hidden)
    _, rop, tor = oracle.moe_dispatch_plan(idx, experts)
    q_ref, s_ref, live = oracle.moe_dispatch_quant(synth.bf16_bits(x), tor, fmt)
    rows = tor.size
    q = torch.full((rows, hidden + qpad), 0x55, dtype=torch.uint8, device="cuda")[:, :hidden]
    sdt = torch.float32 if fmt == fp8rl.SCALE_FP32 else torch.uint8
    s = torch.full(((hidden + 127) // 128, rows), 7, dtype=sdt, device="cuda")
    fp8rl.moe_dispatch_quant(x.cuda(), torch.from_numpy(rop).cuda(), k, fmt, out=(q, s))
    assert fp8rl.fp8rl_sync_status() == 0
    qg, sg = q.contiguous().cpu().numpy(), s.cpu().numpy()
    assert np.array_equal(qg[live], q_ref[live])
    assert np.array_equal(np.ascontiguousarray(sg[:, live]).view(np.uint8),
                          np.ascontiguousarray(s_ref[:, live]).view(np.uint8))
    # rows without a token are left as they were
    assert np.all(qg[~live] == 0x55) and np.all(sg[:, ~live] == 7)


def test_dispatch_then_grouped_gemm_matches_oracle():
    """The whole dispatch path on the GPU: plan, gathered quantisation, the
    grouped GEMM on the plan's offsets; sampled outputs against the oracle."""
    tokens, hidden, n, k, experts = 512, 512, 256, 4, 8
    r = synth.moe_routing(tokens, experts, k, seed=2)
    x = synth.normal_bf16((tokens, hidden), 1.0, 10, "gpu-dispatch-gemm")
    w = synth.moe_expert_weights(n, hidden, experts, 0, 0, "dispatch-gemm")
    wq, sw = fp8rl.quant_weight(w.reshape(experts * n, hidden).cuda())
    wq, sw = wq.reshape(experts, n, hidden), sw.reshape(experts, n // 128, hidden // 128)
    off, rop, tor = fp8rl.moe_plan(torch.from_numpy(r.topk).cuda(), experts)
    xq, sx = fp8rl.moe_dispatch_quant(x.cuda(), rop, k)
    y = fp8rl.grouped_gemm(xq, sx, wq, sw, off)
    assert fp8rl.fp8rl_sync_status() == 0
    off_o, _, tor_o = oracle.moe_dispatch_plan(r.topk, experts)
    xq_o, sx_o, _ = oracle.moe_dispatch_quant(synth.bf16_bits(x), tor_o)
    ref = oracle.grouped_gemm_blockscaled(xq_o, sx_o, wq.cpu().numpy(), sw.cpu().numpy(), off_o)
    got = y.float().cpu().numpy().astype(np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert np.all(np.abs(got - ref) <= 1e-2 * np.abs(ref) + 1e-3 * rms)


def combine_bound(y, rop, gate):
    return oracle.moe_combine(np.abs(y), rop, np.abs(gate))


@pytest.mark.parametrize("tokens,n,k,experts,drop,pad", [
    (4096, 2048, 8, 128, 0.0, 0),   # the MoE layer's down output, T = 4096
    (300, 1000, 3, 9, 0.1, 0),      # n % 8 != 0: scalar tail of each row
    (33, 256, 1, 4, 0.0, 3),        # k = 1; rows not 16-byte aligned: scalar path
    (50, 512, 32, 40, 0.2, 0),      # the largest k
])
def test_combine_within_tolerance(tokens, n, k, experts, drop, pad):
    idx = random_topk(tokens, k, experts, drop, tokens * 3 + n)
    _, rop, _ = oracle.moe_dispatch_plan(idx, experts)
    rng = np.random.default_rng(n)
    gate = rng.random((tokens, k)).astype(np.float32)
    rows = tokens * k
    ld = n + pad
    yfull = synth.normal_bf16((rows, ld), 1.0, 11, "gpu-combine", n)
    y = yfull[:, :n]
    yv = y.float().numpy().astype(np.float64)
    ref = oracle.moe_combine(yv, rop, gate.astype(np.float64))
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -18 * combine_bound(yv, rop, gate.astype(np.float64))
    yd = yfull.cuda()[:, :n]
    out = fp8rl.moe_combine(yd, torch.from_numpy(rop).cuda(), torch.from_numpy(gate).cuda())
    assert fp8rl.fp8rl_sync_status() == 0
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= bound)
    # a token whose every slot was dropped gets exactly zero
    dead = np.all(rop.reshape(tokens, k) < 0, axis=1)
    assert np.all(got[dead] == 0.0)


@pytest.mark.parametrize("keep", [0, 37, 600])
def test_combine_ignores_rows_past_y(keep):
    """y holds only its first `keep` rows: slots naming a row at or past it
    add nothing, as if dropped (keep = 0: y is null, every token zero)."""
    tokens, n, k, experts = 100, 264, 8, 16
    idx = random_topk(tokens, k, experts, 0.1, 21 + keep)
    _, rop, _ = oracle.moe_dispatch_plan(idx, experts)
    gate = np.random.default_rng(keep).random((tokens, k)).astype(np.float32)
    y = synth.normal_bf16((tokens * k, n), 1.0, 14, "gpu-combine-past", keep)[:keep]
    rop_ref = np.where(rop < keep, rop, -1).astype(rop.dtype)
    yv = y.float().numpy().astype(np.float64)
    ref = oracle.moe_combine(yv, rop_ref, gate.astype(np.float64))
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -18 * combine_bound(yv, rop_ref, gate.astype(np.float64))
    yd = y.cuda() if keep else torch.empty((0, n), dtype=torch.bfloat16, device="cuda")
    out = fp8rl.moe_combine(yd, torch.from_numpy(rop).cuda(), torch.from_numpy(gate).cuda())
    assert fp8rl.fp8rl_sync_status() == 0
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= bound)
    if keep == 0:
        assert np.all(got == 0.0)


def test_combine_one_hot_gates_copy_rows_exactly():
    tokens, n, k, experts = 200, 512, 8, 16
    idx = random_topk(tokens, k, experts, 0.0, 5)
    _, rop, _ = oracle.moe_dispatch_plan(idx, experts)
    gate = np.zeros((tokens, k), np.float32)
    pick = np.random.default_rng(6).integers(0, k, tokens)
    gate[np.arange(tokens), pick] = 1.0
    y = synth.normal_bf16((tokens * k, n), 1.0, 12, "gpu-combine-hot")
    out = fp8rl.moe_combine(y.cuda(), torch.from_numpy(rop).cuda(), torch.from_numpy(gate).cuda())
    sel = rop.reshape(tokens, k)[np.arange(tokens), pick]
    assert torch.equal(out.cpu(), y[torch.from_numpy(sel.astype(np.int64))])


def test_rollout_moe_layer_round_trip_with_identity_experts():
    """plan -> dispatch quant -> (identity experts: the dequantised rows as
    bf16) -> combine returns each token row within its quantisation error."""
    tokens, hidden, k, experts = 1024, 512, 8, 32
    r = synth.moe_routing(tokens, experts, k, seed=7)
    x = synth.normal_bf16((tokens, hidden), 1.0, 13, "gpu-roundtrip")
    off, rop, tor = fp8rl.moe_plan(torch.from_numpy(r.topk).cuda(), experts)
    xq, sx = fp8rl.moe_dispatch_quant(x.cuda(), rop, k)
    deq = oracle.dequantize(xq.cpu().numpy(), sx.cpu().numpy().T, 1, 128)
    y = torch.from_numpy(deq.astype(np.float32)).to(torch.bfloat16).cuda()
    out = fp8rl.moe_combine(y, rop, torch.from_numpy(r.gate).cuda())
    assert fp8rl.fp8rl_sync_status() == 0
    xf = x.float().numpy()
    smax = float(sx.max())
    err = np.abs(out.float().cpu().numpy() - xf)
    # E4M3 half-ulp (2^-4 relative) and subnormal floor, then two bf16
    # roundings (the expert output, the combine's result: 2^-8 each)
    assert np.all(err <= 2.0 ** -4 * np.abs(xf) * (1 + 2.0 ** -6) + smax * 2.0 ** -10 + 2.0 ** -7 * np.abs(xf) * 1.1)


def test_moe_entry_points_reject_bad_tensors():
    with pytest.raises(ValueError):
        fp8rl.moe_plan(torch.zeros((4, 2), dtype=torch.int64, device="cuda"), 8)
    with pytest.raises(fp8rl.Fp8rlError):
        fp8rl.moe_plan(torch.zeros((4, 40), dtype=torch.int32, device="cuda"), 8)  # k > 32
    with pytest.raises(ValueError):
        fp8rl.moe_combine(torch.zeros((8, 16), dtype=torch.bfloat16, device="cuda"),
                          torch.zeros(8, dtype=torch.int32, device="cuda"),
                          torch.zeros((4, 2), dtype=torch.float64, device="cuda"))
