"""Pins for the CPU oracle, checked against facts fixed outside the oracle.

Every check here ties the oracle to something other than itself: the format
facts printed on the FP8-RL page ("Prerequisites / FP8 quantisation format"),
closed forms of the E4M3 format, brute force over the whole code table,
invariants of blockwise amax scaling, a hand-worked example, exact integer
arithmetic, and library routines (torch's float8_e4m3fn cast, numpy matmul)
for the special cases that reduce to them.  CPU only.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from fp8_w8a8_rollout_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split()
                out[k] = v
    return out


def torch_decode_all():
    """Library decode of all 256 codes (torch's float8_e4m3fn)."""
    codes = torch.arange(256, dtype=torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def brute_force_encode(values: np.ndarray) -> np.ndarray:
    """Nearest finite code by scanning all 254 finite codes (independent of the
    oracle's bracketing search); ties go to the even code; |v| >= 448 saturates;
    the sign comes from the sign bit."""
    table = torch_decode_all()
    pos = np.arange(127)  # non-negative finite codes 0x00..0x7E
    mags = table[pos]
    v = np.asarray(values, dtype=np.float64)
    a = np.abs(v)
    d = np.abs(a[:, None] - mags[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # among equally near codes prefer the even one
    even = (pos % 2 == 0)[None, :]
    pick_even = cand & even
    has_even = pick_even.any(axis=1)
    code = np.where(has_even, np.argmax(pick_even, axis=1), np.argmax(cand, axis=1))
    code = np.where(a >= 448.0, 126, code)
    sign = np.signbit(v).astype(np.int64) * 128
    return (code + sign).astype(np.uint8)


# --------------------------------------------------------------------------- decode

def test_decode_matches_page_range_and_format_facts():
    facts = read_golden("e4m3_format_facts.txt")
    table = oracle.e4m3_decode_table()
    finite = table[np.isfinite(table)]
    assert finite.max() == float(facts["e4m3_max"])  # page: range about [-448, 448]
    assert finite.min() == float(facts["e4m3_min"])
    assert int(facts["e4m3_exponent_bits"]) + int(facts["e4m3_mantissa_bits"]) + 1 == 8
    assert table[0x7E] == 448.0 and table[0xFE] == -448.0
    assert math.isnan(table[0x7F]) and math.isnan(table[0xFF])
    assert np.isnan(table).sum() == 2  # no infinities, only two NaN codes
    assert table[0x08] == 2.0 ** -6  # smallest normal
    assert table[0x01] == 2.0 ** -9  # smallest subnormal
    assert table[0x00] == 0.0 and not math.copysign(1, table[0x00]) < 0
    assert table[0x80] == 0.0 and math.copysign(1, table[0x80]) < 0
    assert table[0x38] == 1.0  # exponent field 7 = bias
    mags = table[:127]
    assert np.all(np.diff(mags) > 0)  # magnitudes increase strictly with the code
    assert np.array_equal(table[128:255], -table[:127])


def test_decode_matches_library_float8():
    ours = oracle.e4m3_decode_table()
    lib = torch_decode_all()
    fin = ~np.isnan(lib)
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    assert np.array_equal(ours[fin], lib[fin])
    assert np.array_equal(np.signbit(ours[fin]), np.signbit(lib[fin]))


def test_subnormal_spacing_and_binade_spacing():
    table = oracle.e4m3_decode_table()
    # subnormal codes are evenly spaced by 2^-9; each normal binade has 8 codes
    assert np.allclose(np.diff(table[0:9]), 2.0 ** -9, rtol=0, atol=0)
    for e in range(1, 16):
        lo = table[e * 8]
        assert lo == 2.0 ** (e - 7)
        step = 2.0 ** (e - 7 - 3)
        n = 8 if e < 15 else 7
        assert np.all(np.diff(table[e * 8:e * 8 + n]) == step)


# --------------------------------------------------------------------------- encode

def test_encode_roundtrips_every_finite_code():
    table = oracle.e4m3_decode_table()
    for c in range(256):
        if np.isnan(table[c]):
            continue
        assert oracle.e4m3_encode(np.float32(table[c])) == c, hex(c)


def test_encode_midpoints_ties_to_even_and_neighbours():
    table = oracle.e4m3_decode_table()
    for c in range(126):
        lo, hi = table[c], table[c + 1]
        mid = 0.5 * (lo + hi)
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode_f64(mid) == even
        assert oracle.e4m3_encode_f64(-mid) == even | 0x80
        eps = (hi - lo) * 2.0 ** -20
        assert oracle.e4m3_encode_f64(mid - eps) == c
        assert oracle.e4m3_encode_f64(mid + eps) == c + 1
        # the fp32 entry point agrees: every midpoint is an fp32 value
        assert np.float32(mid) == mid
        assert oracle.e4m3_encode(np.float32(mid)) == even


def test_encode_saturates_and_keeps_sign_of_zero():
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(464.0) == 0x7E
    assert oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(-1e30) == 0xFE
    assert oracle.e4m3_encode(432.0) == 0x7E  # tie 416/448 -> even mantissa (448)
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(0.0) == 0x00
    assert oracle.e4m3_encode(-1e-30) == 0x80
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00  # half the smallest subnormal: tie -> 0
    assert oracle.e4m3_encode(np.float32(2.0 ** -10) * np.float32(1 + 2 ** -23)) == 0x01
    tiny = np.frombuffer(np.uint32(1).tobytes(), dtype=np.float32)[0]  # fp32 subnormal
    assert oracle.e4m3_encode(tiny) == 0x00
    assert oracle.e4m3_encode(-tiny) == 0x80


def test_encode_brute_force_all_bf16_values():
    bits = np.arange(65536, dtype=np.uint32) << 16
    v = bits.view(np.float32)
    v = v[np.isfinite(v)]
    ours = oracle.e4m3_encode_array(v)
    ref = brute_force_encode(v.astype(np.float64))
    assert np.array_equal(ours, ref)


def test_encode_matches_library_cast_on_rounding_boundaries():
    """Saturating RNE is the library cast of the clamped value.  The fp32 bit
    patterns cover every sign/exponent/upper-mantissa combination with the low
    bits at the places where rounding decisions change."""
    hi = np.arange(65536, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x1234, 0xC000],
                    dtype=np.uint32)
    bits = (hi[:, None] | lows[None, :]).reshape(-1)
    v = bits.view(np.float32)
    v = v[np.isfinite(v)]
    ours = oracle.e4m3_encode_array(v)
    clamped = torch.from_numpy(v).clamp(-448.0, 448.0)
    lib = clamped.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # the library keeps the sign of zero the same way for finite inputs
    assert np.array_equal(ours, lib)


# --------------------------------------------------------------------------- scales

def test_worked_example_group():
    g = read_golden("quant_worked_example.txt")
    x = np.zeros(128, dtype=np.float32)
    x[0], x[1], x[2], x[3] = 3.0, 1.0, -0.5, -3.0
    x[4] = 131 / 128 * 2.0 ** -10
    x[5] = -0.0
    xb = torch.from_numpy(x[None, :]).to(torch.bfloat16)
    assert float(xb[0, 4]) == x[4]
    q, s = oracle.quant_act_group(synth.bf16_bits(xb))
    assert s.shape == (1, 1)
    assert s.view(np.uint32)[0, 0] == int(g["scale_bits"], 16)
    for key, val in g.items():
        if key.isdigit():
            assert q[0, int(key)] == int(val, 16), key


def test_scale_fp32_closed_form():
    for amax in [448.0, 1.0, 3.0, 0.02, 1e-30, 3.0e38, 2.0 ** -133]:
        a32 = np.float32(amax)
        assert oracle.scale_fp32(a32) == np.float32(a32 / np.float32(448.0))
    assert oracle.scale_fp32(0.0) == 1.0


def test_scale_ue8m0_bounds():
    bits = np.arange(1, 0x7F80, dtype=np.uint32) << 16  # every positive finite bf16
    amaxes = bits.view(np.float32)[::7]
    for a in amaxes:
        e = oracle.scale_ue8m0_exponent(a)
        a = float(a)
        assert -127 <= e <= 127
        if e > -127:
            assert 448.0 * 2.0 ** e >= a > 448.0 * 2.0 ** (e - 1)
        else:
            assert 448.0 * 2.0 ** e >= a
    assert oracle.scale_ue8m0_exponent(448.0) == 0
    assert oracle.scale_ue8m0_exponent(449.0) == 1
    assert oracle.scale_ue8m0_exponent(224.0) == -1
    assert oracle.scale_ue8m0_exponent(0.0) == 0


# --------------------------------------------------------------------------- quantisers

def _blocky_weight(n, k, seed):
    """N(0, 0.02) weights with a distinct magnitude per 128x128 block, so that a
    transposed or shifted block index changes the scale."""
    w = synth.normal_bf16((n, k), 0.02, seed, "pin", n, k).float()
    for i in range((n + 127) // 128):
        for j in range((k + 127) // 128):
            w[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128] *= (1 + i) * (2 + 3 * j)
    return w.to(torch.bfloat16)


@pytest.mark.parametrize("n,k", [(256, 256), (384, 256), (200, 300), (1, 129), (130, 1)])
def test_weight_quant_scales_are_block_amax_over_448(n, k):
    w = _blocky_weight(n, k, 1)
    wf = w.float().numpy()
    q, s = oracle.quant_weight_blockwise(synth.bf16_bits(w))
    assert s.shape == ((n + 127) // 128, (k + 127) // 128)
    for i in range(s.shape[0]):
        for j in range(s.shape[1]):
            blk = wf[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
            amax = np.float32(np.abs(blk).max())
            assert s[i, j] == (np.float32(amax / np.float32(448)) if amax else np.float32(1))
            # invariant: the amax element maps to +-448 exactly
            r, c = np.unravel_index(np.abs(blk).argmax(), blk.shape)
            code = q[i * 128 + r, j * 128 + c]
            if amax:
                assert code in (0x7E, 0xFE)


def test_weight_quant_matches_library_cast_of_fp32_quotient():
    w = _blocky_weight(256, 384, 2)
    q, s = oracle.quant_weight_blockwise(synth.bf16_bits(w))
    wf = w.float().numpy()
    srep = np.repeat(np.repeat(s, 128, axis=0), 128, axis=1)[:256, :384]
    quotient = (wf / srep).astype(np.float32)  # IEEE fp32 division, element by element
    lib = torch.from_numpy(quotient).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(q, lib.numpy())


def test_weight_quant_error_bound():
    w = synth.weight_bf16(256, 384, 3, "pin-err")
    q, s = oracle.quant_weight_blockwise(synth.bf16_bits(w))
    table = oracle.e4m3_decode_table()
    x = w.double().numpy()
    srep = np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1)
    deq = table[q] * srep
    v = np.abs(x / srep)
    # spacing of the E4M3 codes around v: 2^-9 below 2^-6, else 2^(floor(log2 v) - 3)
    with np.errstate(divide="ignore"):
        ulp = np.where(v < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(v, 1e-300))) - 3))
    bound = 0.5 * ulp * srep + 2.0 ** -23 * np.abs(x)
    assert np.all(np.abs(deq - x) <= bound)


def test_all_zero_block_gets_unit_scale_and_zero_codes():
    w, _ = synth.tiny_linear(0)
    for fmt in (oracle.SCALE_FP32, oracle.SCALE_UE8M0):
        q, s = oracle.quant_weight_blockwise(synth.bf16_bits(w), fmt)
        assert np.all(q[0:128, 128:256] == 0)
        if fmt == oracle.SCALE_FP32:
            assert s[0, 1] == 1.0
        else:
            assert s[0, 1] == 127
        assert np.all(q[128:, :] != 0x7F) and np.all(q != 0xFF)


def test_negative_zero_inputs_give_0x80():
    x = torch.zeros((1, 128), dtype=torch.bfloat16)
    x[0, 5] = -0.0
    q, s = oracle.quant_act_group(synth.bf16_bits(x))
    assert q[0, 5] == 0x80 and np.count_nonzero(q) == 1 and s[0, 0] == 1.0


def test_ue8m0_quant_bounds_and_no_saturation():
    w = synth.weight_bf16(256, 256, 4, "pin-ue8m0")
    q, s = oracle.quant_weight_blockwise(synth.bf16_bits(w), oracle.SCALE_UE8M0)
    wf = w.float().numpy()
    table = oracle.e4m3_decode_table()
    for i in range(2):
        for j in range(2):
            blk = wf[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
            amax = float(np.abs(blk).max())
            sc = 2.0 ** (int(s[i, j]) - 127)
            assert sc >= amax / 448 > sc / 2
            qb = q[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
            # saturation only where the exact value is 448 itself
            sat = (qb & 0x7F) == 0x7E
            assert np.all(np.abs(blk[sat].astype(np.float64)) / sc == 448.0)
            # power-of-two scaling is exact, so the codes are the RNE of x / 2^e
            ref = brute_force_encode((blk.astype(np.float64) / sc).reshape(-1)).reshape(128, 128)
            assert np.array_equal(qb, ref)
            assert np.all(np.abs(table[qb] * sc - blk) <= 0.5 * 2.0 ** np.floor(
                np.log2(np.maximum(np.abs(blk) / sc, 2.0 ** -6))) / 8 * sc + 1e-30)


@pytest.mark.parametrize("m,k", [(16, 256), (5, 300), (1, 128), (3, 1)])
def test_act_quant_groups_along_k_with_group_major_scales(m, k):
    x = synth.activation_bf16(m, k, 5, "pin-act")
    xf = x.float().numpy() * (1 + np.arange(m))[:, None].astype(np.float32)
    x = torch.from_numpy(xf).to(torch.bfloat16)
    xf = x.float().numpy()
    q, s = oracle.quant_act_group(synth.bf16_bits(x))
    groups = (k + 127) // 128
    assert s.shape == (groups, m)
    for r in range(m):
        for g in range(groups):
            seg = xf[r, g * 128:(g + 1) * 128]
            amax = np.float32(np.abs(seg).max())
            exp = np.float32(amax / np.float32(448)) if amax else np.float32(1)
            assert s[g, r] == exp
            sq = (seg / exp).astype(np.float32)
            lib = torch.from_numpy(sq).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
            assert np.array_equal(q[r, g * 128:(g + 1) * 128], lib.numpy())


# --------------------------------------------------------------------------- GEMMs

def _integer_operands(m, n, k, seed):
    """E4M3 codes whose values are small integers and power-of-two scales, so
    that every product and partial sum is exact in fp64."""
    rng = np.random.default_rng(seed)
    table = oracle.e4m3_decode_table()
    int_codes = np.array([c for c in range(256)
                          if np.isfinite(table[c]) and table[c] == np.round(table[c])
                          and abs(table[c]) <= 16])
    xq = rng.choice(int_codes, size=(m, k)).astype(np.uint8)
    wq = rng.choice(int_codes, size=(n, k)).astype(np.uint8)
    sx = np.ldexp(1.0, rng.integers(-6, 7, size=(k // 128, m))).astype(np.float32)
    sw = np.ldexp(1.0, rng.integers(-6, 7, size=(n // 128, k // 128))).astype(np.float32)
    return xq, sx, wq, sw, table


def test_gemm_exact_against_integer_matmul():
    m, n, k = 5, 256, 384
    xq, sx, wq, sw, table = _integer_operands(m, n, k, 7)
    y = oracle.gemm_blockscaled(xq, sx, wq, sw)
    xi = table[xq].astype(np.int64)
    wi = table[wq].astype(np.int64)
    ref = np.zeros((m, n), dtype=np.float64)
    for kb in range(k // 128):
        part = xi[:, kb * 128:(kb + 1) * 128] @ wi[:, kb * 128:(kb + 1) * 128].T  # exact int64
        fac = sx[kb][:, None].astype(np.float64) * np.repeat(sw[:, kb], 128)[None, :]
        ref += part.astype(np.float64) * fac
    assert np.array_equal(y, ref)


def test_gemm_matches_library_matmul_of_dequantised_operands():
    m, n, k = 7, 384, 256
    x = synth.activation_bf16(m, k, 8, "pin-gemm")
    w = _blocky_weight(n, k, 9)
    xq, sx = oracle.quant_act_group(synth.bf16_bits(x))
    wq, sw = oracle.quant_weight_blockwise(synth.bf16_bits(w))
    y = oracle.gemm_blockscaled(xq, sx, wq, sw)
    xd = oracle.dequantize(xq, sx.T, 1, 128)
    wd = oracle.dequantize(wq, sw, 128, 128)
    ref = xd @ wd.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    # and it approximates the unquantised product (loosely: E4M3 has 3 mantissa bits)
    exact = x.double().numpy() @ w.double().numpy().T
    rel = np.linalg.norm(y - exact) / np.linalg.norm(exact)
    assert rel < 0.05


def test_gemm_identity_block_returns_dequantised_activations():
    m, k = 4, 128
    x = synth.activation_bf16(m, k, 10, "pin-id")
    xq, sx = oracle.quant_act_group(synth.bf16_bits(x))
    wq = np.zeros((128, 128), dtype=np.uint8)
    np.fill_diagonal(wq, 0x38)  # 1.0
    sw = np.ones((1, 1), dtype=np.float32)
    y = oracle.gemm_blockscaled(xq, sx, wq, sw)
    assert np.array_equal(y, oracle.dequantize(xq, sx.T, 1, 128))


def test_gemm_ue8m0_equals_fp32_with_same_powers_of_two():
    m, n, k = 3, 256, 256
    xq, sx, wq, sw, _ = _integer_operands(m, n, k, 11)
    ex = (np.log2(sx).astype(np.int64) + 127).astype(np.uint8)
    ew = (np.log2(sw).astype(np.int64) + 127).astype(np.uint8)
    y32 = oracle.gemm_blockscaled(xq, sx, wq, sw, oracle.SCALE_FP32)
    yu = oracle.gemm_blockscaled(xq, ex, wq, ew, oracle.SCALE_UE8M0)
    assert np.array_equal(y32, yu)


def test_gemm_sampled_positions_equal_full_product():
    m, n, k = 9, 256, 256
    xq, sx, wq, sw, _ = _integer_operands(m, n, k, 12)
    sx = sx * np.float32(1.37)  # non power of two
    y = oracle.gemm_blockscaled(xq, sx, wq, sw)
    rng = np.random.default_rng(0)
    rows = rng.integers(0, m, 50)
    cols = rng.integers(0, n, 50)
    at = oracle.gemm_blockscaled_at(xq, sx, wq, sw, rows, cols)
    assert np.array_equal(at, y[rows, cols])


def test_grouped_gemm_is_per_expert_gemm_with_empty_experts():
    n, k, e = 256, 256, 4
    counts = [3, 0, 5, 1]
    offsets = synth.routing_with_counts(counts)
    rows = int(offsets[-1])
    rng = np.random.default_rng(13)
    xq, sx, _, _, table = _integer_operands(rows, n, k, 14)
    wq = np.stack([_integer_operands(1, n, k, 20 + i)[2] for i in range(e)])
    sw = np.stack([_integer_operands(1, n, k, 30 + i)[3] for i in range(e)])
    y = oracle.grouped_gemm_blockscaled(xq, sx, wq, sw, offsets)
    for i in range(e):
        a, b = offsets[i], offsets[i + 1]
        if a == b:
            continue
        yi = oracle.gemm_blockscaled(xq[a:b], np.ascontiguousarray(sx[:, a:b]), wq[i], sw[i])
        assert np.array_equal(y[a:b], yi)
    rr = rng.integers(0, rows, 40)
    cc = rng.integers(0, n, 40)
    at = oracle.grouped_gemm_blockscaled_at(xq, sx, wq, sw, offsets, rr, cc)
    assert np.array_equal(at, y[rr, cc])


def test_grouped_gemm_rejects_bad_offsets():
    n = k = 128
    xq = np.zeros((4, k), np.uint8)
    sx = np.ones((1, 4), np.float32)
    wq = np.zeros((2, n, k), np.uint8)
    sw = np.ones((2, 1, 1), np.float32)
    with pytest.raises(ValueError):
        oracle.grouped_gemm_blockscaled(xq, sx, wq, sw, np.array([0, 3, 2], np.int32))
    with pytest.raises(ValueError):
        oracle.grouped_gemm_blockscaled(xq, sx, wq, sw, np.array([0, 1, 3], np.int32))


def test_routing_generator_draws_distinct_topk_with_normalised_gates():
    r = synth.moe_routing(tokens=64, experts=16, topk=4, seed=0)
    assert r.topk.shape == (64, 4) and r.gate.shape == (64, 4)
    assert all(len(set(row)) == 4 for row in r.topk.tolist())
    assert np.allclose(r.gate.sum(axis=1), 1.0, atol=1e-6)
    assert np.all(np.diff(r.gate, axis=1) <= 0)  # descending probability


# --------------------------------------------------------------------------- fused gate-up path (fp32 groups, SwiGLU)

def _fp32_groups(m, k, seed):
    """fp32 values with a wide per-row range and non-bf16 mantissas."""
    rng = np.random.default_rng(seed)
    x = rng.normal(size=(m, k)) * np.exp(rng.normal(size=(m, 1)) * 2.0)
    return x.astype(np.float32)


@pytest.mark.parametrize("m,k", [(4, 256), (3, 300), (2, 128), (1, 5)])
def test_fp32_group_quant_is_rne_of_fp32_quotient(m, k):
    """Codes = library RNE cast of the IEEE fp32 quotient x / s (R2, R3), with
    s = amax / 448 of each 1x128 group computed in fp32 by the library."""
    x = _fp32_groups(m, k, 11)
    q, s = oracle.quant_group_f32(x)
    groups = (k + 127) // 128
    assert s.shape == (groups, m)
    for g in range(groups):
        blk = x[:, g * 128:(g + 1) * 128]
        amax = np.abs(blk).max(axis=1).astype(np.float32)
        assert np.array_equal(s[g], np.where(amax == 0, np.float32(1), amax / np.float32(448)))
        quotient = (blk / s[g][:, None]).astype(np.float32)
        lib = torch.from_numpy(quotient).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        assert np.array_equal(q[:, g * 128:(g + 1) * 128], lib.numpy())


def test_fp32_group_quant_amax_maps_to_448_and_error_bound():
    x = _fp32_groups(8, 384, 12)
    q, s = oracle.quant_group_f32(x)
    table = oracle.e4m3_decode_table()
    srep = np.repeat(s.T.astype(np.float64), 128, axis=1)
    for r in range(8):
        for g in range(3):
            c = int(np.argmax(np.abs(x[r, g * 128:(g + 1) * 128]))) + g * 128
            assert q[r, c] & 0x7F == 0x7E  # the group maximum is exactly +-448
    v = np.abs(x.astype(np.float64) / srep)
    with np.errstate(divide="ignore"):
        ulp = np.where(v < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(v, 1e-300))) - 3))
    assert np.all(np.abs(table[q] * srep - x) <= 0.5 * ulp * srep + 2.0 ** -23 * np.abs(x))


def test_fp32_group_quant_zero_group_and_ue8m0_bounds():
    x = _fp32_groups(3, 256, 13)
    x[1, 128:] = 0.0
    q, s = oracle.quant_group_f32(x)
    assert s[1, 1] == 1.0 and np.all(q[1, 128:] == 0)
    qu, su = oracle.quant_group_f32(x, oracle.SCALE_UE8M0)
    assert su[1, 1] == 127 and np.all(qu[1, 128:] == 0)
    for r in (0, 2):
        for g in range(2):
            blk = x[r, g * 128:(g + 1) * 128].astype(np.float64)
            sc = 2.0 ** (int(su[g, r]) - 127)
            assert sc >= np.abs(blk).max() / 448 > sc / 2
            assert np.array_equal(qu[r, g * 128:(g + 1) * 128], brute_force_encode(blk / sc))


def test_silu_closed_forms():
    x = np.linspace(-30.0, 30.0, 601)
    # x sigmoid(x) - (-x) sigmoid(-x) = x (sigmoid(x) + sigmoid(-x) = 1)
    assert np.allclose(oracle.silu(x) - oracle.silu(-x), x, rtol=0, atol=1e-12)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert oracle.silu(np.array([1.0]))[0] == pytest.approx(math.e / (1.0 + math.e), rel=1e-15)
    assert oracle.silu(np.array([60.0]))[0] == pytest.approx(60.0, rel=1e-15)
    assert abs(oracle.silu(np.array([-800.0]))[0]) == 0.0
    up = np.array([2.0, -3.0, 0.5])
    gate = np.array([1.0, 0.0, -1.0])
    assert np.allclose(oracle.swiglu(gate, up), up * gate / (1.0 + np.exp(-gate)), rtol=1e-15)


def test_gate_up_interleave_is_a_row_permutation_in_128_blocks():
    order = oracle.interleave_gate_up_rows(768)
    assert sorted(order.tolist()) == list(range(768))
    # blocks alternate: gate block b, then up block b
    assert np.array_equal(order[:128], np.arange(128))
    assert np.array_equal(order[128:256], 384 + np.arange(128))
    assert np.array_equal(order[256:384], 128 + np.arange(128))
    assert np.array_equal(order[640:768], 384 + 256 + np.arange(128))


def test_fused_reference_equals_unfused_steps():
    """gemm_swiglu_quant on the interleaved weight = the plain GEMM on [gate; up],
    SiLU(gate) * up, fp32 rounding, group quantisation (each step by hand)."""
    rng = np.random.default_rng(14)
    m, k, inter = 40, 256, 256
    x = torch.from_numpy(rng.normal(size=(m, k)).astype(np.float32)).to(torch.bfloat16)
    w = torch.from_numpy((rng.normal(size=(2 * inter, k)) * 0.05).astype(np.float32)).to(torch.bfloat16)
    xq, sx = oracle.quant_act_group(synth.bf16_bits(x))
    order = oracle.interleave_gate_up_rows(2 * inter)
    wq, sw = oracle.quant_weight_blockwise(synth.bf16_bits(w[torch.from_numpy(order)]))
    h, hq, hs = oracle.gemm_swiglu_quant(xq, sx, wq, sw)
    wq_plain, sw_plain = oracle.quant_weight_blockwise(synth.bf16_bits(w))
    y = oracle.gemm_blockscaled(xq, sx, wq_plain, sw_plain)
    gate, up = y[:, :inter], y[:, inter:]
    h_ref = gate / (1.0 + np.exp(-gate)) * up
    assert np.allclose(h, h_ref, rtol=1e-14, atol=0)
    hq_ref, hs_ref = oracle.quant_group_f32(h_ref.astype(np.float32))
    assert np.array_equal(hq, hq_ref) and np.array_equal(hs, hs_ref)


# --------------------------------------------------------------------------- KV cache (per-step calibration, append)

def _kv(tokens, dim, seed, spread=1.0):
    rng = np.random.default_rng(seed)
    x = rng.normal(size=(tokens, dim)) * spread
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)


def test_kv_calibrate_is_tensor_amax_over_448():
    k, v, q = _kv(50, 256, 21), _kv(50, 256, 22, 3.0), _kv(50, 512, 23, 0.1)
    s = oracle.kv_calibrate(synth.bf16_bits(k), synth.bf16_bits(v), synth.bf16_bits(q))
    for i, t in enumerate((k, v, q)):
        amax = np.float32(t.float().abs().max().item())
        assert s[i] == amax / np.float32(448)
    s0 = oracle.kv_calibrate(synth.bf16_bits(torch.zeros_like(k)), synth.bf16_bits(v))
    assert s0[0] == 1.0 and s0[2] == 0.0


def test_kv_append_codes_slots_and_saturation():
    tokens, dim, slots_total = 40, 256, 64
    k, v = _kv(tokens, dim, 24), _kv(tokens, dim, 25, 2.0)
    s = oracle.kv_calibrate(synth.bf16_bits(k[:20]), synth.bf16_bits(v[:20]))  # calibrated on a prefix
    rng = np.random.default_rng(26)
    slots = rng.permutation(slots_total)[:tokens].astype(np.int32)
    slots[3] = -1        # padding
    slots[7] = 10 ** 6   # outside the cache
    kc = np.full((slots_total, dim), 0x55, np.uint8)
    vc = np.full((slots_total, dim), 0x55, np.uint8)
    oracle.kv_append(synth.bf16_bits(k), synth.bf16_bits(v), slots, kc, vc, s)
    for cache, x, sc in ((kc, k, s[0]), (vc, v, s[1])):
        quotient = (x.float().numpy() / np.float32(sc)).astype(np.float32)  # IEEE fp32 division
        lib = torch.from_numpy(quotient).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        for t in range(tokens):
            if 0 <= slots[t] < slots_total:
                assert np.array_equal(cache[slots[t]], lib[t])
        untouched = np.setdiff1d(np.arange(slots_total), slots[(slots >= 0) & (slots < slots_total)])
        assert np.all(cache[untouched] == 0x55)
    # tokens after the calibration prefix may exceed its range: they saturate
    beyond = np.abs(k.float().numpy()) / s[0] > 448
    if beyond.any():
        t, c = np.argwhere(beyond)[0]
        assert kc[slots[t], c] & 0x7F == 0x7E
    # the calibration tensor's own maximum maps to exactly +-448
    t, c = np.unravel_index(np.argmax(np.abs(k[:20].float().numpy())), (20, dim))
    if 0 <= slots[t] < slots_total:
        assert kc[slots[t], c] & 0x7F == 0x7E


# --------------------------------------------------------------------------- MoE dispatch / combine (routing replay)

def _golden_list(g, key, dtype):
    return np.array([dtype(v) for v in g[key].split(",")])


def test_dispatch_plan_and_combine_worked_example():
    g = read_golden("moe_dispatch_worked_example.txt")
    idx = _golden_list(g, "indices", int).reshape(4, 2)
    off, rop, tor = oracle.moe_dispatch_plan(idx, int(g["experts"]))
    assert off.tolist() == _golden_list(g, "offsets", int).tolist()
    assert rop.tolist() == _golden_list(g, "row_of_pair", int).tolist()
    assert tor.tolist() == _golden_list(g, "token_of_row", int).tolist()
    y = np.array([[r + 1, -(r + 1) / 2] for r in range(8)])
    out = oracle.moe_combine(y, rop, _golden_list(g, "gate", float).reshape(4, 2))
    assert out.reshape(-1).tolist() == _golden_list(g, "combine_out", float).tolist()


@pytest.mark.parametrize("tokens,k,experts,drop", [(64, 8, 16, 0.0), (37, 3, 5, 0.2), (1, 1, 1, 0.0), (0, 8, 4, 0.0)])
def test_dispatch_plan_is_the_stable_sort_by_expert(tokens, k, experts, drop):
    """Equal to numpy's stable argsort of the flattened expert ids (the
    special case the plan reduces to), with dropped pairs left out."""
    rng = np.random.default_rng(tokens * 7 + k)
    idx = rng.integers(0, experts, size=(tokens, k))
    idx[rng.random((tokens, k)) < drop] = -1
    idx[rng.random((tokens, k)) < drop / 2] = experts + 3  # also out of range
    off, rop, tor = oracle.moe_dispatch_plan(idx, experts)
    flat = idx.reshape(-1)
    live = np.flatnonzero((flat >= 0) & (flat < experts))
    order = live[np.argsort(flat[live], kind="stable")]
    assert np.array_equal(np.diff(off), np.bincount(flat[live], minlength=experts))
    assert off[-1] == live.size
    assert np.array_equal(rop[order], np.arange(live.size))  # pair -> row
    assert np.all(rop[np.setdiff1d(np.arange(flat.size), live)] == -1)
    assert np.array_equal(tor[:live.size], order // k) and np.all(tor[live.size:] == -1)


def test_dispatch_quant_rows_equal_each_token_row_quantised_alone():
    tokens, k, experts, hidden = 12, 3, 5, 300
    rng = np.random.default_rng(3)
    idx = rng.integers(-1, experts, size=(tokens, k))
    x = synth.normal_bf16((tokens, hidden), 1.0, 7, "pin-dispatch")
    xb = synth.bf16_bits(x)
    _, _, tor = oracle.moe_dispatch_plan(idx, experts)
    q, s, live = oracle.moe_dispatch_quant(xb, tor)
    for r in np.flatnonzero(live):
        qr, sr = oracle.quant_act_group(xb[tor[r]:tor[r] + 1])
        assert np.array_equal(q[r], qr[0]) and np.array_equal(s[:, r], sr[:, 0])


def test_combine_one_hot_selects_rows_and_ignores_slot_order():
    tokens, k, experts, n = 10, 4, 6, 7
    rng = np.random.default_rng(4)
    idx = np.stack([rng.permutation(experts)[:k] for _ in range(tokens)])
    _, rop, _ = oracle.moe_dispatch_plan(idx, experts)
    y = rng.standard_normal((tokens * k, n))
    hot = np.zeros((tokens, k))
    hot[np.arange(tokens), rng.integers(0, k, tokens)] = 1.0
    out = oracle.moe_combine(y, rop, hot)
    sel = rop.reshape(tokens, k)[hot == 1]
    assert np.array_equal(out, y[sel])
    # permuting each token's slots (indices and gates together) changes nothing but rounding
    gate = rng.random((tokens, k))
    perm = np.stack([rng.permutation(k) for _ in range(tokens)])
    _, rop_p, _ = oracle.moe_dispatch_plan(np.take_along_axis(idx, perm, 1), experts)
    # the same (token, expert) pair owns the same row in both plans, as rows
    # are ordered by token within a segment and a token holds an expert once
    a = oracle.moe_combine(y, rop, gate)
    b = oracle.moe_combine(y, rop_p, np.take_along_axis(gate, perm, 1))
    assert np.allclose(a, b, rtol=1e-14, atol=1e-14)


def test_dispatch_then_identity_experts_then_combine_returns_tokens():
    """With every expert the identity and gates summing to 1, the round trip
    gives back each token row up to its 1x128 quantisation error."""
    tokens, k, experts, hidden = 16, 4, 8, 256
    r = synth.moe_routing(tokens, experts, k, seed=5)
    x = synth.normal_bf16((tokens, hidden), 1.0, 8, "pin-roundtrip")
    xb = synth.bf16_bits(x)
    _, rop, tor = oracle.moe_dispatch_plan(r.topk, experts)
    q, s, _ = oracle.moe_dispatch_quant(xb, tor)
    y = oracle.dequantize(q, s.T, 1, 128)
    out = oracle.moe_combine(y, rop, r.gate.astype(np.float64))
    xf = x.float().numpy().astype(np.float64)
    # per element: half an E4M3 ulp at that magnitude (<= 2^-4 relative) times
    # the weight, plus the subnormal floor scale * 2^-10, summed over slots
    smax = s.max()
    assert np.all(np.abs(out - xf) <= 2.0 ** -4 * np.abs(xf) + smax * 2.0 ** -10 + 1e-6)


# --------------------------------------------------------------------------- TIS weight and mismatch KL

def test_tis_weight_closed_forms_and_truncation():
    lr = np.zeros(6, np.float32)
    lt = np.array([0.0, math.log(1.5), math.log(3.0), -50.0, math.log(2.0) + 1e-3, 10.0], np.float32)
    w = oracle.tis_weights(lt, lr)
    assert w[0] == 1.0
    assert abs(w[1] - 1.5) < 1e-6 and w[2] == 2.0 and w[4] == 2.0 and w[5] == 2.0
    assert abs(w[3] - math.exp(-50.0)) < 1e-30
    # the ratio of probabilities, not of log-probabilities: shifting both sides
    # by the same amount leaves it unchanged
    assert np.allclose(oracle.tis_weights(lt - 3.0, lr - 3.0), w, rtol=1e-6)
    # masked-out tokens weigh 0
    mask = np.array([1, 0, 1, 0, 1, 1], np.uint8)
    assert np.array_equal(oracle.tis_weights(lt, lr, mask), np.where(mask == 1, w, 0.0))


def test_mismatch_kl_constant_gap_mask_and_empty():
    lt = np.full(10, -2.0, np.float32)
    lr = np.full(10, -1.75, np.float32)
    mean, total, count = oracle.mismatch_kl(lt, lr)
    assert (mean, total, count) == (0.25, 2.5, 10)
    mask = np.zeros(10, np.uint8)
    assert oracle.mismatch_kl(lt, lr, mask) == (0.0, 0.0, 0)
    mask[[1, 4]] = 1
    lr2 = lr.copy()
    lr2[0] = 100.0  # masked out: no effect
    assert oracle.mismatch_kl(lt, lr2, mask) == (0.25, 0.5, 2)


def test_mismatch_kl_estimates_kl_of_rollout_from_training_policy():
    """Tokens sampled from the rollout policy p: the mean of log p - log q
    converges to KL(p || q), a closed form over the vocabulary."""
    rng = np.random.default_rng(11)
    vocab, n = 50, 400_000
    p = rng.dirichlet(np.ones(vocab))
    q = 0.8 * p + 0.2 * rng.dirichlet(np.ones(vocab))
    kl = float(np.sum(p * (np.log(p) - np.log(q))))
    tok = rng.choice(vocab, size=n, p=p)
    mean, _, count = oracle.mismatch_kl(np.log(q)[tok], np.log(p)[tok])
    sd = float(np.std(np.log(p)[tok] - np.log(q)[tok]))
    assert count == n and abs(mean - kl) < 5 * sd / math.sqrt(n)
