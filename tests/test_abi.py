"""The C ABI library builds, loads and exports every declared entry point, and
rejects bad arguments on the host before touching the GPU.  CPU only: no call
here reaches a kernel launch."""
import ctypes
import os
import re
import subprocess

import pytest

import fp8_w8a8_rollout_gb300 as fp8rl
from fp8_w8a8_rollout_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_entry_points():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"FP8RL_API\s+[\w\s\*]+?\b(fp8rl_\w+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return fp8rl.load_library()


def test_header_declares_the_path_entry_points():
    names = declared_entry_points()
    for required in ("fp8rl_quant_weight_blockwise", "fp8rl_quant_act_group",
                     "fp8rl_gemm_blockscaled", "fp8rl_grouped_gemm_blockscaled",
                     "fp8rl_quant_weight_blockwise_batched", "fp8rl_sync_status",
                     "fp8rl_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(fp8rl_\w+)", out))
    declared = set(declared_entry_points())
    assert declared <= exported, declared - exported
    for name in declared:
        assert hasattr(lib, name)


def declarations():
    """{name: (return type, [parameter declarations])} of every FP8RL_API
    function in include/*.h."""
    out = {}
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        for ret, name, params in re.findall(r"FP8RL_API\s+([\w\s\*]+?)\b(fp8rl_\w+)\s*\(([^)]*)\)\s*;", text):
            ps = [re.sub(r"\s+", " ", q).strip() for q in params.split(",") if q.strip()]
            out[name] = (re.sub(r"\s+", " ", ret).strip(), [] if ps == ["void"] else ps)
    return out


def _c_type(param):
    """The type of a parameter declaration ('const void* w_bf16' -> 'const void*')."""
    m = re.match(r"^(.*?[\s\*])(\w+)$", param)
    assert m, param
    return m.group(1).strip()


def _ctype_matches(c, ct):
    """Does ctypes type `ct` pass / return C type `c` correctly on this ABI?"""
    c = c.replace("const ", "").replace(" *", "*").strip()
    if c.endswith("*"):
        if c == "char*":
            return ct is ctypes.c_char_p
        return ct is ctypes.c_void_p or (isinstance(ct, type) and issubclass(ct, ctypes._Pointer))
    if c in ("float", "double"):
        return ct is {"float": ctypes.c_float, "double": ctypes.c_double}[c]
    width = {"int64_t": 8, "int32_t": 4, "size_t": 8, "fp8rl_scale_fmt": 4, "fp8rl_status": 4}[c]
    if ct is None or not issubclass(ct, ctypes._SimpleCData):
        return False
    if ct in (ctypes.c_float, ctypes.c_double, ctypes.c_void_p, ctypes.c_char_p, ctypes.c_bool):
        return False
    unsigned = ct(-1).value > 0
    return ctypes.sizeof(ct) == width and unsigned == (c == "size_t")


def test_binding_signatures_match_the_header(lib):
    """ctypes checks no argument list against the C one: every entry point's
    argtypes and restype in the binding must agree with its declaration (count,
    pointer or value, integer width and signedness, float width)."""
    decls = declarations()
    assert len(decls) >= 20
    for name, (ret, params) in decls.items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None, f"{name}: no argtypes in the binding"
        assert len(fn.argtypes) == len(params), (name, len(fn.argtypes), params)
        for i, (decl, ct) in enumerate(zip(params, fn.argtypes)):
            assert _ctype_matches(_c_type(decl), ct), (name, i, decl, ct)
        assert _ctype_matches(ret, fn.restype), (name, ret, fn.restype)


def test_weight_descriptor_layout_matches_the_header():
    """fp8rl_weight_desc and the binding's WeightDesc list the same members
    in the same order with the same types (so the same layout on this ABI)."""
    text = open(os.path.join(ROOT, "include", "fp8rl.h")).read()
    body = re.search(r"typedef struct \{(.*?)\} fp8rl_weight_desc;", text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    members = []
    for stmt in body.split(";"):
        stmt = " ".join(stmt.split())
        if not stmt:
            continue
        m = re.match(r"^(const )?(\w+)(\*?)\s*(.*)$", stmt.replace("* ", "*").replace(" *", "*"))
        ctype = m.group(2) + m.group(3)
        for field in m.group(4).split(","):
            members.append((field.strip().lstrip("*"), ctype))
    fields = fp8rl.WeightDesc._fields_
    assert [n for n, _ in fields] == [n for n, _ in members]
    for (fname, ct), (_, ctype) in zip(fields, members):
        assert _ctype_matches(ctype, ct), (fname, ctype, ct)


def test_library_targets_sm103a_only():
    # the build passes exactly one -gencode, for sm_103a
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings(lib):
    for code, name in fp8rl.STATUS.items():
        assert fp8rl.fp8rl_status_string(code) == name
    assert fp8rl.fp8rl_version() >= 100


def _rc(fn, *args):
    return getattr(fp8rl.load_library(), fn)(*args)


def test_weight_quant_rejects_bad_arguments_on_host(lib):
    a16 = 1 << 20  # an aligned fake address (never dereferenced: validation fails first)
    # null pointers
    assert _rc("fp8rl_quant_weight_blockwise", None, 128, 128, 128, a16, 128, a16, 0, None) == 1
    # negative sizes, short leading dimensions, unknown format
    assert _rc("fp8rl_quant_weight_blockwise", a16, -1, 128, 128, a16, 128, a16, 0, None) == 1
    assert _rc("fp8rl_quant_weight_blockwise", a16, 128, 128, 64, a16, 128, a16, 0, None) == 1
    assert _rc("fp8rl_quant_weight_blockwise", a16, 128, 128, 128, a16, 128, a16, 7, None) == 1
    # misaligned pointers
    assert _rc("fp8rl_quant_weight_blockwise", a16 + 2, 128, 128, 128, a16, 128, a16, 0, None) == 3
    assert _rc("fp8rl_quant_weight_blockwise", a16, 128, 128, 128, a16 + 1, 128, a16, 0, None) == 3
    assert _rc("fp8rl_quant_weight_blockwise", a16, 128, 128, 128, a16, 128, a16 + 2, 0, None) == 3
    # empty work is fine and launches nothing
    assert _rc("fp8rl_quant_weight_blockwise", None, 0, 128, 128, None, 128, None, 0, None) == 0


def test_act_quant_rejects_bad_arguments_on_host(lib):
    a16 = 1 << 20
    assert _rc("fp8rl_quant_act_group", None, 16, 256, 256, a16, 256, a16, 0, None) == 1
    assert _rc("fp8rl_quant_act_group", a16 + 8, 16, 256, 256, a16, 256, a16, 0, None) == 3
    assert _rc("fp8rl_quant_act_group", a16, 0, 256, 256, a16, 256, a16, 0, None) == 0


def test_batched_rejects_bad_descriptors(lib):
    a16 = 1 << 20
    descs = (fp8rl.WeightDesc * 2)()
    descs[0] = fp8rl.WeightDesc(a16, a16, a16, 128, 128, 128, 128)
    descs[1] = fp8rl.WeightDesc(a16 + 2, a16, a16, 128, 128, 128, 128)
    assert _rc("fp8rl_quant_weight_blockwise_batched", descs, 2, 0, None) == 3
    assert _rc("fp8rl_quant_weight_blockwise_batched", None, 1, 0, None) == 1
    assert _rc("fp8rl_quant_weight_blockwise_batched", descs, -1, 0, None) == 1
    assert _rc("fp8rl_quant_weight_blockwise_batched", descs, 0, 0, None) == 0


def test_gemm_rejects_bad_shapes_and_alignment_on_host(lib):
    a16 = 1 << 20
    g = "fp8rl_gemm_blockscaled"
    assert _rc(g, None, a16, a16, a16, a16, 16, 256, 256, 0, None) == 1
    assert _rc(g, a16, a16, a16, a16, a16, 16, 200, 256, 0, None) == 2  # n % 128
    assert _rc(g, a16, a16, a16, a16, a16, 16, 256, 300, 0, None) == 2  # k % 128
    assert _rc(g, a16, a16, a16, a16, a16, -1, 256, 256, 0, None) == 1
    assert _rc(g, a16 + 8, a16, a16, a16, a16, 16, 256, 256, 0, None) == 3
    assert _rc(g, a16, a16, a16, a16, a16 + 2, 16, 256, 256, 0, None) == 3
    assert _rc(g, a16, a16, a16, a16, a16, 16, 256, 256, 9, None) == 1
    assert _rc(g, a16, a16, a16, a16, a16, 0, 256, 256, 0, None) == 0  # m == 0: no-op


def test_act_quant_gemm_rejects_bad_arguments_on_host(lib):
    """fp8rl_gemm_act_quant(x, ldx, wq, w_scale, y, m, n, k, fmt, xq, x_scale,
    stream): the GEMM's checks on its X operands (xq, x_scale), plus x and
    ldx; nothing is launched."""
    a16 = 1 << 20
    g = "fp8rl_gemm_act_quant"
    assert _rc(g, None, 256, a16, a16, a16, 16, 256, 256, 0, a16, a16, None) == 1  # x null
    assert _rc(g, a16, 200, a16, a16, a16, 16, 256, 256, 0, a16, a16, None) == 1  # ldx < k
    assert _rc(g, a16 + 1, 256, a16, a16, a16, 16, 256, 256, 0, a16, a16, None) == 3  # x not 2-byte aligned
    assert _rc(g, a16, 256, a16, a16, a16, 16, 256, 256, 0, None, a16, None) == 1  # xq null
    assert _rc(g, a16, 256, a16, a16, a16, 16, 256, 256, 0, a16 + 8, a16, None) == 3  # xq alignment
    assert _rc(g, a16, 256, a16, a16, a16, 16, 200, 256, 0, a16, a16, None) == 2  # n % 128
    assert _rc(g, a16, 256, a16, a16, a16, 16, 256, 256, 7, a16, a16, None) == 1  # fmt
    assert _rc(g, a16, 256, a16, a16, a16, 0, 256, 256, 0, a16, a16, None) == 0  # m == 0: no-op


def test_workspace_gemm_rejects_bad_arguments_on_host(lib):
    a16 = 1 << 20
    g = "fp8rl_gemm_blockscaled_ws"
    # a null or misaligned workspace, then the checks shared with the plain GEMM
    assert _rc(g, a16, a16, a16, a16, a16, 16, 256, 256, 0, None, 1 << 30, None) == 1
    assert _rc(g, a16, a16, a16, a16, a16, 16, 256, 256, 0, a16 + 16, 1 << 30, None) == 3
    assert _rc(g, a16, a16, a16, a16, a16, 16, 200, 256, 0, a16, 1 << 30, None) == 2
    assert _rc(g, a16, a16, a16, a16, a16, 0, 256, 256, 0, a16, 0, None) == 0  # m == 0: no-op
    assert _rc("fp8rl_gemm_workspace_size", None) == 1


def test_fused_gate_up_rejects_bad_arguments_on_host(lib):
    a16 = 1 << 20
    g = "fp8rl_gemm_swiglu_quant"
    assert _rc(g, None, a16, a16, a16, 16, 128, 256, a16, a16, 0, None) == 1
    assert _rc(g, a16, a16, a16, a16, 16, 100, 256, a16, a16, 0, None) == 2   # inter % 128
    assert _rc(g, a16, a16, a16, a16, 16, 128, 200, a16, a16, 0, None) == 2   # k % 128
    assert _rc(g, a16, a16, a16, a16, 16, 128, 256, a16 + 8, a16, 0, None) == 3  # hq alignment
    assert _rc(g, a16, a16, a16, a16, 16, 128, 256, a16, None, 0, None) == 1
    assert _rc(g, a16, a16, a16, a16, 0, 128, 256, a16, a16, 0, None) == 0    # m == 0: no-op
    gg = "fp8rl_grouped_gemm_swiglu_quant"
    assert _rc(gg, a16, a16, a16, a16, None, 4, 64, 128, 256, a16, a16, 0, None) == 1
    assert _rc(gg, a16, a16, a16, a16, a16, 4, 64, 100, 256, a16, a16, 0, None) == 2
    assert _rc(gg, a16, a16, a16, a16, a16, 4, 0, 128, 256, a16, a16, 0, None) == 0


def test_grouped_gemm_rejects_bad_arguments_on_host(lib):
    a16 = 1 << 20
    g = "fp8rl_grouped_gemm_blockscaled"
    assert _rc(g, a16, a16, a16, a16, None, 4, 64, 256, 256, a16, 0, None) == 1
    assert _rc(g, a16, a16, a16, a16, a16, 0, 64, 256, 256, a16, 0, None) == 1
    assert _rc(g, a16, a16, a16, a16, a16, 4, 64, 200, 256, a16, 0, None) == 2
    assert _rc(g, a16, a16, a16, a16, a16, 4, 64, 256, 256, a16 + 4, 0, None) == 3
    assert _rc(g, a16, a16, a16, a16, a16, 4, 0, 256, 256, a16, 0, None) == 0


def test_codec_entry_rejects_bad_arguments(lib):
    assert _rc("fp8rl_e4m3_encode", None, 10, None, None) == 1
    assert _rc("fp8rl_e4m3_encode", (1 << 20) + 2, 10, 1 << 20, None) == 3
    assert _rc("fp8rl_e4m3_encode", None, 0, None, None) == 0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_build, "LIB", str(tmp_path / "nope.so"))
    monkeypatch.setattr(fp8rl, "_lib", None)
    with pytest.raises(FileNotFoundError):
        fp8rl.load_library()


def test_debug_hook_validates_on_host(lib):
    assert _rc("fp8rl_debug_set", 1, 96) == 1
    assert _rc("fp8rl_debug_set", 3, 0) == 1
    assert _rc("fp8rl_debug_set", 99, 0) == 1
    assert _rc("fp8rl_debug_set", 6, 9) == 1
    assert _rc("fp8rl_debug_set", 6, 4) == 0
    assert _rc("fp8rl_debug_set", 7, 3) == 1
    assert _rc("fp8rl_debug_set", 8, 1025) == 1
    assert _rc("fp8rl_debug_set", 7, 2) == 0
    assert _rc("fp8rl_debug_set", 8, 7) == 0
    assert _rc("fp8rl_debug_set", 9, 3) == 1
    assert _rc("fp8rl_debug_set", 9, 1) == 0
    assert _rc("fp8rl_debug_set", 10, 3) == 1
    assert _rc("fp8rl_debug_set", 10, 2) == 0
    assert _rc("fp8rl_debug_set", 11, 3) == 1
    assert _rc("fp8rl_debug_set", 11, 2) == 0
    assert _rc("fp8rl_debug_set", 11, 1) == 0
    assert _rc("fp8rl_debug_set", 12, 3) == 1
    assert _rc("fp8rl_debug_set", 12, 1) == 0
    assert _rc("fp8rl_debug_set", 13, 2) == 1
    assert _rc("fp8rl_debug_set", 13, 1) == 0
    assert _rc("fp8rl_debug_set", 1, 256) == 0
    assert _rc("fp8rl_debug_set", 0, 0) == 0


def test_debug_hooks_refused_unless_enabled(lib, monkeypatch):
    """Without FP8RL_TEST_HOOKS=1 in the environment every hook but the reset
    is refused (UNSUPPORTED), whatever its value."""
    monkeypatch.delenv("FP8RL_TEST_HOOKS", raising=False)
    for key, value in ((1, 256), (2, 3), (3, 1000), (6, 4), (7, 2), (10, 1)):
        assert _rc("fp8rl_debug_set", key, value) == 4
    monkeypatch.setenv("FP8RL_TEST_HOOKS", "0")
    assert _rc("fp8rl_debug_set", 1, 256) == 4
    assert _rc("fp8rl_debug_set", 0, 0) == 0
    monkeypatch.setenv("FP8RL_TEST_HOOKS", "1")
    assert _rc("fp8rl_debug_set", 1, 256) == 0
    assert _rc("fp8rl_debug_set", 0, 0) == 0


def test_moe_plan_rejects_bad_arguments_on_host(lib):
    ws = lib.fp8rl_moe_plan_workspace_size(4096, 8, 128)
    assert ws >= 4 * 128 and ws % 256 == 0
    assert lib.fp8rl_moe_plan_workspace_size(16, 0, 8) == 0      # topk < 1
    assert lib.fp8rl_moe_plan_workspace_size(16, 33, 8) == 0     # topk > 32
    assert lib.fp8rl_moe_plan_workspace_size(16, 8, 8193) == 0   # too many experts
    fake = 1 << 20  # never dereferenced: every call below fails validation first
    assert _rc("fp8rl_moe_plan", fake, 16, 0, 8, fake, fake, fake, fake, ws, None) == 1
    assert _rc("fp8rl_moe_plan", fake, 16, 8, 0, fake, fake, fake, fake, ws, None) == 1
    assert _rc("fp8rl_moe_plan", fake, 16, 8, 9000, fake, fake, fake, fake, ws, None) == 2
    assert _rc("fp8rl_moe_plan", fake, 1 << 28, 8, 8, fake, fake, fake, fake, ws, None) == 2
    assert _rc("fp8rl_moe_plan", None, 16, 8, 8, fake, fake, fake, fake, ws, None) == 1
    assert _rc("fp8rl_moe_plan", fake, 16, 8, 8, fake, fake, fake, fake, 0, None) == 1  # workspace too small
    small = lib.fp8rl_moe_plan_workspace_size(16, 8, 8)
    assert _rc("fp8rl_moe_plan", fake + 2, 16, 8, 8, fake, fake, fake, fake, small, None) == 3


def test_moe_dispatch_and_combine_reject_bad_arguments_on_host(lib):
    fake = 1 << 20
    q = "fp8rl_moe_dispatch_quant"
    assert _rc(q, fake, 16, 256, 256, fake, 8, 128, fake, 256, fake, 2, None) == 1  # bad format
    assert _rc(q, fake, 16, 256, 100, fake, 8, 128, fake, 256, fake, 0, None) == 1  # ldx < k
    assert _rc(q, fake, 16, 256, 256, fake, 33, 128, fake, 256, fake, 0, None) == 1  # topk > 32
    assert _rc(q, fake, 16, 256, 256, None, 8, 128, fake, 256, fake, 0, None) == 1
    assert _rc(q, fake + 8, 16, 256, 256, fake, 8, 128, fake, 256, fake, 0, None) == 3
    assert _rc(q, fake, 16, 256, 256, fake, 8, 0, fake, 256, fake, 0, None) == 0  # no rows: no-op
    c = "fp8rl_moe_combine"
    assert _rc(c, fake, 128, 256, 256, fake, fake, 16, 0, fake, 256, None) == 1    # topk < 1
    assert _rc(c, fake, 128, 256, 128, fake, fake, 16, 8, fake, 256, None) == 1    # ldy < n
    assert _rc(c, fake, -1, 256, 256, fake, fake, 16, 8, fake, 256, None) == 1     # rows < 0
    assert _rc(c, None, 128, 256, 256, fake, fake, 16, 8, fake, 256, None) == 1    # rows > 0, no y
    assert _rc(c, fake, 1 << 31, 256, 256, fake, fake, 16, 8, fake, 256, None) == 2  # rows >= 2^31
    assert _rc(c, fake + 1, 128, 256, 256, fake, fake, 16, 8, fake, 256, None) == 3
    assert _rc(c, fake, 128, 256, 256, fake, fake, 0, 8, fake, 256, None) == 0     # no tokens: no-op


def test_tis_rejects_bad_arguments_on_host(lib):
    fake = 1 << 20
    ws = lib.fp8rl_tis_workspace_size(1 << 24)
    assert ws >= 16 and lib.fp8rl_tis_workspace_size(-1) == 0
    t = "fp8rl_tis_weights"
    assert _rc(t, fake, fake, None, -1, 2.0, fake, fake, fake, ws, None) == 1
    assert _rc(t, fake, fake, None, 1 << 24, 0.0, fake, fake, fake, ws, None) == 1   # clip <= 0
    assert _rc(t, fake, fake, None, 1 << 24, 2.0, fake, None, fake, ws, None) == 1   # no output
    assert _rc(t, fake, fake, None, 1 << 24, 2.0, fake, fake, fake, 8, None) == 1    # workspace too small
    assert _rc(t, fake + 2, fake, None, 1 << 24, 2.0, fake, fake, fake, ws, None) == 3


def test_kv_rejects_bad_arguments_on_host(lib):
    fake = 1 << 20  # never dereferenced: every call below fails validation first (or has no work)
    c = "fp8rl_kv_calibrate"
    assert _rc(c, fake, fake, fake, -1, 1024, 1024, 1024, 4096, 4096, fake, None) == 1    # tokens < 0
    assert _rc(c, fake, fake, fake, 16, 1024, 1000, 1024, 4096, 4096, fake, None) == 1    # ldk < kv_dim
    assert _rc(c, fake, fake, fake, 16, 1024, 1024, 1024, 4096, 4000, fake, None) == 1    # ldq < q_dim
    assert _rc(c, fake, fake, None, 16, 1024, 1024, 1024, 0, 0, None, None) == 1          # no d_scales
    assert _rc(c, None, fake, None, 16, 1024, 1024, 1024, 0, 0, fake, None) == 1          # tokens, no K
    assert _rc(c, fake, fake, None, 16, 1024, 1024, 1024, 0, 0, fake + 2, None) == 3      # scales misaligned
    assert _rc(c, fake + 1, fake, None, 16, 1024, 1024, 1024, 0, 0, fake, None) == 3      # odd bf16 address
    a = "fp8rl_kv_append"
    assert _rc(a, fake, fake, -1, 1024, 1024, 1024, fake, fake, fake, 1024, 64, fake, None) == 1  # tokens < 0
    assert _rc(a, fake, fake, 16, 1024, 1024, 1024, fake, fake, fake, 1000, 64, fake, None) == 1  # ld_cache < kv_dim
    assert _rc(a, fake, fake, 16, 1024, 1024, 1024, fake, fake, fake, 1024, -1, fake, None) == 1  # num_slots < 0
    assert _rc(a, fake, fake, 16, 1024, 1024, 1024, None, fake, fake, 1024, 64, fake, None) == 1  # no slot map
    assert _rc(a, fake, fake, 16, 1024, 1024, 1024, fake, fake, fake, 1024, 64, None, None) == 1  # no scales
    assert _rc(a, fake, fake, 16, 1024, 1024, 1024, fake + 2, fake, fake, 1024, 64, fake, None) == 3
    assert _rc(a, None, None, 0, 1024, 1024, 1024, None, None, None, 1024, 64, None, None) == 0   # no tokens: no-op


def test_helpers_reject_host_tensors():
    """A host tensor's pointer must never reach a kernel: every tensor helper
    refuses CPU tensors before it loads or calls the library."""
    import torch
    w = torch.zeros((128, 128), dtype=torch.bfloat16)
    u8 = torch.zeros((128, 128), dtype=torch.uint8)
    f32 = torch.ones((1, 1), dtype=torch.float32)
    off = torch.tensor([0, 128], dtype=torch.int32)
    calls = {
        "quant_weight": lambda: fp8rl.quant_weight(w),
        "quant_weights_batched": lambda: fp8rl.quant_weights_batched([w]),
        "quant_act": lambda: fp8rl.quant_act(w),
        "gemm": lambda: fp8rl.gemm(u8, f32, u8, f32),
        "grouped_gemm": lambda: fp8rl.grouped_gemm(u8, f32, u8.view(1, 128, 128), f32.view(1, 1, 1), off),
        "quant_gate_up_interleaved": lambda: fp8rl.quant_gate_up_interleaved(w, w),
        "gemm_swiglu_quant": lambda: fp8rl.gemm_swiglu_quant(u8, f32, u8, f32),
        "grouped_gemm_swiglu_quant": lambda: fp8rl.grouped_gemm_swiglu_quant(
            u8, f32, u8.view(1, 128, 128), f32.view(1, 1, 1), off),
        "kv_calibrate": lambda: fp8rl.kv_calibrate(w, w),
        "kv_append": lambda: fp8rl.kv_append(w, w, torch.zeros(128, dtype=torch.int32), u8, u8, f32),
        "moe_plan": lambda: fp8rl.moe_plan(torch.zeros((64, 2), dtype=torch.int32), 8),
        "moe_dispatch_quant": lambda: fp8rl.moe_dispatch_quant(w, torch.zeros(256, dtype=torch.int32), 2),
        "moe_combine": lambda: fp8rl.moe_combine(w, torch.zeros(8, dtype=torch.int32),
                                                 torch.zeros((4, 2), dtype=torch.float32)),
        "tis_weights": lambda: fp8rl.tis_weights(torch.zeros(8), torch.zeros(8)),
    }
    for name, call in calls.items():
        with pytest.raises(ValueError, match="CUDA tensors"):
            call()


def test_host_sync_rejects_bad_arguments_on_host(lib):
    """fp8rl_quant_weight_host_batched validates everything before it touches
    the device."""
    need = lib.fp8rl_host_sync_staging_bytes(128, 256, 2, 0)
    assert need == 2 * (128 * 256 * 2 + 128 * 256 + 256)
    assert lib.fp8rl_host_sync_staging_bytes(128, 256, 1, 0) == 0   # slots < 2
    assert lib.fp8rl_host_sync_staging_bytes(128, 256, 9, 0) == 0   # slots > 8
    assert lib.fp8rl_host_sync_staging_bytes(0, 256, 2, 0) == 0
    assert lib.fp8rl_host_sync_staging_bytes(128, 256, 2, 2) == 0   # unknown format
    buf = (ctypes.c_uint8 * 4096)()
    d = (fp8rl.WeightDesc * 1)()
    d[0] = fp8rl.WeightDesc(ctypes.addressof(buf), ctypes.addressof(buf), ctypes.addressof(buf), 256, 256, 256, 256)
    staging = 1 << 20  # a 256-byte aligned address, never dereferenced by a rejected call
    f = lib.fp8rl_quant_weight_host_batched
    assert f(d, 1, 2, staging, need, 2, None) == 1           # unknown format
    assert f(None, 1, 0, staging, need, 2, None) == 1        # null descriptors
    assert f(d, -1, 0, staging, need, 2, None) == 1          # negative count
    assert f(d, 1, 0, None, need, 2, None) == 1              # no staging
    assert f(d, 1, 0, staging, need, 1, None) == 1           # slots < 2
    assert f(d, 1, 0, staging, need, 9, None) == 1           # slots > 8
    assert f(d, 1, 0, staging + 16, need, 2, None) == 3      # staging not 256-byte aligned
    assert f(d, 1, 0, staging, need - 512, 2, None) == 2     # a slot cannot hold a block row
    d[0].ldw = 255
    assert f(d, 1, 0, staging, need, 2, None) == 1           # ldw < k
    d[0].ldw, d[0].w_bf16 = 256, None
    assert f(d, 1, 0, staging, need, 2, None) == 1           # null pointer
    assert f(d, 0, 0, staging, need, 2, None) == 0           # count 0: no-op


def test_debug_flavour_builds_with_the_same_entry_points(lib):
    """The FP8RL_DEBUG build (device-side store checks) compiles and exports
    every declared entry point, like the release library."""
    path = _build.build(debug=True)
    assert path == _build.LIB_DEBUG and os.path.exists(path)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(fp8rl_\w+)", out))
    assert set(declared_entry_points()) <= exported


def test_device_check_status_is_named(lib):
    assert lib.fp8rl_status_string(7) == b"FP8RL_ERR_DEVICE_CHECK"
    assert fp8rl.STATUS[7] == "FP8RL_ERR_DEVICE_CHECK"
