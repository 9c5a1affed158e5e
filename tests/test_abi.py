"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function the header declares, sizes workspaces, and rejects bad
arguments synchronously before touching the device."""
import ctypes
import os
import re

import pytest

import mixture_experts_layer_align_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_gb300.h")


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_layer_align_gb300 import build
    build.build()
    return moe.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("moe_route_topk", "moe_align_by_expert", "moe_fused_forward",
              "moe_fused_workspace_size", "moe_status_string", "moe_check_status"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for code in range(7):
        assert moe.status_string(code)
    assert moe.status_string(99) == "unknown status"


def test_workspace_size_grows_with_tokens(lib):
    a = moe.moe_fused_workspace_size(1, 4096, 14336, 8, 2, moe.MOE_DT_FP8_E4M3)
    b = moe.moe_fused_workspace_size(64, 4096, 14336, 8, 2, moe.MOE_DT_FP8_E4M3)
    assert 0 < a < b
    assert b % 256 == 0
    assert moe.moe_fused_workspace_size(1, 128, 128, 4, 5, moe.MOE_DT_FP8_E4M3) == 0  # k > E
    assert moe.moe_fused_workspace_size(1, 128, 128, 2000, 2, moe.MOE_DT_FP8_E4M3) == 0


def test_launch_count(lib):
    fp8, bf16 = moe.MOE_DT_FP8_E4M3, moe.MOE_DT_BF16
    # up to 16 tokens: one front kernel (routing + alignment), gather, GEMM,
    # quant h, GEMM, finalize
    assert moe.moe_fused_launch_count(16, 4096, 14336, 8, 2, fp8) == 6
    assert moe.moe_fused_launch_count(4, 128, 256, 8, 2, bf16) == 5   # no quant of h
    # more tokens: separate router and alignment kernels
    assert moe.moe_fused_launch_count(64, 4096, 14336, 8, 2, fp8) == 7
    assert moe.moe_fused_launch_count(256, 2048, 768, 128, 8, fp8) == 7
    # E > 256: router, alignment, gather, GEMM, quant h, GEMM, finalize
    assert moe.moe_fused_launch_count(4, 2048, 768, 512, 8, fp8) == 7
    # pairs x H > 8M: rows per pair and a combine kernel instead
    assert moe.moe_fused_launch_count(2048, 8192, 256, 8, 1, fp8) == 7
    # 512 x 8 pairs: separate router and alignment kernels
    assert moe.moe_fused_launch_count(512, 2048, 768, 128, 8, fp8) == 7
    # > 4096 pairs: chunk histograms as well; x quantised per token and
    # scattered to its aligned rows in one kernel
    assert moe.moe_fused_launch_count(8192, 2048, 768, 128, 8, fp8) == 8
    assert moe.moe_fused_launch_count(0, 2048, 768, 128, 8, fp8) == 0
    assert moe.moe_fused_launch_count(4, 100, 256, 8, 2, fp8) == -1
    assert moe.moe_fused_launch_count(4, 128, 256, 8, 9, fp8) == -1


def test_inv_rope_argument_checks(lib):
    assert moe.moe_inv_rope_scratch_size(8, 4, 128) > 0
    assert moe.moe_inv_rope_scratch_size(8, 4, 96) == 0     # head size not a power of two
    assert moe.moe_inv_rope_scratch_size(8, 0, 128) == 0
    f = lib.moe_inv_rope_quant_per_head
    assert f(None, None, None, None, 0, 4, 64, 16, None, None, None, 0, None) == 0  # T = 0
    assert f(None, None, None, None, 4, 4, 64, 16, None, None, None, 0, None) == 1
    assert f(ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
             4, 4, 64, 0, ctypes.c_void_p(16), ctypes.c_void_p(16), None, 0, None) == 1  # max_pos
    assert f(ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
             4, 4, 64, 16, ctypes.c_void_p(16), ctypes.c_void_p(16), None, 0, None) == 3  # scratch


def _args(**kw):
    base = dict(x=16, router_logits=16, w13=16, w2=16, w13_scale=16, w2_scale=16,
                weight_dtype=1, T=4, H=128, I=256, E=8, top_k=2, renormalize=1, out=16,
                topk_ids_out=None, topk_w_out=None, counts_out=None, debug_flags=0)
    base.update(kw)
    return moe.MoeFusedArgs(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(top_k=9), 1), (dict(top_k=0), 1), (dict(E=0), 1), (dict(E=1025, top_k=2), 1),
    (dict(T=-1), 1), (dict(H=100), 2), (dict(I=200), 2), (dict(w13_scale=None), 1),
    (dict(weight_dtype=0), 1), (dict(weight_dtype=7), 1), (dict(x=None), 1),
    (dict(x=17), 1), (dict(out=24), 1), (dict(debug_flags=0x4 | 0x8), 1),
])
def test_fused_forward_rejects_bad_arguments(lib, kw, code):
    a = _args(**kw)
    st = lib.moe_fused_forward(ctypes.byref(a), ctypes.c_void_p(256), 1 << 40, None)
    assert st == code


def test_fused_forward_rejects_small_workspace(lib):
    a = _args()
    need = moe.moe_fused_workspace_size(4, 128, 256, 8, 2, moe.MOE_DT_FP8_E4M3)
    assert lib.moe_fused_forward(ctypes.byref(a), ctypes.c_void_p(256), need - 1, None) == 3
    assert lib.moe_fused_forward(ctypes.byref(a), None, need, None) == 3
    assert lib.moe_fused_forward(ctypes.byref(a), ctypes.c_void_p(1024 + 16), need, None) == 3


def test_zero_tokens_is_a_no_op(lib):
    a = _args(T=0)
    assert lib.moe_fused_forward(ctypes.byref(a), None, 0, None) == 0
    assert lib.moe_route_topk(None, 0, 8, 2, 1, None, None, None) == 0


def test_router_and_align_argument_checks(lib):
    assert lib.moe_route_topk(None, 4, 8, 9, 1, None, None, None) == 1
    assert lib.moe_route_topk(None, 4, 8, 2, 1, None, None, None) == 1
    assert lib.moe_align_by_expert(None, 4, 2, 8, 0, None, None, None, None, None, None) == 1
    assert lib.moe_align_by_expert(None, 4, 2, 8, 16, None, None, None, None, None, None) == 1
    assert lib.moe_quantize_e4m3(None, 4, 100, None, None, None, 0, None) == 1


def test_no_device_is_reported_not_faked(lib):
    """Valid arguments on a host without a GPU: the call must fail with a
    CUDA/unsupported status, never pretend to succeed."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("host has a GPU")
    a = _args(weight_dtype=1)
    need = moe.moe_fused_workspace_size(4, 128, 256, 8, 2, 1)
    st = lib.moe_fused_forward(ctypes.byref(a), ctypes.c_void_p(1 << 20), need, None)
    assert st in (2, 4)


def test_binding_constants_match_header():
    """The binding's copies of the header's flag bits, enum values and sizes
    agree with include/moe_gb300.h (read as text)."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    text = open(os.path.join(root, "include", "moe_gb300.h")).read()
    defines = {m.group(1): int(m.group(2), 0)
               for m in re.finditer(r"^#define (MOE_\w+) (0x[0-9a-fA-F]+|\d+)\s*$", text, re.M)}
    enums = {m.group(1): int(m.group(2))
             for m in re.finditer(r"\b(MOE_(?:OK|ERR_\w+|DT_\w+)) = (\d+)", text)}
    for name in ("MOE_DEBUG_FORCE_TIMEOUT", "MOE_DEBUG_TRACE", "MOE_FLAG_TOKENS_IN_M",
                 "MOE_FLAG_WEIGHTS_IN_M", "MOE_FLAG_NO_SM_PAIRS", "MOE_FLAG_ONE_KERNEL"):
        assert getattr(moe, name) == defines[name], name
    assert moe.TRACE_MAX_CTAS == defines["MOE_TRACE_MAX_CTAS"]
    assert len(moe.make_step_events.__defaults__) == 1
    assert moe.make_step_events.__defaults__[0] == defines["MOE_TIMED_EVENTS"]
    assert moe.MOE_OK == enums["MOE_OK"]
    assert moe.MOE_DT_BF16 == enums["MOE_DT_BF16"]
    assert moe.MOE_DT_FP8_E4M3 == enums["MOE_DT_FP8_E4M3"]
    for code, name in moe.STATUS_NAMES.items():
        assert enums[name] == code, name
    # the flag bits are distinct single bits
    flags = [defines[n] for n in defines if n.startswith(("MOE_FLAG_", "MOE_DEBUG_"))
             and n != "MOE_DEBUG_TIMEOUT_MS"]
    assert all(f & (f - 1) == 0 for f in flags) and len(set(flags)) == len(flags)


def test_header_compiles_as_c_and_the_library_links_from_c(lib, tmp_path):
    """A plain C11 program that includes the header, takes the address of
    every declared entry point (so the linker must resolve each one in the
    library) and calls two host-only functions."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = declared_functions()
    src = tmp_path / "abi_check.c"
    src.write_text(
        "#include <stdio.h>\n#include \"moe_gb300.h\"\n"
        "typedef void (*fn_t)(void);\n"
        "static fn_t table[] = {\n" +
        "".join(f"  (fn_t){n},\n" for n in names) +
        "};\n"
        "int main(void) {\n"
        "  printf(\"%d %s %zu\\n\", (int)(sizeof(table) / sizeof(table[0])),\n"
        "         moe_status_string(MOE_OK),\n"
        "         moe_fused_workspace_size(16, 256, 256, 8, 2, MOE_DT_FP8_E4M3));\n"
        "  return 0;\n}\n")
    libdir = os.path.dirname(moe.LIB_PATH)
    exe = tmp_path / "abi_check"
    r = subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-o", str(exe), moe.LIB_PATH, f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    n, status, ws = out.stdout.split()
    assert int(n) == len(names)
    assert status == lib.moe_status_string(0).decode()
    assert int(ws) == lib.moe_fused_workspace_size(16, 256, 256, 8, 2, moe.MOE_DT_FP8_E4M3)
