"""The C ABI library (no GPU needed): it loads, exports every declared symbol,
and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla_decode.h")


@pytest.fixture(scope="module")
def lib():
    from mla_attention_decode_gb300 import binding, build
    build.build()
    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MLA_API\s+[\w\s\*]+?\b(mla_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    assert {"mla_decode_plan", "mla_decode_workspace_bytes", "mla_decode_fwd", "mla_decode_poll_error",
            "mla_status_string", "mla_decode_version"} <= set(names)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in mla_decode.h but not exported"


def test_status_strings(lib):
    from mla_attention_decode_gb300 import binding
    for code in range(0, 8):
        assert binding.mla_status_string(code) != "unknown status"
    assert binding.mla_status_string(99) == "unknown status"
    assert re.fullmatch(r"\d+\.\d+\.\d+", binding.mla_decode_version())


def test_fwd_rejects_bad_arguments_without_cuda(lib):
    from mla_attention_decode_gb300 import binding
    plan = binding.mla_decode_plan([0, 10, 20], "fp8", num_sms=152)
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: validation fails first
    # null plan
    assert lib.mla_decode_fwd(fake, fake, fake, 0, fake, fake, fake, None, 1 / 24, None, fake, 1 << 30, None) == 1
    # null q
    assert lib.mla_decode_fwd(None, fake, fake, 0, fake, fake, fake, None, 1 / 24, ctypes.byref(plan), fake,
                              1 << 30, None) == 1
    # misaligned kv
    assert lib.mla_decode_fwd(fake, P((1 << 20) + 8), fake, 0, fake, fake, fake, None, 1 / 24, ctypes.byref(plan),
                              fake, 1 << 30, None) == 1
    # fp8 without its scale
    assert lib.mla_decode_fwd(fake, fake, None, 0, fake, fake, fake, None, 1 / 24, ctypes.byref(plan), fake,
                              1 << 30, None) == 1
    # workspace too small
    assert lib.mla_decode_fwd(fake, fake, fake, 0, fake, fake, fake, None, 1 / 24, ctypes.byref(plan), fake,
                              16, None) == 3
    # non-finite sm_scale
    assert lib.mla_decode_fwd(fake, fake, fake, 0, fake, fake, fake, None, float("nan"), ctypes.byref(plan), fake,
                              1 << 30, None) == 1
    # mxfp4 with a scale stride below 18
    plan4 = binding.mla_decode_plan([0, 10, 20], "mxfp4", num_sms=152)
    assert lib.mla_decode_fwd(fake, fake, fake, 17, fake, fake, fake, None, 1 / 24, ctypes.byref(plan4), fake,
                              1 << 30, None) == 1


def test_trace_is_off_in_the_normal_build(lib):
    """mla_decode_set_trace records only in the trace build: the normal library
    refuses a buffer and accepts NULL (off)."""
    lib.mla_decode_set_trace.argtypes = [ctypes.c_void_p]
    lib.mla_decode_set_trace.restype = ctypes.c_int
    assert lib.mla_decode_set_trace(ctypes.c_void_p(1 << 20)) == 2
    assert lib.mla_decode_set_trace(None) == 0


def test_empty_batch_is_a_noop(lib):
    from mla_attention_decode_gb300 import binding
    plan = binding.mla_decode_plan([0], "bf16", num_sms=152)
    assert plan.batch == 0 and plan.num_work == 0
    assert lib.mla_decode_fwd(None, None, None, 0, None, None, None, None, 1 / 24, ctypes.byref(plan), None, 0,
                              None) == 0


def test_plan_struct_layout_matches_header(tmp_path):
    """The ctypes mirror of mla_plan has the C header's size and field offsets
    (a plain C program built against include/mla_decode.h prints them)."""
    import shutil
    import subprocess
    from mla_attention_decode_gb300 import binding
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = [name for name, _ in binding.mla_plan._fields_]
    src = tmp_path / "plan_layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "mla_decode.h"\nint main(void) {\n'
                   '  printf("size %zu\\n", sizeof(mla_plan));\n' +
                   "".join(f'  printf("{f} %zu\\n", offsetof(mla_plan, {f}));\n' for f in fields) +
                   "  return 0;\n}\n")
    exe = tmp_path / "plan_layout"
    subprocess.run([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = dict(line.split() for line in subprocess.run([str(exe)], check=True, capture_output=True,
                                                         text=True).stdout.splitlines())
    assert int(out.pop("size")) == ctypes.sizeof(binding.mla_plan)
    for f in fields:
        assert int(out[f]) == getattr(binding.mla_plan, f).offset, f


def test_fwd_rejects_inconsistent_two_token_plans_without_cuda(lib):
    """A two-token plan is e4m3 with q_len 2 and two partial slots per unit;
    any other combination is refused on the host before any CUDA call."""
    from mla_attention_decode_gb300 import binding
    P = ctypes.c_void_p
    fake = P(1 << 20)

    def fwd(plan):
        return lib.mla_decode_fwd(fake, fake, fake, 0, fake, fake, fake, None, 1 / 24, ctypes.byref(plan), fake,
                                  1 << 30, None)

    good = binding.mla_decode_plan_multi([0, 300, 700], 2, "fp8", num_sms=152)
    assert good.tokens_fused == 2 and good.q_len == 2 and good.num_work % 2 == 0
    for field, value in (("tokens_fused", 3), ("tokens_fused", 1), ("q_len", 3), ("kv_dtype", 0), ("num_work", 3)):
        bad = binding.mla_plan.from_buffer_copy(good)
        setattr(bad, field, value)
        assert fwd(bad) == binding.MLA_ERR_INVALID_ARG, (field, value)
    # a one-token plan may not claim two tokens per unit
    one = binding.mla_decode_plan([0, 300, 700], "fp8", num_sms=152)
    one.tokens_fused = 2
    assert fwd(one) == binding.MLA_ERR_INVALID_ARG


def test_fwd_checks_the_mx_scores_field_without_cuda(lib):
    """plan.mx_scores: 0 or 1, and 1 only for MXFP4; the block-scaled form reads
    the cache through a 4-bit tensor map, which needs kv 32-byte aligned."""
    from mla_attention_decode_gb300 import binding
    P = ctypes.c_void_p
    fake = P(1 << 20)

    def fwd(plan, kv=fake):
        return lib.mla_decode_fwd(fake, kv, fake, 18, fake, fake, fake, None, 1 / 24, ctypes.byref(plan), fake,
                                  1 << 30, None)

    mx = binding.mla_decode_plan([0, 300, 700], "mxfp4", num_sms=152)
    assert mx.mx_scores == 0
    for value in (2, -1):
        bad = binding.mla_plan.from_buffer_copy(mx)
        bad.mx_scores = value
        assert fwd(bad) == binding.MLA_ERR_INVALID_ARG, value
    fp8 = binding.mla_decode_plan([0, 300, 700], "fp8", num_sms=152)
    fp8.mx_scores = 1
    assert fwd(fp8) == binding.MLA_ERR_INVALID_ARG
    bs = binding.mla_plan.from_buffer_copy(mx)
    bs.mx_scores = 1
    assert fwd(bs, kv=P((1 << 20) + 16)) == binding.MLA_ERR_INVALID_ARG
