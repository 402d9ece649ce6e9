"""mla_decode_fwd_static: the decode for callers that cannot allocate device
memory (a plugin or custom-operator interface that only hands over inputs and
outputs, or a loop where cudaMalloc's device-wide synchronisation is not
allowed).  It runs the same kernels on the same plan as mla_decode_fwd, only
with the library's own static device workspace, so its output must be
identical, bit for bit, to mla_decode_fwd's (with a caller workspace) on
consecutive calls.

This file is collected last on purpose, and must pass both on its own in a
fresh process and after every other test."""
import pytest
import torch

from mla_attention_decode_gb300 import binding, build, synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()
    assert torch.cuda.is_available()


def _inputs(inp):
    scale = {"bf16": None, "fp8": inp.kv_scale, "mxfp4": inp.block_scales}[inp.kv_dtype]
    return (inp.q.to(DEV), inp.kv.to(DEV), None if scale is None else scale.to(DEV), inp.kv_indptr.to(DEV),
            inp.qo_indptr.to(DEV))


def _reference(inp, plan, q, kv, scale, ind, qo, ss):
    """mla_decode_fwd with a caller-owned workspace."""
    b = plan.batch
    ws = torch.zeros(binding.mla_decode_workspace_bytes(plan), dtype=torch.uint8, device=DEV)
    out = torch.empty(b, 16, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(b, 16, dtype=torch.float32, device=DEV)
    binding.mla_decode_fwd(q, kv, scale, ind, qo, out, lse, plan, ws, scale_stride=ss)
    torch.cuda.synchronize()
    assert binding.mla_decode_poll_error(ws) == 0
    return out.cpu(), lse.cpu()


def _static_calls(plan, q, kv, scale, ind, qo, ss, ref_out, ref_lse, what):
    b = plan.batch
    for call in range(2):
        out = torch.full((b, 16, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
        lse = torch.full((b, 16), float("nan"), dtype=torch.float32, device=DEV)
        err = torch.full((1,), -1, dtype=torch.int32, device=DEV)
        binding.mla_decode_fwd_static(q, kv, scale, ind, qo, out, lse, plan, device_error=err, scale_stride=ss)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"{what} call {call}: device error {int(err.item())}"
        assert torch.equal(out.cpu(), ref_out), f"{what} call {call}: out differs from mla_decode_fwd"
        assert torch.equal(lse.cpu(), ref_lse), f"{what} call {call}: lse differs from mla_decode_fwd"


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "mxfp4"])
def test_static_workspace_matches_caller_workspace(dtype):
    # split and unsplit sequences (the combine stage reads the workspace), an empty one
    inp = synth.make_inputs([1, 700, 0, 3000, 129, 64, 5000], dtype, seed=71)
    q, kv, scale, ind, qo = _inputs(inp)
    ss = int(scale.stride(0)) if dtype == "mxfp4" else 0
    plan = binding.mla_decode_plan(inp.kv_indptr, dtype)
    assert plan.splits_max > 1
    assert binding.mla_decode_workspace_bytes(plan) <= binding.MLA_STATIC_WORKSPACE_BYTES
    ref_out, ref_lse = _reference(inp, plan, q, kv, scale, ind, qo, ss)
    assert torch.all(ref_out[2] == 0), "empty sequence output must be 0"
    _static_calls(plan, q, kv, scale, ind, qo, ss, ref_out, ref_lse, dtype)


def test_static_workspace_after_another_layout():
    """Two layouts in a row share the array: the second call's partials and
    split table replace the first's, and nothing of the first shows."""
    for lens, dtype in (([9000, 10, 4000], "fp8"), ([300] * 20 + [0, 2500], "fp8")):
        inp = synth.make_inputs(lens, dtype, seed=len(lens))
        q, kv, scale, ind, qo = _inputs(inp)
        plan = binding.mla_decode_plan(inp.kv_indptr, dtype)
        ref_out, ref_lse = _reference(inp, plan, q, kv, scale, ind, qo, 0)
        _static_calls(plan, q, kv, scale, ind, qo, 0, ref_out, ref_lse, f"{dtype} {lens[:3]}")


def test_static_workspace_rejects_oversized_plans():
    # 64 sequences forced into 64 splits each: far more partials than the array holds
    plan = binding.mla_decode_plan([8192 * i for i in range(65)], "fp8", num_sms=152, num_splits=64)
    assert binding.mla_decode_workspace_bytes(plan) > binding.MLA_STATIC_WORKSPACE_BYTES
    t = torch.zeros(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(binding.MLAError) as e:
        binding.mla_decode_fwd_static(t, t, t, t, t, t, None, plan)
    assert e.value.status == binding.MLA_ERR_WORKSPACE_TOO_SMALL
