"""mla_decode_fwd_static: the decode for callers that cannot allocate device
memory (a plugin or custom-operator interface that only hands over inputs and
outputs, or a loop where cudaMalloc's device-wide synchronisation is not
allowed).  It runs with the library's own static device workspace; its output
must match mla_decode_fwd's (with a caller workspace) on consecutive calls.

This file is collected last on purpose, and must pass both on its own in a
fresh process and after every other test."""
import numpy as np
import pytest
import torch

from mla_attention_decode_gb300 import binding, build, synth

pytestmark = pytest.mark.gpu

TOL = 2e-2  # the stated rtol = atol of the parity tests


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()
    assert torch.cuda.is_available()


def _inputs(inp, dev):
    scale = inp.kv_scale if inp.kv_dtype == "fp8" else None
    return (inp.q.to(dev), inp.kv.to(dev), None if scale is None else scale.to(dev), inp.kv_indptr.to(dev),
            inp.qo_indptr.to(dev))


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_static_workspace_matches_caller_workspace(dtype):
    # split and unsplit sequences (the combine stage reads the workspace), an empty one
    inp = synth.make_inputs([1, 700, 0, 3000, 129, 64, 5000], dtype, seed=71)
    dev = torch.device("cuda:0")
    q, kv, scale, ind, qo = _inputs(inp, dev)
    plan = binding.mla_decode_plan(inp.kv_indptr, dtype)
    assert plan.splits_max > 1
    assert binding.mla_decode_workspace_bytes(plan) <= binding.MLA_STATIC_WORKSPACE_BYTES
    b = plan.batch
    ws = torch.zeros(binding.mla_decode_workspace_bytes(plan), dtype=torch.uint8, device=dev)
    ref_out = torch.empty(b, 16, 512, dtype=torch.bfloat16, device=dev)
    ref_lse = torch.empty(b, 16, dtype=torch.float32, device=dev)
    binding.mla_decode_fwd(q, kv, scale, ind, qo, ref_out, ref_lse, plan, ws)
    torch.cuda.synchronize()
    assert binding.mla_decode_poll_error(ws) == 0
    ref_out, ref_lse = ref_out.double().cpu().numpy(), ref_lse.double().cpu().numpy()
    for call in range(2):
        out = torch.full((b, 16, 512), float("nan"), dtype=torch.bfloat16, device=dev)
        lse = torch.full((b, 16), float("nan"), dtype=torch.float32, device=dev)
        err = torch.full((1,), -1, dtype=torch.int32, device=dev)
        binding.mla_decode_fwd_static(q, kv, scale, ind, qo, out, lse, plan, device_error=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"call {call}: device error {int(err.item())}"
        got, got_lse = out.double().cpu().numpy(), lse.double().cpu().numpy()
        assert np.all(np.isfinite(got)), f"call {call}: non-finite output"
        np.testing.assert_allclose(got, ref_out, rtol=TOL, atol=TOL, err_msg=f"call {call}: out")
        fin = np.isfinite(ref_lse)
        assert np.array_equal(fin, np.isfinite(got_lse)), f"call {call}: lse finiteness"
        np.testing.assert_allclose(got_lse[fin], ref_lse[fin], rtol=TOL, atol=TOL, err_msg=f"call {call}: lse")
        assert got[2].max() == 0 and got[2].min() == 0, "empty sequence output must be 0"


def test_static_workspace_rejects_oversized_plans():
    # 64 sequences forced into 64 splits each: far more partials than the array holds
    plan = binding.mla_decode_plan([8192 * i for i in range(65)], "fp8", num_sms=152, num_splits=64)
    assert binding.mla_decode_workspace_bytes(plan) > binding.MLA_STATIC_WORKSPACE_BYTES
    dev = torch.device("cuda:0")
    t = torch.zeros(16, dtype=torch.uint8, device=dev)
    with pytest.raises(binding.MLAError) as e:
        binding.mla_decode_fwd_static(t, t, t, t, t, t, None, plan)
    assert e.value.status == binding.MLA_ERR_WORKSPACE_TOO_SMALL
