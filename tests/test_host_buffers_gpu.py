"""The C ABI with pinned host buffers (the q row and index arrays read, out and
lse written by the kernels across the host link): identical bits to the call
with device buffers.  q stays in device memory for bf16 KV, whose kernel
fetches it with bulk copies."""
import pytest
import torch

from mla_attention_decode_gb300 import binding, synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "mxfp4"])
@pytest.mark.parametrize("lens", [[1000, 0, 64, 3000, 1], [257] * 40])
def test_host_buffers_match_device_buffers(dtype, lens):
    inp = synth.make_inputs(lens, dtype, seed=91)
    dec = binding.MLADecoder(inp.kv_indptr, dtype, device=DEV)
    kv = inp.kv.to(DEV)
    scale = {"bf16": None, "fp8": inp.kv_scale, "mxfp4": inp.block_scales}[dtype]
    scale = None if scale is None else scale.to(DEV)
    ss = int(scale.stride(0)) if dtype == "mxfp4" else 0
    b = len(lens)
    out_d = torch.empty(b, 16, 512, dtype=torch.bfloat16, device=DEV)
    lse_d = torch.empty(b, 16, device=DEV)
    binding.mla_decode_fwd(inp.q.to(DEV), kv, scale, inp.kv_indptr.to(DEV), inp.qo_indptr.to(DEV), out_d, lse_d,
                           dec.plan, dec.workspace, scale_stride=ss)
    q = inp.q.to(DEV) if dtype == "bf16" else inp.q.pin_memory()
    ind, qo = inp.kv_indptr.pin_memory(), inp.qo_indptr.pin_memory()
    out_h = torch.full((b, 16, 512), 7, dtype=torch.bfloat16).pin_memory()
    lse_h = torch.full((b, 16), 7.0).pin_memory()
    binding.mla_decode_fwd(q, kv, scale, ind, qo, out_h, lse_h, dec.plan, dec.workspace, scale_stride=ss)
    torch.cuda.synchronize()
    assert dec.poll_error() == 0
    od, ld = out_d.cpu(), lse_d.cpu()
    bad = (out_h != od).any(dim=2).nonzero().tolist()
    assert torch.equal(out_h, od), f"out differs at (seq, head) {bad[:8]} of {len(bad)}; lse equal: {torch.equal(lse_h, ld)}"
    assert torch.equal(lse_h, ld)
