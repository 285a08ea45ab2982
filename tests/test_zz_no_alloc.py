"""The allocation-free attention entry point (for callers that cannot call
cudaMalloc: a host whose memory manager owns all device memory, a plugin
handed no scratch buffer) must give the same results as the workspace entry
point, call after call, although its scratch array keeps the last call's
contents.

This file sorts last so that a run stopping at its first failure has already
run every other test; it must also pass alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from canvas_denoising_gb300 import binding as B
from canvas_denoising_gb300 import synth
from tests.parity import LSE_ABS, assert_rows_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mask", [B.DG_MASK_BIDIR, B.DG_MASK_CAUSAL_BLOCK])
@pytest.mark.parametrize("C,Hq,Hkv,hd,P", [(256, 16, 8, 128, 4096), (100, 6, 3, 64, 700)])
def test_noalloc_matches_workspace_entry_point_twice(lib, mask, C, Hq, Hkv, hd, P):
    assert B.canvas_attn_workspace_size(C, Hq, Hkv, hd, P) > 0  # the shape really uses scratch
    assert B.canvas_attn_workspace_size(C, Hq, Hkv, hd, P) <= B.load().dg_canvas_attn_noalloc_max_scratch()
    k, v = synth.kv_prefix(Hkv, P + C, hd, P, seed=21, device="cuda")
    q, kn, vn = synth.canvas_qkv(C, Hq, Hkv, hd, seed=21, device="cuda")
    ref_out, ref_lse = B.canvas_attn(q, k, v, P, kn, vn, mask=mask)
    for _ in range(2):  # the shared scratch keeps the previous call's contents
        out, lse = B.canvas_attn_noalloc(q, k, v, P, kn, vn, mask=mask)
        torch.cuda.synchronize()
        assert_rows_close(out.float().cpu().numpy().reshape(C * Hq, hd),
                          ref_out.float().cpu().numpy().reshape(C * Hq, hd), what="noalloc out")
        assert np.abs(lse.cpu().numpy() - ref_lse.cpu().numpy()).max() <= LSE_ABS
    assert B.device_status() == B.DG_OK
