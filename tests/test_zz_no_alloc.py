"""dg_attention_noalloc: the step's attention run with the library's static scratch.

The entry point exists for callers that cannot allocate device memory (a
process whose device memory is pre-reserved by another framework, or code that
is only handed fixed buffers).  This file is collected last on purpose.
"""
import ctypes as ct

import numpy as np
import pytest
import torch

from block_diffusion_text_gb300 import synth

from parity import bf16_to_np, check_rel_l2

pytestmark = pytest.mark.gpu


def _call(L, q, K, V, cap, P, k, v, o, B, C, Hq, Hkv, hd):
    p = lambda t: ct.c_void_p(t.data_ptr())
    return L.dg_attention_noalloc(p(q), p(K), p(V), cap, P, p(k), p(v), p(o), B, C, Hq, Hkv, hd,
                                  ct.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_attention_noalloc_matches_step_attention_twice():
    from block_diffusion_text_gb300 import dg
    L = dg.load()
    dims, seed = synth.workload("step_v32k_c256_p2k")  # splits the keys, so the scratch is used
    w = synth.make_weights(dims, seed, device="cuda")
    x, z, a = synth.make_canvas(dims, seed, device="cuda")
    model = dg.Model(dims, w)
    canvas = dg.Canvas(x, z, a)
    out = dg.denoise_step(model, canvas, tau=0.8, b=0.1, seed=seed, step=0, debug=True)
    dbg = out["debug"]
    ref = bf16_to_np(dbg["o"])
    for _ in range(2):
        o = torch.full_like(dbg["o"], float("nan"))
        rc = _call(L, dbg["q"], model.K, model.V, model.cap, dims.P, dbg["k"], dbg["v"], o, dims.B, dims.C,
                   dims.Hq, dims.Hkv, dims.hd)
        assert rc == dg.DG_OK
        torch.cuda.synchronize()
        got = bf16_to_np(o)
        assert np.isfinite(got).all()
        assert check_rel_l2("o", got, ref) <= 1e-2


def test_attention_noalloc_rejects_sizes_beyond_its_scratch():
    """Two canvases of 8 heads over an 8190-key prefix (not a multiple of 128, so the warp-MMA kernel
    with 8 key splits) need 17.0 MB of partials: rejected before any launch.  Every buffer is
    allocated at its full size all the same."""
    from block_diffusion_text_gb300 import dg
    L = dg.load()
    B, C, Hq, Hkv, hd, P = 2, 256, 8, 8, 128, 8190
    bf = dict(dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(B, Hq, C, hd, **bf)
    K = torch.zeros(B, Hkv, P + 2, hd, **bf)
    V = torch.zeros_like(K)
    k = torch.zeros(B, Hkv, C, hd, **bf)
    v = torch.zeros_like(k)
    o = torch.zeros(B * C, Hq * hd, **bf)
    rc = _call(L, q, K, V, P + 2, P, k, v, o, B, C, Hq, Hkv, hd)
    assert rc == dg.DG_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(o).item() == 0
