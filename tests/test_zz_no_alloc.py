"""dg_attention_noalloc: the step's attention run with the library's static scratch.

The entry point exists for callers that cannot allocate device memory (a
process whose device memory is pre-reserved by another framework, or code that
is only handed fixed buffers).  Its results must equal, bit for bit, the
attention inside dg_denoise_step (the same kernels with the same key split,
only the scratch lives elsewhere), on both attention kernels and on calls in a
row (the scratch keeps the previous call's contents), and match the oracle.
This file is collected last on purpose.
"""
import ctypes as ct

import numpy as np
import pytest
import torch

import oracle
from block_diffusion_text_gb300 import synth

from parity import bf16_to_np, check_close_bf16

pytestmark = pytest.mark.gpu


def _call(L, q, K, V, cap, P, k, v, o, B, C, Hq, Hkv, hd):
    p = lambda t: ct.c_void_p(t.data_ptr())
    return L.dg_attention_noalloc(p(q), p(K), p(V), cap, P, p(k), p(v), p(o), B, C, Hq, Hkv, hd,
                                  ct.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("case", ["tensor_core_p2048", "warp_mma_p1000"])
def test_attention_noalloc_equals_step_attention_twice(case):
    """P = 2048 takes the tensor-core kernel, P = 1000 (not a multiple of 128) the warp-MMA kernel;
    both split the keys (5 or more splits), so the partials and their (max, sum) pairs go through
    the static scratch.  Two calls in a row, each bit-identical to the step's own attention output,
    and equal to the oracle's attention within the bf16 operand tolerance."""
    from block_diffusion_text_gb300 import dg
    L = dg.load()
    if case == "tensor_core_p2048":
        dims, seed = synth.workload("step_v32k_c256_p2k")
    else:
        dims, seed = synth.Dims(V=4096, d=256, C=256, B=1, Hq=8, Hkv=2, hd=128, F=256, P=1000, cap=1024), 6
    w = synth.make_weights(dims, seed, device="cpu")
    x, z, a = synth.make_canvas(dims, seed, device="cpu")
    model = dg.Model(dims, {k: t.cuda() for k, t in w.items()})
    canvas = dg.Canvas(x.cuda(), z.cuda(), a.cuda())
    out = dg.denoise_step(model, canvas, tau=0.8, b=0.1, seed=seed, step=0, debug=True)
    torch.cuda.synchronize()
    assert model.status() == 0
    dbg = out["debug"]
    for _ in range(2):
        o = torch.full_like(dbg["o"], float("nan"))
        rc = _call(L, dbg["q"], model.K, model.V, model.cap, dims.P, dbg["k"], dbg["v"], o, dims.B, dims.C,
                   dims.Hq, dims.Hkv, dims.hd)
        assert rc == dg.DG_OK
        assert dg.attention_noalloc_status() == dg.DG_OK
        assert torch.equal(o, dbg["o"])
    ref = oracle.denoise_step(dims, synth.to_numpy_f32(w), x.numpy(), z.float().numpy(), a.numpy(), tau=0.8,
                              b=0.1, seed=seed, step=0, rows=[], want=("o",))
    check_close_bf16("o", bf16_to_np(o), ref["o"])


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
