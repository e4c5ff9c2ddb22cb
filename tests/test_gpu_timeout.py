"""Failure detection on the device without a fault: a bounded wait that runs out.

A kernel waits on an mbarrier phase that nothing completes; the wait gives up after
its limit, the status word reads DG_ERR_TIMEOUT, and the context stays usable: a
denoising step run right after still matches the oracle's entropies."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_timeout_and_leaves_the_context_usable():
    import oracle
    from block_diffusion_text_gb300 import dg, synth
    assert dg.debug_wait_timeout() == dg.DG_ERR_TIMEOUT
    torch.cuda.synchronize()
    dims, seed = synth.workload("tiny_v512_c16")
    w = synth.make_weights(dims, seed, device="cuda")
    x, z, a = synth.make_canvas(dims, seed, device="cuda")
    ref = oracle.denoise_step(dims, synth.to_numpy_f32(w), x.cpu().numpy(), z.float().cpu().numpy(),
                              a.cpu().numpy(), tau=0.8, b=0.1, seed=seed, step=0, want=("H",))
    model = dg.Model(dims, w)
    out = dg.denoise_step(model, dg.Canvas(x, z, a), tau=0.8, b=0.1, seed=seed, step=0)
    torch.cuda.synchronize()
    assert model.status() == 0
    H = out["entropy"].cpu().numpy().reshape(-1)
    assert np.abs(H - np.asarray(ref["H"]).reshape(-1)).max() <= 1e-3
