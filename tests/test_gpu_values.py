"""Device-side value checks: a canvas token outside [0, V) never reaches the embedding gather.

The embedding kernel checks every token it gathers; an out-of-range one is recorded as
DG_ERR_VALUE in the status word and embedded as token 0, so the step reads no memory outside
E and computes exactly what the oracle computes for the canvas with those tokens set to 0."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_out_of_range_tokens_set_value_status_and_embed_token_zero():
    import oracle
    from block_diffusion_text_gb300 import dg, synth
    dims, seed = synth.workload("tiny_v512_c16")
    w = synth.make_weights(dims, seed, device="cuda")
    x, z, a = synth.make_canvas(dims, seed, device="cuda")
    bad = x.clone()
    bad[0, 3] = dims.V
    bad[0, 5] = -5
    x0 = bad.clone()
    x0[0, 3] = 0
    x0[0, 5] = 0
    model = dg.Model(dims, w)
    out = dg.denoise_step(model, dg.Canvas(bad, z.clone(), a), tau=0.8, b=0.1, seed=seed, step=0)
    torch.cuda.synchronize()
    assert model.status() == dg.DG_ERR_VALUE
    ref = oracle.denoise_step(dims, synth.to_numpy_f32(w), x0.cpu().numpy(), z.float().cpu().numpy(),
                              a.cpu().numpy(), tau=0.8, b=0.1, seed=seed, step=0, want=("H",))
    H = out["entropy"].cpu().numpy().reshape(-1)
    assert np.abs(H - np.asarray(ref["H"]).reshape(-1)).max() <= 1e-3
    # the context stays usable: a step on valid tokens with a fresh workspace reports ok
    model2 = dg.Model(dims, w)
    dg.denoise_step(model2, dg.Canvas(x, z.clone(), a), tau=0.8, b=0.1, seed=seed, step=0)
    torch.cuda.synchronize()
    assert model2.status() == dg.DG_OK
