"""The multi-layer stack and its causal prefill / commit through the C ABI against the oracle.

The debug copies of a step (a, q, k, v, o, h) are the last layer's.  Caches
are compared layer by layer with the bf16 operand tolerance: a later piece of
a prefill reads the device's own earlier rows, which may differ from the
oracle's by a rounding step.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from block_diffusion_text_gb300 import synth

from parity import Collect, bf16_to_np, check_close_bf16

from parity import check_entropy
from test_gpu_step import _entropy_given_device_h, _run_and_compare

pytestmark = pytest.mark.gpu


# Every layer adds its bf16 rounding points (a, q, k, v, o, h); fp32 against exact accumulation
# flips a few of them to the other neighbour, and across layers these compound in h.  As in the
# long-canvas case of test_gpu_step, the entropy is compared end to end against a stated bound with
# the rows above 1e-3 counted, and against the oracle's statistics of the device's own h to 1e-3
# (the LM head and the statistics merge); every operand is compared to its bf16 tolerance.
LAYERS_H_BOUND = 4e-3


def test_three_layer_step_warp_mma_attention():
    dims = synth.Dims(V=1000, d=256, C=40, B=2, Hq=4, Hkv=2, hd=64, F=192, P=100, cap=160, L=3)
    g = torch.Generator().manual_seed(31)
    z = (torch.randn(dims.B, dims.C, dims.d, generator=g) * 0.02).to(torch.bfloat16)
    _run_and_compare(dims, 31, tau=0.6, step=2, z_in=z, entropy_given_h=True, e2e_bound=LAYERS_H_BOUND)


def test_two_layer_step_tensor_core_attention():
    dims = synth.Dims(V=1000, d=256, C=100, B=2, Hq=6, Hkv=2, hd=128, F=192, P=256, cap=256, L=2)
    _run_and_compare(dims, 32, tau=0.7, entropy_given_h=True, e2e_bound=LAYERS_H_BOUND)


def test_two_layer_step_split_k_clusters():
    """d = 2048, 128 canvas rows, two layers: each layer's q/k/v projection runs on clusters of four
    K slices (128-column tiles, RoPE in the owner's epilogue), FFW1 on 64-column tiles over four
    slices with GELU; the tensor-core attention reads a 128-row prefix."""
    dims = synth.Dims(V=1000, d=2048, C=64, B=2, Hq=4, Hkv=2, hd=128, F=1024, P=128, cap=192, L=2)
    g = torch.Generator().manual_seed(35)
    z = (torch.randn(dims.B, dims.C, dims.d, generator=g) * 0.02).to(torch.bfloat16)
    _run_and_compare(dims, 35, tau=0.7, step=1, z_in=z, entropy_given_h=True, e2e_bound=LAYERS_H_BOUND)


def _model(dims, seed):
    from block_diffusion_text_gb300 import dg
    w = synth.make_weights(dims, seed, device="cpu")
    return w, dg.Model(dims, {k: v.cuda() for k, v in w.items()}, cache_len=dims.P)


def _check_caches(ck, tag, Kd, Vd, Kr, Vr, rows):
    for l in range(Kr.shape[0]):
        u = 8 * (l + 1)  # layer l's rows carry the rounding of the layers below
        ck(check_close_bf16, f"{tag} K layer {l}", Kd[l][:, :, rows], Kr[l][:, :, rows], ulps=u)
        ck(check_close_bf16, f"{tag} V layer {l}", Vd[l][:, :, rows], Vr[l][:, :, rows], ulps=u)


@pytest.mark.parametrize("hd,d", [(64, 128), (128, 128), (128, 2048)])
def test_prefill_matches_oracle_in_pieces(hd, d):
    """A 100-token prompt into an empty three-layer cache: three pieces of at most C = 40 tokens, each
    attending causally over everything before it; every layer's rows against the oracle's one pass,
    the rows past the prompt untouched, and the length advanced.  At d = 2048 each piece's k/v
    projection runs on split-K clusters."""
    from block_diffusion_text_gb300 import dg
    dims = synth.Dims(V=1000, d=d, C=40, B=2, Hq=4, Hkv=2, hd=hd, F=192, P=0, cap=160, L=3)
    w, model = _model(dims, 33)
    tok = torch.randint(0, dims.V, (dims.B, 100), dtype=torch.int32, generator=torch.Generator().manual_seed(3))
    n = dg.prefill(model, tok.cuda())
    torch.cuda.synchronize()
    assert n == 100 and model.len == 100 and model.status() == 0
    Kr, Vr = oracle.prefill(dims, synth.to_numpy_f32(w), tok.numpy(), P=0)
    Kd, Vd = bf16_to_np(model.K), bf16_to_np(model.V)
    ck = Collect()
    _check_caches(ck, "prefill", Kd, Vd, Kr, Vr, slice(0, 100))
    ck.done()
    assert np.all(Kd[:, :, :, 100:] == 0) and np.all(Vd[:, :, :, 100:] == 0)


def test_step_on_prefilled_cache_then_commit():
    """Two layers: prefill a prompt, run a denoising step on the device's cache (checked against the
    oracle given that cache), commit the step's argmax (checked against the oracle's re-encode from
    the same cache), and the capacity check leaves the cache untouched."""
    from block_diffusion_text_gb300 import dg
    dims = synth.Dims(V=1000, d=256, C=40, B=2, Hq=4, Hkv=2, hd=64, F=192, P=0, cap=140, L=2)
    w, model = _model(dims, 34)
    prompt = torch.randint(0, dims.V, (dims.B, 60), dtype=torch.int32, generator=torch.Generator().manual_seed(4))
    dg.prefill(model, prompt.cuda())
    x, z, a = synth.make_canvas(dims, 34, device="cpu")
    canvas = dg.Canvas(x.cuda(), z.cuda(), a.cuda())
    out = dg.denoise_step(model, canvas, tau=0.8, b=0.1, seed=34, step=0, debug=True)
    torch.cuda.synchronize()
    assert model.status() == 0
    wn = synth.to_numpy_f32(w)
    Kd, Vd = bf16_to_np(model.K), bf16_to_np(model.V)
    d1 = dataclasses.replace(dims, P=60)
    w1 = dict(wn, Kc=Kd.astype(np.float32), Vc=Vd.astype(np.float32))
    ref = oracle.denoise_step(d1, w1, x.numpy(), z.float().numpy(), a.numpy(), tau=0.8, b=0.1, seed=34, step=0,
                              want=("h", "H", "z_out"))
    ck = Collect()
    ck(check_close_bf16, "h", bf16_to_np(out["debug"]["h"]), ref["h"], ulps=16)
    Hd = out["entropy"].cpu().numpy().reshape(-1)
    e2e = float(np.abs(Hd - ref["H"]).max())
    print(f"parity-report entropy end to end: max {e2e:.3e} nats")
    if e2e > LAYERS_H_BOUND:
        ck.errors.append(f"entropy end to end {e2e:.2e}")
    ck(check_entropy, Hd, _entropy_given_device_h(d1, wn, a.numpy(), bf16_to_np(out["debug"]["h"]), 0.8))
    xhat = out["argmax"].clone()
    dg.commit_block(model, xhat)
    torch.cuda.synchronize()
    assert model.len == 100
    Kr, Vr = oracle.prefill(d1, w1, xhat.cpu().numpy(), P=60)
    Kc2, Vc2 = bf16_to_np(model.K), bf16_to_np(model.V)
    _check_caches(ck, "commit", Kc2, Vc2, Kr, Vr, slice(60, 100))
    assert np.array_equal(Kc2[:, :, :, :60], Kd[:, :, :, :60])
    before = model.K.clone()
    with pytest.raises(dg.DgError) as e:
        dg.commit_block(model, xhat)  # 100 + 40 > 140? no; a second one overflows
        dg.commit_block(model, xhat)
    assert e.value.code == dg.DG_ERR_CAPACITY
    torch.cuda.synchronize()
    assert model.len == 140 and torch.equal(model.K[..., :100, :], before[..., :100, :])
    ck.done()
