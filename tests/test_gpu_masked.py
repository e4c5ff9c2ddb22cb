"""Masked confidence decoding (the second sampler) through the C ABI against the oracle.

The oracle's confidence is 1 / Z in double; the device's Z is an fp32 sum, so a
position whose log-confidence lies within 1e-3 (the entropy tolerance, in the
same log units) of the reveal boundary may legitimately swap sides; such
positions are counted and printed.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from block_diffusion_text_gb300 import synth

from parity import Collect, bf16_to_np, check_entropy, check_logits, check_rel_l2

pytestmark = pytest.mark.gpu

LOGZ_TOL = 1e-3


def _setup(dims, seed):
    from block_diffusion_text_gb300 import dg
    w = synth.make_weights(dims, seed, device="cpu")
    x, z, a = synth.make_canvas(dims, seed, device="cpu")
    model = dg.Model(dims, {k: v.cuda() for k, v in w.items()})
    return w, x, z, a, model


def check_reveal(tok_in, tok_dev, rev_dev, ref, mask_id, C):
    """Revealed sets and tokens per canvas; returns the number of excused boundary swaps."""
    tok_in = np.asarray(tok_in).reshape(-1, C)
    tok_dev = np.asarray(tok_dev).reshape(-1, C)
    rev_dev = np.asarray(rev_dev).reshape(-1, C).astype(bool)
    rev_ref = ref["revealed"].reshape(-1, C)
    logZ = np.log(ref["Z"]).reshape(-1, C)
    am = ref["argmax"].reshape(-1, C)
    excused = 0
    for b in range(tok_in.shape[0]):
        unres = tok_in[b] == mask_id
        k = int(rev_ref[b].sum())
        assert int(rev_dev[b].sum()) == k, f"canvas {b}: {int(rev_dev[b].sum())} revealed, oracle {k}"
        order = np.lexsort((np.arange(C), logZ[b]))
        order = order[unres[order]]
        edges = [logZ[b][order[k - 1]]] if k else []
        if k < len(order):
            edges.append(logZ[b][order[k]])
        for i in np.nonzero(rev_dev[b] != rev_ref[b])[0]:
            assert any(abs(logZ[b][i] - e) <= LOGZ_TOL for e in edges), f"canvas {b}: reveal of {i} differs"
            excused += 1
        both = rev_dev[b] & rev_ref[b]
        assert np.array_equal(tok_dev[b][both], am[b][both]), f"canvas {b}: revealed tokens"
        kept = ~rev_dev[b]
        assert np.array_equal(tok_dev[b][kept], tok_in[b][kept]), f"canvas {b}: unrevealed positions changed"
    return excused


def _run_step(dims, seed, N, step, frac_masked, tau=0.8):
    from block_diffusion_text_gb300 import dg
    w, x, z, a, model = _setup(dims, seed)
    mask = dims.V - 1
    g = torch.Generator().manual_seed(seed + 1)
    x = torch.where(torch.rand(x.shape, generator=g) < frac_masked, torch.full_like(x, mask), x)
    zin = (torch.randn(z.shape, generator=g) * 0.02).to(torch.bfloat16) if step else z
    canvas = dg.Canvas(x.cuda(), zin.cuda(), a.cuda())
    out = dg.denoise_step(model, canvas, tau=tau, b=0.0, seed=0, step=step, debug=True, masked=(mask, N))
    torch.cuda.synchronize()
    assert model.status() == 0
    ref = oracle.denoise_step_masked(dims, synth.to_numpy_f32(w), x.numpy(), zin.float().numpy(), a.numpy(),
                                     tau=tau, mask_id=mask, step=step, N=N, want_extra=("logits",))
    ck = Collect()
    ck(check_logits, out["debug"]["logits"].cpu().numpy(), ref["logits"])
    ck(check_entropy, out["entropy"].cpu().numpy().reshape(-1), ref["H"])
    ex = ck(check_reveal, x.numpy(), canvas.tokens.cpu().numpy(), out["accept"].cpu().numpy(), ref, mask, dims.C)
    ck(check_rel_l2, "z", bf16_to_np(canvas.z).reshape(dims.M, dims.d), ref["z_out"])
    ck(check_rel_l2, "u", bf16_to_np(out["debug"]["u"]), ref["u"])

    def counts():
        assert np.array_equal(out["n_acc"].cpu().numpy(), ref["n_rev"])
    ck(counts)
    print(f"parity-report masked step: excused reveal swaps {ex}, revealed {ref['n_rev'].tolist()}")
    ck.done()


def test_masked_step_tiny_all_masked():
    dims, seed = synth.workload("tiny_v512_c16")
    _run_step(dims, seed, N=4, step=0, frac_masked=1.0)


def test_masked_step_ragged_partly_revealed():
    dims = synth.Dims(V=1000, d=128, C=40, B=3, Hq=4, Hkv=2, hd=64, F=192, P=100, cap=160)
    _run_step(dims, 21, N=7, step=3, frac_masked=0.6, tau=0.6)


@pytest.mark.slow
def test_masked_step_v32k():
    dims, seed = synth.workload("step_v32k_c256_p2k")
    _run_step(dims, seed, N=16, step=0, frac_masked=1.0)


def test_masked_loop_reveals_everything_and_follows_the_oracle():
    """dg_denoise_canvas_masked from an all-[MASK] canvas: every step reveals ceil(U / (N - s)),
    nothing is masked at the end, and the canvas equals the oracle's loop run from the same state
    (free-running; the comparison stops at the first excused boundary swap)."""
    from block_diffusion_text_gb300 import dg
    dims = synth.Dims(V=512, d=64, C=16, B=2, Hq=2, Hkv=1, hd=32, F=128, P=32)
    seed, N, tau = 9, 5, 0.8
    w, x, z, a, model = _setup(dims, seed)
    mask = dims.V - 1
    tok0 = dg.canvas_init_masked(dims.B, dims.C, mask)
    assert (tok0 == mask).all()
    canvas = dg.Canvas(tok0.clone(), z.cuda(), a.cuda())
    res = dg.denoise_canvas_masked(model, canvas, mask, N=N, tau=tau)
    torch.cuda.synchronize()
    assert model.status() == 0
    acc = res["accepted"].cpu().numpy()
    U = dims.C
    for s in range(N):
        k = math.ceil(U / (N - s))
        assert (acc[:, s] == k).all(), (s, acc[:, s])
        U -= k
    fin = res["xhat0"].cpu().numpy()
    assert (fin != mask).all() and np.array_equal(fin, canvas.tokens.cpu().numpy())
    assert res["steps_taken"].cpu().tolist() == [N] * dims.B
    # the oracle's loop, step by step
    wn = synth.to_numpy_f32(w)
    tok = np.full((dims.B, dims.C), mask, np.int32)
    zz = z.float().numpy()
    c2 = dg.Canvas(tok0.clone(), z.cuda(), a.cuda())
    for s in range(N):
        ref = oracle.denoise_step_masked(dims, wn, tok, zz, a.numpy(), tau=tau, mask_id=mask, step=s, N=N)
        out = dg.denoise_step(model, c2, tau=tau, b=0.0, seed=0, step=s, masked=(mask, N))
        torch.cuda.synchronize()
        ex = check_reveal(tok, c2.tokens.cpu().numpy(), out["accept"].cpu().numpy(), ref, mask, dims.C)
        if ex:
            print("loop: excused swap at step", s)
            break
        tok = ref["tokens_out"].reshape(dims.B, dims.C)
        zz = ref["z_out"].astype(np.float32).reshape(zz.shape)
        assert np.array_equal(c2.tokens.cpu().numpy(), tok)
    else:
        assert np.array_equal(fin, tok)
