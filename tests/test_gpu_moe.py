"""The MoE FFN of the step (router, expert permutation, grouped expert GEMMs, combine) through the
C ABI against the oracle.

Routing is an integer decision taken from floating-point logits, so it is checked on the device's
own router input x = RMSNorm(h) (a debug copy): the router logits against x . Wr_e in double to fp32
accumulation accuracy (ACC_REL of sum_j |x_j Wr_ej|), the selection against the top_k of those
exact logits (a difference only where two of them lie within twice that bound), and the gates
against their softmax to 1e-5.  End to end, h differs from the oracle's by a rounding step in a few
elements (fp32 against exact accumulation in the attention block), which moves x by a bf16 ulp
there; a row whose selection then differs from the oracle's must have an input that differs and a
near-tie at the first differing rank (within the logit change that input difference causes, in
double); such rows are counted, printed and left out of the element-wise comparisons.  The MoE
block is a second residual block per layer, so the entropy is compared as for the multi-layer
stack: end to end against LAYERS_H_BOUND with the rows above 1e-3 counted, and to 1e-3 against the
oracle's statistics of the device's own h.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from block_diffusion_text_gb300 import synth

from parity import Collect, bf16_to_np, check_close_bf16, check_entropy, check_logits, check_sampler
from test_gpu_layers import LAYERS_H_BOUND
from test_gpu_step import _entropy_given_device_h

pytestmark = pytest.mark.gpu

ACC_REL = 1e-5


def _topk(r, k):
    return np.argsort(-r, axis=1, kind="stable")[:, :k]


def check_routing_given_x(x_dev, Wr, idx_dev, gate_dev, lg_dev, k):
    """Router logits, selection and gates against the exact router of the device's own input."""
    x = np.asarray(x_dev, np.float64)
    W = np.asarray(Wr, np.float64)
    r = x @ W.T
    bound = ACC_REL * (np.abs(x) @ np.abs(W).T)
    err = np.abs(lg_dev - r) / bound
    assert err.max() <= 1.0, f"router logits: {err.max():.3e} of the accumulation bound"
    sel = _topk(r, k)
    n_tie = 0
    for row in np.nonzero(np.any(idx_dev != sel, axis=1))[0]:
        j = int(np.argmax(idx_dev[row] != sel[row]))
        a, b = sel[row, j], idx_dev[row, j]
        assert abs(r[row, a] - r[row, b]) <= 2 * (bound[row, a] + bound[row, b]), f"row {row}: selection"
        n_tie += 1
    keep = np.all(idx_dev == sel, axis=1)
    rs = np.take_along_axis(r, sel, axis=1)
    g = np.exp(rs - rs[:, :1])
    g /= g.sum(axis=1, keepdims=True)
    gerr = np.abs(gate_dev - g)[keep].max(initial=0)
    assert gerr <= 1e-5, f"gates: {gerr:.3e}"
    return n_tie


def routing_moved(x_dev, x_ref, Wr, idx_dev, ref):
    """Rows whose selection differs from the oracle's; each must come from an input difference at a
    near-tie."""
    idx_ref = ref["moe_idx"]
    W = np.asarray(Wr, np.float64)
    moved = np.any(idx_dev != idx_ref, axis=1)
    for row in np.nonzero(moved)[0]:
        dx = np.asarray(x_dev[row], np.float64) - np.asarray(x_ref[row], np.float64)
        assert np.any(dx != 0), f"row {row}: routing differs on the same input"
        shift = np.abs(W @ dx).max()  # how far the input difference moves any logit
        j = int(np.argmax(idx_dev[row] != idx_ref[row]))
        lr = ref["moe_logits"][row]
        a, b = idx_ref[row, j], idx_dev[row, j]
        assert abs(lr[a] - lr[b]) <= 2 * shift + 1e-6 * np.abs(lr).max(), f"row {row}: routing differs"
    return moved


def _run(dims, seed, tau=0.8, b=0.1):
    from block_diffusion_text_gb300 import dg
    w = synth.make_weights(dims, seed, device="cpu")
    x, z, a = synth.make_canvas(dims, seed, device="cpu")
    model = dg.Model(dims, {k: v.cuda() for k, v in w.items()})
    canvas = dg.Canvas(x.cuda(), z.cuda(), a.cuda())
    out = dg.denoise_step(model, canvas, tau=tau, b=b, seed=seed, step=0, debug=True)
    torch.cuda.synchronize()
    assert model.status() == 0
    wn = synth.to_numpy_f32(w)
    ref = oracle.denoise_step(dims, wn, x.numpy(), z.float().numpy(), a.numpy(), tau=tau, b=b, seed=seed, step=0,
                              want=("h", "logits", "H", "top2gap", "argmax", "accept", "cum", "renoise_tok",
                                    "sample_tok", "gumbel_gap", "z_out", "n_acc", "moe_idx", "moe_gate",
                                    "moe_logits", "moe_x"))
    dbg = out["debug"]
    ck = Collect()
    Wr_last = wn["Wr"] if dims.L == 1 else wn["Wr"][dims.L - 1]
    x_dev = bf16_to_np(dbg["moe_x"])
    idx_dev = dbg["moe_idx"].cpu().numpy()
    n_tie = ck(check_routing_given_x, x_dev, Wr_last, idx_dev, dbg["moe_gate"].cpu().numpy(),
               dbg["moe_logits"].cpu().numpy().astype(np.float64), dims.top_k)
    moved = ck(routing_moved, x_dev, ref["moe_x"], Wr_last, idx_dev, ref)
    if moved is None:
        moved = np.zeros(dims.M, bool)
    keep = ~moved
    # every layer's operands pass through bf16: the stack's ulp budget, as for the attention layers
    ck(check_close_bf16, "h", bf16_to_np(dbg["h"])[keep], ref["h"][keep], ulps=8 * dims.L)
    ck(check_logits, dbg["logits"].cpu().numpy()[keep], ref["logits"][keep])
    Hd = out["entropy"].cpu().numpy().reshape(-1).astype(np.float64)
    e2e = np.abs(Hd - ref["H"])[keep]

    def entropy_e2e():
        assert e2e.max(initial=0) <= LAYERS_H_BOUND, f"entropy end to end {e2e.max():.3e}"
    ck(entropy_e2e)
    ck(check_entropy, Hd, _entropy_given_device_h(dims, wn, a.numpy(), bf16_to_np(dbg["h"]), tau))
    stats = ck(check_sampler, out["accept"].cpu().numpy(), canvas.tokens.cpu().numpy(), ref, b, dims.C,
               excuse=moved)
    n_active = len(np.unique(dbg["moe_idx"].cpu().numpy()))
    print(f"parity-report moe {dims.n_exp}x top{dims.top_k} Fe {dims.Fe} L {dims.L}: {n_tie} near-tie selections "
          f"given the device's input; {int(moved.sum())} of {dims.M} rows routed otherwise than the oracle (input "
          f"differences at near-ties); {n_active} experts active; entropy end to end max "
          f"{e2e.max(initial=0):.3e}, {int((e2e > 1e-3).sum())} rows above 1e-3; sampler {stats}")
    ck.done()
    return out, ref


# d = 256 as for the multi-layer stack: the end-to-end entropy bound holds there (see the module note)
MOE_SMALL = synth.Dims(V=1000, d=256, C=40, B=3, Hq=4, Hkv=2, hd=64, F=192, P=100, cap=160, n_exp=16, top_k=4,
                       Fe=128)


def test_moe_step_small():
    _run(MOE_SMALL, 21)


def test_moe_step_every_expert_selected():
    # top_k == n_exp: every expert takes every row (2 M-tiles per expert, the second partial)
    _run(dataclasses.replace(MOE_SMALL, C=70, B=2, n_exp=4, top_k=4), 22)


def test_moe_step_single_expert():
    # n_exp = top_k = 1: gate 1, the routed expert and the shared expert on every row
    _run(dataclasses.replace(MOE_SMALL, n_exp=1, top_k=1, Fe=256), 23)


def test_moe_step_hot_experts_two_layers():
    # two layers with MoE; 64 experts of which 40 are hot, top 8, d = 256
    dims = synth.Dims(V=2048, d=256, C=64, B=2, Hq=4, Hkv=2, hd=64, F=256, P=128, cap=256, L=2, n_exp=64,
                      top_k=8, Fe=256, moe_hot=40)
    _run(dims, 24)


def test_moe_prefill_matches_oracle():
    """Prefill in pieces on a two-layer MoE stack: layer 1's cache rows depend on layer 0's MoE block."""
    from block_diffusion_text_gb300 import dg
    dims = synth.Dims(V=1024, d=128, C=32, B=2, Hq=4, Hkv=2, hd=64, F=128, P=40, cap=160, L=2, n_exp=8, top_k=2,
                      Fe=128)
    w = synth.make_weights(dims, 25, device="cpu")
    model = dg.Model(dims, {k: v.cuda() for k, v in w.items()})
    toks = torch.randint(0, dims.V, (dims.B, 75), generator=torch.Generator().manual_seed(3), dtype=torch.int32)
    dg.prefill(model, toks.cuda())
    torch.cuda.synchronize()
    assert model.status() == 0
    Kr, Vr = oracle.prefill(dims, synth.to_numpy_f32(w), toks.numpy(), dims.P)
    rows = slice(dims.P, dims.P + 75)
    ck = Collect()
    for l in range(dims.L):
        ck(check_close_bf16, f"K layer {l}", bf16_to_np(model.K[l][..., rows, :]).reshape(-1, dims.hd),
           Kr[l][..., rows, :].reshape(-1, dims.hd), ulps=8 * dims.L)
        ck(check_close_bf16, f"V layer {l}", bf16_to_np(model.V[l][..., rows, :]).reshape(-1, dims.hd),
           Vr[l][..., rows, :].reshape(-1, dims.hd), ulps=8 * dims.L)
    ck.done()


@pytest.mark.slow
def test_moe_full_size_sampled_rows():
    """The MoE variant of the loop workload (128 experts, top 8, 84 hot, Fe 768, d 2816, V 262144) at
    a short prefix: routing and h on every row, the vocabulary stages on sampled rows."""
    from block_diffusion_text_gb300 import dg
    dims = synth.Dims(V=262144, d=2816, C=256, B=1, Hq=16, Hkv=8, hd=128, F=1024, P=512, n_exp=128, top_k=8,
                      Fe=768, moe_hot=84)
    seed = 26
    w = synth.make_weights(dims, seed, device="cpu")
    x, z, a = synth.make_canvas(dims, seed, device="cpu")
    model = dg.Model(dims, {k: v.cuda() for k, v in w.items()})
    canvas = dg.Canvas(x.cuda(), z.cuda(), a.cuda())
    out = dg.denoise_step(model, canvas, tau=0.8, b=0.1, seed=seed, step=0, debug=True)
    torch.cuda.synchronize()
    assert model.status() == 0
    rows = [0, 1, 100, 254, 255]
    wn = synth.to_numpy_f32(w)
    ref = oracle.denoise_step(dims, wn, x.numpy(), z.float().numpy(), a.numpy(), tau=0.8, b=0.1,
                              seed=seed, step=0, rows=rows,
                              want=("h", "logits", "H", "argmax", "top2gap", "moe_idx", "moe_gate", "moe_logits",
                                    "moe_x"))
    dbg = out["debug"]
    ck = Collect()
    Wr_last = wn["Wr"] if dims.L == 1 else wn["Wr"][dims.L - 1]
    x_dev = bf16_to_np(dbg["moe_x"])
    idx_dev = dbg["moe_idx"].cpu().numpy()
    n_tie = ck(check_routing_given_x, x_dev, Wr_last, idx_dev, dbg["moe_gate"].cpu().numpy(),
               dbg["moe_logits"].cpu().numpy().astype(np.float64), dims.top_k)
    moved = ck(routing_moved, x_dev, ref["moe_x"], Wr_last, idx_dev, ref)
    if moved is None:
        moved = np.zeros(dims.M, bool)
    keep = ~moved
    ck(check_close_bf16, "h", bf16_to_np(dbg["h"])[keep], ref["h"][keep])
    sel = [r for r in rows if keep[r]]
    li = [rows.index(r) for r in sel]
    ck(check_logits, dbg["logits"][sel].cpu().numpy(), ref["logits"][li])
    e2e = np.abs(out["entropy"].cpu().numpy().reshape(-1)[sel] - ref["H"][sel])

    def entropy_e2e():
        assert e2e.max(initial=0) <= LAYERS_H_BOUND, f"entropy end to end {e2e.max():.3e}"
    ck(entropy_e2e)
    n_active = len(np.unique(dbg["moe_idx"].cpu().numpy()))
    print(f"parity-report moe full size: {n_tie} near-tie selections given the device's input; "
          f"{int(moved.sum())} rows routed otherwise than the oracle; {n_active} experts active; "
          f"entropy end to end max {e2e.max(initial=0):.3e}")
    assert n_active == 84
    ck.done()
