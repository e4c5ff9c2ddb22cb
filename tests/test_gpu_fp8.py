"""The FP8 (E4M3) LM head through the C ABI against the oracle.

Quantization is integer-valued work once the float32 scale is fixed, so the
codes and scales are compared bit for bit.  The step is compared twice:
 - given the device's own h (quantized by the oracle, which the first test
   shows gives the device's codes), the logits to fp32-accumulation accuracy
   and the entropy to the stated 1e-3;
 - end to end against the oracle's FP8 step.  A row whose h differs by a bf16
   ulp between the two sides (the rounding of the attention block) can land
   on another E4M3 code; such rows are counted and printed, their entropy is
   held to a wider stated bound and their argmax to a near-maximum, and they
   are left out of the accept / token decisions; every other row is held to
   the bf16 step's bar.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from block_diffusion_text_gb300 import synth

from parity import (H_TOL, Collect, bf16_to_np, check_argmax, check_entropy, check_logits, check_rel_l2,
                    check_sampler)

pytestmark = pytest.mark.gpu

# fp32 accumulation of exact E4M3 products, then three fp32 scalings: row-relative error bound
FP8_LOGIT_TOL = 1e-4
# entropy end to end on a row whose h took another E4M3 code somewhere (one code step moves a
# logit by about 2^-4 of one of d terms): the multi-layer step's bound
FP8_MOVED_H_BOUND = 4e-3


def _lut():
    return np.array([oracle.e4m3_value(b) for b in range(256)], np.float64)


def _fp8_logits(h, alpha, E8, es, d):
    """l_v = alpha s_h s_v (q_h . q_v) / sqrt(d) in float64, h quantized per row by the oracle."""
    Qh, sh = oracle.quantize_rows_e4m3(np.asarray(h, np.float32))
    lut = _lut()
    hv = lut[Qh]
    acc = np.empty((hv.shape[0], E8.shape[0]))
    for v0 in range(0, E8.shape[0], 16384):  # bounded host memory at a full vocabulary
        acc[:, v0:v0 + 16384] = hv @ lut[E8[v0:v0 + 16384]].T
    al = np.asarray(alpha, np.float64).reshape(-1)
    return (al * sh.astype(np.float64))[:, None] * es.astype(np.float64)[None, :] * acc / math.sqrt(d), Qh


def _matrices(seed):
    g = torch.Generator().manual_seed(seed)
    out = []
    for R, d in ((37, 64), (19, 1024), (5, 2816), (130, 48)):
        X = torch.randn(R, d, generator=g) * torch.exp(torch.randn(R, 1, generator=g) * 3)
        X[0] = 0.0                                  # zero row: scale 0, zero codes
        X[1] = -0.0                                 # negative zeros
        X[2, :] = 1e-3
        X[2, 0] = 1e4                               # one large value: the rest fall to subnormal codes or 0
        X[3, ::2] = -X[3, ::2].abs()                # mixed signs with exact ties in magnitude
        X[3, 1::2] = X[3, ::2].abs()
        out.append(X.to(torch.bfloat16))
    return out


def test_quantize_rows_bit_exact():
    from block_diffusion_text_gb300 import dg
    for X in _matrices(7):
        Q, sc = dg.quantize_rows_e4m3(X.cuda())
        torch.cuda.synchronize()
        Qr, sr = oracle.quantize_rows_e4m3(X.float().numpy())
        n = int((Q.cpu().numpy() != Qr).sum())
        assert n == 0, f"{tuple(X.shape)}: {n} codes differ from the oracle"
        assert np.array_equal(sc.cpu().numpy().view(np.uint32), sr.view(np.uint32)), "scales differ"


def test_quantize_rows_of_a_vocabulary():
    """The codes of a full 262144 x 2816 embedding (the 8-bit copy the FP8 head reads), checked
    on sampled rows, and the zero-row count."""
    from block_diffusion_text_gb300 import dg
    V, d = 262144, 2816
    g = torch.Generator(device="cuda").manual_seed(3)
    E = (torch.randn(V, d, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    Q, sc = dg.quantize_rows_e4m3(E)
    torch.cuda.synchronize()
    rows = np.r_[0:4, V - 4:V, np.random.default_rng(0).integers(0, V, 56)]
    Qr, sr = oracle.quantize_rows_e4m3(E[rows].float().cpu().numpy())
    assert np.array_equal(Q[rows].cpu().numpy(), Qr)
    assert np.array_equal(sc[rows].cpu().numpy(), sr)
    assert int((sc == 0).sum()) == 0


def _run(dims, seed, tau=0.8, b=0.1, rows=None):
    from block_diffusion_text_gb300 import dg
    w = synth.make_weights(dims, seed, device="cpu")
    x, z, a = synth.make_canvas(dims, seed, device="cpu")
    model = dg.Model(dims, {k: v.cuda() for k, v in w.items()}, fp8_head=True)
    canvas = dg.Canvas(x.cuda(), z.cuda(), a.cuda())
    out = dg.denoise_step(model, canvas, tau=tau, b=b, seed=seed, step=0, debug=True)
    torch.cuda.synchronize()
    assert model.status() == 0
    wn = synth.to_numpy_f32(w)
    E8r, esr = oracle.quantize_rows_e4m3(wn["E"])
    ck = Collect()

    def codes_exact():
        assert np.array_equal(model.E8.cpu().numpy(), E8r), "E8 codes"
        assert np.array_equal(model.E8_scale.cpu().numpy(), esr), "E8 scales"
    ck(codes_exact)
    h_dev = bf16_to_np(out["debug"]["h"])
    dev_logits = out["debug"]["logits"].cpu().numpy()
    sel = np.arange(dims.M) if rows is None else np.asarray(rows)
    lg, Qh_dev = _fp8_logits(h_dev[sel], a.numpy().reshape(-1)[sel], E8r, esr, dims.d)

    def logits_given_h():
        err = float(np.max(np.abs(dev_logits[sel] - lg) / np.max(np.abs(lg), axis=1, keepdims=True)))
        print(f"parity-report fp8 logits given device h: max row-relative error {err:.3e}")
        assert err <= FP8_LOGIT_TOL, f"fp8 logits given h: {err:.3e}"
    ck(logits_given_h)
    Hdev = out["entropy"].cpu().numpy().reshape(-1).astype(np.float64)
    ck(check_entropy, Hdev[sel], np.array([oracle.row_stats(r, tau)["H"] for r in lg]))

    ref = oracle.denoise_step(dims, wn, x.numpy(), z.float().numpy(), a.numpy(), tau=tau, b=b, seed=seed, step=0,
                              fp8_head=(E8r, esr), rows=rows,
                              want=("h", "logits", "H", "top2gap", "argmax", "accept", "cum", "renoise_tok",
                                    "sample_tok", "gumbel_gap", "z_out", "n_acc"))
    Qh_ref, _ = oracle.quantize_rows_e4m3(ref["h"][sel].astype(np.float32))
    moved = np.any(Qh_dev != Qh_ref, axis=1)
    keep = ~moved
    # every row: the logits at the bf16 step's 2e-2 row-relative tolerance
    ck(check_logits, dev_logits[sel], ref["logits"])
    e2e = np.abs(Hdev[sel] - ref["H"][sel])
    print(f"parity-report fp8 step: {int(moved.sum())} of {len(sel)} rows with another E4M3 code of h; "
          f"entropy end to end max {e2e[keep].max(initial=0):.3e} (same codes), "
          f"{e2e[moved].max(initial=0):.3e} (other codes)")

    def entropy_e2e():
        assert e2e[keep].max(initial=0) <= H_TOL, "entropy (rows with the same codes of h)"
        assert e2e[moved].max(initial=0) <= FP8_MOVED_H_BOUND, "entropy (rows with other codes of h)"
    ck(entropy_e2e)
    scale = np.max(np.abs(ref["logits"]), axis=1)
    am_dev = out["argmax"].cpu().numpy().reshape(-1)[sel]
    if keep.any():
        ck(check_argmax, am_dev[keep], ref["argmax"][sel][keep], ref["top2gap"][sel][keep], scale[keep])

    def argmax_moved():
        # another code of h moves logits by far less than 1e-2 of the row scale: the device's argmax
        # is a near-maximum of the oracle's row
        for i in np.nonzero(moved)[0]:
            assert ref["logits"][i][am_dev[i]] >= ref["logits"][i].max() - 1e-2 * scale[i], f"argmax row {sel[i]}"
    ck(argmax_moved)
    if rows is None:
        stats = ck(check_sampler, out["accept"].cpu().numpy(), canvas.tokens.cpu().numpy(), ref, b, dims.C,
                   excuse=moved)
        ck(check_rel_l2, "z", bf16_to_np(canvas.z).reshape(dims.M, dims.d), ref["z_out"])
        print(dims, "stats", stats)
    ck.done()


def test_fp8_step_tiny():
    _run(*synth.workload("tiny_v512_c16"))


def test_fp8_step_ragged():
    # K = 128 is one E4M3 stage; V = 1000 leaves a partial vocabulary tile and statistics group
    _run(synth.Dims(V=1000, d=128, C=40, B=3, Hq=4, Hkv=2, hd=64, F=192, P=100, cap=160), 11)


def test_fp8_step_deep_k():
    # d = 704: five full E4M3 stages and a half one (K tail zero-filled by the tensor map)
    _run(synth.Dims(V=4104, d=704, C=64, B=2, Hq=4, Hkv=2, hd=64, F=256, P=128, cap=256), 12)


@pytest.mark.slow
def test_fp8_step_full_vocab_sampled_rows():
    # the full 262144-token vocabulary and d = 2816 of the loop workload, at a short prefix; the
    # oracle evaluates sampled rows only
    dims = synth.Dims(V=262144, d=2816, C=256, B=1, Hq=16, Hkv=8, hd=128, F=1024, P=256, cap=512)
    _run(dims, 2, rows=[0, 1, 77, 128, 200, 254, 255])
