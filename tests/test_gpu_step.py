"""One denoising step through the C ABI against the CPU oracle on the same seeded inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
from block_diffusion_text_gb300 import synth

from parity import (Collect, bf16_to_np, check_argmax, check_entropy, check_logits, check_rel_l2,
                    check_sampler)
from parity import check_close_bf16 as _close

pytestmark = pytest.mark.gpu

# End-to-end entropy bound of the long d = 128 canvas case (see test_long_canvas_entropy_given_h).
LONG_CANVAS_H_BOUND = 2e-3

RAGGED = synth.Dims(V=1000, d=128, C=40, B=3, Hq=4, Hkv=2, hd=64, F=192, P=100, cap=160)
# head dim 128 with a prefix that is a multiple of 128: the tensor-core attention kernel, with a partial
# canvas key block (C = 100) and a 3-head group whose 300 query rows leave a partial third Q tile and an
# empty fourth one (Q tiles go in pairs)
RAGGED_TC = synth.Dims(V=1000, d=128, C=100, B=2, Hq=6, Hkv=2, hd=128, F=192, P=256, cap=256)


def _setup(dims, seed, alpha=None):
    from block_diffusion_text_gb300 import dg
    w = synth.make_weights(dims, seed, device="cpu")
    x, z, a = synth.make_canvas(dims, seed, device="cpu")
    if alpha is not None:
        a = torch.full_like(a, alpha)
    model = dg.Model(dims, {k: v.cuda() for k, v in w.items()})
    canvas = dg.Canvas(x.cuda(), z.cuda(), a.cuda())
    return w, x, z, a, model, canvas


def _entropy_given_device_h(dims, w, alpha, h_dev, tau):
    """The oracle's tempered-softmax entropy of logits formed from the device's own h."""
    import oracle
    E = np.asarray(w["E"], np.float64)
    al = np.asarray(alpha, np.float64).reshape(-1)
    logits = al[:, None] * (np.asarray(h_dev, np.float64) @ E.T) / math.sqrt(dims.d)
    return np.array([oracle.row_stats(r, tau)["H"] for r in logits])


def _run_and_compare(dims, seed, tau=0.8, b=0.1, step=0, alpha=None, z_in=None, prev=None,
                     entropy_given_h=False, e2e_bound=None):
    from block_diffusion_text_gb300 import dg
    w, x, z, a, model, canvas = _setup(dims, seed, alpha)
    if z_in is not None:
        z = z_in
        canvas.z.copy_(z.cuda())
    if prev is not None:
        canvas.prev_argmax.copy_(torch.as_tensor(prev).cuda())
    out = dg.denoise_step(model, canvas, tau=tau, b=b, seed=seed, step=step, debug=True)
    torch.cuda.synchronize()
    assert model.status() == 0
    wn = synth.to_numpy_f32(w)
    ref = oracle.denoise_step(dims, wn, x.numpy(), z.float().numpy(), a.numpy(), tau=tau, b=b, seed=seed,
                              step=step, prev_argmax=prev,
                              want=("a", "q", "k", "v", "o", "h", "logits", "H", "m", "Z", "top2gap",
                                    "argmax", "accept", "cum", "rank", "renoise_tok", "sample_tok",
                                    "gumbel_gap", "tokens_out", "u", "g", "z_out", "n_acc", "meanH",
                                    "stop"))
    dbg = out["debug"]
    B, C, Hq, Hkv, hd = dims.B, dims.C, dims.Hq, dims.Hkv, dims.hd
    ck = Collect()
    ul = 8 * dims.L  # the last layer's operands carry every earlier layer's rounding

    def check_close_bf16(name, got, ref_):
        return _close(name, got, ref_, ulps=ul)
    # a = RMSNorm(E[x] + z) is the correctly rounded bf16 of its definition on both sides; a deeper
    # layer's input RMSNorm(h) is compared like the other operands (h itself is within tolerance)
    def a_exact():
        n = int((bf16_to_np(dbg["a"]) != ref["a"]).sum())
        assert n == 0, f"a: {n} elements differ from the oracle"
    if dims.L == 1:
        ck(a_exact)
    else:
        ck(check_close_bf16, "a", bf16_to_np(dbg["a"]), ref["a"])
    q = bf16_to_np(dbg["q"]).reshape(B, Hq, C, hd).transpose(0, 2, 1, 3).reshape(B * C, Hq * hd)
    ck(check_close_bf16, "q", q, ref["q"])
    k = bf16_to_np(dbg["k"]).reshape(B, Hkv, C, hd).transpose(0, 2, 1, 3).reshape(B * C, Hkv * hd)
    ck(check_close_bf16, "k", k, ref["k"])
    v = bf16_to_np(dbg["v"]).reshape(B, Hkv, C, hd).transpose(0, 2, 1, 3).reshape(B * C, Hkv * hd)
    ck(check_close_bf16, "v", v, ref["v"])
    ck(check_close_bf16, "o", bf16_to_np(dbg["o"]), ref["o"])
    ck(check_close_bf16, "h", bf16_to_np(dbg["h"]), ref["h"])
    ck(check_logits, dbg["logits"].cpu().numpy(), ref["logits"])
    if entropy_given_h:
        Hg = out["entropy"].cpu().numpy().reshape(-1).astype(np.float64)
        # end to end: the documented bound of this case, with the rows past 1e-3 counted and printed
        e2e = np.abs(Hg - ref["H"])
        print(f"parity-report entropy end to end: max {e2e.max():.3e} nats, "
              f"{int((e2e > 1e-3).sum())} of {e2e.size} rows above 1e-3")

        bound = LONG_CANVAS_H_BOUND if e2e_bound is None else e2e_bound

        def e2e_within():
            assert e2e.max() <= bound, f"entropy end to end {e2e.max():.3e} > {bound}"
        ck(e2e_within)
        # given the device's own h: the LM head and the statistics merge, to the stated 1e-3
        ck(check_entropy, Hg, _entropy_given_device_h(dims, synth.to_numpy_f32(w), a.numpy(), bf16_to_np(dbg["h"]),
                                                      tau))
    else:
        ck(check_entropy, out["entropy"].cpu().numpy().reshape(-1), ref["H"])
    scale = np.max(np.abs(ref["logits"]), axis=1)
    n_am = ck(check_argmax, out["argmax"].cpu().numpy(), ref["argmax"], ref["top2gap"], scale)
    stats = ck(check_sampler, out["accept"].cpu().numpy(), canvas.tokens.cpu().numpy(), ref, b, C)
    # u, g, z: the stated relative-L2 tolerance (a chain of three bf16 roundings)
    ck(check_rel_l2, "u", bf16_to_np(dbg["u"]), ref["u"])
    ck(check_rel_l2, "g", bf16_to_np(dbg["g"]), ref["g"])
    zz = bf16_to_np(canvas.z).reshape(B * C, dims.d)
    ck(check_rel_l2, "z", zz, ref["z_out"])
    # per-canvas scalars
    def scalars():
        if stats and stats["boundary_excused"] == 0:
            assert np.array_equal(out["n_acc"].cpu().numpy(), ref["n_acc"]), (out["n_acc"], ref["n_acc"])
        assert np.allclose(out["mean_H"].cpu().numpy(), ref["meanH"], atol=1e-3), "mean_H"
        if n_am == 0:
            assert np.array_equal(out["stop"].cpu().numpy(), ref["stop"]), "stop"
            assert np.array_equal(canvas.prev_argmax.cpu().numpy().reshape(-1), ref["argmax"]), "prev"
    ck(scalars)
    print(dims, "stats", stats, "n_acc", out["n_acc"].cpu().numpy(), ref["n_acc"])
    ck.done()
    return out, ref, stats


def test_tiny_step():
    dims, seed = synth.workload("tiny_v512_c16")
    _run_and_compare(dims, seed)


def test_tiny_step_sharp_alpha_accepts_all():
    dims, seed = synth.workload("tiny_v512_c16")
    out, ref, stats = _run_and_compare(dims, seed, alpha=64.0, tau=0.4)
    assert stats["accepted"] == dims.C


def test_ragged_step_later_step_with_z():
    # several canvases, a vocabulary that leaves a partial tile, M not a multiple of 128
    seed = 11
    g = torch.Generator().manual_seed(5)
    z = (torch.randn(RAGGED.B, RAGGED.C, RAGGED.d, generator=g) * 0.02).to(torch.bfloat16)
    prev = np.random.default_rng(1).integers(0, RAGGED.V, size=(RAGGED.B, RAGGED.C)).astype(np.int32)
    _run_and_compare(RAGGED, seed, tau=0.55, step=3, z_in=z, prev=prev)


def test_ragged_step_tensor_core_attention():
    seed = 12
    g = torch.Generator().manual_seed(6)
    z = (torch.randn(RAGGED_TC.B, RAGGED_TC.C, RAGGED_TC.d, generator=g) * 0.02).to(torch.bfloat16)
    _run_and_compare(RAGGED_TC, seed, tau=0.7, step=2, z_in=z)


def test_long_canvas_entropy_given_h():
    # 600 rows of a d = 128 model with sharp alpha: a few q / k / v elements round to the other bf16
    # neighbour than the oracle's (fp32 against exact accumulation), which moves h by an ulp in a few
    # places and the end-to-end entropy by up to ~1.4e-3 nats (the logit scale alpha / (tau sqrt d)
    # is 2.4x that of the d = 1024 workload).  Every other quantity is compared end to end; the
    # entropy end to end against LONG_CANVAS_H_BOUND with the rows above 1e-3 counted, and against
    # the oracle's statistics of the device's own h (the LM head and the statistics merge) to 1e-3.
    dims = synth.Dims(V=1000, d=128, C=300, B=2, Hq=4, Hkv=2, hd=64, F=192, P=64, cap=64)
    _run_and_compare(dims, 14, tau=0.6, entropy_given_h=True)


def test_gumbel_search_flat_rows_every_group():
    """V = 131072 (1024 statistics groups), near-flat rows and b large enough that every position is
    accepted: every group of a row can hold the Gumbel-max winner, so the search passes its list of
    candidate groups and scans all of them; the sampled tokens against the oracle's."""
    dims = synth.Dims(V=131072, d=64, C=16, B=1, Hq=2, Hkv=1, hd=32, F=64, P=32)
    out, ref, stats = _run_and_compare(dims, 17, tau=0.8, b=1e9, alpha=0.5)
    assert stats["accepted"] == dims.C


def test_step_events_eager_and_captured():
    """Per-kernel events through the ABI: recorded by a host-launched step and by a replayed graph of
    the same step, every timed slot's pair recorded in order (non-negative elapsed time), and the
    step's results unchanged by the events."""
    from block_diffusion_text_gb300 import dg
    dims, seed = synth.workload("tiny_v512_c16")
    slots = [k for k in dg.PROF_SLOTS if k != "moe"]

    def events():
        ev = [None] * (2 * len(dg.PROF_SLOTS))
        for k in slots:
            i = dg.PROF_SLOTS.index(k)
            for e in (0, 1):
                ev[2 * i + e] = torch.cuda.Event(enable_timing=True)
                ev[2 * i + e].record()
        return ev

    outs = []
    for use_events in (False, True):
        _, _, _, _, model, canvas = _setup(dims, seed)
        ev = events() if use_events else None
        out = dg.denoise_step(model, canvas, tau=0.7, b=0.1, seed=seed, step=0, events=ev)
        torch.cuda.synchronize()
        assert model.status() == 0
        if use_events:
            for k in slots:
                i = dg.PROF_SLOTS.index(k)
                assert ev[2 * i].elapsed_time(ev[2 * i + 1]) >= 0.0, k
        outs.append((canvas.tokens.cpu(), canvas.z.cpu(), out["entropy"].cpu()))
        if use_events:  # the same step captured with its events, then replayed
            ev2 = events()
            g = torch.cuda.CUDAGraph()
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.graph(g, stream=s):
                dg.denoise_step(model, canvas, tau=0.7, b=0.1, seed=seed, step=1, events=ev2)
            g.replay()
            torch.cuda.synchronize()
            assert model.status() == 0
            for k in slots:
                i = dg.PROF_SLOTS.index(k)
                assert ev2[2 * i].elapsed_time(ev2[2 * i + 1]) >= 0.0, k
    for x, y in zip(outs[0], outs[1]):
        assert torch.equal(x, y)


@pytest.mark.parametrize("hd", [32, 64])
def test_split_k_clusters_small_heads(hd):
    """d = 2048 with 128 canvas rows: the q/k/v projection (64-column tiles, heads of 32 or 64) and
    FFW1 (GELU) run split over K on clusters of four CTAs that sum their slices in shared memory."""
    dims = synth.Dims(V=2000, d=2048, C=64, B=2, Hq=4, Hkv=2, hd=hd, F=1024, P=100, cap=160)
    g = torch.Generator().manual_seed(7)
    z = (torch.randn(dims.B, dims.C, dims.d, generator=g) * 0.02).to(torch.bfloat16)
    _run_and_compare(dims, 15 + hd, tau=0.7, step=1, z_in=z)


def test_tensor_core_attention_canvas_tail():
    dims = synth.Dims(V=512, d=64, C=40, B=1, Hq=2, Hkv=2, hd=128, F=64, P=128, cap=128)
    _run_and_compare(dims, 13)


@pytest.mark.slow
def test_sharp_rows_tempered():
    """alpha = 64 at tau = 0.4: each row's own token sits ~160 nats above the rest (the widest
    logit range of the method's schedule), every row near zero entropy and accepted; every row is
    compared end to end at V = 32768."""
    dims, seed = synth.workload("step_v32k_c256_p2k")
    _run_and_compare(dims, seed, alpha=64.0, tau=0.4)


@pytest.mark.slow
def test_single_step_v32k():
    dims, seed = synth.workload("step_v32k_c256_p2k")
    out, ref, stats = _run_and_compare(dims, seed)
    print("accepted", stats)
