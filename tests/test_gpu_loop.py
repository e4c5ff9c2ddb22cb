"""Canvas initialisation, the annealed loop, the commit and determinism, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from block_diffusion_text_gb300 import synth

from parity import (Collect, bf16_to_np, boundary_excused, check_close_bf16, check_entropy, check_logits,
                    check_rel_l2, check_sampler, GUMBEL_GAP_TOL)

pytestmark = pytest.mark.gpu

TINY = synth.workload("tiny_v512_c16")[0]


def _model(dims, seed, alpha=None):
    from block_diffusion_text_gb300 import dg
    w = synth.make_weights(dims, seed, device="cpu")
    x, z, a = synth.make_canvas(dims, seed, device="cpu")
    if alpha is not None:
        a = torch.full_like(a, alpha)
    model = dg.Model(dims, {k: v.cuda() for k, v in w.items()})
    return w, x, z, a, model


def test_canvas_init_matches_oracle():
    from block_diffusion_text_gb300 import dg
    for (B, C, V, seed, block) in ((3, 40, 1000, 5, 2), (1, 256, 262144, 2, 0), (8, 256, 32768, 4, 3)):
        t = dg.canvas_init(B, C, V, seed, block)
        torch.cuda.synchronize()
        assert np.array_equal(t.cpu().numpy(), oracle.canvas_init(B, C, V, seed, block))


def test_loop_sharp_alpha_converges_at_step_one():
    from block_diffusion_text_gb300 import dg
    w, x, z, a, model = _model(TINY, 5, alpha=64.0)
    canvas = dg.Canvas(x.cuda(), z.cuda(), a.cuda())
    res = dg.denoise_canvas(model, canvas, seed=5, N=48)
    torch.cuda.synchronize()
    assert model.status() == 0
    ref = oracle.denoise_canvas(TINY, synth.to_numpy_f32(w), x.numpy(), a.numpy(), seed=5, N=48)
    assert res["steps_taken"].cpu().tolist() == ref["steps_taken"].tolist() == [2]
    assert res["converged"].cpu().tolist() == [1]
    acc = res["accepted"].cpu().numpy()
    assert acc[0, 0] == TINY.C and acc[0, 1] == TINY.C and (acc[0, 2:] == -1).all()
    assert np.array_equal(res["xhat0"].cpu().numpy(), ref["xhat0"])


def test_loop_canvases_stop_independently():
    """Three canvases in one batch: the sharp first and last stop at step 1 (adaptive stop), the
    middle one runs every step.  Stopped canvases are left untouched by the later steps (their
    tokens, z and x0 equal the oracle's frozen state) while the batch goes on."""
    from block_diffusion_text_gb300 import dg
    dims = synth.Dims(V=512, d=64, C=16, B=3, Hq=2, Hkv=1, hd=32, F=128, P=32)
    N = 6
    w, x, z, a, model = _model(dims, 8)
    a[0] = 64.0
    a[2] = 64.0
    canvas = dg.Canvas(x.cuda(), z.cuda(), a.cuda())
    res = dg.denoise_canvas(model, canvas, seed=8, N=N)
    torch.cuda.synchronize()
    assert model.status() == 0
    ref = oracle.denoise_canvas(dims, synth.to_numpy_f32(w), x.numpy(), a.numpy(), seed=8, N=N)
    steps = res["steps_taken"].cpu().numpy()
    assert steps.tolist() == ref["steps_taken"].tolist()
    assert res["converged"].cpu().tolist() == ref["converged"].tolist()
    assert steps[0] == steps[2] == 2 and steps[1] > 2  # the batch outlives its stopped canvases
    acc = res["accepted"].cpu().numpy()
    tok = canvas.tokens.cpu().numpy()
    zz = bf16_to_np(canvas.z).reshape(dims.B, dims.C, dims.d)
    for b in (0, 2):
        assert np.array_equal(acc[b], ref["accepted"][b]), b
        assert (acc[b, 2:] == -1).all()
        assert np.array_equal(res["xhat0"][b].cpu().numpy(), ref["xhat0"][b])
        assert np.array_equal(tok[b], ref["tokens"][b])
        assert check_rel_l2(f"z canvas {b}", zz[b], ref["z"][b]) <= 1e-2
    assert (acc[1] >= 0).all()


def test_loop_stops_launching_once_every_canvas_stopped():
    """With sharp alpha every canvas stops at step 1.  Outside a capture the loop reads the 4-byte
    stopped count after step 1 and enqueues nothing more, so the 48-step loop costs about two steps
    and a flag read, not 48 steps of kernels that exit at once; the result equals the oracle's."""
    import time
    from block_diffusion_text_gb300 import dg
    dims, seed = synth.workload("step_v32k_c256_p2k")
    w, x, z, a, model = _model(dims, seed, alpha=64.0)
    c = dg.Canvas(x.cuda(), z.cuda(), a.cuda())
    for s in range(3):
        dg.denoise_step(model, c, tau=0.8, b=0.1, seed=seed, step=s)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s in range(8):
        dg.denoise_step(model, c, tau=0.8, b=0.1, seed=seed, step=s)
    torch.cuda.synchronize()
    t_step = (time.perf_counter() - t0) / 8
    times = []
    for _ in range(3):
        canvas = dg.Canvas(x.cuda(), z.cuda(), a.cuda())
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        res = dg.denoise_canvas(model, canvas, seed=seed, N=48)
        torch.cuda.synchronize()
        times.append(time.perf_counter() - t0)
    assert model.status() == 0
    assert res["steps_taken"].cpu().tolist() == [2] and res["converged"].cpu().tolist() == [1]
    acc = res["accepted"].cpu().numpy()
    assert (acc[0, :2] >= 0).all() and (acc[0, 2:] == -1).all()
    print(f"loop {min(times) * 1e3:.3f} ms, one step {t_step * 1e3:.3f} ms")
    assert min(times) < 8 * t_step


def _step_by_step(dims, seed, N, alpha=None):
    """GPU and oracle loops side by side, each from its own state; returns per-step agreement."""
    from block_diffusion_text_gb300 import dg
    w, x, z, a, model = _model(dims, seed, alpha)
    wn = synth.to_numpy_f32(w)
    canvas = dg.Canvas(x.cuda(), z.cuda(), a.cuda())
    taus = dg.tau_schedule(N)
    ox, oz, oprev = x.numpy().copy(), z.float().numpy().copy(), None
    agree = []
    for s in range(N):
        out = dg.denoise_step(model, canvas, tau=taus[s], b=0.1, seed=seed, step=s)
        torch.cuda.synchronize()
        ref = oracle.denoise_step(dims, wn, ox, oz, a.numpy(), tau=taus[s], b=0.1, seed=seed, step=s,
                                  prev_argmax=oprev)
        gt = canvas.tokens.cpu().numpy().reshape(-1)
        ex = boundary_excused(ref["H"], ref["cum"], ref["accept"], 0.1, dims.C)
        acc_g = out["accept"].cpu().numpy().reshape(-1).astype(bool)
        same_acc = np.array_equal(acc_g, ref["accept"])
        samp_ok = np.all((gt == ref["tokens_out"]) | (acc_g & (ref["gumbel_gap"] < GUMBEL_GAP_TOL)))
        agree.append(dict(step=s, tokens_equal=bool(np.array_equal(gt, ref["tokens_out"])),
                          accept_equal=same_acc, excusable=bool(ex.any() or not samp_ok),
                          n_acc=(int(out["n_acc"][0]), int(ref["n_acc"][0]))))
        if not agree[-1]["tokens_equal"]:
            break
        zg = bf16_to_np(canvas.z).reshape(dims.M, dims.d)
        assert check_rel_l2("z", zg, ref["z_out"]) <= 1e-2
        ox = ref["tokens_out"].reshape(x.shape).astype(np.int32)
        oz = ref["z_out"].astype(np.float32).reshape(z.shape)
        oprev = ref["argmax"].reshape(x.shape)
    return agree, model, w, x, z, a


def test_loop_trajectory_follows_oracle():
    agree, *_ = _step_by_step(TINY, 3, N=6)
    print(agree)
    for r in agree:
        assert r["tokens_equal"] or r["excusable"], r


def test_denoise_canvas_equals_step_by_step():
    from block_diffusion_text_gb300 import dg
    N = 5
    w, x, z, a, model = _model(TINY, 7)
    c1 = dg.Canvas(x.cuda(), z.cuda(), a.cuda())
    res = dg.denoise_canvas(model, c1, seed=7, N=N)
    c2 = dg.Canvas(x.cuda(), z.cuda(), a.cuda())
    taus = dg.tau_schedule(N)
    for s in range(N):
        dg.denoise_step(model, c2, tau=taus[s], b=0.1, seed=7, step=s)
    torch.cuda.synchronize()
    assert torch.equal(c1.tokens, c2.tokens)
    assert torch.equal(c1.z, c2.z)
    assert torch.equal(res["xhat0"], c2.prev_argmax)
    assert res["steps_taken"].item() == N and res["converged"].item() == 0


def test_step_is_deterministic():
    from block_diffusion_text_gb300 import dg
    dims = synth.Dims(V=1000, d=128, C=40, B=3, Hq=4, Hkv=2, hd=64, F=192, P=100, cap=160)
    w, x, z, a, model = _model(dims, 2)
    outs = []
    for _ in range(2):
        c = dg.Canvas(x.cuda(), z.cuda(), a.cuda())
        o = dg.denoise_step(model, c, tau=0.7, b=0.1, seed=2, step=1)
        torch.cuda.synchronize()
        outs.append((c.tokens.clone(), c.z.clone(), o["entropy"].clone()))
    for t1, t2 in zip(*outs):
        assert torch.equal(t1, t2)


def test_commit_matches_oracle_and_checks_capacity():
    from block_diffusion_text_gb300 import dg
    dims = synth.Dims(V=1000, d=128, C=40, B=2, Hq=4, Hkv=2, hd=64, F=192, P=100, cap=180)
    w, x, z, a, model = _model(dims, 9)
    toks = torch.randint(0, dims.V, (dims.B, dims.C), dtype=torch.int32, generator=torch.Generator().manual_seed(1))
    dg.commit_block(model, toks.cuda())
    torch.cuda.synchronize()
    assert model.len == dims.P + dims.C
    wn = synth.to_numpy_f32(w)
    Kr, Vr = oracle.commit(dims, wn["E"], wn["Wk"], wn["Wv"], toks.numpy(), wn["Kc"], wn["Vc"], P=dims.P)
    K = bf16_to_np(model.K)
    V = bf16_to_np(model.V)
    assert np.array_equal(K[:, :, :dims.P], Kr[:, :, :dims.P])
    sl = slice(dims.P, dims.P + dims.C)
    check_close_bf16("k", K[:, :, sl], Kr[:, :, sl])
    check_close_bf16("v", V[:, :, sl], Vr[:, :, sl])
    assert np.all(K[:, :, dims.P + dims.C:] == 0)
    before = model.K.clone()
    with pytest.raises(dg.DgError) as e:
        dg.commit_block(model, toks.cuda())  # 140 + 40 > 180? no: fits; commit twice more
        dg.commit_block(model, toks.cuda())
    assert e.value.code == dg.DG_ERR_CAPACITY
    torch.cuda.synchronize()
    assert model.len == dims.P + 2 * dims.C
    assert torch.equal(model.K[:, :, :dims.P + dims.C], before[:, :, :dims.P + dims.C])


def _check_sampled_rows(ck, dims, wn, x0, z0, alpha, prev, out, canvas, seed, step, tau, block=0,
                        all_rows=False):
    """One device step against the oracle run from the same state (tokens x0, z0, previous argmax,
    the prefix cache in wn).  Sampled rows (including the last row, whose logits span the LM head's
    final half tiles like every row's) get the logits at the 2e-2 tolerance.  With all_rows the
    oracle runs the vocabulary stages on every row, and entropy, z, argmax and the accept / renoise
    decisions with the renoised and sampled tokens are compared on every row (check_sampler: exact,
    with counted boundary and Gumbel-gap excuses); otherwise the sampled rows get those checks and
    the acceptance invariants are checked on the device's own entropies.  Returns (n_acc per
    canvas, counts of excused positions)."""
    M = dims.M
    rows = sorted({0, 1, M // 3, M // 2 + 7, M - 1})
    want = ("h", "H", "m", "argmax", "top2gap", "sample_tok", "gumbel_gap", "renoise_tok", "z_out")
    if all_rows:
        want = want + ("accept", "cum", "tokens_out", "n_acc")
    ref = oracle.denoise_step(dims, wn, x0, z0, alpha, tau=tau, b=0.1, seed=seed, step=step, block=block,
                              prev_argmax=prev, rows=None if all_rows else rows, want=want)
    ref_l = oracle.denoise_step(dims, wn, x0, z0, alpha, tau=tau, b=0.1, seed=seed, step=step, block=block,
                                prev_argmax=prev, rows=rows, want=("logits",))["logits"]
    H = out["entropy"].cpu().numpy().reshape(-1)
    am = out["argmax"].cpu().numpy().reshape(-1)
    acc = out["accept"].cpu().numpy().reshape(-1).astype(bool)
    tok = canvas.tokens.cpu().numpy().reshape(-1)
    tag = f"step {step}"
    chk = list(range(M)) if all_rows else rows
    ck(check_close_bf16, f"h ({tag})", bf16_to_np(out["debug"]["h"])[chk], ref["h"][chk])
    ck(check_entropy, H[chk], ref["H"][chk])
    zz = bf16_to_np(canvas.z).reshape(M, dims.d)
    ck(check_rel_l2, f"z ({tag})", zz[chk], ref["z_out"][chk])
    logits = out["debug"]["logits"][rows].cpu().numpy()
    ck(check_logits, logits, ref_l)
    counts = dict(boundary_excused=0, sample_excused=0, argmax_excused=0)
    # row scale of the argmax excuse: the largest |logit| where the logits were fetched, else the row's
    # largest logit (m is the maximum of l / tau)
    scale = np.abs(np.asarray(ref["m"], np.float64)) * tau
    scale[rows] = np.abs(ref_l).max(axis=1)
    for r in chk:
        if am[r] != ref["argmax"][r]:
            if ref["top2gap"][r] < 1e-4 * scale[r]:
                counts["argmax_excused"] += 1
            else:
                ck.errors.append(f"{tag}: argmax row {r}")
    if all_rows:
        st = ck(check_sampler, acc, tok, ref, 0.1, dims.C)
        if st:
            counts.update(boundary_excused=st["boundary_excused"], sample_excused=st["sample_excused"])
        if counts["boundary_excused"] == 0 and not np.array_equal(out["n_acc"].cpu().numpy(), ref["n_acc"]):
            ck.errors.append(f"{tag}: n_acc {out['n_acc'].cpu().numpy()} vs {ref['n_acc']}")
    else:
        for r in rows:
            if acc[r]:
                if tok[r] != ref["sample_tok"][r]:
                    if ref["gumbel_gap"][r] >= GUMBEL_GAP_TOL:
                        ck.errors.append(f"{tag}: sample row {r}")
                    else:
                        counts["sample_excused"] += 1
            elif tok[r] != ref["renoise_tok"][r]:
                ck.errors.append(f"{tag}: renoise row {r}")
    # acceptance invariants on the device's own entropies, per canvas
    for b in range(dims.B):
        Hb = H[b * dims.C:(b + 1) * dims.C].astype(np.float64)
        ab = acc[b * dims.C:(b + 1) * dims.C]
        order = np.lexsort((np.arange(dims.C), Hb))
        n = int(ab.sum())
        if set(np.nonzero(ab)[0]) != set(order[:n]):
            ck.errors.append(f"{tag}, canvas {b}: accepted set is not a sorted prefix")
        if Hb[ab].sum() > 0.1 + 1e-6:
            ck.errors.append(f"{tag}, canvas {b}: accepted entropy {Hb[ab].sum()} > b")
        if n < dims.C and Hb[ab].sum() + Hb[order[n]] <= 0.1 - 1e-6:
            ck.errors.append(f"{tag}, canvas {b}: prefix not maximal")
        if n != int(out["n_acc"][b]):
            ck.errors.append(f"{tag}, canvas {b}: n_acc")
    print(f"parity-report {tag}: rows checked {len(chk)}, excused {counts}")
    return out["n_acc"].cpu().tolist(), counts


@pytest.mark.slow
@pytest.mark.parametrize("name", ["loop_v262k_c256_p8k", "prefix_p131k_v32k_c256", "blocks_b8_v32k_p4k"])
def test_full_size_step_all_rows(name):
    """Full-size step in the launch configuration of the benchmark against the oracle on every row:
    entropy, z, argmax and the accept / renoise decisions with their tokens (excused positions
    counted and printed), logits on sampled rows."""
    from block_diffusion_text_gb300 import dg
    dims, seed = synth.workload(name)
    dev = torch.device("cuda")
    w = synth.make_weights(dims, seed, device=dev)
    x, z, a = synth.make_canvas(dims, seed, device=dev)
    x0, z0 = x.clone(), z.clone()
    model = dg.Model(dims, w)
    canvas = dg.Canvas(x, z, a)
    out = dg.denoise_step(model, canvas, tau=0.8, b=0.1, seed=seed, step=0, debug=True)
    torch.cuda.synchronize()
    assert model.status() == 0
    ck = Collect()
    n_acc, counts = _check_sampled_rows(ck, dims, synth.to_numpy_f32(w), x0.cpu().numpy(),
                                        z0.float().cpu().numpy(), a.cpu().numpy(), None, out, canvas, seed, 0,
                                        0.8, all_rows=True)
    print(name, "accepted per canvas", n_acc, "excused", counts)
    ck.done()


@pytest.mark.slow
def test_full_size_loop_teacher_forced():
    """The 48-step annealed loop at V = 262144, C = 256, P = 8192: steps 0, 1, 24 and 47 checked
    against the oracle run from the device's own state before that step (free-running
    trajectories may part after an excused mismatch, so they are not compared)."""
    from block_diffusion_text_gb300 import dg
    dims, seed = synth.workload("loop_v262k_c256_p8k")
    N = 48
    dev = torch.device("cuda")
    w = synth.make_weights(dims, seed, device=dev)
    x, z, a = synth.make_canvas(dims, seed, device=dev)
    model = dg.Model(dims, w)
    canvas = dg.Canvas(x, z, a)
    wn = synth.to_numpy_f32(w)
    taus = dg.tau_schedule(N)
    ck = Collect()
    log = []
    for s in range(N):
        check = s in (0, 1, N // 2, N - 1)
        if check:
            x0 = canvas.tokens.cpu().numpy().copy()
            z0 = canvas.z.float().cpu().numpy().copy()
            prev = canvas.prev_argmax.cpu().numpy().copy() if s > 0 else None
        out = dg.denoise_step(model, canvas, tau=taus[s], b=0.1, seed=seed, step=s, debug=check)
        if check:
            torch.cuda.synchronize()
            assert model.status() == 0
            log.append((s, _check_sampled_rows(ck, dims, wn, x0, z0, a.cpu().numpy(), prev, out, canvas, seed,
                                               s, taus[s])[0]))
    print("accepted per checked step", log)
    ck.done()


@pytest.mark.slow
def test_full_size_blocks_commit_teacher_forced():
    """8 canvases at V = 32768: block 0 runs the annealed loop (adaptive stop), its x0 is committed
    (checked against the oracle's re-encode of the same tokens), and step 0 of block 1 on the
    committed cache is checked against the oracle given that cache."""
    import dataclasses
    from block_diffusion_text_gb300 import dg
    dims, seed = synth.workload("blocks_b8_v32k_p4k")
    dev = torch.device("cuda")
    w = synth.make_weights(dims, seed, device=dev)
    x, z, a = synth.make_canvas(dims, seed, device=dev)
    model = dg.Model(dims, w)
    wn = synth.to_numpy_f32(w)
    canvas = dg.Canvas(dg.canvas_init(dims.B, dims.C, dims.V, seed, 0), z.clone(), a)
    res = dg.denoise_canvas(model, canvas, seed=seed, block=0, N=48)
    xhat0 = res["xhat0"].clone()
    dg.commit_block(model, xhat0)
    torch.cuda.synchronize()
    assert model.status() == 0 and model.len == dims.P + dims.C
    Kr, Vr = oracle.commit(dims, wn["E"], wn["Wk"], wn["Wv"], xhat0.cpu().numpy(), wn["Kc"], wn["Vc"], P=dims.P)
    K, V = bf16_to_np(model.K), bf16_to_np(model.V)
    sl = slice(dims.P, dims.P + dims.C)
    assert np.array_equal(K[:, :, :dims.P], Kr[:, :, :dims.P])
    ck = Collect()
    ck(check_close_bf16, "committed k", K[:, :, sl], Kr[:, :, sl])
    ck(check_close_bf16, "committed v", V[:, :, sl], Vr[:, :, sl])
    # block 1, step 0, on the device's committed cache
    d1 = dataclasses.replace(dims, P=dims.P + dims.C)
    w1 = dict(wn, Kc=K, Vc=V)
    c1 = dg.Canvas(dg.canvas_init(dims.B, dims.C, dims.V, seed, 1), torch.zeros_like(z), a)
    x0 = c1.tokens.cpu().numpy().copy()
    out = dg.denoise_step(model, c1, tau=0.8, b=0.1, seed=seed, step=0, block=1, debug=True)
    torch.cuda.synchronize()
    assert model.status() == 0
    n_acc, _ = _check_sampled_rows(ck, d1, w1, x0, np.zeros((dims.B, dims.C, dims.d), np.float32),
                                   a.cpu().numpy(), None, out, c1, seed, 0, 0.8, block=1)
    print("block 0 steps", res["steps_taken"].cpu().tolist(), "block 1 step 0 accepted", n_acc)
    ck.done()


def test_steps_captured_in_a_cuda_graph_match_eager_steps():
    from block_diffusion_text_gb300 import dg
    dims, seed = synth.workload("step_v32k_c256_p2k")
    w, x, z, a, model = _model(dims, seed)
    taus = dg.tau_schedule(48)
    eager = dg.Canvas(x.cuda(), z.cuda(), a.cuda())
    out = None
    for s in range(3):
        out = dg.denoise_step(model, eager, tau=taus[s], b=0.1, seed=seed, step=s, out=out)
    torch.cuda.synchronize()
    graphed = dg.Canvas(x.cuda(), z.cuda(), a.cuda())
    out2 = dg.denoise_step(model, dg.Canvas(x.cuda(), z.cuda(), a.cuda()), tau=0.8, b=0.1, seed=seed, step=0)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=cap):
        for s in range(3):
            dg.denoise_step(model, graphed, tau=taus[s], b=0.1, seed=seed, step=s, out=out2)
    g.replay()
    torch.cuda.synchronize()
    assert model.status() == 0
    assert torch.equal(graphed.tokens, eager.tokens)
    assert torch.equal(graphed.z, eager.z)
    assert torch.equal(out2["entropy"], out["entropy"])
