"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: published
known answers, closed forms, invariants, library routines that the operation
reduces to in a special case, or brute force on tiny inputs.
"""
import dataclasses
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
from block_diffusion_text_gb300 import synth

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


# --------------------------------------------------------------- Philox -----
def _kat(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "philox4x64_10_kat.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            w = [int(t, 16) for t in line.split()]
            rows.append((w[0:4], w[4:6], w[6:10]))
    return rows


def test_philox_known_answers(golden_dir):
    rows = _kat(golden_dir)
    assert len(rows) == 3
    for ctr, key, want in rows:
        got = [int(x) for x in oracle.philox4x64_10(ctr, key)]
        assert got == want


def test_philox_matches_numpy():
    # numpy's Philox (4x64, 10 rounds) bumps its 256-bit counter before each
    # block, so the block of counter c is produced from state c - 1.
    rng = np.random.default_rng(123)
    for _ in range(200):
        ctr = [int(x) for x in rng.integers(0, 2**64, size=4, dtype=np.uint64)]
        key = [int(x) for x in rng.integers(0, 2**64, size=2, dtype=np.uint64)]
        c = (sum(w << (64 * i) for i, w in enumerate(ctr)) - 1) % (1 << 256)
        cw = np.array([(c >> (64 * i)) & (2**64 - 1) for i in range(4)], dtype=np.uint64)
        want = np.random.Philox(key=np.array(key, dtype=np.uint64), counter=cw).random_raw(4)
        got = oracle.philox4x64_10(ctr, key)
        assert [int(x) for x in got] == [int(x) for x in want]


def test_philox_word_streams_differ():
    a = oracle.philox_word(5, 0, 3, 0, 7, 0, 0)
    b = oracle.philox_word(5, 0, 3, 0, 7, 0, 1)
    c = oracle.philox_word(5, 0, 4, 0, 7, 0, 1)
    d = oracle.philox_word(5, 1, 3, 0, 7, 0, 1)
    assert len({a, b, c, d}) == 4
    # four consecutive vocabulary indices share one Philox block
    blk = oracle.philox4x64_10([1, 7, (0 << 32) | 3, (0 << 32) | 0], [5, 0])
    for v in range(4, 8):
        assert oracle.philox_word(5, 0, 3, 0, 7, v, 0) == int(blk[v & 3])


# ------------------------------------------------------- uniform tokens -----
def test_uniform_token_exact_high_word():
    rng = np.random.default_rng(1)
    for _ in range(1000):
        w = int(rng.integers(0, 2**64, dtype=np.uint64))
        V = int(rng.integers(1, 2**31 - 1))
        assert oracle.uniform_token(w, V) == (w * V) >> 64
    assert oracle.uniform_token(2**64 - 1, 262144) == 262143
    assert oracle.uniform_token(0, 262144) == 0


def test_uniform_tokens_chi_square():
    from scipy import stats
    V, n = 512, 400_000
    t = oracle.uniform_many(V, 11, n)
    assert t.min() >= 0 and t.max() < V
    counts = np.bincount(t, minlength=V)
    chi2 = ((counts - n / V) ** 2 / (n / V)).sum()
    p = stats.chi2.sf(chi2, V - 1)
    assert p > 1e-4, (chi2, p)


def test_canvas_init_in_range_and_seeded():
    a = oracle.canvas_init(2, 64, 1000, seed=3, block=0)
    b = oracle.canvas_init(2, 64, 1000, seed=3, block=1)
    assert a.min() >= 0 and a.max() < 1000
    assert not np.array_equal(a, b)
    assert np.array_equal(a, oracle.canvas_init(2, 64, 1000, seed=3, block=0))


# ---------------------------------------------------------------- Gumbel ----
def test_gumbel_moments():
    g = oracle.gumbel_many(3, 1_000_000).astype(np.float64)
    assert np.isfinite(g).all()
    assert abs(g.mean() - 0.5772156649) < 5e-3          # Euler-Mascheroni constant
    assert abs(g.var() - math.pi ** 2 / 6) < 2e-2
    assert g.min() >= -2.82 and g.max() <= 16.7


def test_gumbel_max_law():
    # argmax(s + G) is distributed as softmax(s) (the Gumbel-max trick).
    from scipy import stats
    s = np.array([0.0, 1.0, -0.5, 2.0, 0.3, -1.0, 1.5, 0.7])
    n = 200_000
    t = oracle.gumbel_argmax_many(s, 9, n)
    p = np.exp(s - s.max())
    p /= p.sum()
    counts = np.bincount(t, minlength=s.size)
    chi2 = ((counts - n * p) ** 2 / (n * p)).sum()
    assert stats.chi2.sf(chi2, s.size - 1) > 1e-4, (counts, n * p)


def test_gumbel_argmax_of_one_hot_row():
    s = np.full(1000, -1e4)
    s[417] = 0.0
    i, gap = oracle.gumbel_argmax(s, seed=1, pos=3)
    assert i == 417 and gap > 1e3


# ---------------------------------------------------------- bf16 rounding ---
def test_round_bf16_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(5000).astype(np.float32),
                        (rng.standard_normal(1000) * 1e-30).astype(np.float32),
                        (rng.standard_normal(1000) * 1e30).astype(np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.round_bf16(float(v)) for v in x])
    assert np.array_equal(got, want)
    # ties go to even
    assert oracle.round_bf16(1.0 + 2 ** -8) == 1.0
    assert oracle.round_bf16(1.0 + 3 * 2 ** -8) == 1.0 + 2 ** -6


# ------------------------------------------------------------- RMSNorm ------
def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(1024) * 3.0
    y = oracle.rmsnorm(x, 1e-6)
    ms = np.mean(x * x)
    assert abs(np.sqrt(np.mean(y * y)) - np.sqrt(ms / (ms + 1e-6))) < 1e-12
    y2 = oracle.rmsnorm(5.0 * x, 0.0)
    assert np.allclose(y2, oracle.rmsnorm(x, 0.0), rtol=1e-13, atol=0)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (1024,), eps=1e-6).numpy()
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- RoPE ------
def test_rope_complex_form_and_norm():
    rng = np.random.default_rng(3)
    hd = 32
    x = rng.standard_normal(hd)
    pos = 123.0
    y = oracle.rope(x, pos, 10000.0)
    # complex form: (x_j + i x_{j+hd/2}) * exp(i pos base^(-2j/hd))
    zc = (x[: hd // 2] + 1j * x[hd // 2:]) * np.exp(1j * pos * 10000.0 ** (-2.0 * np.arange(hd // 2) / hd))
    assert np.allclose(y, np.concatenate([zc.real, zc.imag]), rtol=0, atol=1e-12)
    assert abs(np.linalg.norm(y) - np.linalg.norm(x)) < 1e-12
    assert np.array_equal(oracle.rope(x, 0.0, 10000.0), x)


def test_rope_relative_position():
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    d1 = oracle.rope(q, 1000.0, 10000.0) @ oracle.rope(k, 990.0, 10000.0)
    d2 = oracle.rope(q, 20.0, 10000.0) @ oracle.rope(k, 10.0, 10000.0)
    assert abs(d1 - d2) < 1e-10


# ---------------------------------------------------------------- GELU ------
def test_gelu_matches_torch():
    xs = np.linspace(-6, 6, 241)
    want = torch.nn.functional.gelu(torch.from_numpy(xs), approximate="none").numpy()
    got = np.array([oracle.gelu(v) for v in xs])
    assert np.allclose(got, want, rtol=1e-14, atol=1e-15)


# ------------------------------------------------------------- entropy ------
def test_entropy_uniform_row_is_log_v():
    for V in (512, 32768):
        st = oracle.row_stats(np.full(V, 0.37), 0.8)
        assert abs(st["H"] - math.log(V)) < 1e-12
        assert st["argmax"] == 0


def test_entropy_two_level_closed_form():
    V, tau = 512, 0.8
    for a in (0.5, 3.0, 20.0, 80.0):
        l = np.zeros(V)
        l[7] = a * tau  # s = l / tau puts one logit at a and V-1 at 0
        Z = math.exp(a) + V - 1
        want = math.log(Z) - a * math.exp(a) / Z
        st = oracle.row_stats(l, tau)
        assert abs(st["H"] - want) < 1e-12
        assert st["argmax"] == 7


def test_entropy_matches_scipy_and_bounds():
    from scipy import special, stats
    rng = np.random.default_rng(5)
    for tau in (0.8, 0.4):
        l = rng.standard_normal(4096) * 4.0
        st = oracle.row_stats(l, tau)
        p = special.softmax(l / tau)
        assert abs(st["H"] - stats.entropy(p)) < 1e-10
        assert 0.0 <= st["H"] <= math.log(l.size)
        assert st["argmax"] == int(np.argmax(l))
        assert abs(st["m"] - l.max() / tau) < 1e-12
        # temperature enters only through l / tau
        st2 = oracle.row_stats(l / tau, 1.0)
        assert abs(st2["H"] - st["H"]) < 1e-12


# ---------------------------------------------------------- acceptance ------
def test_accept_bruteforce_max_cardinality():
    # Accepting the smallest entropies first maximises how many positions fit
    # in the budget; brute force over every subset confirms the count, and the
    # accepted set is the sorted prefix of that size.
    rng = np.random.default_rng(6)
    for trial in range(300):
        C = int(rng.integers(1, 11))
        H = rng.exponential(0.04, size=C)
        if trial % 5 == 0:
            H[rng.integers(0, C)] = H[rng.integers(0, C)]  # ties
        b = 0.1
        best = 0
        for r in range(C + 1):
            for S in itertools.combinations(range(C), r):
                if sum(H[list(S)]) <= b + 1e-15:
                    best = max(best, r)
        res = oracle.accept(H, b)
        assert res["n"] == best
        order = sorted(range(C), key=lambda i: (H[i], i))
        assert set(np.nonzero(res["accept"])[0]) == set(order[: res["n"]])
        if res["n"] < C:
            assert H[res["accept"]].sum() + H[order[res["n"]]] > b


def test_accept_edge_cases():
    assert oracle.accept([0.2, 0.3, math.log(512)], 0.1)["n"] == 0          # H_min > b
    assert oracle.accept([0.01, 0.02, 0.03], 0.1)["n"] == 3                 # sum <= b
    r = oracle.accept([0.05, 0.05], 0.1)                                    # sum == b
    assert r["n"] == 2
    r = oracle.accept([0.06, 0.06, 0.06], 0.1)                              # equal, ties by index
    assert list(r["accept"]) == [True, False, False]
    r = oracle.accept(np.full(16, math.log(512)), 0.1)                      # uniform rows
    assert r["n"] == 0


# ---------------------------------------------------------- attention -------
def test_attention_matches_sdpa():
    rng = np.random.default_rng(7)
    hd = 16
    for P, C in ((8, 4), (0, 5), (33, 1)):
        q = rng.standard_normal(hd)
        Kp, Vp = rng.standard_normal((P, hd)), rng.standard_normal((P, hd))
        Kc, Vc = rng.standard_normal((C, hd)), rng.standard_normal((C, hd))
        Kp32, Vp32 = Kp.astype(np.float32), Vp.astype(np.float32)
        o = oracle.attend_row(q, Kp32, Vp32, Kc, Vc)
        K = torch.from_numpy(np.concatenate([Kp32.astype(np.float64), Kc]))
        Vv = torch.from_numpy(np.concatenate([Vp32.astype(np.float64), Vc]))
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q)[None, None, None], K[None, None], Vv[None, None])[0, 0, 0].numpy()
        assert np.allclose(o, ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------ the whole step ------
TINY = synth.workload("tiny_v512_c16")[0]


def _tiny_inputs(dtype=torch.float32, alpha=None, seed=0, dims=TINY):
    w = synth.to_numpy_f32(synth.make_weights(dims, seed, dtype=dtype))
    x, z, a = synth.make_canvas(dims, seed, dtype=dtype)
    if alpha is not None:
        a = torch.full_like(a, alpha)
    return w, x.numpy(), z.to(torch.float32).numpy(), a.numpy()


def _torch_forward(dims, w, x, z, mirror):
    """Independent float64 composition of library routines for a1..a4."""
    f = lambda k: torch.from_numpy(w[k]).double()
    rb = (lambda t: t.to(torch.bfloat16).double()) if mirror else (lambda t: t)
    B, C, d, Hq, Hkv, hd, P = dims.B, dims.C, dims.d, dims.Hq, dims.Hkv, dims.hd, dims.P
    e = f("E")[torch.from_numpy(x).long()] + torch.from_numpy(z).double()
    a = rb(torch.nn.functional.rms_norm(e, (d,), eps=dims.rms_eps))
    q = (a @ f("Wq").T).view(B, C, Hq, hd).transpose(1, 2)
    k = (a @ f("Wk").T).view(B, C, Hkv, hd).transpose(1, 2)
    v = rb((a @ f("Wv").T).view(B, C, Hkv, hd).transpose(1, 2))
    pos = torch.arange(P, P + C, dtype=torch.float64)
    ang = pos[:, None] * dims.rope_base ** (-2.0 * torch.arange(hd // 2, dtype=torch.float64) / hd)
    rot = torch.polar(torch.ones_like(ang), ang)

    def rope(t):
        c = torch.complex(t[..., : hd // 2], t[..., hd // 2:]) * rot
        return torch.cat([c.real, c.imag], -1)

    q, k = rb(rope(q)), rb(rope(k))
    Kall = torch.cat([f("Kc")[:, :, :P], k], 2)
    Vall = torch.cat([f("Vc")[:, :, :P], v], 2)
    rep = Hq // Hkv
    o = torch.nn.functional.scaled_dot_product_attention(
        q, Kall.repeat_interleave(rep, 1), Vall.repeat_interleave(rep, 1))
    o = rb(o.transpose(1, 2).reshape(B, C, Hq * hd))
    h = rb(a + o @ f("Wo").T)
    return a.reshape(B * C, d), o.reshape(B * C, -1), h.reshape(B * C, d)


@pytest.mark.parametrize("mirror", [False, True])
def test_step_forward_matches_library_composition(mirror):
    dtype = torch.bfloat16 if mirror else torch.float32
    w, x, z, a = _tiny_inputs(dtype)
    out = oracle.denoise_step(TINY, w, x, z, a, tau=0.8, b=0.1, seed=0, step=0,
                              mirror_bf16=mirror, want=("a", "o", "h"), nthreads=2)
    ra, ro, rh = _torch_forward(TINY, w, x, z, mirror)
    tol = 1e-10 if not mirror else 1e-2  # bf16 mirrors may flip one ulp at a rounding edge
    assert np.allclose(out["a"], ra.numpy(), rtol=0, atol=tol)
    assert np.allclose(out["o"], ro.numpy(), rtol=0, atol=tol)
    assert np.allclose(out["h"], rh.numpy(), rtol=0, atol=tol * 4)
    if mirror:
        assert np.mean(np.abs(out["h"] - rh.numpy()) > 0) < 0.01


def test_step_vocab_stages_match_library_composition():
    from scipy import special, stats
    w, x, z, a = _tiny_inputs(torch.float32, seed=1)
    tau = 0.6
    out = oracle.denoise_step(TINY, w, x, z, a, tau=tau, b=0.1, seed=4, step=2, mirror_bf16=False,
                              want=("h", "logits", "H", "argmax", "u", "g", "z_out"), nthreads=2)
    h = out["h"]
    l = a.reshape(-1, 1) * (h @ w["E"].astype(np.float64).T) / math.sqrt(TINY.d)
    assert np.allclose(out["logits"], l, rtol=1e-12, atol=1e-12)
    p = special.softmax(l / tau, axis=1)
    assert np.allclose(out["H"], stats.entropy(p, axis=1), atol=1e-10)
    assert np.array_equal(out["argmax"], np.argmax(l, axis=1))
    u = p @ w["E"].astype(np.float64)
    assert np.allclose(out["u"], u, atol=1e-12)
    g = torch.nn.functional.gelu(torch.from_numpy(u) @ torch.from_numpy(w["W1"]).double().T).numpy()
    assert np.allclose(out["g"], g, atol=1e-12)
    assert np.allclose(out["z_out"], g @ w["W2"].astype(np.float64).T, atol=1e-12)


def test_step_sampler_invariants():
    w, x, z, a = _tiny_inputs(torch.bfloat16, seed=2)
    out = oracle.denoise_step(TINY, w, x, z, a, tau=0.8, b=0.1, seed=9, step=3, nthreads=2)
    H, acc = out["H"], out["accept"]
    order = sorted(range(TINY.C), key=lambda i: (H[i], i))
    n = int(out["n_acc"][0])
    assert n == acc.sum()
    assert set(np.nonzero(acc)[0]) == set(order[:n])
    assert H[acc].sum() <= 0.1
    if n < TINY.C:
        assert H[acc].sum() + H[order[n]] > 0.1
    for i in range(TINY.C):
        want = out["sample_tok"][i] if acc[i] else out["renoise_tok"][i]
        assert out["tokens_out"][i] == want
        assert out["renoise_tok"][i] == oracle.uniform_token(
            oracle.philox_word(9, 0, 3, 0, i, 0, 1), TINY.V)
    assert abs(out["meanH"][0] - H.mean()) < 1e-12


def test_step_samples_follow_the_tempered_softmax():
    """a7 as the step composes it: an accepted position takes argmax_v (l_v / tau + G_v), so over many
    seeds the sampled token of a row is distributed as softmax(l / tau) (the Gumbel-max law applied to
    the tempered logits, [TR] step 3 samples from p0).  The same draws reject softmax(l): a step that
    perturbed l instead of l / tau fails here."""
    from scipy import special, stats
    dims = synth.Dims(V=8, d=64, C=16, B=1, Hq=2, Hkv=1, hd=32, F=64, P=4)
    w, x, z, a = _tiny_inputs(torch.float32, alpha=1.0, seed=11, dims=dims)
    tau, n = 0.4, 600
    draws = np.empty((n, dims.C), np.int64)
    logits = None
    for k in range(n):
        o = oracle.denoise_step(dims, w, x, z, a, tau=tau, b=0.1, seed=1000 + k, step=0, mirror_bf16=False,
                                want=("logits", "sample_tok"), nthreads=1)
        draws[k] = o["sample_tok"]
        if logits is None:
            logits = o["logits"]
        else:
            assert np.array_equal(logits, o["logits"])  # the seed moves only the noise

    def pvalue(p):
        stat = 0.0
        for i in range(dims.C):
            e = n * p[i]
            stat += float((((np.bincount(draws[:, i], minlength=dims.V) - e) ** 2) / e).sum())
        return stats.chi2.sf(stat, dims.C * (dims.V - 1))

    p_tau, p_one = special.softmax(logits / tau, axis=1), special.softmax(logits, axis=1)
    assert np.abs(p_tau - p_one).max() > 0.2  # the two laws are far apart: the test has power
    assert pvalue(p_tau) > 1e-4
    assert pvalue(p_one) < 1e-12


def test_step_uniform_logits_accept_nothing():
    # alpha -> 0 makes every logit row uniform: H = log V > b, nothing accepted.
    w, x, z, a = _tiny_inputs(torch.float32, alpha=1e-12)
    out = oracle.denoise_step(TINY, w, x, z, a, tau=0.8, b=0.1, seed=0, step=0, mirror_bf16=False)
    assert np.allclose(out["H"], math.log(TINY.V), atol=1e-9)
    assert out["n_acc"][0] == 0 and not out["accept"].any()
    assert abs(out["meanH"][0] - math.log(TINY.V)) < 1e-9
    # and u is the mean embedding row
    assert np.allclose(out["u"], w["E"].astype(np.float64).mean(0)[None], atol=1e-9)


def test_step_one_hot_p0_gives_embedding_row():
    # very sharp logits make p0 one-hot, so p0 . E is the row of E at the argmax.
    w, x, z, a = _tiny_inputs(torch.float32, alpha=1e5)
    out = oracle.denoise_step(TINY, w, x, z, a, tau=0.4, b=0.1, seed=0, step=0, mirror_bf16=False)
    E = w["E"].astype(np.float64)
    assert np.allclose(out["u"], E[out["argmax"]], rtol=0, atol=1e-6)
    assert np.all(out["H"] < 1e-6)
    # every position fits in the budget and samples its argmax
    assert out["accept"].all()
    assert np.array_equal(out["tokens_out"], out["argmax"])


def test_rows_mode_agrees_with_full_mode():
    w, x, z, a = _tiny_inputs(torch.bfloat16, seed=3)
    full = oracle.denoise_step(TINY, w, x, z, a, tau=0.7, b=0.1, seed=1, step=1, nthreads=3,
                               want=oracle._WANT_ALL)
    rows = [15, 0, 5]
    part = oracle.denoise_step(TINY, w, x, z, a, tau=0.7, b=0.1, seed=1, step=1, rows=rows,
                               want=("H", "argmax", "sample_tok", "z_out", "logits"), nthreads=1)
    assert np.array_equal(part["logits"], full["logits"][rows])  # rows mode: logits in the rows' order
    for r in rows:
        assert part["H"][r] == full["H"][r]
        assert part["argmax"][r] == full["argmax"][r]
        assert part["sample_tok"][r] == full["sample_tok"][r]
        assert np.array_equal(part["z_out"][r], full["z_out"][r])


def test_thread_count_bit_identical():
    w, x, z, a = _tiny_inputs(torch.bfloat16, seed=4)
    r1 = oracle.denoise_step(TINY, w, x, z, a, tau=0.8, b=0.1, seed=2, step=0, nthreads=1)
    r4 = oracle.denoise_step(TINY, w, x, z, a, tau=0.8, b=0.1, seed=2, step=0, nthreads=4)
    for k in r1:
        assert np.array_equal(r1[k], r4[k]), k


# -------------------------------------------------------- loop and commit ---
def test_loop_sharp_alpha_stops_at_step_one(golden_dir):
    # With alpha = 64 every row is confident: all positions are accepted, the
    # argmax repeats, mean entropy is below the threshold, and the stop test
    # fires at the first step where it can (step index 1).
    w, x, z, a = _tiny_inputs(torch.bfloat16, alpha=64.0, seed=5)
    r = oracle.denoise_canvas(TINY, w, x, a, seed=5, N=48)
    assert r["converged"][0] == 1
    assert r["steps_taken"][0] == 2
    assert r["accepted"][0, 0] == TINY.C and r["accepted"][0, 2] == -1


def test_loop_matches_manual_steps_with_linear_anneal(golden_dir):
    table = {}
    with open(os.path.join(golden_dir, "sampler_table2.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                table[k] = float(v)
    N = 4
    tau0, tau1 = table["tau_start"], table["tau_end"]
    w, x, z, a = _tiny_inputs(torch.bfloat16, seed=6)
    loop = oracle.denoise_canvas(TINY, w, x, a, seed=8, N=N, tau0=tau0, tau1=tau1,
                                 b=table["entropy_budget"], stop_H=table["stop_mean_entropy"])
    taus = [tau0 + (tau1 - tau0) * s / (N - 1) for s in range(N)]
    assert taus[0] == 0.8 and abs(taus[-1] - 0.4) < 1e-15
    # the oracle's schedule: the printed endpoints, equal steps in between
    ot = oracle.tau_schedule(48, tau0, tau1)
    assert ot[0] == tau0 and abs(ot[-1] - tau1) < 1e-15
    assert np.ptp(np.diff(ot)) < 1e-15 and abs(np.diff(ot)[0] - (tau1 - tau0) / 47) < 1e-15
    assert np.array_equal(oracle.tau_schedule(N, tau0, tau1), np.array(taus))
    xx, zz, prev = x.copy(), z.copy(), None
    for s in range(N):
        o = oracle.denoise_step(TINY, w, xx, zz, a, tau=taus[s], b=0.1, seed=8, step=s,
                                prev_argmax=prev)
        xx = o["tokens_out"].reshape(x.shape)
        zz = o["z_out"].astype(np.float32).reshape(z.shape)
        prev = o["argmax"].reshape(x.shape)
        assert loop["accepted"][0, s] == o["n_acc"][0]
    assert loop["steps_taken"][0] == N and loop["converged"][0] == 0
    assert np.array_equal(loop["tokens"], xx)
    assert np.array_equal(loop["xhat0"], prev)


def test_commit_appends_reencoded_kv():
    dims = synth.Dims(V=512, d=64, C=16, B=2, Hq=2, Hkv=1, hd=32, F=128, P=32, cap=64)
    w = synth.to_numpy_f32(synth.make_weights(dims, 3, dtype=torch.float32))
    toks = np.random.default_rng(0).integers(0, 512, size=(2, 16)).astype(np.int32)
    Kc, Vc = oracle.commit(dims, w["E"], w["Wk"], w["Wv"], toks, w["Kc"], w["Vc"], P=32,
                           mirror_bf16=False)
    assert np.array_equal(Kc[:, :, :32], w["Kc"][:, :, :32])
    assert np.all(Kc[:, :, 48:] == 0)
    a = torch.nn.functional.rms_norm(torch.from_numpy(w["E"]).double()[torch.from_numpy(toks).long()],
                                     (64,), eps=1e-6)
    k = (a @ torch.from_numpy(w["Wk"]).double().T).numpy()
    v = (a @ torch.from_numpy(w["Wv"]).double().T).numpy()
    for bb in range(2):
        for i in range(16):
            kr = oracle.rope(k[bb, i], 32 + i, 10000.0)
            assert np.allclose(Kc[bb, 0, 32 + i], kr, atol=1e-6)
            assert np.allclose(Vc[bb, 0, 32 + i], v[bb, i], atol=1e-6)
    with pytest.raises(ValueError):
        oracle.commit(dims, w["E"], w["Wk"], w["Wv"], toks, w["Kc"], w["Vc"], P=60)


# ------------------------------------------- masked confidence decoding ---
def test_reveal_matches_topk():
    """or_reveal reveals the k = min(ceil(U / (N - step)), U) still-masked positions of highest
    confidence 1 / Z with their argmax candidates: compared with torch.topk over the confidences
    (resolved positions at -1, the form of the pages' generate()), on random canvases with distinct
    confidences."""
    rng = np.random.default_rng(7)
    C, V, mask = 64, 1000, 999
    for trial in range(200):
        N = int(rng.integers(1, 12))
        step = int(rng.integers(0, N))
        tokens = rng.integers(0, V - 1, size=C).astype(np.int32)
        tokens[rng.random(C) < rng.random()] = mask
        Z = 1.0 + rng.random(C) * 50.0
        am = rng.integers(0, V - 1, size=C).astype(np.int32)
        new, rev, k = oracle.reveal(Z, am, tokens, mask, step, N)
        unresolved = tokens == mask
        U = int(unresolved.sum())
        assert k == min(math.ceil(U / (N - step)), U)
        conf = torch.from_numpy(np.where(unresolved, 1.0 / Z, -1.0))
        want = tokens.copy()
        if k:
            chosen = conf.topk(k).indices.numpy()
            want[chosen] = am[chosen]
        assert np.array_equal(new, want)
        assert set(np.nonzero(rev)[0]) == (set(chosen.tolist()) if k else set())


def test_reveal_ties_and_edges():
    # equal confidences: the lower position first; nothing masked: nothing changes; the last
    # step reveals every remaining position
    Z = np.array([2.0, 1.0, 1.0, 3.0, 1.0])
    am = np.array([10, 11, 12, 13, 14], np.int32)
    tok = np.full(5, 99, np.int32)
    new, rev, k = oracle.reveal(Z, am, tok, 99, 3, 5)  # ceil(5 / 2) = 3
    assert k == 3 and new.tolist() == [99, 11, 12, 99, 14]
    new2, rev2, k2 = oracle.reveal(Z, am, new, 99, 4, 5)
    assert k2 == 2 and (new2 != 99).all()
    same, rev3, k3 = oracle.reveal(Z, am, new2, 99, 0, 5)
    assert k3 == 0 and np.array_equal(same, new2) and not rev3.any()


def test_reveal_loop_invariants():
    """The masked loop through the oracle's step: every step reveals ceil(U / (N - step)) positions,
    revealed positions keep their tokens, nothing is masked after the last step, and each revealed
    token is the argmax of its position at the step that revealed it."""
    dims = synth.Dims(V=512, d=64, C=16, B=2, Hq=2, Hkv=1, hd=32, F=128, P=32)
    w, x, z, a = _tiny_inputs(torch.bfloat16, seed=4, dims=dims)
    mask = dims.V - 1
    N = 5
    tok = np.full((dims.B, dims.C), mask, np.int32)
    zz = np.zeros_like(z)
    for s in range(N):
        o = oracle.denoise_step_masked(dims, w, tok, zz, a, tau=0.8, mask_id=mask, step=s, N=N)
        new = o["tokens_out"].reshape(dims.B, dims.C)
        for bb in range(dims.B):
            U = int((tok[bb] == mask).sum())
            assert o["n_rev"][bb] == math.ceil(U / (N - s))
            kept = tok[bb] != mask
            assert np.array_equal(new[bb][kept], tok[bb][kept])
            r = o["revealed"].reshape(dims.B, dims.C)[bb]
            assert np.array_equal(new[bb][r], o["argmax"].reshape(dims.B, dims.C)[bb][r])
        tok = new
        zz = o["z_out"].astype(np.float32).reshape(z.shape)
    assert (tok != mask).all()


def test_excluded_token_is_removed_from_the_softmax():
    """exclude_tok: the row statistics and p0 . E equal those of the softmax over the other tokens
    (scipy softmax of the logits with that entry removed); the logits output keeps the raw value."""
    from scipy import special, stats
    w, x, z, a = _tiny_inputs(torch.float32, seed=5)
    tau, ex = 0.7, 37
    out = oracle.denoise_step(TINY, w, x, z, a, tau=tau, b=0.1, seed=1, step=0, mirror_bf16=False,
                              want=("logits", "H", "Z", "argmax", "u"), exclude_tok=ex)
    l = out["logits"]
    keep = np.arange(TINY.V) != ex
    p = special.softmax(l[:, keep] / tau, axis=1)
    assert np.allclose(out["H"], stats.entropy(p, axis=1), atol=1e-10)
    assert np.allclose(out["u"], p @ w["E"].astype(np.float64)[keep], atol=1e-12)
    am = np.argmax(l[:, keep], axis=1)
    assert np.array_equal(out["argmax"], np.where(am >= ex, am + 1, am))
    assert np.allclose(1.0 / out["Z"], p.max(axis=1), rtol=1e-12)


# ---------------------------------------- multi-layer stack and causal prefill ---
ML = synth.Dims(V=300, d=64, C=12, B=2, Hq=4, Hkv=2, hd=16, F=64, P=10, cap=40, L=3)


def _rope_t(t, pos, hd, base):
    ang = pos[:, None] * base ** (-2.0 * torch.arange(hd // 2, dtype=torch.float64) / hd)
    rot = torch.polar(torch.ones_like(ang), ang)
    c = torch.complex(t[..., : hd // 2], t[..., hd // 2:]) * rot
    return torch.cat([c.real, c.imag], -1)


def _torch_layers(dims, w, a, Kc, Vc, P, n, mask=None, write_cache=False):
    """Float64 composition of the attention stack with library routines (rms_norm, SDPA, complex
    RoPE): a [B, n, d] into layer 0; per layer q, k, v of a_l, attention over [cache rows 0..P-1 ;
    the n new rows] with an optional boolean mask, h_l = a_l + o Wo^T, a_{l+1} = rms_norm(h_l).
    Returns the last h and the new rows' (k, v) of every layer."""
    f = lambda t: torch.from_numpy(np.asarray(t)).double()
    B, d, Hq, Hkv, hd = dims.B, dims.d, dims.Hq, dims.Hkv, dims.hd
    pos = torch.arange(P, P + n, dtype=torch.float64)
    rep = Hq // Hkv
    kv = []
    h = None
    for l in range(dims.L):
        if l > 0:
            a = torch.nn.functional.rms_norm(h, (d,), eps=dims.rms_eps)
        q = _rope_t((a @ f(w["Wq"][l]).T).view(B, n, Hq, hd).transpose(1, 2), pos, hd, dims.rope_base)
        k = _rope_t((a @ f(w["Wk"][l]).T).view(B, n, Hkv, hd).transpose(1, 2), pos, hd, dims.rope_base)
        v = (a @ f(w["Wv"][l]).T).view(B, n, Hkv, hd).transpose(1, 2)
        kv.append((k, v))
        Kall = torch.cat([f(Kc[l])[:, :, :P], k], 2)
        Vall = torch.cat([f(Vc[l])[:, :, :P], v], 2)
        o = torch.nn.functional.scaled_dot_product_attention(
            q, Kall.repeat_interleave(rep, 1), Vall.repeat_interleave(rep, 1), attn_mask=mask)
        h = a + o.transpose(1, 2).reshape(B, n, Hq * hd) @ f(w["Wo"][l]).T
    return h, kv


def test_multilayer_step_matches_library_composition():
    """L = 3: the oracle step's h (last layer), entropy and u equal a float64 composition of library
    routines, each layer over its own prefix cache."""
    from scipy import special, stats
    w, x, z, al = _tiny_inputs(torch.float32, seed=12, dims=ML)
    tau = 0.7
    out = oracle.denoise_step(ML, w, x, z, al, tau=tau, b=0.1, seed=0, step=0, mirror_bf16=False,
                              want=("h", "logits", "H", "u"), nthreads=2)
    e = torch.from_numpy(w["E"]).double()[torch.from_numpy(x).long()] + torch.from_numpy(z).double()
    a0 = torch.nn.functional.rms_norm(e, (ML.d,), eps=ML.rms_eps)
    h, _ = _torch_layers(ML, w, a0, w["Kc"], w["Vc"], ML.P, ML.C)
    h = h.reshape(ML.M, ML.d).numpy()
    assert np.allclose(out["h"], h, rtol=0, atol=1e-10)
    l = al.reshape(-1, 1) * (h @ w["E"].astype(np.float64).T) / math.sqrt(ML.d)
    p = special.softmax(l / tau, axis=1)
    assert np.allclose(out["H"], stats.entropy(p, axis=1), atol=1e-9)
    assert np.allclose(out["u"], p @ w["E"].astype(np.float64), atol=1e-10)
    # one layer of the stack: the single-layer step on that layer's weights and cache
    one = dataclasses.replace(ML, L=1)
    w1 = {k: (v[0] if k in ("Wq", "Wk", "Wv", "Wo", "Kc", "Vc") else v) for k, v in w.items()}
    o1 = oracle.denoise_step(one, w1, x, z, al, tau=tau, b=0.1, seed=0, step=0, mirror_bf16=False, want=("h",))
    h1, _ = _torch_layers(one, {k: (v[None] if k in ("Wq", "Wk", "Wv", "Wo") else v) for k, v in w1.items()},
                          a0, w["Kc"][:1], w["Vc"][:1], ML.P, ML.C)
    assert np.allclose(o1["h"], h1.reshape(ML.M, ML.d).numpy(), rtol=0, atol=1e-10)


def _prefill_inputs(seed=13, n=7):
    w, _, _, _ = _tiny_inputs(torch.float32, seed=seed, dims=ML)
    tok = np.random.default_rng(seed).integers(0, ML.V, size=(ML.B, n)).astype(np.int32)
    return w, tok


def test_prefill_matches_causal_composition():
    """or_prefill: the appended K/V of every layer equal a float64 composition with an explicit causal
    mask (token i sees the cached rows and the new tokens 0..i); rows outside the block are untouched."""
    w, tok = _prefill_inputs()
    n = tok.shape[1]
    Kn, Vn = oracle.prefill(ML, w, tok, P=ML.P, mirror_bf16=False)
    e = torch.from_numpy(w["E"]).double()[torch.from_numpy(tok).long()]
    a0 = torch.nn.functional.rms_norm(e, (ML.d,), eps=ML.rms_eps)
    mask = torch.ones(n, ML.P + n, dtype=torch.bool)
    mask[:, ML.P:] = torch.tril(torch.ones(n, n, dtype=torch.bool))
    _, kv = _torch_layers(ML, w, a0, w["Kc"], w["Vc"], ML.P, n, mask=mask)
    # the caches are float32 arrays: the appended rows carry their float32 rounding (~6e-8
    # relative), which the deeper layers then read back
    for l, (k, v) in enumerate(kv):
        assert np.allclose(Kn[l][:, :, ML.P:ML.P + n], k.numpy(), rtol=1e-6, atol=1e-6), l
        assert np.allclose(Vn[l][:, :, ML.P:ML.P + n], v.numpy(), rtol=1e-6, atol=1e-6), l
    assert np.array_equal(Kn[:, :, :, :ML.P], w["Kc"][:, :, :, :ML.P])
    assert np.array_equal(Kn[:, :, :, ML.P + n:], w["Kc"][:, :, :, ML.P + n:])


def test_prefill_is_causal_and_chunked_prefill_is_one_piece():
    """Changing token j leaves every layer's K/V of positions before j unchanged and changes the
    deeper layers' K/V after j (they attend over it); layer 0's K/V of a position depend on that token
    only.  Prefill in two pieces equals prefill in one (the second piece attends over the first)."""
    w, tok = _prefill_inputs(seed=14)
    n, j = tok.shape[1], 3
    K1, V1 = oracle.prefill(ML, w, tok, P=ML.P, mirror_bf16=False)
    t2 = tok.copy()
    t2[:, j] = (t2[:, j] + 1) % ML.V
    K2, _ = oracle.prefill(ML, w, t2, P=ML.P, mirror_bf16=False)
    blk = slice(ML.P, ML.P + n)
    for l in range(ML.L):
        d = np.abs(K1[l][:, :, blk] - K2[l][:, :, blk]).max(axis=(1, 3))  # [B, n]
        assert (d[:, :j] == 0).all(), l
        assert (d[:, j] > 0).all(), l
        if l == 0:
            assert (d[:, j + 1:] == 0).all()
        else:
            assert (d[:, j + 1:] > 0).all(), l
    wa = dict(w)
    Ka, Va = oracle.prefill(ML, wa, tok[:, :4], P=ML.P, mirror_bf16=False)
    wa["Kc"], wa["Vc"] = Ka, Va
    Kb, Vb = oracle.prefill(ML, wa, tok[:, 4:], P=ML.P + 4, mirror_bf16=False)
    assert np.array_equal(Kb, K1) and np.array_equal(Vb, V1)


def test_one_layer_commit_is_the_prefill_of_one_block():
    one = synth.Dims(V=300, d=64, C=12, B=2, Hq=4, Hkv=2, hd=16, F=64, P=10, cap=40)
    w, _, _, _ = _tiny_inputs(torch.bfloat16, seed=15, dims=one)
    tok = np.random.default_rng(15).integers(0, one.V, size=(one.B, one.C)).astype(np.int32)
    Kc, Vc = oracle.commit(one, w["E"], w["Wk"], w["Wv"], tok, w["Kc"], w["Vc"], P=one.P)
    Kp, Vp = oracle.prefill(one, w, tok, P=one.P)
    assert np.array_equal(Kc, Kp) and np.array_equal(Vc, Vp)



# ----------------------------------------------------------------- E4M3 ---
def test_round_e4m3_matches_torch():
    """Round to nearest even in E4M3 equals torch's float8_e4m3fn conversion below the saturation
    point (torch gives NaN past the range; this rounding saturates at 448)."""
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.uniform(-463.9, 463.9, 20000), rng.standard_normal(20000) * 1e-2,
                        rng.standard_normal(5000) * 1e-3, np.arange(-448, 449, 0.5),
                        (np.arange(1, 64) + 0.5) * 2.0 ** -9])  # subnormal ties
    x = x.astype(np.float32)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.round_e4m3(float(v)) for v in x])
    assert np.array_equal(got, want)
    assert oracle.round_e4m3(464.0) == 448.0 and oracle.round_e4m3(-1e9) == -448.0
    assert oracle.round_e4m3(463.99) == 448.0


def test_e4m3_codes_decode_like_torch():
    codes = np.array([c for c in range(256) if (c & 0x7f) != 0x7f], np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_value(int(c)) for c in codes])
    assert np.array_equal(got, want)


def test_quantize_rows_e4m3_matches_torch():
    """Codes and scales equal the same definition written with torch float32 arithmetic
    (scale = absmax / 448, codes of x * (448 / absmax)); decoded rows are within E4M3's relative step."""
    rng = np.random.default_rng(4)
    X = (rng.standard_normal((64, 200)) * rng.uniform(0.01, 10, (64, 1))).astype(np.float32)
    X[5] = 0.0
    Q, sc = oracle.quantize_rows_e4m3(X)
    t = torch.from_numpy(X)
    amax = t.abs().amax(dim=1)
    inv = torch.where(amax > 0, torch.tensor(448.0) / amax, torch.zeros_like(amax))
    want_q = (t * inv[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    want_q[5] = 0
    assert np.array_equal(Q, want_q)
    assert np.array_equal(sc, (amax / 448.0).numpy())
    dq = torch.from_numpy(Q).view(torch.float8_e4m3fn).double().numpy() * sc[:, None]
    assert np.all(np.abs(dq - X) <= 2.0 ** -4 * np.abs(X) + 2.0 ** -9 * sc[:, None] + 1e-30)


def test_fp8_head_logits_are_the_quantized_product():
    """With an FP8 head the oracle's logits are alpha s_h s_v (q_h . q_v) / sqrt(d) for h quantized per
    row (recomputed here with numpy from the oracle's h and the quantizer), and the contraction
    keeps the bf16 E."""
    from scipy import special
    w, x, z, a = _tiny_inputs(torch.bfloat16, seed=6)
    E8, sE = oracle.quantize_rows_e4m3(w["E"])
    tau = 0.8
    out = oracle.denoise_step(TINY, w, x, z, a, tau=tau, b=0.1, seed=1, step=0, want=("h", "logits", "u"),
                              fp8_head=(E8, sE))
    hq, hs = oracle.quantize_rows_e4m3(out["h"].astype(np.float32))
    dec = lambda q: torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy()
    l = a.reshape(-1, 1) * (hs[:, None].astype(np.float64) * sE[None, :].astype(np.float64) *
                            (dec(hq) @ dec(E8).T)) / math.sqrt(TINY.d)
    assert np.allclose(out["logits"], l, rtol=1e-12, atol=1e-12)
    p = special.softmax(l / tau, axis=1)
    assert np.allclose(out["u"], np.vectorize(oracle.round_bf16)(p @ w["E"].astype(np.float64)), atol=2e-3)


# ------------------------------------------------------------------ MoE FFN ----
# The DiffusionGemma backbone's FFN (the "文本 Diffusion 模型" survey page, §11: 128 experts per
# layer, 8 routed plus one shared; §13: router top-k, expert GEMM, token permutation).  The pins below fix the routing, the
# gates, the experts' orientation and the residual against closed forms and library routines.
MOE = synth.Dims(V=300, d=64, C=12, B=2, Hq=4, Hkv=2, hd=16, F=64, P=10, cap=40, n_exp=16, top_k=4, Fe=32)


def _moe_dims(**kw):
    return dataclasses.replace(MOE, **kw)


def _gelu1():
    return 0.5 * (1.0 + math.erf(1.0 / math.sqrt(2.0)))  # GELU(1)


def _probe_experts(dims, logit_of):
    """Weights whose routed expert e maps x = ones(d) to GELU(1) e_e (unit vector on output column e)
    and whose router gives expert e the logit logit_of[e]; the shared expert is zero."""
    NE, d, Fe = dims.n_exp, dims.d, dims.Fe
    Wr = np.zeros((NE, d), np.float32)
    for e in range(NE):
        Wr[e, :] = np.float32(logit_of[e]) / d  # x = ones: r_e = d * (logit / d)
    We1 = np.zeros((NE + 1, Fe, d), np.float32)
    We2 = np.zeros((NE + 1, d, Fe), np.float32)
    for e in range(NE):
        We1[e, 0, 0] = 1.0   # hidden unit 0 = GELU(x_0) = GELU(1)
        We2[e, e, 0] = 1.0   # output column e
    return Wr, We1, We2


def test_moe_gates_and_routing_closed_form():
    """x = RMSNorm(ones) = ones (eps 0); selected logits ln 4, ln 2, 0, 0 among negatives: the gates
    are 4/8, 2/8, 1/8, 1/8 and y lands on exactly the selected experts' columns."""
    dims = _moe_dims(rms_eps=0.0)
    lg = np.full(dims.n_exp, -5.0)
    lg[[9, 2, 13, 6]] = [math.log(4), math.log(2), 0.0, 0.0]
    Wr, We1, We2 = _probe_experts(dims, lg)
    h = np.ones((3, dims.d))
    out = oracle.moe_ffn(dims, Wr, We1, We2, h, mirror_bf16=False)
    assert out["idx"].tolist() == [[9, 2, 6, 13]] * 3  # rank order; the tie 0 = 0 in index order
    np.testing.assert_allclose(out["gate"], [[0.5, 0.25, 0.125, 0.125]] * 3, rtol=1e-6)
    y = out["h"] - h
    want = np.zeros(dims.d)
    want[[9, 2, 6, 13]] = np.array([0.5, 0.25, 0.125, 0.125]) * _gelu1()
    np.testing.assert_allclose(y, np.tile(want, (3, 1)), rtol=1e-6, atol=1e-12)


def test_moe_top1_and_ties():
    """top_k = 1 gives gate 1 exactly; with top_k = 2 and three equal logits the two lowest indices
    are taken with gates 1/2 each."""
    d1 = _moe_dims(rms_eps=0.0, top_k=1)
    lg = np.linspace(-1, 1, d1.n_exp)
    Wr, We1, We2 = _probe_experts(d1, lg)
    out = oracle.moe_ffn(d1, Wr, We1, We2, np.ones((1, d1.d)), mirror_bf16=False)
    assert out["idx"][0, 0] == d1.n_exp - 1 and out["gate"][0, 0] == 1.0
    d2 = _moe_dims(rms_eps=0.0, top_k=2)
    lg = np.full(d2.n_exp, -3.0)
    lg[[7, 3, 11]] = 1.0
    Wr, We1, We2 = _probe_experts(d2, lg)
    out = oracle.moe_ffn(d2, Wr, We1, We2, np.ones((1, d2.d)), mirror_bf16=False)
    assert out["idx"][0].tolist() == [3, 7]
    assert out["gate"][0].tolist() == [0.5, 0.5]


def test_moe_identical_experts_reduce_to_dense_ffn():
    """With every routed expert equal, the gates sum to one whatever the router does: the block is
    h + FFN(x) + FFN_shared(x), x = rms_norm(h), composed here from torch's rms_norm and GELU."""
    dims = MOE
    rng = np.random.default_rng(5)
    d, Fe, NE = dims.d, dims.Fe, dims.n_exp
    A = (rng.standard_normal((Fe, d)) / math.sqrt(d)).astype(np.float32)
    Bm = (rng.standard_normal((d, Fe)) / math.sqrt(Fe)).astype(np.float32)
    S1 = (rng.standard_normal((Fe, d)) / math.sqrt(d)).astype(np.float32)
    S2 = (rng.standard_normal((d, Fe)) / math.sqrt(Fe)).astype(np.float32)
    Wr = (rng.standard_normal((NE, d)) / math.sqrt(d)).astype(np.float32)
    We1 = np.concatenate([np.repeat(A[None], NE, 0), S1[None]])
    We2 = np.concatenate([np.repeat(Bm[None], NE, 0), S2[None]])
    h = rng.standard_normal((20, d))
    out = oracle.moe_ffn(dims, Wr, We1, We2, h, mirror_bf16=False)
    ht = torch.from_numpy(h)
    x = torch.nn.functional.rms_norm(ht, (d,), eps=dims.rms_eps)
    gelu = torch.nn.functional.gelu
    ffn = lambda W1, W2: gelu(x @ torch.from_numpy(W1).double().T) @ torch.from_numpy(W2).double().T
    ref = (ht + ffn(A, Bm) + ffn(S1, S2)).numpy()
    np.testing.assert_allclose(out["h"], ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out["gate"].sum(axis=1), 1.0, rtol=1e-14)
    # the router logits are x . Wr_e
    np.testing.assert_allclose(out["logits"], (x @ torch.from_numpy(Wr).double().T).numpy(), rtol=1e-12,
                               atol=1e-12)


def test_moe_expert_permutation_invariance():
    """Relabelling the routed experts (router rows and expert matrices alike) leaves the output
    unchanged and relabels the selection."""
    dims = MOE
    w = synth.to_numpy_f32(synth.make_weights(dims, 3))
    rng = np.random.default_rng(9)
    perm = rng.permutation(dims.n_exp)
    h = rng.standard_normal((24, dims.d))
    a = oracle.moe_ffn(dims, w["Wr"], w["We1"], w["We2"], h)
    ext = np.r_[perm, dims.n_exp]
    b = oracle.moe_ffn(dims, w["Wr"][perm], w["We1"][ext], w["We2"][ext], h)
    np.testing.assert_array_equal(a["h"], b["h"])
    np.testing.assert_array_equal(a["idx"], perm[b["idx"]])


def test_moe_hot_experts_bound_the_canvas_activation():
    """The synthetic router's cold experts (row norm / 64) never reach a top-8 of 84 unit-spread
    logits: a 256-token canvas activates exactly the hot set (the pages' 84 of 128)."""
    dims = dataclasses.replace(MOE, d=128, n_exp=128, top_k=8, moe_hot=84)
    w = synth.to_numpy_f32(synth.make_weights(dims, 4))
    h = np.random.default_rng(1).standard_normal((256, dims.d))
    x = torch.nn.functional.rms_norm(torch.from_numpy(h), (dims.d,), eps=dims.rms_eps).numpy()
    r = x @ w["Wr"].astype(np.float64).T
    top = np.argsort(-r, axis=1, kind="stable")[:, :8]
    assert len(np.unique(top)) == 84


def test_moe_in_the_step_follows_the_attention_block():
    """The step with an MoE layer: its h is the MoE block applied to the attention block's h (the
    same step without MoE), and the routing outputs are that block's."""
    dims = MOE
    w = synth.to_numpy_f32(synth.make_weights(dims, 6))
    x, z, a = synth.make_canvas(dims, 6)
    base = dataclasses.replace(dims, n_exp=0, top_k=0, Fe=0)
    r0 = oracle.denoise_step(base, w, x.numpy(), z.float().numpy(), a.numpy(), tau=0.8, b=0.1, seed=1, step=0,
                             want=("h",))
    r1 = oracle.denoise_step(dims, w, x.numpy(), z.float().numpy(), a.numpy(), tau=0.8, b=0.1, seed=1, step=0,
                             want=("h", "moe_idx", "moe_gate", "H"))
    m = oracle.moe_ffn(dims, w["Wr"], w["We1"], w["We2"], r0["h"])
    np.testing.assert_array_equal(r1["h"], m["h"])
    np.testing.assert_array_equal(r1["moe_idx"], m["idx"])
    np.testing.assert_array_equal(r1["moe_gate"], m["gate"])


def test_moe_prefill_feeds_the_next_layer_only():
    """Prefill with two layers and MoE: layer 0's cache rows do not depend on the MoE weights, layer
    1's do (the MoE output is the next layer's input)."""
    dims = dataclasses.replace(MOE, L=2)
    w = synth.to_numpy_f32(synth.make_weights(dims, 8))
    toks = np.random.default_rng(2).integers(0, dims.V, (dims.B, 5)).astype(np.int32)
    K1, V1 = oracle.prefill(dims, w, toks, dims.P)
    w2 = dict(w)
    w2["We2"] = w["We2"] * 2
    K2, V2 = oracle.prefill(dims, w2, toks, dims.P)
    rows = slice(dims.P, dims.P + 5)
    np.testing.assert_array_equal(K1[0][..., rows, :], K2[0][..., rows, :])
    assert np.abs(K1[1][..., rows, :] - K2[1][..., rows, :]).max() > 1e-3
