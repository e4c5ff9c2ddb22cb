"""Comparison helpers for device-vs-oracle parity.

Tolerances (from the problem statement): logits max error relative to the
row's largest |logit| 2e-2, entropy absolute 1e-3 nats, z (and u) relative L2
1e-2.  Accept / renoise decisions and renoised tokens must match exactly,
except positions whose cumulative entropy lies within 1e-3 of the budget, or
whose entropy lies within the entropy tolerance of the first rejected
position's (an order tie across the boundary); those are counted.  A sampled
token of an accepted position may differ only where the oracle's two best
Gumbel-perturbed scores are closer than 1e-2.  An argmax may differ only
where the oracle's two largest logits are closer than 1e-4 of the row scale.
"""
from __future__ import annotations

import numpy as np
import torch

LOGIT_TOL = 2e-2
H_TOL = 1e-3
Z_TOL = 1e-2
BOUNDARY_TOL = 1e-3
GUMBEL_GAP_TOL = 1e-2


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


def rel_l2(got, ref) -> float:
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def check_close_bf16(name, got, ref, tol=Z_TOL, ulps=8):
    """Stored bf16 operands: relative L2 within tol, and no element off by more than
    `ulps` bf16 ulps of (|ref| + rms(ref) / 4) (the floor absorbs cancellation in sums).
    8 for one layer; deeper layers' operands carry the earlier layers' rounding as well."""
    got, ref = np.asarray(got, np.float64).reshape(-1), np.asarray(ref, np.float64).reshape(-1)
    r = rel_l2(got, ref)
    assert r <= tol, f"{name}: rel L2 {r:.3e} > {tol}"
    rms = float(np.sqrt(np.mean(ref * ref))) + 1e-30
    worst = float(np.max(np.abs(got - ref) / (np.abs(ref) + 0.25 * rms)))
    assert worst <= ulps * 2.0 ** -8, f"{name}: worst element error {worst:.3e}"
    return r


def check_rel_l2(name, got, ref, tol=Z_TOL):
    r = rel_l2(got, ref)
    assert r <= tol, f"{name}: rel L2 {r:.3e} > {tol}"
    return r


class Collect:
    """Runs checks and keeps every failure, so one run reports all of them."""

    def __init__(self):
        self.errors = []

    def __call__(self, fn, *args, **kw):
        try:
            return fn(*args, **kw)
        except AssertionError as e:
            self.errors.append(str(e))
            return None

    def done(self):
        assert not self.errors, "; ".join(self.errors)


def check_logits(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    rowmax = np.max(np.abs(ref), axis=1, keepdims=True)
    err = float(np.max(np.abs(got - ref) / rowmax))
    assert err <= LOGIT_TOL, f"logits: max row-relative error {err:.3e}"
    return err


def check_entropy(got, ref):
    err = float(np.max(np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))))
    assert err <= H_TOL, f"entropy: max abs error {err:.3e} nats"
    return err


def check_argmax(got, ref, top2gap, logits_scale):
    got, ref = np.asarray(got).reshape(-1), np.asarray(ref).reshape(-1)
    bad = np.nonzero(got != ref)[0]
    excused = [i for i in bad if top2gap[i] < 1e-4 * max(logits_scale[i], 1e-30)]
    assert len(bad) == len(excused), f"argmax: {len(bad) - len(excused)} unexcused mismatches"
    return len(excused)


def boundary_excused(H, cum, accept, b, C):
    """Positions whose acceptance may legitimately flip under rounding."""
    H = np.asarray(H).reshape(-1, C)
    cum = np.asarray(cum).reshape(-1, C)
    acc = np.asarray(accept).reshape(-1, C).astype(bool)
    ex = np.zeros_like(acc)
    for bb in range(H.shape[0]):
        ex[bb] |= np.abs(cum[bb] - b) <= BOUNDARY_TOL
        rej = ~acc[bb]
        if rej.any() and acc[bb].any():
            first_rej = np.argmin(np.where(rej, cum[bb], np.inf))
            last_acc = np.argmax(np.where(acc[bb], cum[bb], -np.inf))
            h0 = H[bb, first_rej]
            near = np.abs(H[bb] - h0) <= H_TOL
            if abs(H[bb, last_acc] - h0) <= H_TOL:
                ex[bb] |= near
    return ex.reshape(-1)


def check_sampler(got_accept, got_tokens, ref, b, C, excuse=None):
    """Accept decisions and next tokens against the oracle's full-mode outputs.

    excuse: optional boolean mask of positions whose inputs legitimately differ
    between the two sides (their decisions are not compared)."""
    ga = np.asarray(got_accept).reshape(-1).astype(bool)
    gt = np.asarray(got_tokens).reshape(-1)
    ra = ref["accept"].reshape(-1).astype(bool)
    ex = boundary_excused(ref["H"], ref["cum"], ra, b, C)
    if excuse is not None:
        ex = ex | np.asarray(excuse, bool).reshape(-1)
    bad_acc = np.nonzero((ga != ra) & ~ex)[0]
    assert len(bad_acc) == 0, f"accept: {len(bad_acc)} unexcused mismatches at {bad_acc[:8]}"
    same = (ga == ra)
    # rejected on both sides: renoised token, exact
    rej = same & ~ga
    bad_tok = np.nonzero(rej & (gt != ref["renoise_tok"]))[0]
    assert len(bad_tok) == 0, f"renoise tokens differ at {bad_tok[:8]}"
    # accepted on both sides: Gumbel-max sample
    acc = same & ga
    diff = acc & (gt != ref["sample_tok"])
    if excuse is not None:
        diff &= ~np.asarray(excuse, bool).reshape(-1)
    unexcused = np.nonzero(diff & (ref["gumbel_gap"] >= GUMBEL_GAP_TOL))[0]
    assert len(unexcused) == 0, f"sampled tokens differ at {unexcused[:8]}"
    return dict(boundary_excused=int((ex & (ga != ra)).sum()), sample_excused=int(diff.sum()),
                accepted=int(ga.sum()))
