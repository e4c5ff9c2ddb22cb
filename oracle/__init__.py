"""CPU oracle for the block-diffusion denoising step (test infrastructure).

This package is test infrastructure.  Only the tests, the smoke check and the
CPU-baseline leg of the benchmark may import it; the device library never does.
It wraps the plain double-precision C++ restatement in ``dg_oracle.cpp`` with
ctypes and numpy marshalling.  The shared library is compiled on first use
with the host C++ compiler (it builds the same on x86-64 and aarch64).
"""
from __future__ import annotations

import ctypes as ct
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dg_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libdg_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle library (g++, -O2, no fast-math, no FP contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
               "-fno-fast-math", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Dims(ct.Structure):
    _fields_ = [("V", ct.c_int32), ("d", ct.c_int32), ("C", ct.c_int32), ("B", ct.c_int32),
                ("Hq", ct.c_int32), ("Hkv", ct.c_int32), ("hd", ct.c_int32), ("F", ct.c_int32),
                ("P", ct.c_int32), ("cap", ct.c_int32), ("rope_base", ct.c_double),
                ("rms_eps", ct.c_double), ("mirror_bf16", ct.c_int32), ("L", ct.c_int32),
                ("n_exp", ct.c_int32), ("top_k", ct.c_int32), ("Fe", ct.c_int32)]


_F = ct.POINTER(ct.c_float)
_D = ct.POINTER(ct.c_double)
_I = ct.POINTER(ct.c_int32)
_U8 = ct.POINTER(ct.c_uint8)


class StepIn(ct.Structure):
    _fields_ = [("E", _F), ("Wq", _F), ("Wk", _F), ("Wv", _F), ("Wo", _F), ("W1", _F), ("W2", _F),
                ("Kc", _F), ("Vc", _F), ("x", _I), ("z", _F), ("alpha", _F), ("prev_argmax", _I),
                ("tau", ct.c_double), ("b", ct.c_double), ("stop_H", ct.c_double),
                ("seed", ct.c_uint64), ("step", ct.c_int32), ("block", ct.c_int32), ("exclude_tok", ct.c_int32),
                ("E8", _U8), ("E8_scale", _F), ("Wr", _F), ("We1", _F), ("We2", _F)]


class StepOut(ct.Structure):
    _fields_ = [("a", _D), ("q", _D), ("k", _D), ("v", _D), ("o", _D), ("h", _D), ("logits", _D),
                ("H", _D), ("m", _D), ("Z", _D), ("top2gap", _D), ("argmax", _I), ("accept", _U8),
                ("cum", _D), ("rank", _I), ("renoise_tok", _I), ("sample_tok", _I),
                ("gumbel_gap", _D), ("tokens_out", _I), ("u", _D), ("g", _D), ("z_out", _D),
                ("n_acc", _I), ("meanH", _D), ("stop", _I), ("moe_idx", _I), ("moe_gate", _D),
                ("moe_logits", _D), ("moe_x", _D)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ct.CDLL(build())
            L.or_philox4x64_10.argtypes = [ct.POINTER(ct.c_uint64), ct.POINTER(ct.c_uint64),
                                           ct.POINTER(ct.c_uint64)]
            L.or_philox_word.argtypes = [ct.c_uint64, ct.c_int32, ct.c_int32, ct.c_int32, ct.c_int32,
                                         ct.c_int64, ct.c_int32]
            L.or_philox_word.restype = ct.c_uint64
            L.or_uniform_token.argtypes = [ct.c_uint64, ct.c_int32]
            L.or_uniform_token.restype = ct.c_int32
            L.or_prefill.argtypes = [ct.POINTER(Dims), _F, _F, _F, _F, _F, ct.c_void_p, _I, ct.c_int32, _F, _F,
                                     ct.c_int32]
            L.or_moe_ffn.argtypes = [ct.POINTER(Dims), _F, _F, _F, _D, ct.c_int64, _I, _D, _D, ct.c_int32]
            L.or_moe_ffn.restype = ct.c_int
            L.or_prefill.restype = ct.c_int
            L.or_reveal.argtypes = [_D, _I, _I, ct.c_int32, ct.c_int32, ct.c_int32, ct.c_int32, _U8]
            L.or_reveal.restype = ct.c_int32
            L.or_round_e4m3.argtypes = [ct.c_double]
            L.or_round_e4m3.restype = ct.c_double
            L.or_e4m3_value.argtypes = [ct.c_uint8]
            L.or_e4m3_value.restype = ct.c_double
            L.or_quantize_rows_e4m3.argtypes = [_F, ct.c_int64, ct.c_int64, _U8, _F]
            L.or_tau.argtypes = [ct.c_double, ct.c_double, ct.c_int32, ct.c_int32]
            L.or_tau.restype = ct.c_double
            L.or_gumbel.argtypes = [ct.c_uint64]
            L.or_gumbel.restype = ct.c_float
            L.or_gumbel_argmax.argtypes = [_D, ct.c_int64, ct.c_uint64, ct.c_int32, ct.c_int32,
                                           ct.c_int32, ct.c_int32, _D]
            L.or_gumbel_argmax.restype = ct.c_int32
            L.or_gumbel_argmax_many.argtypes = [_D, ct.c_int64, ct.c_uint64, ct.c_int32, _I]
            L.or_uniform_many.argtypes = [ct.c_int32, ct.c_uint64, ct.c_int32, _I]
            L.or_gumbel_many.argtypes = [ct.c_uint64, ct.c_int64, _F]
            L.or_canvas_init.argtypes = [_I, ct.c_int32, ct.c_int32, ct.c_int32, ct.c_uint64, ct.c_int32]
            L.or_rmsnorm.argtypes = [_D, ct.c_int32, ct.c_double, _D]
            L.or_rope.argtypes = [_D, ct.c_int32, ct.c_double, ct.c_double]
            L.or_gelu.argtypes = [ct.c_double]
            L.or_gelu.restype = ct.c_double
            L.or_row_stats.argtypes = [_D, ct.c_int64, ct.c_double, _D, _D, _D, _I, _D]
            L.or_accept.argtypes = [_D, ct.c_int32, ct.c_double, _U8, _D, _I]
            L.or_accept.restype = ct.c_int32
            L.or_attend_row.argtypes = [_D, _F, _F, ct.c_int64, _D, _D, ct.c_int64, ct.c_int32, _D]
            L.or_denoise_step.argtypes = [ct.POINTER(Dims), ct.POINTER(StepIn), ct.POINTER(StepOut),
                                          _I, ct.c_int32, ct.c_int32]
            L.or_denoise_canvas.argtypes = [ct.POINTER(Dims)] + [_F] * 9 + [
                _I, _F, _F, ct.c_int32, ct.c_double, ct.c_double, ct.c_double, ct.c_double,
                ct.c_uint64, ct.c_int32, _I, _I, _I, _I, ct.c_int32]
            L.or_commit.argtypes = [ct.POINTER(Dims), _F, _F, _F, _I, _F, _F, ct.c_int32]
            L.or_round_bf16.argtypes = [ct.c_double]
            L.or_round_bf16.restype = ct.c_double
            _lib = L
    return _lib


def _p(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctype)


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# ----------------------------------------------------------------- scalars --
def philox4x64_10(ctr, key):
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint64))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint64))
    out = np.zeros(4, dtype=np.uint64)
    lib().or_philox4x64_10(_p(c, ct.POINTER(ct.c_uint64)), _p(k, ct.POINTER(ct.c_uint64)),
                           _p(out, ct.POINTER(ct.c_uint64)))
    return out


def philox_word(seed, block, step, batch, pos, v, stream) -> int:
    return int(lib().or_philox_word(seed, block, step, batch, pos, v, stream))


def uniform_token(w: int, V: int) -> int:
    return int(lib().or_uniform_token(w, V))


def gumbel(w: int) -> float:
    return float(lib().or_gumbel(w))


def gumbel_argmax(s, seed, block=0, step=0, batch=0, pos=0):
    s = np.ascontiguousarray(np.asarray(s, dtype=np.float64))
    gap = ct.c_double()
    i = lib().or_gumbel_argmax(_p(s, _D), s.size, seed, block, step, batch, pos, ct.byref(gap))
    return int(i), gap.value


def gumbel_argmax_many(s, seed, npos):
    s = np.ascontiguousarray(np.asarray(s, dtype=np.float64))
    out = np.zeros(npos, dtype=np.int32)
    lib().or_gumbel_argmax_many(_p(s, _D), s.size, seed, npos, _p(out, _I))
    return out


def uniform_many(V, seed, npos):
    out = np.zeros(npos, dtype=np.int32)
    lib().or_uniform_many(V, seed, npos, _p(out, _I))
    return out


def gumbel_many(seed, n):
    out = np.zeros(n, dtype=np.float32)
    lib().or_gumbel_many(seed, n, _p(out, _F))
    return out


def round_e4m3(x: float) -> float:
    return float(lib().or_round_e4m3(float(x)))


def e4m3_value(b: int) -> float:
    return float(lib().or_e4m3_value(int(b)))


def quantize_rows_e4m3(X):
    """Per-row E4M3 codes and scales of a float32 matrix [R, d] (or_quantize_rows_e4m3)."""
    Xf = _f32(X)
    R, d = Xf.shape
    Q = np.zeros((R, d), np.uint8)
    sc = np.zeros(R, np.float32)
    lib().or_quantize_rows_e4m3(_p(Xf, _F), R, d, _p(Q, _U8), _p(sc, _F))
    return Q, sc


def round_bf16(x: float) -> float:
    return float(lib().or_round_bf16(x))


def canvas_init(B, C, V, seed, block=0):
    t = np.zeros((B, C), dtype=np.int32)
    lib().or_canvas_init(_p(t, _I), B, C, V, seed, block)
    return t


# ---------------------------------------------------------- small pieces ----
def rmsnorm(x, eps=1e-6):
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    y = np.zeros_like(x)
    lib().or_rmsnorm(_p(x, _D), x.size, eps, _p(y, _D))
    return y


def rope(x, pos, base=10000.0):
    y = np.ascontiguousarray(np.array(x, dtype=np.float64))
    lib().or_rope(_p(y, _D), y.size, float(pos), float(base))
    return y


def gelu(x: float) -> float:
    return float(lib().or_gelu(float(x)))


def row_stats(logits, tau):
    l = np.ascontiguousarray(np.asarray(logits, dtype=np.float64))
    H, m, Z, g = (ct.c_double(), ct.c_double(), ct.c_double(), ct.c_double())
    am = ct.c_int32()
    lib().or_row_stats(_p(l, _D), l.size, float(tau), ct.byref(H), ct.byref(m), ct.byref(Z),
                       ct.byref(am), ct.byref(g))
    return dict(H=H.value, m=m.value, Z=Z.value, argmax=am.value, top2gap=g.value)


def accept(H, b):
    Hh = np.ascontiguousarray(np.asarray(H, dtype=np.float64))
    C = Hh.size
    acc = np.zeros(C, dtype=np.uint8)
    cum = np.zeros(C, dtype=np.float64)
    rank = np.zeros(C, dtype=np.int32)
    n = lib().or_accept(_p(Hh, _D), C, float(b), _p(acc, _U8), _p(cum, _D), _p(rank, _I))
    return dict(n=int(n), accept=acc.astype(bool), cum=cum, rank=rank)


def reveal(Z, argmax, tokens, mask_id, step, N):
    """Masked confidence decoding of one step (or_reveal): returns (new tokens, revealed mask, k)."""
    Zh = np.ascontiguousarray(np.asarray(Z, dtype=np.float64))
    am = np.ascontiguousarray(np.asarray(argmax, dtype=np.int32))
    tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32)).copy()
    rev = np.zeros(Zh.size, dtype=np.uint8)
    k = lib().or_reveal(_p(Zh, _D), _p(am, _I), _p(tok, _I), Zh.size, int(mask_id), int(step), int(N), _p(rev, _U8))
    if k < 0:
        raise ValueError("oracle reveal: bad arguments")
    return tok, rev.astype(bool), int(k)


def denoise_step_masked(dims, w, x, z, alpha, tau, mask_id, step, N, mirror_bf16=True, nthreads=None,
                        want_extra=(), fp8_head=None):
    """One step of masked confidence decoding: the forward and self-conditioning of denoise_step
    with the [MASK] token excluded from the softmax (not a prediction target), then or_reveal per
    canvas in place of the uniform-state accept / renoise."""
    out = denoise_step(dims, w, x, z, alpha, tau=tau, b=0.0, seed=0, step=0, mirror_bf16=mirror_bf16,
                       want=("H", "Z", "m", "argmax", "top2gap", "z_out", "u") + tuple(want_extra),
                       nthreads=nthreads, exclude_tok=mask_id, fp8_head=fp8_head)
    B, C = dims.B, dims.C
    tok = np.asarray(x, np.int32).reshape(B, C).copy()
    rev = np.zeros((B, C), bool)
    ks = []
    for bb in range(B):
        t, r, k = reveal(out["Z"][bb * C:(bb + 1) * C], out["argmax"][bb * C:(bb + 1) * C], tok[bb], mask_id,
                         step, N)
        tok[bb], rev[bb] = t, r
        ks.append(k)
    out["tokens_out"] = tok.reshape(-1)
    out["revealed"] = rev.reshape(-1)
    out["n_rev"] = np.array(ks, np.int32)
    return out


def attend_row(q, Kp, Vp, Kc, Vc):
    q = np.ascontiguousarray(np.asarray(q, dtype=np.float64))
    hd = q.size
    Kp = _f32(Kp).reshape(-1, hd)
    Vp = _f32(Vp).reshape(-1, hd)
    Kc = np.ascontiguousarray(np.asarray(Kc, dtype=np.float64)).reshape(-1, hd)
    Vc = np.ascontiguousarray(np.asarray(Vc, dtype=np.float64)).reshape(-1, hd)
    o = np.zeros(hd, dtype=np.float64)
    lib().or_attend_row(_p(q, _D), _p(Kp, _F), _p(Vp, _F), Kp.shape[0], _p(Kc, _D), _p(Vc, _D),
                        Kc.shape[0], hd, _p(o, _D))
    return o


# ------------------------------------------------------------- the step -----
def _dims(dims, mirror_bf16: bool, P=None):
    return Dims(V=dims.V, d=dims.d, C=dims.C, B=dims.B, Hq=dims.Hq, Hkv=dims.Hkv, hd=dims.hd,
                F=dims.F, P=dims.P if P is None else P, cap=dims.cap, rope_base=dims.rope_base,
                rms_eps=dims.rms_eps, mirror_bf16=1 if mirror_bf16 else 0, L=getattr(dims, "L", 1),
                n_exp=getattr(dims, "n_exp", 0), top_k=getattr(dims, "top_k", 0), Fe=getattr(dims, "Fe", 0))


class _MoeW(ct.Structure):
    _fields_ = [("Wr", _F), ("We1", _F), ("We2", _F)]


_WANT_ALL = ("a", "q", "k", "v", "o", "h", "logits", "H", "m", "Z", "top2gap", "argmax", "accept",
             "cum", "rank", "renoise_tok", "sample_tok", "gumbel_gap", "tokens_out", "u", "g",
             "z_out", "n_acc", "meanH", "stop")


def denoise_step(dims, w, x, z, alpha, tau, b, seed, step, block=0, prev_argmax=None,
                 stop_H=0.005, mirror_bf16=True, rows=None, want=None, nthreads=None, exclude_tok=-1,
                 fp8_head=None):
    """Run one oracle denoising step.

    dims: an object with V, d, C, B, Hq, Hkv, hd, F, P, cap, rope_base, rms_eps.
    w: dict of float32 numpy arrays E, Wq, Wk, Wv, Wo, W1, W2, Kc, Vc.
    x [B, C] int32, z [B, C, d] float32, alpha [B, C] float32.
    rows: optional list of global rows (b * C + i) for the vocabulary stages.
    fp8_head: optional (E8 uint8 [V, d], scale float32 [V]) from quantize_rows_e4m3(E): the LM head
    in FP8 (h quantized per row the same way); the embedding and p0 . E keep E.
    want: names of outputs to return (default: everything except logits).  In rows mode the
    logits are returned for the listed rows only, in their order ([len(rows), V]).
    """
    B, C, d, V, F = dims.B, dims.C, dims.d, dims.V, dims.F
    M, nq, nkv = B * C, dims.Hq * dims.hd, dims.Hkv * dims.hd
    if want is None:
        want = tuple(n for n in _WANT_ALL if n != "logits")
    nl = M if rows is None else len(rows)
    shapes = dict(a=(M, d), q=(M, nq), k=(M, nkv), v=(M, nkv), o=(M, nq), h=(M, d), logits=(nl, V),
                  H=(M,), m=(M,), Z=(M,), top2gap=(M,), argmax=(M,), accept=(M,), cum=(M,),
                  rank=(M,), renoise_tok=(M,), sample_tok=(M,), gumbel_gap=(M,), tokens_out=(M,),
                  u=(M, d), g=(M, F), z_out=(M, d), n_acc=(B,), meanH=(B,), stop=(B,))
    ne, tk = getattr(dims, "n_exp", 0), getattr(dims, "top_k", 0)
    shapes.update(moe_idx=(M, tk), moe_gate=(M, tk), moe_logits=(M, ne), moe_x=(M, d))
    types = dict(argmax=np.int32, accept=np.uint8, rank=np.int32, renoise_tok=np.int32,
                 sample_tok=np.int32, tokens_out=np.int32, n_acc=np.int32, stop=np.int32, moe_idx=np.int32)
    outs = {}
    so = StepOut()
    ctmap = {np.float64: _D, np.int32: _I, np.uint8: _U8}
    for n in want:
        t = types.get(n, np.float64)
        arr = np.zeros(shapes[n], dtype=t)
        outs[n] = arr
        setattr(so, n, _p(arr, ctmap[t]))
    keep = [_f32(w[k]) for k in ("E", "Wq", "Wk", "Wv", "Wo", "W1", "W2", "Kc", "Vc")]
    xx, zz, aa = _i32(x), _f32(z), _f32(alpha)
    pa = _i32(prev_argmax) if prev_argmax is not None else None
    e8 = es = None
    if fp8_head is not None:
        e8 = np.ascontiguousarray(np.asarray(fp8_head[0], np.uint8))
        es = _f32(fp8_head[1])
    mw = [_f32(w[k]) if k in w else None for k in ("Wr", "We1", "We2")] if ne > 0 else [None] * 3
    si = StepIn(*[_p(a, _F) for a in keep], _p(xx, _I), _p(zz, _F), _p(aa, _F),
                _p(pa, _I) if pa is not None else None, float(tau), float(b), float(stop_H),
                int(seed), int(step), int(block), int(exclude_tok),
                _p(e8, _U8) if e8 is not None else None, _p(es, _F) if es is not None else None,
                *[_p(a, _F) if a is not None else None for a in mw])
    rr = _i32(rows) if rows is not None else None
    nrows = 0 if rr is None else rr.size
    if rr is not None and rr.size == 0:
        rr = np.zeros(1, dtype=np.int32)  # non-null pointer: front stages only
    D = _dims(dims, mirror_bf16)
    rc = lib().or_denoise_step(ct.byref(D), ct.byref(si), ct.byref(so),
                               _p(rr, _I) if rr is not None else None,
                               nrows, nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle denoise_step: bad arguments")
    if "accept" in outs:
        outs["accept"] = outs["accept"].astype(bool)
    return outs


def moe_ffn(dims, Wr, We1, We2, h, mirror_bf16=True, nthreads=None):
    """The MoE FFN of one layer on rows h [n, d] (or_moe_ffn).  dims carries d, rms_eps, n_exp,
    top_k, Fe; Wr [n_exp, d], We1 [n_exp + 1, Fe, d], We2 [n_exp + 1, d, Fe] (index n_exp: the
    shared expert).  Returns dict(h=h + y, idx [n, top_k], gate [n, top_k], logits [n, n_exp])."""
    hh = np.ascontiguousarray(np.array(h, dtype=np.float64))
    n = hh.shape[0]
    idx = np.zeros((n, dims.top_k), np.int32)
    gate = np.zeros((n, dims.top_k))
    logits = np.zeros((n, dims.n_exp))
    D = _dims(dims, mirror_bf16, P=0)
    arrs = [_f32(Wr), _f32(We1), _f32(We2)]
    rc = lib().or_moe_ffn(ct.byref(D), *[_p(a, _F) for a in arrs], _p(hh, _D), n, _p(idx, _I), _p(gate, _D),
                          _p(logits, _D), nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle moe_ffn: bad arguments")
    return dict(h=hh, idx=idx, gate=gate, logits=logits)


def tau_schedule(N=48, tau0=0.8, tau1=0.4):
    """Temperatures of steps 0..N-1 of the linear anneal (or_tau)."""
    return np.array([lib().or_tau(float(tau0), float(tau1), int(N), s) for s in range(N)])


def denoise_canvas(dims, w, x0, alpha, seed, N=48, tau0=0.8, tau1=0.4, b=0.1, stop_H=0.005,
                   block=0, z0=None, mirror_bf16=True, nthreads=None):
    B, C, d = dims.B, dims.C, dims.d
    x = _i32(x0).copy().reshape(B, C)
    z = _f32(np.zeros((B, C, d)) if z0 is None else z0).copy()
    al = _f32(alpha)
    keep = [_f32(w[k]) for k in ("E", "Wq", "Wk", "Wv", "Wo", "W1", "W2", "Kc", "Vc")]
    steps = np.zeros(B, dtype=np.int32)
    conv = np.zeros(B, dtype=np.int32)
    acc = np.zeros((B, N), dtype=np.int32)
    xhat = np.zeros((B, C), dtype=np.int32)
    D = _dims(dims, mirror_bf16)
    rc = lib().or_denoise_canvas(ct.byref(D), *[_p(a, _F) for a in keep], _p(x, _I), _p(z, _F),
                                 _p(al, _F), N, tau0, tau1, b, stop_H, int(seed), int(block),
                                 _p(steps, _I), _p(conv, _I), _p(acc, _I), _p(xhat, _I),
                                 nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle denoise_canvas: bad arguments")
    return dict(tokens=x, z=z, steps_taken=steps, converged=conv, accepted=acc, xhat0=xhat)


def commit(dims, E, Wk, Wv, tokens, Kc, Vc, P, mirror_bf16=True, nthreads=None):
    """Append the re-encoded K/V of `tokens` [B, C] at rows P..P+C-1 (one layer); returns new (Kc, Vc)."""
    Kc = _f32(Kc).copy()
    Vc = _f32(Vc).copy()
    D = _dims(dims, mirror_bf16, P=P)
    rc = lib().or_commit(ct.byref(D), _p(_f32(E), _F), _p(_f32(Wk), _F), _p(_f32(Wv), _F),
                         _p(_i32(tokens), _I), _p(Kc, _F), _p(Vc, _F), nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle commit: cache capacity exceeded")
    return Kc, Vc


def prefill(dims, w, tokens, P, mirror_bf16=True, nthreads=None):
    """Causal re-encode of tokens [B, n] appended at rows P..P+n-1 of every layer's cache (or_prefill).
    w: E, Wq, Wk, Wv, Wo (stacked [L, ...] when L > 1), Kc, Vc ([L, B, Hkv, cap, hd] or [B, Hkv, cap, hd]).
    Returns the new (Kc, Vc) with the shape of w's."""
    Kc = _f32(w["Kc"]).copy()
    Vc = _f32(w["Vc"]).copy()
    tok = _i32(tokens)
    n = tok.shape[-1] if tok.ndim > 1 else tok.size // dims.B
    D = _dims(dims, mirror_bf16, P=P)
    mw = None
    if getattr(dims, "n_exp", 0) > 0:
        arrs = [_f32(w[k]) for k in ("Wr", "We1", "We2")]
        mw = _MoeW(*[_p(a, _F) for a in arrs])
    rc = lib().or_prefill(ct.byref(D), *[_p(_f32(w[k]), _F) for k in ("E", "Wq", "Wk", "Wv", "Wo")],
                          ct.byref(mw) if mw is not None else None,
                          _p(tok, _I), int(n), _p(Kc, _F), _p(Vc, _F), nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle prefill: cache capacity exceeded")
    return Kc, Vc
