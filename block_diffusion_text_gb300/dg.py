"""Python binding of libdg (ctypes).

Argument marshalling only: every step of the path runs in the CUDA kernels of
libdg.  PyTorch supplies device memory and the current stream.  The binding
fails loudly if the library has not been built (there is no CPU fallback).
The functions ``dg_*`` of the C ABI are reachable as ``lib().dg_*``; the
helpers below take torch tensors.
"""
from __future__ import annotations

import ctypes as ct
import math
import os
import threading
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libdg.so")
_lock = threading.Lock()
_lib = None

DG_OK, DG_ERR_ARG, DG_ERR_SHAPE, DG_ERR_CAPACITY, DG_ERR_WORKSPACE, DG_ERR_CUDA, DG_ERR_TIMEOUT, DG_ERR_VALUE = range(8)

# Every function the C header declares (checked by the tests).
EXPORTS = ("dg_status_string", "dg_workspace_size", "dg_read_status", "dg_tau", "dg_canvas_init",
           "dg_denoise_step", "dg_denoise_canvas", "dg_commit_block", "dg_debug_gemm",
           "dg_attention_noalloc", "dg_attention_noalloc_status", "dg_debug_wait_timeout",
           "dg_canvas_init_masked", "dg_denoise_step_masked", "dg_denoise_canvas_masked", "dg_prefill",
           "dg_quantize_rows_e4m3")


class DgError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


class dg_dims(ct.Structure):
    _fields_ = [("V", ct.c_int32), ("d", ct.c_int32), ("C", ct.c_int32), ("B", ct.c_int32),
                ("Hq", ct.c_int32), ("Hkv", ct.c_int32), ("hd", ct.c_int32), ("F", ct.c_int32),
                ("rope_base", ct.c_float), ("rms_eps", ct.c_float), ("L", ct.c_int32),
                ("n_exp", ct.c_int32), ("top_k", ct.c_int32), ("Fe", ct.c_int32)]


class dg_model(ct.Structure):
    _fields_ = [("dims", dg_dims)] + [(n, ct.c_void_p) for n in ("E", "Wq", "Wk", "Wv", "Wo", "W1", "W2",
                                                                 "E8", "E8_scale", "Wr", "We1", "We2")]


class dg_kv_cache(ct.Structure):
    _fields_ = [("K", ct.c_void_p), ("V", ct.c_void_p), ("cap", ct.c_int32), ("len", ct.c_int32)]


class dg_canvas(ct.Structure):
    _fields_ = [("tokens", ct.c_void_p), ("z", ct.c_void_p), ("alpha", ct.c_void_p),
                ("prev_argmax", ct.c_void_p)]


class dg_step_debug(ct.Structure):
    _fields_ = [(n, ct.c_void_p) for n in ("a", "q", "k", "v", "o", "h", "u", "g", "logits", "moe_idx", "moe_gate",
                                           "moe_logits", "moe_x")]


class dg_step_out(ct.Structure):
    _fields_ = [(n, ct.c_void_p) for n in ("entropy", "argmax", "accept", "n_acc", "mean_H", "stop")] + [
        ("debug", ct.POINTER(dg_step_debug)), ("events", ct.POINTER(ct.c_void_p))]


# Kernel slots of one step (dg_step_out.events), in launch order.
PROF_SLOTS = ("embed", "qkv", "attn", "oproj", "lmhead", "stats", "sampler", "p0", "selfcond",
              "reduce", "ffw1", "ffw2", "moe")


class dg_sched(ct.Structure):
    _fields_ = [("tau0", ct.c_float), ("tau1", ct.c_float), ("N", ct.c_int32), ("b", ct.c_float),
                ("stop_H", ct.c_float)]


class dg_canvas_result(ct.Structure):
    _fields_ = [(n, ct.c_void_p) for n in ("steps_taken", "converged", "accepted", "xhat0")]


def load():
    """Load libdg.so; raises if it is missing (build it with __graft_entry__.build())."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libdg is not built ({LIB_PATH} missing); run __graft_entry__.build()")
            L = ct.CDLL(LIB_PATH)
            L.dg_status_string.restype = ct.c_char_p
            L.dg_status_string.argtypes = [ct.c_int32]
            for name in EXPORTS[1:]:
                getattr(L, name).restype = ct.c_int32
            L.dg_workspace_size.argtypes = [ct.POINTER(dg_dims), ct.c_int32, ct.POINTER(ct.c_size_t)]
            L.dg_read_status.argtypes = [ct.c_void_p, ct.POINTER(ct.c_int32), ct.c_void_p]
            L.dg_tau.argtypes = [ct.POINTER(dg_sched), ct.c_int32, ct.POINTER(ct.c_float)]
            L.dg_attention_noalloc_status.argtypes = [ct.POINTER(ct.c_int32), ct.c_void_p]
            L.dg_canvas_init_masked.argtypes = [ct.c_void_p, ct.c_int32, ct.c_int32, ct.c_int32, ct.c_void_p]
            L.dg_denoise_step_masked.argtypes = [ct.POINTER(dg_model), ct.POINTER(dg_kv_cache),
                                                 ct.POINTER(dg_canvas), ct.c_float, ct.c_int32, ct.c_int32,
                                                 ct.c_int32, ct.c_void_p, ct.c_size_t, ct.POINTER(dg_step_out),
                                                 ct.c_void_p]
            L.dg_denoise_canvas_masked.argtypes = [ct.POINTER(dg_model), ct.POINTER(dg_kv_cache),
                                                   ct.POINTER(dg_canvas), ct.POINTER(dg_sched), ct.c_int32,
                                                   ct.c_void_p, ct.c_size_t, ct.POINTER(dg_canvas_result),
                                                   ct.c_void_p]
            L.dg_canvas_init.argtypes = [ct.c_void_p, ct.c_int32, ct.c_int32, ct.c_int32, ct.c_uint64,
                                         ct.c_int32, ct.c_void_p]
            L.dg_denoise_step.argtypes = [ct.POINTER(dg_model), ct.POINTER(dg_kv_cache),
                                          ct.POINTER(dg_canvas), ct.c_float, ct.c_float, ct.c_uint64,
                                          ct.c_int32, ct.c_int32, ct.c_void_p, ct.c_size_t,
                                          ct.POINTER(dg_step_out), ct.c_void_p]
            L.dg_denoise_canvas.argtypes = [ct.POINTER(dg_model), ct.POINTER(dg_kv_cache),
                                            ct.POINTER(dg_canvas), ct.POINTER(dg_sched), ct.c_uint64,
                                            ct.c_int32, ct.c_void_p, ct.c_size_t,
                                            ct.POINTER(dg_canvas_result), ct.c_void_p]
            L.dg_commit_block.argtypes = [ct.POINTER(dg_model), ct.POINTER(dg_kv_cache), ct.c_void_p,
                                          ct.c_void_p, ct.c_size_t, ct.c_void_p]
            L.dg_prefill.argtypes = [ct.POINTER(dg_model), ct.POINTER(dg_kv_cache), ct.c_void_p, ct.c_int32,
                                     ct.c_void_p, ct.c_size_t, ct.c_void_p]
            L.dg_debug_wait_timeout.argtypes = [ct.POINTER(ct.c_int32), ct.c_void_p]
            L.dg_quantize_rows_e4m3.argtypes = [ct.c_void_p, ct.c_int32, ct.c_int32, ct.c_void_p, ct.c_void_p,
                                                ct.c_void_p]
            L.dg_debug_gemm.argtypes = [ct.c_void_p, ct.c_void_p, ct.c_void_p, ct.c_int32, ct.c_int32,
                                        ct.c_int32, ct.c_int32, ct.c_void_p]
            L.dg_attention_noalloc.argtypes = [ct.c_void_p, ct.c_void_p, ct.c_void_p, ct.c_int32, ct.c_int32,
                                               ct.c_void_p, ct.c_void_p, ct.c_void_p, ct.c_int32, ct.c_int32,
                                               ct.c_int32, ct.c_int32, ct.c_int32, ct.c_void_p]
            _lib = L
    return _lib


lib = load


def status_string(code: int) -> str:
    try:
        return load().dg_status_string(code).decode()
    except Exception:  # library missing while formatting an error
        return "status"


def _check(code, what):
    if code != DG_OK:
        raise DgError(code, what)


def _ptr(t):
    return None if t is None else ct.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ct.c_void_p(s.cuda_stream)


def make_dims(d) -> dg_dims:
    return dg_dims(V=d.V, d=d.d, C=d.C, B=d.B, Hq=d.Hq, Hkv=d.Hkv, hd=d.hd, F=d.F,
                   rope_base=d.rope_base, rms_eps=d.rms_eps, L=getattr(d, "L", 1),
                   n_exp=getattr(d, "n_exp", 0), top_k=getattr(d, "top_k", 0), Fe=getattr(d, "Fe", 0))


def workspace_size(dims, cap: int) -> int:
    n = ct.c_size_t()
    _check(load().dg_workspace_size(ct.byref(make_dims(dims)), int(cap), ct.byref(n)), "dg_workspace_size")
    return n.value


class Model:
    """Weights (bf16 device tensors, [out][in]) and the prefix cache of a batch of canvases."""

    def __init__(self, dims, w: dict, cache_len: int | None = None, fp8_head: bool = False):
        """fp8_head: quantize E per row to E4M3 (quantize_rows_e4m3) and take the
        LM head's logits on the FP8 tensor cores; E8 / E8_scale are then kept
        here as the codes and scales."""
        self.dims = dims
        self.w = w
        self.K, self.V = w["Kc"], w["Vc"]
        self.cap = self.K.shape[-2]
        self.len = dims.P if cache_len is None else cache_len
        self.E8 = self.E8_scale = None
        if fp8_head:
            self.E8, self.E8_scale = quantize_rows_e4m3(w["E"])
        self.s = dg_model(make_dims(dims), *[ct.c_void_p(w[k].data_ptr()) for k in
                                             ("E", "Wq", "Wk", "Wv", "Wo", "W1", "W2")],
                          ct.c_void_p(self.E8.data_ptr() if fp8_head else None),
                          ct.c_void_p(self.E8_scale.data_ptr() if fp8_head else None),
                          *[ct.c_void_p(w[k].data_ptr() if k in w else None) for k in ("Wr", "We1", "We2")])
        self.ws_bytes = workspace_size(dims, self.cap)
        # zero-initialised: the first word is the device status word
        self.ws = torch.zeros(self.ws_bytes + 256, dtype=torch.uint8, device=self.K.device)
        off = (-self.ws.data_ptr()) % 256
        self.ws_ptr = ct.c_void_p(self.ws.data_ptr() + off)

    def cache(self) -> dg_kv_cache:
        key = (self.K.data_ptr(), self.V.data_ptr(), self.cap, self.len)
        if getattr(self, "_cache_key", None) != key:
            self._cache_s = dg_kv_cache(ct.c_void_p(key[0]), ct.c_void_p(key[1]), self.cap, self.len)
            self._cache_key = key
        return self._cache_s

    def workspace_for(self, cap: int):
        """(pointer, bytes) of a workspace for a cache of `cap` rows: the model's own when that is
        large enough, else one allocated once per capacity (a commit into a larger cache)."""
        if cap <= self.cap:
            return self.ws_ptr, self.ws_bytes
        extra = getattr(self, "_ws_extra", {})
        if cap not in extra:
            nb = workspace_size(self.dims, cap)
            t = torch.zeros(nb + 256, dtype=torch.uint8, device=self.K.device)
            extra[cap] = (t, ct.c_void_p(t.data_ptr() + (-t.data_ptr()) % 256), nb)
            self._ws_extra = extra
        return extra[cap][1], extra[cap][2]

    def status(self) -> int:
        """The device status word (first non-zero over the model's workspaces)."""
        for ptr in [self.ws_ptr] + [e[1] for e in getattr(self, "_ws_extra", {}).values()]:
            st = ct.c_int32()
            _check(load().dg_read_status(ptr, ct.byref(st), _stream()), "dg_read_status")
            if st.value:
                return st.value
        return 0


@dataclass
class Canvas:
    tokens: torch.Tensor          # int32 [B, C]
    z: torch.Tensor               # bf16 [B, C, d]
    alpha: torch.Tensor           # fp32 [B, C]
    prev_argmax: torch.Tensor | None = None

    def __post_init__(self):
        if self.prev_argmax is None:
            self.prev_argmax = torch.zeros_like(self.tokens)

    def struct(self) -> dg_canvas:
        key = (self.tokens.data_ptr(), self.z.data_ptr(), self.alpha.data_ptr(), self.prev_argmax.data_ptr())
        if getattr(self, "_key", None) != key:
            self._s = dg_canvas(*[ct.c_void_p(p) for p in key])
            self._key = key
        return self._s


_STEP_OUT_CACHE: dict = {}


def denoise_step(model: Model, canvas: Canvas, tau: float, b: float, seed: int, step: int, block: int = 0,
                 debug: bool = False, stream=None, events=None, out=None, masked=None) -> dict:
    """One denoising step (dg_denoise_step); updates canvas in place, returns outputs.

    events: optional list of 2 * len(PROF_SLOTS) recorded torch.cuda.Event (per-kernel timing).
    out: optional dict of preallocated output tensors (as returned by a previous call).
    masked: optional (mask_id, N): a step of masked confidence decoding (dg_denoise_step_masked)
    instead; b, seed and block are then not used.
    """
    d = model.dims
    dev = canvas.tokens.device
    M = d.B * d.C
    if out is None:
        out = dict(entropy=torch.empty(d.B, d.C, dtype=torch.float32, device=dev),
                   argmax=torch.empty(d.B, d.C, dtype=torch.int32, device=dev),
                   accept=torch.empty(d.B, d.C, dtype=torch.uint8, device=dev),
                   n_acc=torch.empty(d.B, dtype=torch.int32, device=dev),
                   mean_H=torch.empty(d.B, dtype=torch.float32, device=dev),
                   stop=torch.empty(d.B, dtype=torch.int32, device=dev))
    keys = ("entropy", "argmax", "accept", "n_acc", "mean_H", "stop")
    ptrs = tuple(out[k].data_ptr() for k in keys)
    so = _STEP_OUT_CACHE.get(ptrs) if events is None and not debug else None
    if so is None:
        so = dg_step_out(*[ct.c_void_p(p) for p in ptrs])
        if events is None and not debug:
            _STEP_OUT_CACHE.clear()  # one entry: the output set of the latest plain call
            _STEP_OUT_CACHE[ptrs] = so
    if events is not None:
        if len(events) != 2 * len(PROF_SLOTS):
            raise ValueError(f"events: expected {2 * len(PROF_SLOTS)} entries, got {len(events)}")
        arr = (ct.c_void_p * len(events))(*[ct.c_void_p(e.cuda_event if e is not None else 0) for e in events])
        so.events = ct.cast(arr, ct.POINTER(ct.c_void_p))
    dbg = None
    if debug:
        bf = dict(dtype=torch.bfloat16, device=dev)
        dbg_t = dict(a=torch.empty(M, d.d, **bf), q=torch.empty(d.B, d.Hq, d.C, d.hd, **bf),
                     k=torch.empty(d.B, d.Hkv, d.C, d.hd, **bf), v=torch.empty(d.B, d.Hkv, d.C, d.hd, **bf),
                     o=torch.empty(M, d.Hq * d.hd, **bf), h=torch.empty(M, d.d, **bf),
                     u=torch.empty(M, d.d, **bf), g=torch.empty(M, d.F, **bf),
                     logits=torch.empty(M, d.V, dtype=torch.float32, device=dev))
        ne, tk = getattr(d, "n_exp", 0), getattr(d, "top_k", 0)
        if ne > 0:
            dbg_t.update(moe_idx=torch.empty(M, tk, dtype=torch.int32, device=dev),
                         moe_gate=torch.empty(M, tk, dtype=torch.float32, device=dev),
                         moe_logits=torch.empty(M, ne, dtype=torch.float32, device=dev),
                         moe_x=torch.empty(M, d.d, **bf))
        dbg = dg_step_debug(*[_ptr(dbg_t.get(k)) for k in ("a", "q", "k", "v", "o", "h", "u", "g", "logits",
                                                            "moe_idx", "moe_gate", "moe_logits", "moe_x")])
        so.debug = ct.pointer(dbg)
        out["debug"] = dbg_t
    cs = canvas.struct()
    cache = model.cache()
    if masked is not None:
        mask_id, N = masked
        rc = load().dg_denoise_step_masked(ct.byref(model.s), ct.byref(cache), ct.byref(cs), float(tau),
                                           int(mask_id), int(step), int(N), model.ws_ptr, model.ws_bytes,
                                           ct.byref(so), _stream(stream))
        _check(rc, "dg_denoise_step_masked")
        return out
    rc = load().dg_denoise_step(ct.byref(model.s), ct.byref(cache), ct.byref(cs), float(tau), float(b),
                                int(seed), int(step), int(block), model.ws_ptr, model.ws_bytes,
                                ct.byref(so), _stream(stream))
    _check(rc, "dg_denoise_step")
    return out


def tau(step: int, N: int = 48, tau0: float = 0.8, tau1: float = 0.4) -> float:
    """Temperature of step `step` of the annealed schedule, as the library computes it (dg_tau)."""
    t = ct.c_float()
    _check(load().dg_tau(ct.byref(dg_sched(tau0, tau1, N, 0.1, 0.005)), int(step), ct.byref(t)), "dg_tau")
    return t.value


def tau_schedule(N=48, tau0=0.8, tau1=0.4):
    """Temperatures of steps 0..N-1 (dg_tau for each step)."""
    return [tau(s, N, tau0, tau1) for s in range(N)]


def denoise_canvas(model: Model, canvas: Canvas, seed: int, block: int = 0, N: int = 48, tau0: float = 0.8,
                   tau1: float = 0.4, b: float = 0.1, stop_H: float = 0.005, stream=None) -> dict:
    """The annealed loop (dg_denoise_canvas); returns device tensors of the result."""
    d = model.dims
    dev = canvas.tokens.device
    res = dict(steps_taken=torch.empty(d.B, dtype=torch.int32, device=dev),
               converged=torch.empty(d.B, dtype=torch.int32, device=dev),
               accepted=torch.empty(d.B, N, dtype=torch.int32, device=dev),
               xhat0=torch.empty(d.B, d.C, dtype=torch.int32, device=dev))
    rs = dg_canvas_result(*[_ptr(res[k]) for k in ("steps_taken", "converged", "accepted", "xhat0")])
    sched = dg_sched(tau0, tau1, N, b, stop_H)
    cs = canvas.struct()
    cache = model.cache()
    rc = load().dg_denoise_canvas(ct.byref(model.s), ct.byref(cache), ct.byref(cs), ct.byref(sched), int(seed),
                                  int(block), model.ws_ptr, model.ws_bytes, ct.byref(rs), _stream(stream))
    _check(rc, "dg_denoise_canvas")
    return res


def denoise_canvas_masked(model: Model, canvas: Canvas, mask_id: int, N: int = 16, tau: float = 1.0,
                          stream=None) -> dict:
    """Masked confidence decoding loop (dg_denoise_canvas_masked): N steps at temperature tau."""
    d = model.dims
    dev = canvas.tokens.device
    res = dict(steps_taken=torch.empty(d.B, dtype=torch.int32, device=dev),
               converged=torch.empty(d.B, dtype=torch.int32, device=dev),
               accepted=torch.empty(d.B, N, dtype=torch.int32, device=dev),
               xhat0=torch.empty(d.B, d.C, dtype=torch.int32, device=dev))
    rs = dg_canvas_result(*[_ptr(res[k]) for k in ("steps_taken", "converged", "accepted", "xhat0")])
    sched = dg_sched(tau, tau, N, 0.0, 0.0)
    cs = canvas.struct()
    cache = model.cache()
    rc = load().dg_denoise_canvas_masked(ct.byref(model.s), ct.byref(cache), ct.byref(cs), ct.byref(sched),
                                         int(mask_id), model.ws_ptr, model.ws_bytes, ct.byref(rs), _stream(stream))
    _check(rc, "dg_denoise_canvas_masked")
    return res


def canvas_init_masked(B, C, mask_id, device="cuda", stream=None) -> torch.Tensor:
    """A canvas of [MASK] tokens (dg_canvas_init_masked)."""
    t = torch.empty(B, C, dtype=torch.int32, device=device)
    _check(load().dg_canvas_init_masked(_ptr(t), B, C, int(mask_id), _stream(stream)), "dg_canvas_init_masked")
    return t


def commit_block(model: Model, tokens: torch.Tensor, stream=None, cache=None) -> int:
    """Append the re-encoded K/V of tokens [B, C] to the cache (dg_commit_block).

    cache: optional (K, V, len) of another cache with the model's layout ([B, Hkv, cap, hd] bf16);
    by default the model's own cache, whose length is advanced.  Returns the new length."""
    if cache is None:
        cs = model.cache()
    else:
        K, V, n = cache
        cs = dg_kv_cache(ct.c_void_p(K.data_ptr()), ct.c_void_p(V.data_ptr()), K.shape[-2], int(n))
    ws, wsb = model.workspace_for(cs.cap)
    rc = load().dg_commit_block(ct.byref(model.s), ct.byref(cs), _ptr(tokens), ws, wsb, _stream(stream))
    _check(rc, "dg_commit_block")
    if cache is None:
        model.len = cs.len
    return cs.len


def prefill(model: Model, tokens: torch.Tensor, stream=None) -> int:
    """Causal prefill of tokens [B, n] into every layer's cache (dg_prefill); returns the new length."""
    cache = model.cache()
    tok = tokens.contiguous()
    rc = load().dg_prefill(ct.byref(model.s), ct.byref(cache), _ptr(tok), int(tok.shape[-1]), model.ws_ptr,
                           model.ws_bytes, _stream(stream))
    _check(rc, "dg_prefill")
    model.len = cache.len
    return cache.len


def canvas_init(B, C, V, seed, block=0, device="cuda", stream=None) -> torch.Tensor:
    t = torch.empty(B, C, dtype=torch.int32, device=device)
    _check(load().dg_canvas_init(_ptr(t), B, C, V, int(seed), int(block), _stream(stream)), "dg_canvas_init")
    return t


def debug_gemm(A: torch.Tensor, Bm: torch.Tensor, b_mn_major: int = 0, stream=None) -> torch.Tensor:
    """fp32 A B^T on the tensor-core engine; B is [N][K] (b_mn_major 0, 3 on CTA pairs, 5-8 on
    the cluster split-K engine) or [K][N] (1 or 2, or 4 on CTA pairs)."""
    M, K = A.shape
    N = Bm.shape[0] if b_mn_major in (0, 3, 5, 6, 7, 8) else Bm.shape[1]
    D = torch.empty(M, N, dtype=torch.float32, device=A.device)
    _check(load().dg_debug_gemm(_ptr(A), _ptr(Bm), _ptr(D), M, N, K, b_mn_major, _stream(stream)),
           "dg_debug_gemm")
    return D


def debug_wait_timeout(stream=None) -> int:
    """Run the never-satisfied bounded wait (dg_debug_wait_timeout); returns the status word it left."""
    st = ct.c_int32(-1)
    _check(load().dg_debug_wait_timeout(ct.byref(st), _stream(stream)), "dg_debug_wait_timeout")
    return st.value


def attention_noalloc(q, K, V, cache_len, k, v, o=None, stream=None) -> torch.Tensor:
    """Step attention with the library's static scratch (dg_attention_noalloc), for callers
    that cannot allocate device memory; q [B,Hq,C,hd], K/V [B,Hkv,cap,hd], k/v [B,Hkv,C,hd]."""
    B, Hq, C, hd = q.shape
    Hkv, cap = K.shape[1], K.shape[2]
    if o is None:
        o = torch.empty(B * C, Hq * hd, dtype=q.dtype, device=q.device)
    _check(load().dg_attention_noalloc(_ptr(q), _ptr(K), _ptr(V), cap, int(cache_len), _ptr(k), _ptr(v), _ptr(o),
                                       B, C, Hq, Hkv, hd, _stream(stream)), "dg_attention_noalloc")
    return o


def attention_noalloc_status(stream=None) -> int:
    """Status word of the last attention_noalloc call on this device (synchronises the stream)."""
    st = ct.c_int32(-1)
    _check(load().dg_attention_noalloc_status(ct.byref(st), _stream(stream)), "dg_attention_noalloc_status")
    return st.value


def quantize_rows_e4m3(X: torch.Tensor, stream=None):
    """Per-row E4M3 codes (uint8 [R, d]) and scales (fp32 [R]) of a bf16 matrix X [R, d]."""
    assert X.dtype == torch.bfloat16 and X.dim() == 2 and X.is_contiguous()
    R, d = X.shape
    Q = torch.empty((R, d), dtype=torch.uint8, device=X.device)
    sc = torch.empty(R, dtype=torch.float32, device=X.device)
    _check(load().dg_quantize_rows_e4m3(_ptr(X), R, d, _ptr(Q), _ptr(sc), _stream(stream)),
           "dg_quantize_rows_e4m3")
    return Q, sc
