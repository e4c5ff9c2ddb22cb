"""The C-ABI library without a GPU: it loads, exports every declared symbol, and
rejects bad arguments with the documented codes before touching the device.
Device pointers passed here are never dereferenced: every call takes an error
path that returns before any CUDA call."""
import ctypes as ct
import dataclasses
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dg():
    import __graft_entry__ as g
    from block_diffusion_text_gb300 import dg as _dg
    if not os.path.exists(_dg.LIB_PATH):
        g.build_cuda()
    _dg.load()
    return _dg


def _declared():
    with open(os.path.join(ROOT, "include", "dg.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"DG_API[^;(]*?\b(dg_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("dg_denoise_step", "dg_denoise_canvas", "dg_commit_block", "dg_workspace_size"):
        assert n in names


def test_library_exports_every_declared_symbol(dg):
    lib = ct.CDLL(dg.LIB_PATH)
    for n in _declared():
        assert hasattr(lib, n), n
    assert set(_declared()) == set(dg.EXPORTS)


def test_status_strings(dg):
    L = dg.load()
    seen = {L.dg_status_string(c).decode() for c in range(8)}
    assert len(seen) == 8
    assert L.dg_status_string(99).decode() == "unknown status"


def _dims(**kw):
    from block_diffusion_text_gb300 import synth
    d = synth.workload("step_v32k_c256_p2k")[0]
    from dataclasses import replace
    return replace(d, **kw)


def test_workspace_size_validates_dims(dg):
    L = dg.load()
    n = ct.c_size_t()
    assert L.dg_workspace_size(ct.byref(dg.make_dims(_dims())), 2048, ct.byref(n)) == dg.DG_OK
    assert n.value > 2 * 256 * 32768  # holds at least the exp(s - m) tiles
    bad = [(dict(V=1001), dg.DG_ERR_SHAPE), (dict(hd=96), dg.DG_ERR_SHAPE), (dict(Hq=6, Hkv=4), dg.DG_ERR_ARG),
           (dict(C=2048), dg.DG_ERR_SHAPE), (dict(d=1000), dg.DG_ERR_SHAPE), (dict(F=100), dg.DG_ERR_SHAPE),
           (dict(B=0), dg.DG_ERR_ARG)]
    for kw, code in bad:
        assert L.dg_workspace_size(ct.byref(dg.make_dims(_dims(**kw))), 2048, ct.byref(n)) == code, kw
    assert L.dg_workspace_size(None, 2048, ct.byref(n)) == dg.DG_ERR_ARG
    assert L.dg_workspace_size(ct.byref(dg.make_dims(_dims())), -1, ct.byref(n)) == dg.DG_ERR_ARG
    # grows with the cache capacity (attention partials are sized for it)
    n2 = ct.c_size_t()
    L.dg_workspace_size(ct.byref(dg.make_dims(_dims())), 131072, ct.byref(n2))
    assert n2.value >= n.value


FAKE = 1 << 20  # a non-null address that is never dereferenced on these paths


def _structs(dg, dims, ws_bytes=None, cap=2048, length=2048):
    m = dg.dg_model(dg.make_dims(dims), *[ct.c_void_p(FAKE)] * 7)
    c = dg.dg_kv_cache(ct.c_void_p(FAKE), ct.c_void_p(FAKE), cap, length)
    cv = dg.dg_canvas(*[ct.c_void_p(FAKE)] * 4)
    L = dg.load()
    n = ct.c_size_t()
    L.dg_workspace_size(ct.byref(dg.make_dims(dims)), cap, ct.byref(n))
    return m, c, cv, n.value if ws_bytes is None else ws_bytes


def test_step_argument_errors(dg):
    L = dg.load()
    dims = _dims()
    m, c, cv, wsb = _structs(dg, dims)
    ws = ct.c_void_p(1 << 30)
    call = lambda m_, c_, cv_, tau, ws_, wsb_: L.dg_denoise_step(
        m_, c_, cv_, tau, 0.1, 1, 0, 0, ws_, wsb_, None, None)
    assert call(None, ct.byref(c), ct.byref(cv), 0.8, ws, wsb) == dg.DG_ERR_ARG
    assert call(ct.byref(m), None, ct.byref(cv), 0.8, ws, wsb) == dg.DG_ERR_ARG
    assert call(ct.byref(m), ct.byref(c), None, 0.8, ws, wsb) == dg.DG_ERR_ARG
    assert call(ct.byref(m), ct.byref(c), ct.byref(cv), 0.0, ws, wsb) == dg.DG_ERR_ARG
    assert call(ct.byref(m), ct.byref(c), ct.byref(cv), 0.8, ws, wsb - 1) == dg.DG_ERR_WORKSPACE
    assert call(ct.byref(m), ct.byref(c), ct.byref(cv), 0.8, ct.c_void_p((1 << 30) + 8), wsb) == \
        dg.DG_ERR_WORKSPACE
    assert call(ct.byref(m), ct.byref(c), ct.byref(cv), 0.8, None, wsb) == dg.DG_ERR_ARG
    c_bad = dg.dg_kv_cache(ct.c_void_p(FAKE), ct.c_void_p(FAKE), 100, 200)   # len > cap
    assert call(ct.byref(m), ct.byref(c_bad), ct.byref(cv), 0.8, ws, wsb) == dg.DG_ERR_ARG
    m_null = dg.dg_model(dg.make_dims(dims), *([ct.c_void_p(FAKE)] * 6 + [None]))
    assert call(ct.byref(m_null), ct.byref(c), ct.byref(cv), 0.8, ws, wsb) == dg.DG_ERR_ARG


def test_canvas_loop_argument_errors(dg):
    L = dg.load()
    dims = _dims()
    m, c, cv, wsb = _structs(dg, dims)
    ws = ct.c_void_p(1 << 30)
    res = dg.dg_canvas_result(*[ct.c_void_p(FAKE)] * 4)
    for sched in (dg.dg_sched(0.8, 0.4, 0, 0.1, 0.005), dg.dg_sched(0.0, 0.4, 48, 0.1, 0.005),
                  dg.dg_sched(0.8, 0.4, 48, -1.0, 0.005)):
        assert L.dg_denoise_canvas(ct.byref(m), ct.byref(c), ct.byref(cv), ct.byref(sched), 1, 0, ws, wsb,
                                   ct.byref(res), None) == dg.DG_ERR_ARG
    good = dg.dg_sched(0.8, 0.4, 48, 0.1, 0.005)
    assert L.dg_denoise_canvas(ct.byref(m), ct.byref(c), ct.byref(cv), ct.byref(good), 1, 0, ws, wsb,
                               None, None) == dg.DG_ERR_ARG


def test_commit_capacity_is_checked_before_any_write(dg):
    L = dg.load()
    dims = _dims()
    m, c, cv, wsb = _structs(dg, dims, cap=2100, length=2048)  # 2048 + 256 > 2100
    ws = ct.c_void_p(1 << 30)
    assert L.dg_commit_block(ct.byref(m), ct.byref(c), ct.c_void_p(FAKE), ws, wsb, None) == dg.DG_ERR_CAPACITY
    assert c.len == 2048
    assert L.dg_commit_block(ct.byref(m), ct.byref(c), None, ws, wsb, None) == dg.DG_ERR_ARG


def test_small_entry_points_validate(dg):
    L = dg.load()
    assert L.dg_canvas_init(None, 1, 16, 512, 0, 0, None) == dg.DG_ERR_ARG
    assert L.dg_canvas_init(ct.c_void_p(FAKE), 1, 0, 512, 0, 0, None) == dg.DG_ERR_ARG
    st = ct.c_int32()
    assert L.dg_read_status(None, ct.byref(st), None) == dg.DG_ERR_ARG
    assert L.dg_debug_gemm(None, None, None, 1, 8, 8, 0, None) == dg.DG_ERR_ARG
    assert L.dg_debug_wait_timeout(None, None) == dg.DG_ERR_ARG
    assert L.dg_debug_gemm(ct.c_void_p(FAKE), ct.c_void_p(FAKE), ct.c_void_p(FAKE), 4, 12, 8, 0, None) == \
        dg.DG_ERR_SHAPE
    assert L.dg_debug_gemm(ct.c_void_p(FAKE), ct.c_void_p(FAKE), ct.c_void_p(FAKE), 4, 16, 64, 9, None) == \
        dg.DG_ERR_ARG
    # the cluster split-K modes need a 64-wide K block per slice
    for mode, k in ((5, 64), (6, 192), (7, 64), (8, 192)):
        assert L.dg_debug_gemm(ct.c_void_p(FAKE), ct.c_void_p(FAKE), ct.c_void_p(FAKE), 4, 16, k, mode, None) == \
            dg.DG_ERR_SHAPE
    f = ct.c_void_p(FAKE)
    assert L.dg_attention_noalloc(f, f, f, 100, 50, f, f, f, 1, 16, 2, 1, 96, None) == dg.DG_ERR_SHAPE
    assert L.dg_attention_noalloc(f, f, f, 100, 200, f, f, f, 1, 16, 2, 1, 32, None) == dg.DG_ERR_ARG
    assert L.dg_attention_noalloc(None, f, f, 100, 50, f, f, f, 1, 16, 2, 1, 32, None) == dg.DG_ERR_ARG
    # sizes the step rejects are rejected here too, before any CUDA call
    assert L.dg_attention_noalloc(f, f, f, 100, 50, f, f, f, 1, 2048, 2, 1, 32, None) == dg.DG_ERR_SHAPE
    assert L.dg_attention_noalloc(f, f, f, 100, 50, f, f, f, 2048, 1024, 2, 1, 32, None) == dg.DG_ERR_SHAPE
    assert L.dg_attention_noalloc(f, f, f, 100, 50, f, f, f, 2, 16, 32768, 1, 32, None) == dg.DG_ERR_SHAPE
    big = 2 ** 31 - 1
    assert L.dg_attention_noalloc(f, f, f, big, big - 8, f, f, f, 1, 16, 2, 1, 32, None) == dg.DG_ERR_SHAPE
    assert L.dg_attention_noalloc_status(None, None) == dg.DG_ERR_ARG


def test_tau_schedule_is_the_linear_anneal(dg):
    """dg_tau: tau0 at step 0, tau1 at step N-1, linear in between ([TR] Table 2: 0.8 -> 0.4 over
    48 steps); arguments outside the schedule are rejected."""
    L = dg.load()
    t = ct.c_float()
    sched = dg.dg_sched(0.8, 0.4, 48, 0.1, 0.005)
    got = []
    for s in range(48):
        assert L.dg_tau(ct.byref(sched), s, ct.byref(t)) == dg.DG_OK
        got.append(t.value)
    assert got[0] == pytest.approx(0.8, abs=1e-7) and got[-1] == pytest.approx(0.4, abs=1e-7)
    steps = [got[s + 1] - got[s] for s in range(47)]
    assert max(steps) == pytest.approx(min(steps), abs=1e-6)
    assert steps[0] == pytest.approx(-0.4 / 47, abs=1e-6)
    import oracle
    assert got == pytest.approx(list(oracle.tau_schedule(48, 0.8, 0.4)), abs=1e-7)
    one = dg.dg_sched(0.7, 0.4, 1, 0.1, 0.005)
    assert L.dg_tau(ct.byref(one), 0, ct.byref(t)) == dg.DG_OK and t.value == pytest.approx(0.7)
    for s in (-1, 48):
        assert L.dg_tau(ct.byref(sched), s, ct.byref(t)) == dg.DG_ERR_ARG
    assert L.dg_tau(None, 0, ct.byref(t)) == dg.DG_ERR_ARG
    assert L.dg_tau(ct.byref(sched), 0, None) == dg.DG_ERR_ARG
    assert L.dg_tau(ct.byref(dg.dg_sched(0.0, 0.4, 48, 0.1, 0.005)), 0, ct.byref(t)) == dg.DG_ERR_ARG


def test_masked_entry_points_validate(dg):
    L = dg.load()
    dims = _dims()
    m, c, cv, wsb = _structs(dg, dims)
    ws = ct.c_void_p(1 << 30)
    call = lambda tau, mask, step, N: L.dg_denoise_step_masked(ct.byref(m), ct.byref(c), ct.byref(cv), tau, mask,
                                                               step, N, ws, wsb, None, None)
    assert call(0.0, 5, 0, 4) == dg.DG_ERR_ARG
    assert call(0.8, -1, 0, 4) == dg.DG_ERR_ARG
    assert call(0.8, dims.V, 0, 4) == dg.DG_ERR_ARG
    assert call(0.8, 5, 4, 4) == dg.DG_ERR_ARG
    assert call(0.8, 5, 0, 0) == dg.DG_ERR_ARG
    res = dg.dg_canvas_result(*[ct.c_void_p(FAKE)] * 4)
    sched = dg.dg_sched(0.8, 0.8, 16, 0.0, 0.0)
    assert L.dg_denoise_canvas_masked(ct.byref(m), ct.byref(c), ct.byref(cv), ct.byref(sched), dims.V, ws, wsb,
                                      ct.byref(res), None) == dg.DG_ERR_ARG
    assert L.dg_denoise_canvas_masked(ct.byref(m), ct.byref(c), ct.byref(cv), ct.byref(sched), 5, ws, wsb,
                                      None, None) == dg.DG_ERR_ARG
    assert L.dg_canvas_init_masked(None, 1, 16, 5, None) == dg.DG_ERR_ARG
    assert L.dg_canvas_init_masked(ct.c_void_p(FAKE), 1, 16, -1, None) == dg.DG_ERR_ARG


def test_layers_and_prefill_validate(dg):
    L = dg.load()
    n = ct.c_size_t()
    for bad in (0, 65):
        dd = dg.make_dims(_dims())
        dd.L = bad
        assert L.dg_workspace_size(ct.byref(dd), 2048, ct.byref(n)) == dg.DG_ERR_ARG
    dims = _dims()
    m, c, cv, wsb = _structs(dg, dims, cap=2100, length=2048)
    ws = ct.c_void_p(1 << 30)
    assert L.dg_prefill(ct.byref(m), ct.byref(c), ct.c_void_p(FAKE), 0, ws, wsb, None) == dg.DG_ERR_ARG
    assert L.dg_prefill(ct.byref(m), ct.byref(c), None, 10, ws, wsb, None) == dg.DG_ERR_ARG
    assert L.dg_prefill(ct.byref(m), ct.byref(c), ct.c_void_p(FAKE), 53, ws, wsb, None) == dg.DG_ERR_CAPACITY
    assert c.len == 2048


def test_fp8_head_entry_points_validate(dg):
    """dg_quantize_rows_e4m3 argument checks, and a model whose FP8 head has codes but no scales (or
    misaligned codes) is rejected before any launch."""
    L = dg.load()
    f = ct.c_void_p(FAKE)
    assert L.dg_quantize_rows_e4m3(None, 4, 64, f, f, None) == dg.DG_ERR_ARG
    assert L.dg_quantize_rows_e4m3(f, 4, 64, None, f, None) == dg.DG_ERR_ARG
    assert L.dg_quantize_rows_e4m3(f, 4, 64, f, None, None) == dg.DG_ERR_ARG
    assert L.dg_quantize_rows_e4m3(f, -1, 64, f, f, None) == dg.DG_ERR_ARG
    assert L.dg_quantize_rows_e4m3(ct.c_void_p(FAKE + 8), 4, 64, f, f, None) == dg.DG_ERR_ARG
    assert L.dg_quantize_rows_e4m3(f, 4, 40, f, f, None) == dg.DG_ERR_SHAPE
    assert L.dg_quantize_rows_e4m3(f, 4, 0, f, f, None) == dg.DG_ERR_SHAPE
    dims = _dims()
    m, c, cv, wsb = _structs(dg, dims)
    ws = ct.c_void_p(1 << 30)
    for e8, es in ((f, None), (None, f), (ct.c_void_p(FAKE + 8), f)):
        m.E8, m.E8_scale = e8, es
        assert L.dg_denoise_step(ct.byref(m), ct.byref(c), ct.byref(cv), 0.8, 0.1, 1, 0, 0, ws, wsb, None,
                                 None) == dg.DG_ERR_ARG


def test_moe_dims_and_weights_validate(dg):
    L = dg.load()
    n = ct.c_size_t()
    base = _dims()

    def ws_rc(**kw):
        dd = dg.make_dims(base)
        for k, v in kw.items():
            setattr(dd, k, v)
        return L.dg_workspace_size(ct.byref(dd), 2048, ct.byref(n))
    assert ws_rc(n_exp=128, top_k=8, Fe=768) == dg.DG_OK
    assert ws_rc(n_exp=128, top_k=0, Fe=768) == dg.DG_ERR_ARG
    assert ws_rc(n_exp=4, top_k=5, Fe=768) == dg.DG_ERR_ARG
    assert ws_rc(n_exp=257, top_k=8, Fe=768) == dg.DG_ERR_ARG
    assert ws_rc(n_exp=128, top_k=17, Fe=768) == dg.DG_ERR_ARG
    assert ws_rc(n_exp=-1) == dg.DG_ERR_ARG
    assert ws_rc(n_exp=128, top_k=8, Fe=700) == dg.DG_ERR_SHAPE
    assert ws_rc(n_exp=128, top_k=8, Fe=768, d=1088) == dg.DG_ERR_SHAPE   # d not a multiple of 128
    assert ws_rc(n_exp=128, top_k=8, Fe=768, B=17) == dg.DG_ERR_SHAPE    # B * C > 4096
    dims = dataclasses.replace(base, n_exp=16, top_k=4, Fe=128)
    m, c, cv, wsb = _structs(dg, dims)
    ws = ct.c_void_p(1 << 30)
    m.Wr, m.We1, m.We2 = ct.c_void_p(FAKE), None, ct.c_void_p(FAKE)
    assert L.dg_denoise_step(ct.byref(m), ct.byref(c), ct.byref(cv), 0.8, 0.1, 1, 0, 0, ws, wsb, None,
                             None) == dg.DG_ERR_ARG
