"""ctypes binding of libdgcanvas: the same names as the C ABI, argument
marshalling only (every step of the path runs in the library's kernels).

Tensors are torch tensors already on the GPU; PyTorch provides device
memory and streams, nothing else. Every call checks shapes, dtypes and
contiguity, passes raw pointers, and raises DGError on a non-zero status.
Loading fails loudly if the library has not been built: there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

DG_OK = 0
DG_ERR_INVALID_ARG, DG_ERR_UNSUPPORTED, DG_ERR_WORKSPACE, DG_ERR_CUDA, DG_ERR_TIMEOUT, DG_ERR_DEVICE_BOUNDS = (
    -1, -2, -3, -4, -5, -6)
DG_BF16, DG_F32 = 0, 1
DG_MASK_BIDIR, DG_MASK_CAUSAL_BLOCK = 0, 1

_c_int, _c_i64, _c_u64, _c_u32, _c_f, _c_sz, _p = (ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32,
                                                   ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p)

_SIGS = {
    "dg_status_string": (ctypes.c_char_p, [_c_int]),
    "dg_device_status": (_c_int, [_p]),
    "dg_canvas_attn_workspace_size": (_c_sz, [_c_int, _c_int, _c_int, _c_int, _c_i64, _c_int]),
    "dg_canvas_attn": (_c_int, [_p, _p, _p, _c_i64, _c_i64, _p, _p, _p, _p, _c_int, _c_int, _c_int, _c_int, _c_f,
                                _c_int, _c_int, _p, _c_sz, _p]),
    "dg_canvas_attn_noalloc": (_c_int, [_p, _p, _p, _c_i64, _c_i64, _p, _p, _p, _p, _c_int, _c_int, _c_int, _c_int,
                                        _c_f, _c_int, _c_int, _p]),
    "dg_canvas_attn_noalloc_max_scratch": (_c_sz, []),
    "dg_vocab_step_workspace_size": (_c_sz, [_c_int, _c_int, _c_int, _c_int]),
    "dg_vocab_step_plan": (_c_int, [_c_int, _c_int, _c_int, _c_int, _p]),
    "dg_vocab_step": (_c_int, [_p, _p, _c_int, _c_int, _c_int, _c_int, _p, _p, _p, _p, _p, _c_sz, _p]),
    "dg_vocab_step_renoise": (_c_int, [_p, _p, _c_int, _c_int, _c_int, _c_int, _p, _p, _p, _p, _p, _c_f, _c_u64,
                                       _c_u32, _c_i64, _p, _p, _c_sz, _p]),
    "dg_renoise": (_c_int, [_p, _p, _p, _c_int, _c_int, _c_f, _c_u64, _c_u32, _c_i64, _p, _p]),
    "dg_canvas_init": (_c_int, [_p, _c_int, _c_int, _c_u64, _c_i64, _p]),
    "dg_kv_append": (_c_int, [_p, _p, _c_i64, ctypes.POINTER(_c_i64), _p, _p, _c_int, _c_int, _c_int, _c_int, _p,
                              _c_int, _p, _p, _p, _c_sz, _p]),
    "dg_selfcond_input": (_c_int, [_p, _p, _p, _p, _c_int, _c_int, _c_int, _c_int, _p]),
    "dg_token_prob": (_c_int, [_p, _p, _p, _p, _p, _c_int, _c_int, _c_int, _c_int, _p]),
    "dg_unmask": (_c_int, [_p, _p, _p, _c_int, ctypes.c_int32, _c_f, _p, _p]),
    "dg_canvas_fill": (_c_int, [_p, _c_int, ctypes.c_int32, _p]),
    "dg_count_flags": (_c_int, [_p, _c_int, _p, _p]),
    "dg_canvas_attn_devlen": (_c_int, [_p, _p, _p, _c_i64, _p, _c_i64, _p, _p, _p, _p, _c_int, _c_int, _c_int, _c_int,
                                       _c_f, _c_int, _c_int, _p, _c_sz, _p]),
    "dg_canvas_init_devpos": (_c_int, [_p, _c_int, _c_int, _c_u64, _p, _p]),
    "dg_vocab_step_renoise_devpos": (_c_int, [_p, _p, _c_int, _c_int, _c_int, _c_int, _p, _p, _p, _p, _p, _c_f,
                                              _c_u64, _c_u32, _p, _p, _p, _c_sz, _p]),
    "dg_kv_append_devlen": (_c_int, [_p, _p, _c_i64, _p, _p, _p, _c_int, _c_int, _c_int, _c_int, _p]),
    "dg_debug_inject": (_c_int, [_c_int, _c_int]),
}

EXPORTS = tuple(_SIGS)


class DGError(RuntimeError):
    def __init__(self, fn, code, text):
        super().__init__(f"{fn} failed: {text} ({code})")
        self.code = code


_LIB = None


def load(path: str | None = None):
    """Loads libdgcanvas (built in-tree by canvas_denoising_gb300.build)."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    path = path or _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libdgcanvas is not built ({path} missing): run "
                           "`python -m canvas_denoising_gb300.build` or __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == _build.LIB:
        _LIB = lib
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn, code):
    if code != DG_OK:
        raise DGError(fn, code, load().dg_status_string(code).decode())


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return DG_BF16
    if t.dtype == torch.float32:
        return DG_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _need(t, name, device=True):
    if t is None:
        return
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def status_string(code: int) -> str:
    return load().dg_status_string(code).decode()


def device_status(stream=None) -> int:
    return load().dg_device_status(_stream(stream))


# ------------------------------------------------------------------ attention
def canvas_attn_workspace_size(C, Hq, Hkv, hd, prefix_len, dtype=DG_BF16) -> int:
    return load().dg_canvas_attn_workspace_size(C, Hq, Hkv, hd, prefix_len, dtype)


def canvas_attn(q, k_cache, v_cache, prefix_len, k_canvas, v_canvas, out=None, lse=None, scale=-1.0,
                mask=DG_MASK_BIDIR, workspace=None, stream=None):
    """q [C][Hq][hd]; caches [Hkv][cap][hd]; canvas K/V [Hkv][C][hd]. Returns (out, lse)."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (k_canvas, "k_canvas"), (v_canvas, "v_canvas")):
        _need(t, n)
    C, Hq, hd = q.shape
    Hkv, cap = k_cache.shape[0], k_cache.shape[1]
    dt = _dtype_code(q)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, C), dtype=torch.float32, device=q.device)
    ws_need = canvas_attn_workspace_size(C, Hq, Hkv, hd, prefix_len, dt)
    if workspace is None and ws_need:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().dg_canvas_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), cap, prefix_len, _ptr(k_canvas),
                               _ptr(v_canvas), _ptr(out), _ptr(lse), C, Hq, Hkv, hd, float(scale), dt, mask,
                               _ptr(workspace), ws_bytes, _stream(stream))
    _check("dg_canvas_attn", rc)
    return out, lse


def canvas_attn_noalloc(q, k_cache, v_cache, prefix_len, k_canvas, v_canvas, out=None, lse=None, scale=-1.0,
                        mask=DG_MASK_BIDIR, stream=None):
    """dg_canvas_attn without a workspace: for callers that cannot allocate
    device memory (the scratch is a fixed array inside the library)."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (k_canvas, "k_canvas"), (v_canvas, "v_canvas")):
        _need(t, n)
    C, Hq, hd = q.shape
    Hkv, cap = k_cache.shape[0], k_cache.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, C), dtype=torch.float32, device=q.device)
    rc = load().dg_canvas_attn_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), cap, prefix_len, _ptr(k_canvas),
                                       _ptr(v_canvas), _ptr(out), _ptr(lse), C, Hq, Hkv, hd, float(scale),
                                       _dtype_code(q), mask, _stream(stream))
    _check("dg_canvas_attn_noalloc", rc)
    return out, lse


# ------------------------------------------------------------------ vocabulary step
def vocab_step_workspace_size(C, V, d, dtype=DG_BF16) -> int:
    return load().dg_vocab_step_workspace_size(C, V, d, dtype)


def vocab_step_plan(C, V, d, dtype=DG_BF16) -> dict:
    """The launch plan dg_vocab_step uses on the current device."""
    buf = (ctypes.c_int32 * 6)()
    _check("dg_vocab_step_plan", load().dg_vocab_step_plan(C, V, d, dtype, ctypes.cast(buf, ctypes.c_void_p)))
    return dict(zip(("producers", "consumers", "vocab_split", "cluster_pairs", "ctas", "vocab_tiles"), list(buf)))


def vocab_step(h, emb, argmax=None, conf=None, lse=None, selfcond=None, workspace=None, want_selfcond=True,
               stream=None):
    """h [C][d], emb [V][d]. Returns (argmax int32, conf f32, lse f32, selfcond)."""
    _need(h, "h")
    _need(emb, "emb")
    C, d = h.shape
    V = emb.shape[0]
    dt = _dtype_code(h)
    dev = h.device
    argmax = torch.empty(C, dtype=torch.int32, device=dev) if argmax is None else argmax
    conf = torch.empty(C, dtype=torch.float32, device=dev) if conf is None else conf
    lse = torch.empty(C, dtype=torch.float32, device=dev) if lse is None else lse
    if selfcond is None and want_selfcond:
        selfcond = torch.empty((C, d), dtype=h.dtype, device=dev)
    need = vocab_step_workspace_size(C, V, d, dt)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().dg_vocab_step(_ptr(h), _ptr(emb), C, V, d, dt, _ptr(argmax), _ptr(conf), _ptr(lse), _ptr(selfcond),
                              _ptr(workspace), ws_bytes, _stream(stream))
    _check("dg_vocab_step", rc)
    return argmax, conf, lse, selfcond


def vocab_step_renoise(h, emb, tokens, threshold, seed, step, abs_pos0, argmax=None, conf=None, lse=None,
                       selfcond=None, renoised=None, workspace=None, stream=None):
    """dg_vocab_step and dg_renoise in one call (re-noise fused into the last kernel)."""
    _need(h, "h")
    _need(emb, "emb")
    _need(tokens, "tokens")
    C, d = h.shape
    V = emb.shape[0]
    dt = _dtype_code(h)
    dev = h.device
    argmax = torch.empty(C, dtype=torch.int32, device=dev) if argmax is None else argmax
    conf = torch.empty(C, dtype=torch.float32, device=dev) if conf is None else conf
    lse = torch.empty(C, dtype=torch.float32, device=dev) if lse is None else lse
    selfcond = torch.empty((C, d), dtype=h.dtype, device=dev) if selfcond is None else selfcond
    need = vocab_step_workspace_size(C, V, d, dt)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().dg_vocab_step_renoise(_ptr(h), _ptr(emb), C, V, d, dt, _ptr(argmax), _ptr(conf), _ptr(lse),
                                      _ptr(selfcond), _ptr(tokens), float(threshold), seed, step, abs_pos0,
                                      _ptr(renoised), _ptr(workspace), ws_bytes, _stream(stream))
    _check("dg_vocab_step_renoise", rc)
    return argmax, conf, lse, selfcond


# ------------------------------------------------------------------ re-noise / init
def renoise(tokens, argmax, conf, V, threshold, seed, step, abs_pos0, renoised=None, stream=None):
    for t, n in ((tokens, "tokens"), (argmax, "argmax"), (conf, "conf"), (renoised, "renoised")):
        _need(t, n)
    C = tokens.shape[0]
    rc = load().dg_renoise(_ptr(tokens), _ptr(argmax), _ptr(conf), C, V, float(threshold), seed, step, abs_pos0,
                           _ptr(renoised), _stream(stream))
    _check("dg_renoise", rc)
    return tokens


def canvas_init(tokens, V, seed, abs_pos0, stream=None):
    _need(tokens, "tokens")
    rc = load().dg_canvas_init(_ptr(tokens), tokens.shape[0], V, seed, abs_pos0, _stream(stream))
    _check("dg_canvas_init", rc)
    return tokens


# ------------------------------------------------------------------ KV append
def kv_append(k_cache, v_cache, length: int, k_new, v_new, q_new=None, out=None, lse=None, workspace=None,
              stream=None):
    """Appends [Hkv][C][hd] rows at `length`; returns (new_length, out, lse)."""
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (k_new, "k_new"), (v_new, "v_new"), (q_new, "q_new")):
        _need(t, n)
    Hkv, cap, hd = k_cache.shape
    C = k_new.shape[1]
    dt = _dtype_code(k_cache)
    Hq = 0
    if q_new is not None:
        Hq = q_new.shape[1]
        if out is None:
            out = torch.empty_like(q_new)
        if lse is None:
            lse = torch.empty((Hq, C), dtype=torch.float32, device=q_new.device)
        need = canvas_attn_workspace_size(C, Hq, Hkv, hd, length, dt)
        if workspace is None and need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q_new.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    n = ctypes.c_int64(length)
    rc = load().dg_kv_append(_ptr(k_cache), _ptr(v_cache), cap, ctypes.byref(n), _ptr(k_new), _ptr(v_new), C, Hkv, hd,
                             dt, _ptr(q_new), Hq, _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, _stream(stream))
    _check("dg_kv_append", rc)
    return n.value, out, lse


# ------------------------------------------------------------------ next to the step
def selfcond_input(tokens, emb, selfcond=None, x=None, stream=None):
    """x[i] = emb[tokens[i]] + selfcond[i] (the next step's stand-in input)."""
    for t, n in ((tokens, "tokens"), (emb, "emb"), (selfcond, "selfcond"), (x, "x")):
        _need(t, n)
    C = tokens.shape[0]
    V, d = emb.shape
    if x is None:
        x = torch.empty((C, d), dtype=emb.dtype, device=emb.device)
    rc = load().dg_selfcond_input(_ptr(tokens), _ptr(emb), _ptr(selfcond), _ptr(x), C, V, d, _dtype_code(emb),
                                  _stream(stream))
    _check("dg_selfcond_input", rc)
    return x


def token_prob(h, emb, tokens, lse, prob=None, stream=None):
    """prob[i] = exp(h[i] . emb[tokens[i]] - lse[i]): the current token's probability."""
    for t, n in ((h, "h"), (emb, "emb"), (tokens, "tokens"), (lse, "lse"), (prob, "prob")):
        _need(t, n)
    C, d = h.shape
    V = emb.shape[0]
    if prob is None:
        prob = torch.empty(C, dtype=torch.float32, device=h.device)
    rc = load().dg_token_prob(_ptr(h), _ptr(emb), _ptr(tokens), _ptr(lse), _ptr(prob), C, V, d, _dtype_code(h),
                              _stream(stream))
    _check("dg_token_prob", rc)
    return prob


def unmask(tokens, argmax, conf, mask_id, threshold, unmasked=None, stream=None):
    for t, n in ((tokens, "tokens"), (argmax, "argmax"), (conf, "conf"), (unmasked, "unmasked")):
        _need(t, n)
    rc = load().dg_unmask(_ptr(tokens), _ptr(argmax), _ptr(conf), tokens.shape[0], int(mask_id), float(threshold),
                          _ptr(unmasked), _stream(stream))
    _check("dg_unmask", rc)
    return tokens


def canvas_fill(tokens, value, stream=None):
    _need(tokens, "tokens")
    rc = load().dg_canvas_fill(_ptr(tokens), tokens.shape[0], int(value), _stream(stream))
    _check("dg_canvas_fill", rc)
    return tokens


def count_flags(flags, count=None, stream=None):
    """Device-side count of non-zero flags (an int32 tensor of one element)."""
    _need(flags, "flags")
    if count is None:
        count = torch.empty(1, dtype=torch.int32, device=flags.device)
    rc = load().dg_count_flags(_ptr(flags), flags.shape[0], _ptr(count), _stream(stream))
    _check("dg_count_flags", rc)
    return count


# ------------------------------------------------------------------ device-side cache length
def canvas_attn_devlen(q, k_cache, v_cache, prefix_len_dev, prefix_max, k_canvas, v_canvas, out=None, lse=None,
                       scale=-1.0, mask=DG_MASK_BIDIR, workspace=None, stream=None):
    """dg_canvas_attn with the prefix length in a device int64 tensor of one element."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (k_canvas, "k_canvas"),
                 (v_canvas, "v_canvas"), (prefix_len_dev, "prefix_len_dev")):
        _need(t, n)
    C, Hq, hd = q.shape
    Hkv, cap = k_cache.shape[0], k_cache.shape[1]
    dt = _dtype_code(q)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((Hq, C), dtype=torch.float32, device=q.device) if lse is None else lse
    need = canvas_attn_workspace_size(C, Hq, Hkv, hd, prefix_max, dt)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().dg_canvas_attn_devlen(_ptr(q), _ptr(k_cache), _ptr(v_cache), cap, _ptr(prefix_len_dev), prefix_max,
                                      _ptr(k_canvas), _ptr(v_canvas), _ptr(out), _ptr(lse), C, Hq, Hkv, hd,
                                      float(scale), dt, mask, _ptr(workspace), ws_bytes, _stream(stream))
    _check("dg_canvas_attn_devlen", rc)
    return out, lse


def canvas_init_devpos(tokens, V, seed, abs_pos0_dev, stream=None):
    _need(tokens, "tokens")
    rc = load().dg_canvas_init_devpos(_ptr(tokens), tokens.shape[0], V, seed, _ptr(abs_pos0_dev), _stream(stream))
    _check("dg_canvas_init_devpos", rc)
    return tokens


def vocab_step_renoise_devpos(h, emb, tokens, threshold, seed, step, abs_pos0_dev, argmax, conf, lse, selfcond,
                              renoised, workspace, stream=None):
    C, d = h.shape
    V = emb.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().dg_vocab_step_renoise_devpos(_ptr(h), _ptr(emb), C, V, d, _dtype_code(h), _ptr(argmax), _ptr(conf),
                                             _ptr(lse), _ptr(selfcond), _ptr(tokens), float(threshold), seed, step,
                                             _ptr(abs_pos0_dev), _ptr(renoised), _ptr(workspace), ws_bytes,
                                             _stream(stream))
    _check("dg_vocab_step_renoise_devpos", rc)
    return tokens


def kv_append_devlen(k_cache, v_cache, len_dev, k_new, v_new, stream=None):
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (k_new, "k_new"), (v_new, "v_new")):
        _need(t, n)
    Hkv, cap, hd = k_cache.shape
    rc = load().dg_kv_append_devlen(_ptr(k_cache), _ptr(v_cache), cap, _ptr(len_dev), _ptr(k_new), _ptr(v_new),
                                    k_new.shape[1], Hkv, hd, _dtype_code(k_cache), _stream(stream))
    _check("dg_kv_append_devlen", rc)


# ------------------------------------------------------------------ failure injection (tests)
INJECT_NONE, INJECT_ATTN_ARRIVAL, INJECT_VOCAB_READY = 0, 1, 2


def debug_inject(kind: int, wait_ms: int = 0):
    """The next launch of the named kernel withholds one cross-CTA arrival, so
    its bounded waits expire (DG_ERR_TIMEOUT) after `wait_ms`."""
    _check("dg_debug_inject", load().dg_debug_inject(int(kind), int(wait_ms)))
