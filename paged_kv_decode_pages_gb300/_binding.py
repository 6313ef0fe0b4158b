"""ctypes binding of libpkv (include/pkv.h).  Argument marshalling only: torch
tensors become device pointers, the current torch CUDA stream becomes the
``stream`` argument, and a non-zero status raises ``PkvError``.  There is no
fallback of any kind: without the library (or a GPU) every call raises."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

KIND_OTHER, KIND_AUDIO, KIND_STOP = 0, 1, 2
CODE_PAD = -1  # PKV_CODE_PAD

_P = ctypes.c_void_p
_I = ctypes.c_int
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_U32 = ctypes.c_uint32
_F = ctypes.c_float
_SZ = ctypes.c_size_t


class pkv_cache_t(ctypes.Structure):
    _fields_ = [("num_layers", _I32), ("num_pages", _I32), ("page_size", _I32),
                ("num_kv_heads", _I32), ("head_dim", _I32)]


class pkv_sample_ext_t(ctypes.Structure):
    _fields_ = [("min_p", _P), ("rep_penalty", _P), ("rep_window", _P), ("history", _P),
                ("hist_len", _P), ("hist_cap", _I32), ("logprob_raw", _P),
                ("logprob_proc", _P)]


# every symbol include/pkv.h declares, with its ctypes signature
SIGNATURES = {
    "pkv_version": (ctypes.c_char_p, []),
    "pkv_error_string": (ctypes.c_char_p, [_I]),
    "pkv_num_dev_error_bits": (_I, []),
    "pkv_last_cuda_error": (_I, []),
    "pkv_cuda_error_name": (ctypes.c_char_p, [_I]),
    "pkv_kv_append": (_I, [ctypes.POINTER(pkv_cache_t), _P, _I, _P, _P, _P, _I, _P, _P, _I, _P,
                           _P]),
    "pkv_decode_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "pkv_selftest_wait_timeout": (_I, [ctypes.c_ulonglong, _P, _P]),
    "pkv_paged_decode_attn": (_I, [ctypes.POINTER(pkv_cache_t), _P, _I, _P, _I, _F, _P, _I, _P,
                                   _P, _I, _P, _I, _P, _P, _SZ, _P, _P]),
    "pkv_paged_decode_attn_static": (_I, [ctypes.POINTER(pkv_cache_t), _P, _I, _P, _I, _F, _P,
                                          _I, _P, _P, _I, _P, _I, _P, _P, _P]),
    "pkv_decode_plan": (_I, [ctypes.POINTER(pkv_cache_t), _I, _I, _P, _P, _I, _P, _SZ, _P, _P]),
    "pkv_paged_decode_attn_planned": (_I, [ctypes.POINTER(pkv_cache_t), _P, _I, _P, _I, _F, _P,
                                           _I, _P, _P, _I, _P, _I, _P, _P, _SZ, _P, _P]),
    "pkv_kv_append_tokens": (_I, [ctypes.POINTER(pkv_cache_t), _P, _I, _P, _P, _I, _P, _P, _I,
                                  _P, _P, _I, _P, _P]),
    "pkv_prefill_workspace_bytes": (_SZ, [_I]),
    "pkv_prefill_attn": (_I, [ctypes.POINTER(pkv_cache_t), _P, _I, _P, _I, _F, _I, _P, _P, _I, _P,
                              _P, _I, _P, _P, _P, _SZ, _P, _P]),
    "pkv_sample_workspace_bytes": (_SZ, [_I, _I]),
    "pkv_seeded_sample": (_I, [_P, _I64, _I, _I, _P, _P, _I, _P, _P, _P, _P, _P, _U32, _I, _P,
                               _I, _I32, _I32, _P, _P, _P, _SZ, _P, _P]),
    "pkv_sample_ext_workspace_bytes": (_SZ, [_I, _I]),
    "pkv_seeded_sample_ext": (_I, [_P, _I64, _I, _I, _P, _P, _I, _P, _P, _P, _P, _P, _U32, _I,
                                   _P, _I, _I32, _I32, _P, _P, ctypes.POINTER(pkv_sample_ext_t),
                                   _P, _SZ, _P, _P]),
    "pkv_frame_workspace_bytes": (_SZ, [_I, _I, _I]),
    "pkv_codebook_frame_sample": (_I, [_P, _P, _I, _I, _I, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P,
                                       _P, _SZ, _P, _P]),
    "pkv_frame_sample_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "pkv_frame_sample": (_I, [_P, _I, _I32, _P, _P, _I, _I, _I, _P, _P, _I, _P, _P, _P, _P, _P,
                              _P, _P, _P, _SZ, _P, _P]),
}

_lock = threading.Lock()
_lib = None


class PkvError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        msg = "%s failed: %s (status %d)" % (fn, error_string(status), status)
        self.cuda_error = 0
        if status == 3:  # PKV_ERR_CUDA: name the CUDA runtime's error
            lib = load()
            self.cuda_error = int(lib.pkv_last_cuda_error())
            if self.cuda_error:
                msg += ": %s (%d)" % (lib.pkv_cuda_error_name(self.cuda_error).decode(),
                                      self.cuda_error)
        super().__init__(msg)


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libpkv.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if build_if_missing and not _build.up_to_date():
                _build.build()
            if not os.path.exists(path):
                raise RuntimeError("libpkv.so is missing (%s); run paged_kv_decode_pages_gb300."
                                   "build.build()" % path)
            L = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def version() -> str:
    return load().pkv_version().decode()


def error_string(status: int) -> str:
    return load().pkv_error_string(int(status)).decode()


def _check(fn, status):
    if status != 0:
        raise PkvError(fn, status)


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _geom(cache):
    L, P, two, ps, hkv, d = cache.shape
    assert two == 2, "cache dim 2 must be 2 (K, V)"
    return pkv_cache_t(L, P, ps, hkv, d)


def _req(t, dtype, name, cuda=True):
    import torch
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if cuda and not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    return t


# ---------------------------------------------------------------------------
def kv_append(cache, layer, k, v, page_table, seq_lens, active, err_word=None, stream=None):
    import torch
    _req(cache, torch.bfloat16, "cache")
    _req(k, torch.bfloat16, "k")
    _req(v, torch.bfloat16, "v")
    _req(page_table, torch.int32, "page_table")
    _req(seq_lens, torch.int32, "seq_lens")
    _req(active, torch.int32, "active")
    g = _geom(cache)
    st = load().pkv_kv_append(ctypes.byref(g), _ptr(cache), int(layer), _ptr(k), _ptr(v),
                              _ptr(page_table), page_table.shape[1], _ptr(seq_lens),
                              _ptr(active), seq_lens.shape[0], _ptr(err_word), _stream(stream))
    _check("pkv_kv_append", st)


def decode_workspace_bytes(batch, num_qo_heads, head_dim, max_pages, page_size=16) -> int:
    return int(load().pkv_decode_workspace_bytes(batch, num_qo_heads, head_dim, max_pages,
                                                 page_size))


def paged_decode_attn(cache, layer, q, page_table, seq_lens, active, out, workspace,
                      lse=None, sm_scale=None, err_word=None, stream=None, planned=False):
    """pkv_paged_decode_attn, or with planned=True pkv_paged_decode_attn_planned
    (the workspace then holds a plan from decode_plan for this batch)."""
    import torch
    _req(cache, torch.bfloat16, "cache")
    _req(q, torch.bfloat16, "q")
    _req(page_table, torch.int32, "page_table")
    _req(seq_lens, torch.int32, "seq_lens")
    _req(active, torch.int32, "active")
    if out.dtype not in (torch.bfloat16, torch.float32) or not out.is_contiguous():
        raise TypeError("out must be a contiguous bf16 or fp32 tensor")
    g = _geom(cache)
    B, Hq, D = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / (D ** 0.5)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    name = "pkv_paged_decode_attn_planned" if planned else "pkv_paged_decode_attn"
    st = getattr(load(), name)(
        ctypes.byref(g), _ptr(cache), int(layer), _ptr(q), Hq, float(sm_scale), _ptr(page_table),
        page_table.shape[1], _ptr(seq_lens), _ptr(active), B, _ptr(out),
        int(out.dtype == torch.float32), _ptr(lse), _ptr(workspace), ws_bytes, _ptr(err_word),
        _stream(stream))
    _check(name, st)


def paged_decode_attn_planned(cache, layer, q, page_table, seq_lens, active, out, workspace,
                              lse=None, sm_scale=None, err_word=None, stream=None):
    """pkv_paged_decode_attn_planned: one layer's attention on the plan that
    decode_plan wrote into the workspace."""
    paged_decode_attn(cache, layer, q, page_table, seq_lens, active, out, workspace, lse=lse,
                      sm_scale=sm_scale, err_word=err_word, stream=stream, planned=True)


def decode_plan(cache, num_qo_heads, max_pages, seq_lens, active, workspace, err_word=None,
                stream=None):
    """pkv_decode_plan: the batch's attention schedule, once per step, for
    paged_decode_attn(..., planned=True) calls of every layer."""
    import torch
    _req(cache, torch.bfloat16, "cache")
    _req(seq_lens, torch.int32, "seq_lens")
    _req(active, torch.int32, "active")
    g = _geom(cache)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().pkv_decode_plan(ctypes.byref(g), int(num_qo_heads), int(max_pages),
                                _ptr(seq_lens), _ptr(active), seq_lens.shape[0],
                                _ptr(workspace), ws_bytes, _ptr(err_word), _stream(stream))
    _check("pkv_decode_plan", st)


def selftest_wait_timeout(limit_ns, err_word, stream=None):
    """pkv_selftest_wait_timeout: the kernels' bounded wait run on an
    mbarrier nothing completes; sets the timeout bit of err_word."""
    import torch
    _req(err_word, torch.int32, "err_word")
    st = load().pkv_selftest_wait_timeout(int(limit_ns), _ptr(err_word), _stream(stream))
    _check("pkv_selftest_wait_timeout", st)


STATIC_SCRATCH_BYTES = 32 << 20  # PKV_ATTN_STATIC_SCRATCH_BYTES


def paged_decode_attn_static(cache, layer, q, page_table, seq_lens, active, out, lse=None,
                             sm_scale=None, err_word=None, stream=None):
    """pkv_paged_decode_attn_static: the same attention with the library's
    own device scratch, for callers that have no device memory to lend."""
    import torch
    _req(cache, torch.bfloat16, "cache")
    _req(q, torch.bfloat16, "q")
    _req(page_table, torch.int32, "page_table")
    _req(seq_lens, torch.int32, "seq_lens")
    _req(active, torch.int32, "active")
    if out.dtype not in (torch.bfloat16, torch.float32) or not out.is_contiguous():
        raise TypeError("out must be a contiguous bf16 or fp32 tensor")
    g = _geom(cache)
    B, Hq, D = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / (D ** 0.5)
    st = load().pkv_paged_decode_attn_static(
        ctypes.byref(g), _ptr(cache), int(layer), _ptr(q), Hq, float(sm_scale), _ptr(page_table),
        page_table.shape[1], _ptr(seq_lens), _ptr(active), B, _ptr(out),
        int(out.dtype == torch.float32), _ptr(lse), _ptr(err_word), _stream(stream))
    _check("pkv_paged_decode_attn_static", st)


def kv_append_tokens(cache, layer, k, v, qo_indptr, page_table, seq_lens, active, err_word=None,
                     stream=None):
    """The packed new tokens k, v (bf16 [T, Hkv, D]) of a prefill / mixed step
    into their positions (request b: rows qo_indptr[b] .. qo_indptr[b+1],
    ending at position seq_lens[b] - 1)."""
    import torch
    _req(cache, torch.bfloat16, "cache")
    for t, nm in ((k, "k"), (v, "v")):
        _req(t, torch.bfloat16, nm)
    for t, nm in ((qo_indptr, "qo_indptr"), (page_table, "page_table"), (seq_lens, "seq_lens"),
                  (active, "active")):
        _req(t, torch.int32, nm)
    g = _geom(cache)
    st = load().pkv_kv_append_tokens(ctypes.byref(g), _ptr(cache), int(layer), _ptr(k), _ptr(v),
                                     k.shape[0], _ptr(qo_indptr), _ptr(page_table),
                                     page_table.shape[1], _ptr(seq_lens), _ptr(active),
                                     seq_lens.shape[0], _ptr(err_word), _stream(stream))
    _check("pkv_kv_append_tokens", st)


def prefill_workspace_bytes(batch) -> int:
    return int(load().pkv_prefill_workspace_bytes(batch))


def prefill_attn(cache, layer, q, qo_indptr, page_table, seq_lens, active, out, workspace,
                 lse=None, sm_scale=None, err_word=None, stream=None):
    """Causal attention of the packed new tokens q (bf16 [T, Hq, D]) over the
    paged cache into out (bf16 [T, Hq, D]); lse fp32 [T, Hq] optional."""
    import torch
    _req(cache, torch.bfloat16, "cache")
    _req(q, torch.bfloat16, "q")
    _req(out, torch.bfloat16, "out")
    for t, nm in ((qo_indptr, "qo_indptr"), (page_table, "page_table"), (seq_lens, "seq_lens"),
                  (active, "active")):
        _req(t, torch.int32, nm)
    if lse is not None:
        _req(lse, torch.float32, "lse")
    g = _geom(cache)
    T, Hq, D = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / (D ** 0.5)
    st = load().pkv_prefill_attn(ctypes.byref(g), _ptr(cache), int(layer), _ptr(q), Hq,
                                 float(sm_scale), T, _ptr(qo_indptr), _ptr(page_table),
                                 page_table.shape[1], _ptr(seq_lens), _ptr(active),
                                 seq_lens.shape[0], _ptr(out), _ptr(lse), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _ptr(err_word),
                                 _stream(stream))
    _check("pkv_prefill_attn", st)


def sample_workspace_bytes(batch, vocab) -> int:
    return int(load().pkv_sample_workspace_bytes(batch, vocab))


def seeded_sample(logits, slots, active, seeds, steps, temperature, top_k, top_p, out_tok,
                  out_kind, workspace, salt=0, advance=True, stop_tokens=None, audio_lo=0,
                  audio_hi=0, err_word=None, stream=None):
    import torch
    if logits.dtype != torch.float32 or logits.stride(-1) != 1 or not logits.is_cuda:
        raise TypeError("logits must be a CUDA fp32 tensor with unit last stride")
    B, V = logits.shape
    for t, dt, nm in ((slots, torch.int32, "slots"), (active, torch.int32, "active"),
                      (seeds, torch.uint64, "seeds"), (steps, torch.int64, "steps"),
                      (temperature, torch.float32, "temperature"), (top_k, torch.int32, "top_k"),
                      (top_p, torch.float32, "top_p"), (out_tok, torch.int32, "out_tok"),
                      (out_kind, torch.int32, "out_kind")):
        _req(t, dt, nm)
    n_stop = 0 if stop_tokens is None else stop_tokens.numel()
    st = load().pkv_seeded_sample(
        _ptr(logits), logits.stride(0), B, V, _ptr(slots), _ptr(active), seeds.numel(),
        _ptr(seeds), _ptr(steps), _ptr(temperature), _ptr(top_k), _ptr(top_p), int(salt),
        int(bool(advance)), _ptr(stop_tokens) if n_stop else None, n_stop, int(audio_lo),
        int(audio_hi), _ptr(out_tok), _ptr(out_kind), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(err_word), _stream(stream))
    _check("pkv_seeded_sample", st)


def sample_ext_workspace_bytes(batch, vocab) -> int:
    return int(load().pkv_sample_ext_workspace_bytes(batch, vocab))


def seeded_sample_ext(logits, slots, active, seeds, steps, temperature, top_k, top_p, out_tok,
                      out_kind, workspace, min_p=None, rep_penalty=None, rep_window=None,
                      history=None, hist_len=None, logprob_raw=None, logprob_proc=None, salt=0,
                      advance=True, stop_tokens=None, audio_lo=0, audio_hi=0, err_word=None,
                      stream=None):
    """seeded_sample with the further settings (each None = off): min_p,
    rep_penalty fp32 [num_slots], rep_window int32 [num_slots], the token
    ring history int32 [num_slots, cap] with hist_len int32 [num_slots]
    (appended to when advance), and the fp32 [B] log-prob outputs."""
    import torch
    if logits.dtype != torch.float32 or logits.stride(-1) != 1 or not logits.is_cuda:
        raise TypeError("logits must be a CUDA fp32 tensor with unit last stride")
    B, V = logits.shape
    for t, dt, nm in ((slots, torch.int32, "slots"), (active, torch.int32, "active"),
                      (seeds, torch.uint64, "seeds"), (steps, torch.int64, "steps"),
                      (temperature, torch.float32, "temperature"), (top_k, torch.int32, "top_k"),
                      (top_p, torch.float32, "top_p"), (out_tok, torch.int32, "out_tok"),
                      (out_kind, torch.int32, "out_kind")):
        _req(t, dt, nm)
    for t, dt, nm in ((min_p, torch.float32, "min_p"), (rep_penalty, torch.float32, "rep_penalty"),
                      (rep_window, torch.int32, "rep_window"), (history, torch.int32, "history"),
                      (hist_len, torch.int32, "hist_len"),
                      (logprob_raw, torch.float32, "logprob_raw"),
                      (logprob_proc, torch.float32, "logprob_proc")):
        if t is not None:
            _req(t, dt, nm)
    cap = 0
    if history is not None:
        if history.dim() != 2 or history.shape[1] < 1 or hist_len is None:
            raise ValueError("history must be [num_slots, cap >= 1] and comes with hist_len")
        cap = history.shape[1]
    ext = pkv_sample_ext_t(_ptr(min_p), _ptr(rep_penalty), _ptr(rep_window), _ptr(history),
                           _ptr(hist_len), cap, _ptr(logprob_raw), _ptr(logprob_proc))
    n_stop = 0 if stop_tokens is None else stop_tokens.numel()
    st = load().pkv_seeded_sample_ext(
        _ptr(logits), logits.stride(0), B, V, _ptr(slots), _ptr(active), seeds.numel(),
        _ptr(seeds), _ptr(steps), _ptr(temperature), _ptr(top_k), _ptr(top_p), int(salt),
        int(bool(advance)), _ptr(stop_tokens) if n_stop else None, n_stop, int(audio_lo),
        int(audio_hi), _ptr(out_tok), _ptr(out_kind), ctypes.byref(ext), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(err_word), _stream(stream))
    _check("pkv_seeded_sample_ext", st)


def frame_workspace_bytes(n_codebooks, batch, vocab) -> int:
    return int(load().pkv_frame_workspace_bytes(n_codebooks, batch, vocab))


def codebook_frame_sample(base, fb, slots, active, seeds, steps, temperature, top_k, top_p,
                          out_codes, out_kind, workspace, err_word=None, stream=None):
    import torch
    _req(base, torch.float32, "base")
    if fb is not None:
        _req(fb, torch.float32, "fb")
    n_cb, B, V = base.shape
    for t, dt, nm in ((slots, torch.int32, "slots"), (active, torch.int32, "active"),
                      (seeds, torch.uint64, "seeds"), (steps, torch.int64, "steps"),
                      (temperature, torch.float32, "temperature"), (top_k, torch.int32, "top_k"),
                      (top_p, torch.float32, "top_p"), (out_codes, torch.int32, "out_codes"),
                      (out_kind, torch.int32, "out_kind")):
        _req(t, dt, nm)
    st = load().pkv_codebook_frame_sample(
        _ptr(base), _ptr(fb), n_cb, B, V, _ptr(slots), _ptr(active), seeds.numel(), _ptr(seeds),
        _ptr(steps), _ptr(temperature), _ptr(top_k), _ptr(top_p), _ptr(out_codes),
        _ptr(out_kind), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(err_word), _stream(stream))
    _check("pkv_codebook_frame_sample", st)


def frame_sample_workspace_bytes(n_codebooks, batch, vocab, ctrl_vocab) -> int:
    return int(load().pkv_frame_sample_workspace_bytes(n_codebooks, batch, vocab, ctrl_vocab))


def frame_sample(ctrl, stop_ctrl, base, fb, slots, active, seeds, steps, temperature, top_k,
                 top_p, out_rows, out_kind, workspace, err_word=None, stream=None):
    """pkv_frame_sample: channel 0 (stop/continue, from ``ctrl`` [B, Vc])
    then the codebooks; out_rows int32 [B, 1 + n_codebooks]."""
    import torch
    _req(ctrl, torch.float32, "ctrl")
    _req(base, torch.float32, "base")
    if fb is not None:
        _req(fb, torch.float32, "fb")
    n_cb, B, V = base.shape
    for t, dt, nm in ((slots, torch.int32, "slots"), (active, torch.int32, "active"),
                      (seeds, torch.uint64, "seeds"), (steps, torch.int64, "steps"),
                      (temperature, torch.float32, "temperature"), (top_k, torch.int32, "top_k"),
                      (top_p, torch.float32, "top_p"), (out_rows, torch.int32, "out_rows"),
                      (out_kind, torch.int32, "out_kind")):
        _req(t, dt, nm)
    st = load().pkv_frame_sample(
        _ptr(ctrl), ctrl.shape[1], int(stop_ctrl), _ptr(base), _ptr(fb), n_cb, B, V, _ptr(slots),
        _ptr(active), seeds.numel(), _ptr(seeds), _ptr(steps), _ptr(temperature), _ptr(top_k),
        _ptr(top_p), _ptr(out_rows), _ptr(out_kind), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(err_word), _stream(stream))
    _check("pkv_frame_sample", st)
