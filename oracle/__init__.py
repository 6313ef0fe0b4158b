"""Plain fp64 CPU oracle of the paged-KV decode step.

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference arm of ``bench.py`` may import this package;
the product path (``paged_kv_decode_pages_gb300``) never does, and this
package never imports it.  The arithmetic lives in ``pkv_oracle.c``; this
module only builds it with gcc and marshals numpy arrays through ctypes.

Sources it follows (page title, section):
  * "Adding a Model" (vox-serve docs), "How a program runs" and "1. The model
    code": the cache layout [num_layers, num_pages, 2, page_size,
    num_kv_heads, head_dim], set_kv_cache / run, padding entries on page 0,
    per-request seeded sampling, out_tok / out_kind;
  * "Supported Models" (mstar docs), "Fish Audio S2-Pro notes" and
    "Chatterbox notes": sampling order, top-p boundary, greedy conventions;
  * MOSS-TTS-Local on SGLang-Omni (mosi.cn blog), model and "AR Engine"
    sections: the frame-local loop over 12 codebooks.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libpkv_oracle.so")

KIND_OTHER, KIND_AUDIO, KIND_STOP = 0, 1, 2

_lock = threading.Lock()
_lib = None


def _try_compile(flags):
    cc = os.environ.get("CC", "gcc")
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = [cc, "-O2", "-std=c11", "-shared", "-fPIC", *flags, _SRC, "-o", tmp, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        return r.stderr
    os.replace(tmp, _LIB_PATH)
    return None


def build(force: bool = False) -> str:
    """Compile pkv_oracle.c into oracle/_build/libpkv_oracle.so (gcc, OpenMP if
    the compiler has it).  Returns the library path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    err = _try_compile(["-fopenmp"])
    if err is not None:
        err2 = _try_compile([])
        if err2 is not None:
            raise RuntimeError("oracle build failed:\n" + err + "\n" + err2)
    return _LIB_PATH


class SampleInfo(ctypes.Structure):
    _fields_ = [
        ("token", ctypes.c_int32),
        ("n_kept", ctypes.c_int32),
        ("greedy", ctypes.c_int32),
        ("pad_", ctypes.c_int32),
        ("top2_gap_rel", ctypes.c_double),
        ("member_margin", ctypes.c_double),
        ("logprob_raw", ctypes.c_double),
        ("logprob_proc", ctypes.c_double),
    ]


_INFO_DTYPE = np.dtype([
    ("token", np.int32), ("n_kept", np.int32), ("greedy", np.int32),
    ("pad_", np.int32), ("top2_gap_rel", np.float64), ("member_margin", np.float64),
    ("logprob_raw", np.float64), ("logprob_proc", np.float64),
])

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_U32 = ctypes.c_uint32
_U64 = ctypes.c_uint64
_F = ctypes.c_float
_D = ctypes.c_double


class using_library:
    """Context manager: route every oracle call through another build of
    pkv_oracle.c (the mutation tests plant mistakes in a copy)."""

    def __init__(self, path):
        self.path = path
        self.saved = None

    def __enter__(self):
        global _lib
        with _lock:
            self.saved = _lib
            _lib = _load(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self.saved
        return False


def compile_variant(src_text: str, out_path: str) -> None:
    """Compile a modified copy of the oracle source (used by the mutation
    tests only)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(src_text)
    cc = os.environ.get("CC", "gcc")
    r = subprocess.run([cc, "-O1", "-std=c11", "-shared", "-fPIC", src, "-o", out_path, "-lm"],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(r.stderr)


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _load(build())
    return _lib


def _load(path):
    L = ctypes.CDLL(path)
    L.pkvo_num_threads.restype = _I
    L.pkvo_set_num_threads.argtypes = [_I]
    L.pkvo_kv_append.restype = _I
    L.pkvo_kv_append.argtypes = [_P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _I, _P, _P, _I]
    L.pkvo_kv_append_tokens.restype = _I
    L.pkvo_kv_append_tokens.argtypes = [_P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _P,
                                        _I]
    L.pkvo_prefill_attn.restype = _I
    L.pkvo_prefill_attn.argtypes = [_P, _I, _I, _I, _I, _I, _I, _P, _I, _D, _P, _P, _I, _P, _P,
                                    _I, _P, _P]
    L.pkvo_paged_decode_attn.restype = _I
    L.pkvo_paged_decode_attn.argtypes = [_P, _I, _I, _I, _I, _I, _I, _P, _I, _D,
                                         _P, _I, _P, _P, _I, _P, _P]
    L.pkvo_philox4x64_10.argtypes = [_P, _P, _P]
    L.pkvo_uniform.restype = _D
    L.pkvo_uniform.argtypes = [_U64, _U32, _I64, _I64]
    L.pkvo_gumbel.restype = _D
    L.pkvo_gumbel.argtypes = [_U64, _U32, _I64, _I64]
    L.pkvo_sample_row.restype = ctypes.c_int32
    L.pkvo_sample_row.argtypes = [_P, _I, _U64, _I64, _U32, _F, ctypes.c_int32, _F,
                                  ctypes.POINTER(SampleInfo)]
    L.pkvo_token_kind.restype = ctypes.c_int32
    L.pkvo_token_kind.argtypes = [ctypes.c_int32, _P, _I, ctypes.c_int32, ctypes.c_int32]
    L.pkvo_seeded_sample.restype = _I
    L.pkvo_seeded_sample.argtypes = [_P, _I64, _I, _I, _P, _P, _I, _P, _P, _P, _P, _P,
                                     _U32, _I, _P, _I, ctypes.c_int32, ctypes.c_int32,
                                     _P, _P, _P]
    L.pkvo_codebook_frame_sample.restype = _I
    L.pkvo_codebook_frame_sample.argtypes = [_P, _P, _I, _I, _I, _P, _P, _I, _P, _P,
                                             _P, _P, _P, _P, _P, _P]
    L.pkvo_sample_row_ext.restype = ctypes.c_int32
    L.pkvo_sample_row_ext.argtypes = [_P, _I, _U64, _I64, _U32, _F, ctypes.c_int32, _F, _F, _F,
                                      _P, _I, ctypes.POINTER(SampleInfo)]
    L.pkvo_seeded_sample_ext.restype = _I
    L.pkvo_seeded_sample_ext.argtypes = [_P, _I64, _I, _I, _P, _P, _I, _P, _P, _P, _P, _P, _P,
                                         _P, _P, _P, _P, _I, _U32, _I, _P, _P, _P, _P]
    L.pkvo_frame_sample.restype = _I
    L.pkvo_frame_sample.argtypes = [_P, _I, ctypes.c_int32, _P, _P, _I, _I, _I, _P, _P, _I,
                                    _P, _P, _P, _P, _P, _P, _P, _P]
    return L


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def num_threads() -> int:
    return lib().pkvo_num_threads()


def set_num_threads(n: int) -> None:
    lib().pkvo_set_num_threads(int(n))


# --------------------------------------------------------------------------
# KV append
# --------------------------------------------------------------------------
def kv_append(cache_bits, layer, k_bits, v_bits, page_table, seq_lens, active):
    """In place on ``cache_bits`` (uint16 bf16 bits, shape
    [L, P, 2, ps, Hkv, D], C-contiguous).  k_bits / v_bits: uint16 [B, Hkv, D].
    Returns the count of rejected active rows."""
    assert cache_bits.dtype == np.uint16 and cache_bits.flags.c_contiguous
    L, P, two, ps, Hkv, D = cache_bits.shape
    assert two == 2
    k = _c(k_bits, np.uint16)
    v = _c(v_bits, np.uint16)
    pt = _c(page_table, np.int32)
    sl = _c(seq_lens, np.int32)
    ac = _c(active, np.int32)
    B = sl.shape[0]
    return lib().pkvo_kv_append(_ptr(cache_bits), L, P, ps, Hkv, D, int(layer), _ptr(k), _ptr(v),
                                _ptr(pt), pt.shape[1], _ptr(sl), _ptr(ac), B)


# --------------------------------------------------------------------------
# Paged decode attention
# --------------------------------------------------------------------------
def paged_decode_attn(cache_bits, layer, q_bits, page_table, seq_lens, active, sm_scale=None):
    """Returns (out fp64 [B, Hq, D], lse fp64 [B, Hq], n_bad_rows)."""
    assert cache_bits.dtype == np.uint16 and cache_bits.flags.c_contiguous
    L, P, two, ps, Hkv, D = cache_bits.shape
    q = _c(q_bits, np.uint16)
    B, Hq, Dq = q.shape
    assert Dq == D and Hq % Hkv == 0
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    pt = _c(page_table, np.int32)
    sl = _c(seq_lens, np.int32)
    ac = _c(active, np.int32)
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    bad = lib().pkvo_paged_decode_attn(_ptr(cache_bits), L, P, ps, Hkv, D, int(layer), _ptr(q), Hq,
                                       float(sm_scale), _ptr(pt), pt.shape[1], _ptr(sl), _ptr(ac),
                                       B, _ptr(out), _ptr(lse))
    return out, lse, bad


# --------------------------------------------------------------------------
# Prefill / mixed steps: ragged new tokens per request
# --------------------------------------------------------------------------
def kv_append_tokens(cache_bits, layer, k_bits, v_bits, qo_indptr, page_table, seq_lens, active):
    """In place on ``cache_bits``.  k_bits / v_bits: uint16 [T, Hkv, D] with
    request b's new tokens at rows [qo_indptr[b], qo_indptr[b+1]), ending at
    position seq_lens[b] - 1.  Returns the count of rejected active requests."""
    assert cache_bits.dtype == np.uint16 and cache_bits.flags.c_contiguous
    L, P, two, ps, Hkv, D = cache_bits.shape
    k = _c(k_bits, np.uint16)
    v = _c(v_bits, np.uint16)
    ind = _c(qo_indptr, np.int32)
    pt = _c(page_table, np.int32)
    sl = _c(seq_lens, np.int32)
    ac = _c(active, np.int32)
    B = sl.shape[0]
    assert ind.shape[0] == B + 1 and k.shape[0] >= ind[-1]
    return lib().pkvo_kv_append_tokens(_ptr(cache_bits), L, P, ps, Hkv, D, int(layer), _ptr(k),
                                       _ptr(v), _ptr(ind), _ptr(pt), pt.shape[1], _ptr(sl),
                                       _ptr(ac), B)


def prefill_attn(cache_bits, layer, q_bits, qo_indptr, page_table, seq_lens, active,
                 sm_scale=None):
    """Causal attention of the new tokens (q_bits uint16 [T, Hq, D]) over the
    paged cache.  Returns (out fp64 [T, Hq, D], lse fp64 [T, Hq], n_bad)."""
    assert cache_bits.dtype == np.uint16 and cache_bits.flags.c_contiguous
    L, P, two, ps, Hkv, D = cache_bits.shape
    q = _c(q_bits, np.uint16)
    T, Hq, Dq = q.shape
    assert Dq == D and Hq % Hkv == 0
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    ind = _c(qo_indptr, np.int32)
    pt = _c(page_table, np.int32)
    sl = _c(seq_lens, np.int32)
    ac = _c(active, np.int32)
    B = sl.shape[0]
    assert ind.shape[0] == B + 1 and int(ind[-1]) <= T
    out = np.zeros((T, Hq, D), np.float64)
    lse = np.full((T, Hq), -np.inf, np.float64)
    bad = lib().pkvo_prefill_attn(_ptr(cache_bits), L, P, ps, Hkv, D, int(layer), _ptr(q), Hq,
                                  float(sm_scale), _ptr(ind), _ptr(pt), pt.shape[1], _ptr(sl),
                                  _ptr(ac), B, _ptr(out), _ptr(lse))
    return out, lse, bad


# --------------------------------------------------------------------------
# Philox / Gumbel
# --------------------------------------------------------------------------
def philox4x64_10(key, counter):
    k = np.ascontiguousarray(key, np.uint64)
    c = np.ascontiguousarray(counter, np.uint64)
    out = np.zeros(4, np.uint64)
    lib().pkvo_philox4x64_10(_ptr(k), _ptr(c), _ptr(out))
    return out


def uniform(seed, salt, token, step):
    return lib().pkvo_uniform(int(seed), int(salt), int(token), int(step))


def gumbel(seed, salt, token, step):
    return lib().pkvo_gumbel(int(seed), int(salt), int(token), int(step))


# --------------------------------------------------------------------------
# Sampling
# --------------------------------------------------------------------------
def sample_row(logits, seed, step, salt, temperature, top_k, top_p):
    """One row; returns (token, info dict)."""
    x = _c(logits, np.float32)
    info = SampleInfo()
    tok = lib().pkvo_sample_row(_ptr(x), x.shape[0], int(seed), int(step), int(salt),
                                float(temperature), int(top_k), float(top_p), ctypes.byref(info))
    return int(tok), {f: getattr(info, f) for f, _ in SampleInfo._fields_ if f != "pad_"}


def sample_row_ext(logits, seed, step, salt, temperature, top_k, top_p, min_p=0.0,
                   rep_penalty=1.0, pen_tokens=()):
    """One row with the further controls (repetition penalty over
    ``pen_tokens``, min_p) and log-probs; returns (token, info dict)."""
    x = _c(logits, np.float32)
    pt = np.ascontiguousarray(pen_tokens, np.int32)
    info = SampleInfo()
    tok = lib().pkvo_sample_row_ext(_ptr(x), x.shape[0], int(seed), int(step), int(salt),
                                    float(temperature), int(top_k), float(top_p), float(min_p),
                                    float(rep_penalty), _ptr(pt) if pt.size else None, pt.size,
                                    ctypes.byref(info))
    return int(tok), {f: getattr(info, f) for f, _ in SampleInfo._fields_ if f != "pad_"}


def seeded_sample_ext(logits, slots, active, seeds, steps, temperature, top_k, top_p,
                      min_p=None, rep_penalty=None, rep_window=None, history=None,
                      hist_len=None, salt=0, advance=True):
    """seeded_sample with min_p / repetition penalty (per slot, each None =
    off), the per-slot history ring ``history`` int32 [num_slots, cap] and
    ``hist_len`` int32 [num_slots] (updated in place when advance, like
    ``steps``).  Returns (out_tok, logprob_raw, logprob_proc, info, n_bad)."""
    x = _c(logits, np.float32)
    B, V = x.shape
    sl = _c(slots, np.int32)
    ac = _c(active, np.int32)
    sd = _c(seeds, np.uint64)
    assert steps.dtype == np.int64 and steps.flags.c_contiguous
    tp = _c(temperature, np.float32)
    tk = _c(top_k, np.int32)
    pp = _c(top_p, np.float32)
    mp = None if min_p is None else _c(min_p, np.float32)
    rp = None if rep_penalty is None else _c(rep_penalty, np.float32)
    rw = None if rep_window is None else _c(rep_window, np.int32)
    cap = 0
    if history is not None:
        assert history.dtype == np.int32 and history.flags.c_contiguous
        assert hist_len.dtype == np.int32 and hist_len.flags.c_contiguous
        cap = history.shape[1]
    out_tok = np.zeros(B, np.int32)
    lraw = np.zeros(B, np.float32)
    lproc = np.zeros(B, np.float32)
    info = np.zeros(B, _INFO_DTYPE)
    bad = lib().pkvo_seeded_sample_ext(_ptr(x), V, B, V, _ptr(sl), _ptr(ac), sd.shape[0],
                                       _ptr(sd), _ptr(steps), _ptr(tp), _ptr(tk), _ptr(pp),
                                       _ptr(mp), _ptr(rp), _ptr(rw), _ptr(history), _ptr(hist_len),
                                       cap, int(salt), int(bool(advance)), _ptr(out_tok),
                                       _ptr(lraw), _ptr(lproc), _ptr(info))
    return out_tok, lraw, lproc, info, bad


def token_kind(tok, stop_tokens=(), audio_lo=0, audio_hi=0):
    st = np.ascontiguousarray(stop_tokens, np.int32)
    return int(lib().pkvo_token_kind(int(tok), _ptr(st) if st.size else None, st.size,
                                     int(audio_lo), int(audio_hi)))


def seeded_sample(logits, slots, active, seeds, steps, temperature, top_k, top_p, salt=0,
                  advance=True, stop_tokens=(), audio_lo=0, audio_hi=0):
    """logits fp32 [B, V].  ``steps`` (int64 [num_slots]) is updated in place
    when advance.  Returns (out_tok, out_kind, info structured array, n_bad)."""
    x = _c(logits, np.float32)
    B, V = x.shape
    sl = _c(slots, np.int32)
    ac = _c(active, np.int32)
    sd = _c(seeds, np.uint64)
    assert steps.dtype == np.int64 and steps.flags.c_contiguous
    tp = _c(temperature, np.float32)
    tk = _c(top_k, np.int32)
    pp = _c(top_p, np.float32)
    st = np.ascontiguousarray(stop_tokens, np.int32)
    out_tok = np.zeros(B, np.int32)
    out_kind = np.zeros(B, np.int32)
    info = np.zeros(B, _INFO_DTYPE)
    bad = lib().pkvo_seeded_sample(_ptr(x), V, B, V, _ptr(sl), _ptr(ac), sd.shape[0], _ptr(sd),
                                   _ptr(steps), _ptr(tp), _ptr(tk), _ptr(pp), int(salt),
                                   int(bool(advance)), _ptr(st) if st.size else None, st.size,
                                   int(audio_lo), int(audio_hi), _ptr(out_tok), _ptr(out_kind),
                                   _ptr(info))
    return out_tok, out_kind, info, bad


def codebook_frame_sample(base, fb, slots, active, seeds, steps, temperature, top_k, top_p):
    """base fp32 [n_cb, B, V]; fb fp32 [n_cb, V, V] or None.  ``steps`` is
    advanced in place once per frame for active rows.  Returns
    (out_codes [B, n_cb], out_kind [B], info [B, n_cb], n_bad)."""
    bs = _c(base, np.float32)
    n_cb, B, V = bs.shape
    f = None if fb is None else _c(fb, np.float32)
    if f is not None:
        assert f.shape == (n_cb, V, V)
    sl = _c(slots, np.int32)
    ac = _c(active, np.int32)
    sd = _c(seeds, np.uint64)
    assert steps.dtype == np.int64 and steps.flags.c_contiguous
    tp = _c(temperature, np.float32)
    tk = _c(top_k, np.int32)
    pp = _c(top_p, np.float32)
    codes = np.zeros((B, n_cb), np.int32)
    kind = np.zeros(B, np.int32)
    info = np.zeros((B, n_cb), _INFO_DTYPE)
    bad = lib().pkvo_codebook_frame_sample(_ptr(bs), _ptr(f), n_cb, B, V, _ptr(sl), _ptr(ac),
                                           sd.shape[0], _ptr(sd), _ptr(steps), _ptr(tp), _ptr(tk),
                                           _ptr(pp), _ptr(codes), _ptr(kind), _ptr(info))
    return codes, kind, info, bad


CODE_PAD = -1  # codebook channels of a frame that stopped


def frame_sample(ctrl, stop_ctrl, base, fb, slots, active, seeds, steps, temperature, top_k,
                 top_p):
    """A full frame row per active row: ctrl fp32 [B, Vc] is sampled on
    channel 0 (salt 0); a sampled ``stop_ctrl`` fills the codebook channels
    with CODE_PAD and gives kind STOP, else channels 1..n_cb are the
    codebook_frame_sample codes and the kind is AUDIO.  base fp32
    [n_cb, B, V]; fb fp32 [n_cb, V, V] or None.  ``steps`` is advanced in
    place once per frame for active rows.  Returns (out_rows [B, 1 + n_cb],
    out_kind [B], info [B, 1 + n_cb], n_bad)."""
    ct = _c(ctrl, np.float32)
    bs = _c(base, np.float32)
    n_cb, B, V = bs.shape
    assert ct.shape[0] == B
    Vc = ct.shape[1]
    f = None if fb is None else _c(fb, np.float32)
    if f is not None:
        assert f.shape == (n_cb, V, V)
    sl = _c(slots, np.int32)
    ac = _c(active, np.int32)
    sd = _c(seeds, np.uint64)
    assert steps.dtype == np.int64 and steps.flags.c_contiguous
    tp = _c(temperature, np.float32)
    tk = _c(top_k, np.int32)
    pp = _c(top_p, np.float32)
    rows = np.zeros((B, 1 + n_cb), np.int32)
    kind = np.zeros(B, np.int32)
    info = np.zeros((B, 1 + n_cb), _INFO_DTYPE)
    bad = lib().pkvo_frame_sample(_ptr(ct), Vc, int(stop_ctrl), _ptr(bs), _ptr(f), n_cb, B, V,
                                  _ptr(sl), _ptr(ac), sd.shape[0], _ptr(sd), _ptr(steps),
                                  _ptr(tp), _ptr(tk), _ptr(pp), _ptr(rows), _ptr(kind),
                                  _ptr(info))
    return rows, kind, info, bad


def have_compiler() -> bool:
    return shutil.which(os.environ.get("CC", "gcc")) is not None
