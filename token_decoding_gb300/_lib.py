"""ctypes binding of libmars (argument marshalling only).

Every function here checks tensor shapes / dtypes / devices, then calls the
C entry point of the same name with raw device pointers and the current CUDA
stream.  All computation happens in the CUDA kernels of libmars.so; there is
no fallback of any kind: if the library is not built, or a call fails, a
RuntimeError is raised.
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmars.so")

MARS_OK = 0
MARS_ERR_INVALID_ARG = 1
MARS_ERR_WORKSPACE_TOO_SMALL = 2
MARS_ERR_CUDA = 3
MARS_ERR_UNSUPPORTED_DEVICE = 4
MARS_ERR_SCRATCH_LIMIT = 5
MARS_ERR_SCRATCH_NOT_READY = 6

MARS_ACCEPT_MARGIN = 1
MARS_ACCEPT_BATCH_MIN = 2
MARS_ACCEPT_DEFERRED = 4

MARS_DEV_CAPACITY = 1
MARS_DEV_LEN_RANGE = 2
MARS_DEV_TIMEOUT = 4

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t

_SIGNATURES = {
    "mars_status_string": (ctypes.c_char_p, [_I]),
    "mars_version": (_I, []),
    "mars_last_cuda_error": (ctypes.c_char_p, []),
    "mars_train_attn": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P]),
    "mars_train_attn_bwd_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "mars_train_attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _SZ, _P, _P]),
    "mars_decode_attn_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "mars_decode_attn": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P]),
    "mars_decode_attn_deferred": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P]),
    "mars_accept_workspace_size": (_SZ, [_I, _I, _I]),
    "mars_accept": (_I, [_P, _I, _I, _I, _F, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "mars_accept_margin": (_I, [_P, _I, _I, _I, _F, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "mars_accept_ex": (_I, [_P, _I, _I, _I, _F, _I, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "mars_accept_noalloc": (_I, [_P, _I, _I, _I, _F, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P]),
    "mars_selftest_wait_timeout": (_I, [_I, ctypes.c_uint, _P, _P, _P]),
    "mars_lm_head_accept_workspace_size": (_SZ, [_I, _I, _I]),
    "mars_lm_head_accept": (_I, [_P, _P, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _SZ,
                                 _P]),
}

_lib = None


class MarsError(RuntimeError):
    def __init__(self, fn, code):
        detail = f"; CUDA: {last_cuda_error()}" if code == MARS_ERR_CUDA else ""
        super().__init__(f"{fn} failed: {code} ({status_string(code)}){detail}")
        self.code = code


def lib() -> ctypes.CDLL:
    """The loaded libmars.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m token_decoding_gb300.build` "
                "(or __graft_entry__.build()); there is no fallback path")
        _lib = ctypes.CDLL(LIB_PATH)
    return _lib


_fns = {}


def _fn(name):
    """The C entry point `name` with its ctypes signature (resolved on first use)."""
    f = _fns.get(name)
    if f is None:
        f = getattr(lib(), name)
        res, args = _SIGNATURES[name]
        f.restype = res
        f.argtypes = args
        _fns[name] = f
    return f


def status_string(code: int) -> str:
    return _fn("mars_status_string")(int(code)).decode()


def last_cuda_error() -> str:
    return _fn("mars_last_cuda_error")().decode()


def version() -> int:
    return int(_fn("mars_version")())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, dtype, shape, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _call(name, *args):
    rc = _fn(name)(*args)
    if rc != MARS_OK:
        raise MarsError(name, rc)


def train_attn(q, k, v, L: int, B: int, scale: float | None = None, o=None, lse=None, status=None,
               want_lse: bool = False, stream=None):
    """MARS masked attention over z = [x ; x~] (see include/mars.h: mars_train_attn).

    q [b, 2L, Hq, D], k/v [b, 2L, Hkv, D] bf16 CUDA tensors.  Returns o (and lse
    when ``want_lse`` or ``lse`` is given).
    """
    nb, n2, hq, d = q.shape
    hkv = k.shape[2]
    dev = q.device
    _check(q, "q", torch.bfloat16, (nb, 2 * L, hq, d))
    _check(k, "k", torch.bfloat16, (nb, 2 * L, hkv, d), dev)
    _check(v, "v", torch.bfloat16, (nb, 2 * L, hkv, d), dev)
    if scale is None:
        scale = d ** -0.5
    if o is None:
        o = torch.empty_like(q)
    _check(o, "o", torch.bfloat16, q.shape, dev)
    if lse is None and want_lse:
        lse = torch.empty((nb, hq, 2 * L), dtype=torch.float32, device=dev)
    if lse is not None:
        _check(lse, "lse", torch.float32, (nb, hq, 2 * L), dev)
    if status is not None:
        _check(status, "status", torch.int32, (1,), dev)
    _call("mars_train_attn", _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), nb, L, B, hq, hkv, d, float(scale),
          _ptr(status), _stream(stream))
    return (o, lse) if lse is not None else o


def train_attn_bwd_workspace_size(batch: int, L: int, Hq: int, Hkv: int, D: int) -> int:
    return int(_fn("mars_train_attn_bwd_workspace_size")(batch, L, Hq, Hkv, D))


def train_attn_bwd(q, k, v, o, dout, lse, L: int, B: int, scale: float | None = None, dq=None, dk=None, dv=None,
                   workspace=None, status=None, stream=None):
    """Gradients of train_attn (include/mars.h: mars_train_attn_bwd).

    q, o, dout [b, 2L, Hq, D], k, v [b, 2L, Hkv, D] bf16; lse [b, Hq, 2L] fp32
    from the forward.  Returns (dq, dk, dv) in the shapes of q, k, v."""
    nb, n2, hq, d = q.shape
    hkv = k.shape[2]
    dev = q.device
    _check(q, "q", torch.bfloat16, (nb, 2 * L, hq, d))
    for t, name in ((o, "o"), (dout, "dout")):
        _check(t, name, torch.bfloat16, q.shape, dev)
    _check(k, "k", torch.bfloat16, (nb, 2 * L, hkv, d), dev)
    _check(v, "v", torch.bfloat16, (nb, 2 * L, hkv, d), dev)
    _check(lse, "lse", torch.float32, (nb, hq, 2 * L), dev)
    if scale is None:
        scale = d ** -0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(dq, "dq", torch.bfloat16, q.shape, dev)
    _check(dk, "dk", torch.bfloat16, k.shape, dev)
    _check(dv, "dv", torch.bfloat16, v.shape, dev)
    if workspace is None:
        n = int(_fn("mars_train_attn_bwd_workspace_size")(nb, L, hq, hkv, d))
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
    if status is not None:
        _check(status, "status", torch.int32, (1,), dev)
    _call("mars_train_attn_bwd", _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
          _ptr(dv), nb, L, B, hq, hkv, d, float(scale), _ptr(workspace), workspace.numel(), _ptr(status),
          _stream(stream))
    return dq, dk, dv


def decode_attn_workspace_size(batch: int, B: int, Hq: int, D: int, max_len: int) -> int:
    """Workspace bytes of decode_attn (include/mars.h: always 0, the merge stays in the cluster)."""
    return int(_fn("mars_decode_attn_workspace_size")(batch, B, Hq, D, max_len))


def decode_attn(q, k_new, v_new, k_cache, v_cache, cache_len, max_len: int, scale: float | None = None, o=None,
                status=None, stream=None):
    """Attention of one sliding-window decode step (include/mars.h: mars_decode_attn)."""
    nb, bq, hq, d = q.shape
    hkv = k_new.shape[2]
    cap = k_cache.shape[2]
    dev = q.device
    _check(q, "q", torch.bfloat16, (nb, bq, hq, d))
    _check(k_new, "k_new", torch.bfloat16, (nb, bq, hkv, d), dev)
    _check(v_new, "v_new", torch.bfloat16, (nb, bq, hkv, d), dev)
    _check(k_cache, "k_cache", torch.bfloat16, (nb, hkv, cap, d), dev)
    _check(v_cache, "v_cache", torch.bfloat16, (nb, hkv, cap, d), dev)
    _check(cache_len, "cache_len", torch.int32, (nb,), dev)
    if scale is None:
        scale = d ** -0.5
    if o is None:
        o = torch.empty_like(q)
    _check(o, "o", torch.bfloat16, q.shape, dev)
    if status is not None:
        _check(status, "status", torch.int32, (1,), dev)
    _call("mars_decode_attn", _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(cache_len),
          nb, bq, hq, hkv, d, cap, int(max_len), float(scale), _ptr(o), _ptr(status), _stream(stream))
    return o


def decode_attn_deferred(q, k_new, v_new, k_cache, v_cache, cache_len, pending, max_len: int,
                         scale: float | None = None, o=None, status=None, stream=None):
    """Decode step of the deferred-KV sampler (include/mars.h: mars_decode_attn_deferred).

    q [b, 2B, Hq, D], k_new / v_new [b, 2B, Hkv, D]: slots 0..B-1 are the previous
    step's committed tokens (valid below pending[b]), slots B..2B-1 the new
    placeholders.  The valid pending K/V rows are written into k_cache / v_cache
    at cache_len; cache_len is not changed here.  Returns o [b, 2B, Hq, D]."""
    nb, s2, hq, d = q.shape
    if s2 % 2:
        raise ValueError(f"q must carry 2B slots, got {s2}")
    hkv = k_new.shape[2]
    cap = k_cache.shape[2]
    dev = q.device
    _check(q, "q", torch.bfloat16, (nb, s2, hq, d))
    _check(k_new, "k_new", torch.bfloat16, (nb, s2, hkv, d), dev)
    _check(v_new, "v_new", torch.bfloat16, (nb, s2, hkv, d), dev)
    _check(k_cache, "k_cache", torch.bfloat16, (nb, hkv, cap, d), dev)
    _check(v_cache, "v_cache", torch.bfloat16, (nb, hkv, cap, d), dev)
    _check(cache_len, "cache_len", torch.int32, (nb,), dev)
    _check(pending, "pending", torch.int32, (nb,), dev)
    if scale is None:
        scale = d ** -0.5
    if o is None:
        o = torch.empty_like(q)
    _check(o, "o", torch.bfloat16, q.shape, dev)
    if status is not None:
        _check(status, "status", torch.int32, (1,), dev)
    _call("mars_decode_attn_deferred", _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
          _ptr(cache_len), _ptr(pending), nb, s2 // 2, hq, hkv, d, cap, int(max_len), float(scale), _ptr(o),
          _ptr(status), _stream(stream))
    return o


def accept_workspace_size(batch: int, B: int, V: int) -> int:
    return int(_fn("mars_accept_workspace_size")(batch, B, V))


def accept_workspace(batch: int, B: int, V: int, device) -> torch.Tensor:
    """A workspace for accept (one partial result per 16 KB slice of logits)."""
    n = accept_workspace_size(batch, B, V)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device)


def accept(logits, tau: float, k_new, v_new, k_cache, v_cache, cache_len, workspace=None, tokens=None, conf=None,
           n_commit=None, status=None, stream=None, gate: str = "prob", batch_min: bool = False):
    """Greedy tokens, confidences, left-to-right commit and KV append
    (include/mars.h: mars_accept_ex; gate="margin" makes conf p1 - p2,
    batch_min=True commits the batch-minimum count for every sequence).
    Returns (tokens, conf, n_commit); k_cache, v_cache and cache_len are
    updated in place."""
    if gate not in ("prob", "margin"):
        raise ValueError(f"gate must be 'prob' or 'margin', got {gate!r}")
    nb, bq, V = logits.shape
    hkv, d = k_new.shape[2], k_new.shape[3]
    cap = k_cache.shape[2]
    dev = logits.device
    _check(logits, "logits", torch.bfloat16, (nb, bq, V))
    _check(k_new, "k_new", torch.bfloat16, (nb, bq, hkv, d), dev)
    _check(v_new, "v_new", torch.bfloat16, (nb, bq, hkv, d), dev)
    _check(k_cache, "k_cache", torch.bfloat16, (nb, hkv, cap, d), dev)
    _check(v_cache, "v_cache", torch.bfloat16, (nb, hkv, cap, d), dev)
    _check(cache_len, "cache_len", torch.int32, (nb,), dev)
    if workspace is None:
        workspace = accept_workspace(nb, bq, V, dev)
    if tokens is None:
        tokens = torch.empty((nb, bq), dtype=torch.int32, device=dev)
    if conf is None:
        conf = torch.empty((nb, bq), dtype=torch.float32, device=dev)
    if n_commit is None:
        n_commit = torch.empty((nb,), dtype=torch.int32, device=dev)
    _check(tokens, "tokens", torch.int32, (nb, bq), dev)
    _check(conf, "conf", torch.float32, (nb, bq), dev)
    _check(n_commit, "n_commit", torch.int32, (nb,), dev)
    if status is not None:
        _check(status, "status", torch.int32, (1,), dev)
    flags = (MARS_ACCEPT_MARGIN if gate == "margin" else 0) | (MARS_ACCEPT_BATCH_MIN if batch_min else 0)
    _call("mars_accept_ex", _ptr(logits), nb, bq, V, float(tau), flags, _ptr(k_new), _ptr(v_new), _ptr(k_cache),
          _ptr(v_cache), _ptr(cache_len), hkv, d, cap, _ptr(tokens), _ptr(conf), _ptr(n_commit), _ptr(status),
          _ptr(workspace), workspace.numel(), _stream(stream))
    return tokens, conf, n_commit


def accept_deferred(logits, tau: float, cache_len, n_commit, cap: int, workspace=None, tokens=None, conf=None,
                    status=None, stream=None, gate: str = "prob", batch_min: bool = False):
    """Acceptance step of the deferred-KV sampler (include/mars.h: mars_accept_ex
    with MARS_ACCEPT_DEFERRED).  n_commit holds the previous step's count on
    entry (the rows the deferred decode step just wrote): cache_len advances by
    it, and n_commit is overwritten with this step's count.  No K/V is copied.
    Returns (tokens, conf, n_commit)."""
    if gate not in ("prob", "margin"):
        raise ValueError(f"gate must be 'prob' or 'margin', got {gate!r}")
    nb, bq, V = logits.shape
    dev = logits.device
    _check(logits, "logits", torch.bfloat16, (nb, bq, V))
    _check(cache_len, "cache_len", torch.int32, (nb,), dev)
    _check(n_commit, "n_commit", torch.int32, (nb,), dev)
    if workspace is None:
        workspace = accept_workspace(nb, bq, V, dev)
    if tokens is None:
        tokens = torch.empty((nb, bq), dtype=torch.int32, device=dev)
    if conf is None:
        conf = torch.empty((nb, bq), dtype=torch.float32, device=dev)
    _check(tokens, "tokens", torch.int32, (nb, bq), dev)
    _check(conf, "conf", torch.float32, (nb, bq), dev)
    if status is not None:
        _check(status, "status", torch.int32, (1,), dev)
    flags = (MARS_ACCEPT_DEFERRED | (MARS_ACCEPT_MARGIN if gate == "margin" else 0)
             | (MARS_ACCEPT_BATCH_MIN if batch_min else 0))
    _call("mars_accept_ex", _ptr(logits), nb, bq, V, float(tau), flags, None, None, None, None, _ptr(cache_len),
          0, 0, int(cap), _ptr(tokens), _ptr(conf), _ptr(n_commit), _ptr(status), _ptr(workspace),
          workspace.numel(), _stream(stream))
    return tokens, conf, n_commit


def accept_noalloc(logits, tau: float, k_new, v_new, k_cache, v_cache, cache_len, tokens, conf, n_commit,
                   status=None, stream=None):
    """mars_accept for callers that cannot allocate device memory (include/mars.h:
    mars_accept_noalloc).  Every output buffer is supplied by the caller; the
    library uses its own fixed scratch, so nothing is allocated here either.
    Returns (tokens, conf, n_commit); k_cache, v_cache and cache_len are
    updated in place."""
    nb, bq, V = logits.shape
    hkv, d = k_new.shape[2], k_new.shape[3]
    cap = k_cache.shape[2]
    dev = logits.device
    _check(logits, "logits", torch.bfloat16, (nb, bq, V))
    _check(k_new, "k_new", torch.bfloat16, (nb, bq, hkv, d), dev)
    _check(v_new, "v_new", torch.bfloat16, (nb, bq, hkv, d), dev)
    _check(k_cache, "k_cache", torch.bfloat16, (nb, hkv, cap, d), dev)
    _check(v_cache, "v_cache", torch.bfloat16, (nb, hkv, cap, d), dev)
    _check(cache_len, "cache_len", torch.int32, (nb,), dev)
    _check(tokens, "tokens", torch.int32, (nb, bq), dev)
    _check(conf, "conf", torch.float32, (nb, bq), dev)
    _check(n_commit, "n_commit", torch.int32, (nb,), dev)
    if status is not None:
        _check(status, "status", torch.int32, (1,), dev)
    _call("mars_accept_noalloc", _ptr(logits), nb, bq, V, float(tau), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
          _ptr(v_cache), _ptr(cache_len), hkv, d, cap, _ptr(tokens), _ptr(conf), _ptr(n_commit), _ptr(status),
          _stream(stream))
    return tokens, conf, n_commit


def selftest_wait_timeout(withhold: bool, spin_limit: int, status, elapsed_ns=None, stream=None):
    """Run the library's bounded pipeline wait on the device (include/mars.h:
    mars_selftest_wait_timeout).  status: int32 [1] CUDA tensor (MARS_DEV_TIMEOUT is
    OR-ed in when the wait gives up); elapsed_ns: optional int64 [1] CUDA tensor."""
    _check(status, "status", torch.int32, (1,))
    if elapsed_ns is not None:
        _check(elapsed_ns, "elapsed_ns", torch.int64, (1,), status.device)
    _call("mars_selftest_wait_timeout", 1 if withhold else 0, int(spin_limit), _ptr(status), _ptr(elapsed_ns),
          _stream(stream))


def lm_head_accept_workspace(batch: int, B: int, V: int, device) -> torch.Tensor:
    """A workspace for lm_head_accept (one partial per row and vocabulary range)."""
    n = int(_fn("mars_lm_head_accept_workspace_size")(batch, B, V))
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def lm_head_accept(hidden, weight, tau: float, k_new, v_new, k_cache, v_cache, cache_len, workspace=None,
                   tokens=None, conf=None, n_commit=None, status=None, stream=None):
    """The LM head of the proposal positions fused with accept (include/mars.h:
    mars_lm_head_accept): hidden [b, B, K], weight [V, K] bf16.  Returns (tokens,
    conf, n_commit); k_cache, v_cache and cache_len are updated in place."""
    nb, bq, K = hidden.shape
    V = weight.shape[0]
    hkv, d = k_new.shape[2], k_new.shape[3]
    cap = k_cache.shape[2]
    dev = hidden.device
    _check(hidden, "hidden", torch.bfloat16, (nb, bq, K))
    _check(weight, "weight", torch.bfloat16, (V, K), dev)
    _check(k_new, "k_new", torch.bfloat16, (nb, bq, hkv, d), dev)
    _check(v_new, "v_new", torch.bfloat16, (nb, bq, hkv, d), dev)
    _check(k_cache, "k_cache", torch.bfloat16, (nb, hkv, cap, d), dev)
    _check(v_cache, "v_cache", torch.bfloat16, (nb, hkv, cap, d), dev)
    _check(cache_len, "cache_len", torch.int32, (nb,), dev)
    if workspace is None:
        workspace = lm_head_accept_workspace(nb, bq, V, dev)
    tokens = torch.empty((nb, bq), dtype=torch.int32, device=dev) if tokens is None else tokens
    conf = torch.empty((nb, bq), dtype=torch.float32, device=dev) if conf is None else conf
    n_commit = torch.empty((nb,), dtype=torch.int32, device=dev) if n_commit is None else n_commit
    _check(tokens, "tokens", torch.int32, (nb, bq), dev)
    _check(conf, "conf", torch.float32, (nb, bq), dev)
    _check(n_commit, "n_commit", torch.int32, (nb,), dev)
    if status is not None:
        _check(status, "status", torch.int32, (1,), dev)
    _call("mars_lm_head_accept", _ptr(hidden), _ptr(weight), nb, bq, K, V, float(tau), _ptr(k_new), _ptr(v_new),
          _ptr(k_cache), _ptr(v_cache), _ptr(cache_len), hkv, d, cap, _ptr(tokens), _ptr(conf), _ptr(n_commit),
          _ptr(status), _ptr(workspace), workspace.numel(), _stream(stream))
    return tokens, conf, n_commit
