"""ctypes binding of ``librlk_logp.so``: argument marshalling only.

Every step of the operator runs in the library's CUDA kernels; this module
turns torch tensors into device pointers, picks the current CUDA stream and
allocates outputs when the caller does not pass them.  There is no fallback:
if the library is missing or a call fails, an exception is raised.
"""

from __future__ import annotations

import ctypes
import os

from .build import LIB

VOCAB_PADDED = 152576
VOCAB_REAL = 151936
NUM_SHARDS = 8
SHARD_WIDTH = 19072

RLK_OK, RLK_EINVAL, RLK_EALIGN, RLK_ECUDA = 0, 1, 2, 3


class RlkError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"rlk status {status}: {message}")
        self.status = status


class LogpArgs(ctypes.Structure):
    _fields_ = [
        ("logits", ctypes.c_void_p),
        ("T", ctypes.c_int64),
        ("row_stride", ctypes.c_int64),
        ("vocab_real", ctypes.c_int32),
        ("vocab_padded", ctypes.c_int32),
        ("target", ctypes.c_void_p),
        ("temperature", ctypes.c_void_p),
        ("temperature_scalar", ctypes.c_float),
        ("top_p", ctypes.c_void_p),
        ("top_p_scalar", ctypes.c_float),
        ("top_k", ctypes.c_void_p),
        ("top_k_scalar", ctypes.c_int32),
        ("err_count", ctypes.c_void_p),
    ]


class ShardArgs(ctypes.Structure):
    _fields_ = [
        ("logits", ctypes.c_void_p),
        ("T", ctypes.c_int64),
        ("row_stride", ctypes.c_int64),
        ("shard", ctypes.c_int32),
        ("target", ctypes.c_void_p),
        ("temperature", ctypes.c_void_p),
        ("temperature_scalar", ctypes.c_float),
        ("top_p", ctypes.c_void_p),
        ("top_p_scalar", ctypes.c_float),
        ("top_k", ctypes.c_void_p),
        ("top_k_scalar", ctypes.c_int32),
        ("err_count", ctypes.c_void_p),
    ]


COMPUTE = ("rlk_logp_full", "rlk_logp_restricted", "rlk_logp_pair", "rlk_logp_kl", "rlk_logp_kl_ref",
           "rlk_logp_kl_host",
           "rlk_logp_backward", "rlk_logp_pair_save", "rlk_logp_backward_saved", "rlk_sample",
           "rlk_sample_noalloc", "rlk_linear_logp", "rlk_linear_logp_pair",
           "rlk_logp_shard_summary", "rlk_logp_shard_counts", "rlk_logp_merge",
           "rlk_logp_merge_resumable", "rlk_logp_shard_counts_window",
           "rlk_sqnorm_accumulate", "rlk_sqnorm_finalize", "rlk_grad_norm")
RLK_GRAD_BF16, RLK_GRAD_F32 = 0, 1
EXPORTS = COMPUTE + ("rlk_status_string", "rlk_last_error", "rlk_abi_version")

_lib = None


def load_library(path: str = LIB) -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"CUDA library {path} is missing: run "
                          "`python -c 'import __graft_entry__ as g; g.build()'` first")
    lib = ctypes.CDLL(path)
    P, VP = ctypes.POINTER, ctypes.c_void_p
    A = P(LogpArgs)
    lib.rlk_logp_full.argtypes = [A, VP, VP]
    lib.rlk_logp_restricted.argtypes = [A, VP, VP, VP]
    lib.rlk_logp_pair.argtypes = [A, VP, VP, VP, VP]
    lib.rlk_logp_kl.argtypes = [A, VP, ctypes.c_int64, VP, VP, VP, VP, VP, VP]
    lib.rlk_logp_kl_ref.argtypes = [A, VP, VP, VP, VP]
    lib.rlk_logp_kl_host.argtypes = [A, VP, ctypes.c_int64, VP, VP, VP, VP, VP, VP, ctypes.c_int32, VP, VP]
    lib.rlk_logp_backward.argtypes = [A, VP, VP, VP, ctypes.c_int64, ctypes.c_int32, VP, VP, VP, VP]
    lib.rlk_logp_pair_save.argtypes = [A, VP, VP, VP, VP, VP]
    lib.rlk_sample.argtypes = [A, ctypes.c_uint64, VP, VP, VP, VP, VP, VP, VP, VP]
    lib.rlk_sample_noalloc.argtypes = [A, ctypes.c_uint64, VP, VP, VP, VP, VP, VP, VP]
    i64 = ctypes.c_int64
    lib.rlk_linear_logp.argtypes = [VP, i64, i64, i64, VP, i64, VP, VP, ctypes.c_float, VP, VP, VP, VP]
    lib.rlk_linear_logp_pair.argtypes = [VP, i64, i64, i64, VP, i64, VP, VP, ctypes.c_float, VP,
                                         ctypes.c_float, VP, ctypes.c_int32, VP, VP, VP, VP, VP, VP]
    lib.rlk_logp_backward_saved.argtypes = [A, VP, VP, VP, VP, ctypes.c_int64, ctypes.c_int32, VP]
    SA = P(ShardArgs)
    lib.rlk_logp_shard_summary.argtypes = [SA, VP, VP, VP, VP, VP, VP]
    lib.rlk_logp_shard_counts.argtypes = [SA, VP, VP, VP, VP, VP, VP]
    f32, i32 = ctypes.c_float, ctypes.c_int32
    lib.rlk_logp_merge.argtypes = [VP, VP, VP, VP, ctypes.c_int64, VP, VP, f32, VP, f32, VP, i32,
                                   VP, i32, VP, VP, VP, VP]
    lib.rlk_logp_merge_resumable.argtypes = [VP, VP, VP, VP, ctypes.c_int64, VP, VP, f32, VP, f32, VP,
                                             i32, VP, i32, VP, VP, VP, VP, VP, VP]
    lib.rlk_logp_shard_counts_window.argtypes = [SA, VP, VP, VP, VP]
    lib.rlk_sqnorm_accumulate.argtypes = [VP, i64, i32, VP, VP]
    lib.rlk_sqnorm_finalize.argtypes = [VP, VP, VP]
    lib.rlk_grad_norm.argtypes = [VP, i64, i32, VP, VP, VP]
    for f in COMPUTE:
        getattr(lib, f).restype = ctypes.c_int
    lib.rlk_status_string.argtypes = [ctypes.c_int]
    lib.rlk_status_string.restype = ctypes.c_char_p
    lib.rlk_last_error.argtypes = []
    lib.rlk_last_error.restype = ctypes.c_char_p
    lib.rlk_abi_version.argtypes = []
    lib.rlk_abi_version.restype = ctypes.c_int
    if lib.rlk_abi_version() != 5:
        raise ImportError("librlk_logp.so ABI version mismatch")
    _lib = lib
    return lib


def check(status: int) -> None:
    if status != RLK_OK:
        msg = load_library().rlk_last_error().decode()
        raise RlkError(status, msg)


# ------------------------------------------------------------ torch marshalling

def _torch():
    import torch
    return torch


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _param(v, T, dtype, name):
    """(device pointer or None, scalar) for a per-row tensor or a Python scalar."""
    torch = _torch()
    if isinstance(v, torch.Tensor):
        if v.dtype != dtype or v.dim() != 1 or v.shape[0] != T or not v.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape [{T}]")
        if not v.is_cuda:
            raise ValueError(f"{name} must live on the GPU")
        return v.data_ptr(), 0
    return None, v


def make_args(logits, target, temperature=1.0, top_p=1.0, top_k=-1, err_count=None) -> LogpArgs:
    """target may be None only for the sampler (which has no target)."""
    torch = _torch()
    if logits.dtype != torch.bfloat16 or logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be a bf16 [T, >=152576] tensor with unit column stride")
    if logits.shape[1] < VOCAB_PADDED:
        raise ValueError(f"logits must have at least {VOCAB_PADDED} columns")
    T = logits.shape[0]
    if target is not None and (target.dtype != torch.int32 or target.shape != (T,)
                               or not target.is_contiguous()):
        raise ValueError("target must be a contiguous int32 tensor of shape [T]")
    a = LogpArgs()
    a.logits = logits.data_ptr() if T else None
    a.T = T
    a.row_stride = logits.stride(0) if T else VOCAB_PADDED
    a.vocab_real = VOCAB_REAL
    a.vocab_padded = VOCAB_PADDED
    a.target = _ptr(target) if T and target is not None else None
    a.temperature, a.temperature_scalar = _param(temperature, T, torch.float32, "temperature")
    a.top_p, a.top_p_scalar = _param(top_p, T, torch.float32, "top_p")
    a.top_k, a.top_k_scalar = _param(top_k, T, torch.int32, "top_k")
    a.err_count = _ptr(err_count)
    return a


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _empty(T, dtype, like):
    return _torch().empty((T,), dtype=dtype, device=like.device)


def logp_full(logits, target, temperature=1.0, *, out=None, err_count=None, stream=None):
    """Full-vocabulary logprob of each row's target (float32 [T])."""
    lib = load_library()
    torch = _torch()
    a = make_args(logits, target, temperature, 1.0, -1, err_count)
    out = _empty(a.T, torch.float32, logits) if out is None else out
    check(lib.rlk_logp_full(ctypes.byref(a), _ptr(out), _stream(stream)))
    return out


def logp_pair(logits, target, temperature=1.0, top_p=1.0, top_k=-1, *, out_full=None,
              out_restr=None, out_support=None, err_count=None, stream=None):
    """(full, restricted, support) of each row's target in one pass."""
    lib = load_library()
    torch = _torch()
    a = make_args(logits, target, temperature, top_p, top_k, err_count)
    out_full = _empty(a.T, torch.float32, logits) if out_full is None else out_full
    out_restr = _empty(a.T, torch.float32, logits) if out_restr is None else out_restr
    out_support = _empty(a.T, torch.int32, logits) if out_support is None else out_support
    check(lib.rlk_logp_pair(ctypes.byref(a), _ptr(out_full), _ptr(out_restr), _ptr(out_support),
                            _stream(stream)))
    return out_full, out_restr, out_support


def logp_restricted(logits, target, temperature=1.0, top_p=1.0, top_k=-1, *, out=None,
                    out_support=None, err_count=None, stream=None):
    """(restricted, support) of each row's target."""
    lib = load_library()
    torch = _torch()
    a = make_args(logits, target, temperature, top_p, top_k, err_count)
    out = _empty(a.T, torch.float32, logits) if out is None else out
    out_support = _empty(a.T, torch.int32, logits) if out_support is None else out_support
    check(lib.rlk_logp_restricted(ctypes.byref(a), _ptr(out), _ptr(out_support), _stream(stream)))
    return out, out_support


def logp_kl(logits, ref_logits, target, temperature=1.0, top_p=1.0, top_k=-1, *, out_full=None,
            out_restr=None, out_support=None, out_full_ref=None, out_kl=None, err_count=None,
            stream=None):
    """Policy (full, restricted, support), reference full logprob, and the KL term
    full_policy - full_ref of each row's target."""
    lib = load_library()
    torch = _torch()
    a = make_args(logits, target, temperature, top_p, top_k, err_count)
    if ref_logits.dtype != torch.bfloat16 or ref_logits.shape[0] != a.T or ref_logits.stride(1) != 1:
        raise ValueError("ref_logits must be a bf16 [T, >=152576] tensor like logits")
    outs = [o if o is not None else _empty(a.T, dt, logits) for o, dt in
            ((out_full, torch.float32), (out_restr, torch.float32), (out_support, torch.int32),
             (out_full_ref, torch.float32), (out_kl, torch.float32))]
    check(lib.rlk_logp_kl(ctypes.byref(a), ref_logits.data_ptr() if a.T else None,
                          ref_logits.stride(0) if a.T else VOCAB_PADDED,
                          *[_ptr(o) for o in outs], _stream(stream)))
    return tuple(outs)


def logp_kl_host_workspace_bytes(T: int) -> int:
    """RLK_LOGP_KL_HOST_WORKSPACE_BYTES(T): both logits tensors, the targets and five outputs."""
    return T * 2 * VOCAB_PADDED * 2 + 6 * ((T * 4 + 255) // 256 * 256)


def logp_kl_host(logits, ref_logits, target, temperature=1.0, top_p=1.0, top_k=-1, *, out_full=None,
                 out_restr=None, out_support=None, out_full_ref=None, out_kl=None, workspace=None,
                 chunks=8, copy_stream=None, err_count=None, stream=None, device=None):
    """logp_kl on host-resident inputs (pinned CPU tensors: logits and ref_logits
    bf16 [T, >=152576], target int32 [T]): the copies in run on ``copy_stream``
    beside the passes, range by range.  Per-row parameters, if tensors, are on
    the GPU.  Returns pinned CPU tensors (full, restricted, support, full_ref,
    kl), valid once ``stream`` has completed."""
    lib = load_library()
    torch = _torch()
    for t, name in ((logits, "logits"), (ref_logits, "ref_logits"), (target, "target")):
        if t.is_cuda:
            raise ValueError(f"{name} must be a host (CPU) tensor")
    a = make_args(logits, target, temperature, top_p, top_k, err_count)
    if ref_logits.dtype != torch.bfloat16 or ref_logits.shape[0] != a.T or ref_logits.stride(1) != 1 \
            or ref_logits.shape[1] < VOCAB_PADDED:
        raise ValueError("ref_logits must be a bf16 [T, >=152576] tensor like logits")
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    outs = [o if o is not None else torch.empty((a.T,), dtype=dt, pin_memory=True) for o, dt in
            ((out_full, torch.float32), (out_restr, torch.float32), (out_support, torch.int32),
             (out_full_ref, torch.float32), (out_kl, torch.float32))]
    if workspace is None:
        workspace = torch.empty(logp_kl_host_workspace_bytes(a.T), dtype=torch.uint8, device=dev)
    if workspace.numel() * workspace.element_size() < logp_kl_host_workspace_bytes(a.T) or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor of at least logp_kl_host_workspace_bytes(T) bytes")
    check(lib.rlk_logp_kl_host(ctypes.byref(a), ref_logits.data_ptr() if a.T else None,
                               ref_logits.stride(0) if a.T else VOCAB_PADDED,
                               *[_ptr(o) for o in outs], workspace.data_ptr() if a.T else None,
                               int(chunks), _stream(stream),
                               copy_stream.cuda_stream if copy_stream is not None else None))
    return tuple(outs)


def logp_kl_ref(ref_logits, target, full_policy, temperature=1.0, *, out_full_ref=None,
                out_kl=None, stream=None):
    """Reference pass alone: (full_ref, kl = full_policy - full_ref) of each row's target."""
    lib = load_library()
    torch = _torch()
    a = make_args(ref_logits, target, temperature, 1.0, -1, None)
    if full_policy.dtype != torch.float32 or full_policy.shape != (a.T,):
        raise ValueError("full_policy must be a float32 tensor of shape [T]")
    out_full_ref = _empty(a.T, torch.float32, ref_logits) if out_full_ref is None else out_full_ref
    out_kl = _empty(a.T, torch.float32, ref_logits) if out_kl is None else out_kl
    check(lib.rlk_logp_kl_ref(ctypes.byref(a), _ptr(full_policy), _ptr(out_full_ref), _ptr(out_kl),
                              _stream(stream)))
    return out_full_ref, out_kl


# ------------------------------------------------------------ vocabulary-sharded form

def make_shard_args(shard_logits, shard, target, temperature=1.0, top_p=1.0, top_k=-1,
                    err_count=None) -> ShardArgs:
    torch = _torch()
    if shard_logits.dtype != torch.bfloat16 or shard_logits.dim() != 2 or shard_logits.stride(1) != 1:
        raise ValueError("shard logits must be a bf16 [T, >=19072] tensor with unit column stride")
    if shard_logits.shape[1] < SHARD_WIDTH:
        raise ValueError(f"shard logits must have at least {SHARD_WIDTH} columns")
    T = shard_logits.shape[0]
    if target.dtype != torch.int32 or target.shape != (T,) or not target.is_contiguous():
        raise ValueError("target must be a contiguous int32 tensor of shape [T]")
    a = ShardArgs()
    a.logits = shard_logits.data_ptr() if T else None
    a.T = T
    a.row_stride = shard_logits.stride(0) if T else SHARD_WIDTH
    a.shard = shard
    a.target = _ptr(target) if T else None
    a.temperature, a.temperature_scalar = _param(temperature, T, torch.float32, "temperature")
    a.top_p, a.top_p_scalar = _param(top_p, T, torch.float32, "top_p")
    a.top_k, a.top_k_scalar = _param(top_k, T, torch.int32, "top_k")
    a.err_count = _ptr(err_count)
    return a


SHARD_CHUNKS = 2384


def shard_summary(shard_logits, shard, target, temperature=1.0, top_p=1.0, top_k=-1, *,
                  out_max, out_sumexp, out_aux, out_target_logit, out_chunk_max=None, err_count=None,
                  stream=None):
    """Phase 1 on one shard: per-row (max, sum-exp, aux) into the given [T]
    views, the target logit for rows whose target lies in this shard, and
    optionally each 16-byte chunk's maximum (int16 [T, 2384], bf16 bits)."""
    lib = load_library()
    a = make_shard_args(shard_logits, shard, target, temperature, top_p, top_k, err_count)
    check(lib.rlk_logp_shard_summary(ctypes.byref(a), _ptr(out_max), _ptr(out_sumexp), _ptr(out_aux),
                                     _ptr(out_target_logit), _ptr(out_chunk_max), _stream(stream)))


def shard_counts(shard_logits, shard, target, maxes, sumexps, aux, temperature=1.0, top_p=1.0,
                 top_k=-1, *, out_counts, chunk_max=None, stream=None):
    """Phase 2 on one shard: exact per-key counts [T, 1024] on each row's
    window; with phase 1's chunk maxima only the chunks reaching it are read."""
    lib = load_library()
    a = make_shard_args(shard_logits, shard, target, temperature, top_p, top_k, None)
    check(lib.rlk_logp_shard_counts(ctypes.byref(a), _ptr(maxes), _ptr(sumexps), _ptr(aux),
                                    _ptr(chunk_max), _ptr(out_counts), _stream(stream)))


def logp_merge(maxes, sumexps, aux, target_logit, target, temperature=1.0, top_p=1.0, top_k=-1, *,
               counts=None, out_full=None, out_restr=None, out_support=None, stream=None):
    """Merge of the gathered [8, T] summaries: full logprob, and with counts
    ([1 or 8, T, 1024]) the restricted logprob and support."""
    lib = load_library()
    torch = _torch()
    T = target.shape[0]
    tp, ts = _param(temperature, T, torch.float32, "temperature")
    pp, ps = _param(top_p, T, torch.float32, "top_p")
    kp, ks = _param(top_k, T, torch.int32, "top_k")
    out_full = _empty(T, torch.float32, maxes) if out_full is None else out_full
    if counts is not None:
        out_restr = _empty(T, torch.float32, maxes) if out_restr is None else out_restr
        out_support = _empty(T, torch.int32, maxes) if out_support is None else out_support
    nc = 0 if counts is None else counts.shape[0]
    check(lib.rlk_logp_merge(_ptr(maxes), _ptr(sumexps), _ptr(aux), _ptr(target_logit), T,
                             _ptr(target), tp, ts, pp, ps, kp, ks, _ptr(counts), nc,
                             _ptr(out_full), _ptr(out_restr), _ptr(out_support), _stream(stream)))
    return (out_full,) if counts is None else (out_full, out_restr, out_support)


MERGE_STATE_WORDS = 5        # rlk_merge_state: 40 bytes per row, as int64 words
MAX_RESUME_ROUNDS = 2 * 64 + 2


def merge_state(T, device):
    """A zeroed per-row resolution state (rlk_merge_state [T]) for the resumable merge."""
    return _torch().zeros((T, MERGE_STATE_WORDS), dtype=_torch().int64, device=device)


def shard_counts_window(shard_logits, shard, target, state, *, out_counts, chunk_max=None,
                        stream=None):
    """Counts [T, 1024] of one shard's tokens on each pending row's next window
    (the window its state names; zeros for rows that are not pending)."""
    lib = load_library()
    a = make_shard_args(shard_logits, shard, target, 1.0, 1.0, -1, None)
    check(lib.rlk_logp_shard_counts_window(ctypes.byref(a), _ptr(state), _ptr(chunk_max),
                                           _ptr(out_counts), _stream(stream)))


def logp_merge_resumable(maxes, sumexps, aux, target_logit, target, temperature=1.0, top_p=1.0,
                         top_k=-1, *, counts, state, out_full, out_restr, out_support,
                         out_pending=None, stream=None):
    """One round of the resumable merge: resolves what the given counts allow
    and records the next window of the rows that stay pending."""
    lib = load_library()
    torch = _torch()
    T = target.shape[0]
    tp, ts = _param(temperature, T, torch.float32, "temperature")
    pp, ps = _param(top_p, T, torch.float32, "top_p")
    kp, ks = _param(top_k, T, torch.int32, "top_k")
    check(lib.rlk_logp_merge_resumable(_ptr(maxes), _ptr(sumexps), _ptr(aux), _ptr(target_logit), T,
                                       _ptr(target), tp, ts, pp, ps, kp, ks, _ptr(counts),
                                       counts.shape[0], _ptr(state), _ptr(out_full), _ptr(out_restr),
                                       _ptr(out_support), _ptr(out_pending), _stream(stream)))


def logp_sharded(shards, target, temperature=1.0, top_p=1.0, top_k=-1, *, restricted=True,
                 chunk_maxima=True, resolve=True, err_count=None, stream=None):
    """All phases over 8 shard buffers (shard r holds vocabulary columns
    [19072 r, 19072 (r+1))): summaries, then counts when restricted (reading
    only the chunks whose phase-1 maximum reaches the window, unless
    ``chunk_maxima`` is False), then the merge.  With ``resolve`` (the
    default) rows whose support reaches below the first window are carried
    through lower windows (counts + resumable merge rounds, each round
    reading the number of pending rows on the host) until every row is
    resolved; without it such rows keep support -2.  Returns (full,) or
    (full, restricted, support)."""
    torch = _torch()
    if len(shards) != NUM_SHARDS:
        raise ValueError(f"expected {NUM_SHARDS} shard tensors")
    T = target.shape[0]
    dev = shards[0].device
    maxes = torch.empty((NUM_SHARDS, T), dtype=torch.float32, device=dev)
    sumexps = torch.empty_like(maxes)
    aux = torch.empty((NUM_SHARDS, T), dtype=torch.int32, device=dev)
    xt = torch.empty((T,), dtype=torch.float32, device=dev)
    pk = (top_p, top_k) if restricted else (1.0, -1)
    cmax = (torch.empty((NUM_SHARDS, T, SHARD_CHUNKS), dtype=torch.int16, device=dev)
            if restricted and chunk_maxima else None)
    for r, sh in enumerate(shards):
        shard_summary(sh, r, target, temperature, *pk, out_max=maxes[r], out_sumexp=sumexps[r],
                      out_aux=aux[r], out_target_logit=xt,
                      out_chunk_max=None if cmax is None else cmax[r], err_count=err_count,
                      stream=stream)
    counts = None
    if restricted:
        counts = torch.empty((NUM_SHARDS, T, 1024), dtype=torch.int32, device=dev)
        for r, sh in enumerate(shards):
            shard_counts(sh, r, target, maxes, sumexps, aux, temperature, top_p, top_k,
                         out_counts=counts[r], chunk_max=None if cmax is None else cmax[r],
                         stream=stream)
    if not (restricted and resolve and T > 0):
        return logp_merge(maxes, sumexps, aux, xt, target, temperature, *pk, counts=counts,
                          stream=stream)
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    state = merge_state(T, dev)
    pending = torch.zeros(1, dtype=torch.int32, device=dev)
    full = torch.empty(T, dtype=torch.float32, device=dev)
    restr = torch.empty(T, dtype=torch.float32, device=dev)
    support = torch.empty(T, dtype=torch.int32, device=dev)
    for rnd in range(MAX_RESUME_ROUNDS + 1):
        if rnd > 0:
            for r, sh in enumerate(shards):
                shard_counts_window(sh, r, target, state, out_counts=counts[r],
                                    chunk_max=None if cmax is None else cmax[r], stream=stream)
        with torch.cuda.stream(st):
            pending.zero_()
        logp_merge_resumable(maxes, sumexps, aux, xt, target, temperature, top_p, top_k,
                             counts=counts, state=state, out_full=full, out_restr=restr,
                             out_support=support, out_pending=pending, stream=stream)
        with torch.cuda.stream(st):
            left = int(pending.item())
        if left == 0:
            return full, restr, support
    raise RlkError(f"{left} rows still pending after {MAX_RESUME_ROUNDS} windows")


# ------------------------------------------------------------ backward

def logp_backward(logits, target, temperature=1.0, top_p=1.0, top_k=-1, *, grad_full=None,
                  grad_restr=None, dtype=None, out=None, out_full=None, out_restr=None,
                  out_support=None, err_count=None, stream=None):
    """Gradient of grad_full * full + grad_restr * restr with respect to the
    logits ([T, 152576], bf16 unless ``dtype`` is torch.float32), recomputing
    the forward in the same pass (optional forward outputs)."""
    lib = load_library()
    torch = _torch()
    a = make_args(logits, target, temperature, top_p, top_k, err_count)
    for g, name in ((grad_full, "grad_full"), (grad_restr, "grad_restr")):
        if g is not None and (g.dtype != torch.float32 or g.shape != (a.T,) or not g.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous float32 tensor of shape [T]")
    if out is None:
        dtype = torch.bfloat16 if dtype is None else dtype
        out = torch.empty((a.T, VOCAB_PADDED), dtype=dtype, device=logits.device)
    if out.dtype not in (torch.bfloat16, torch.float32) or out.dim() != 2 or out.stride(1) != 1:
        raise ValueError("out must be a bf16 or float32 [T, >=152576] tensor with unit column stride")
    gd = RLK_GRAD_F32 if out.dtype == torch.float32 else RLK_GRAD_BF16
    check(lib.rlk_logp_backward(ctypes.byref(a), _ptr(grad_full), _ptr(grad_restr),
                                out.data_ptr() if a.T else None,
                                out.stride(0) if a.T else VOCAB_PADDED, gd, _ptr(out_full),
                                _ptr(out_restr), _ptr(out_support), _stream(stream)))
    return out


def logp_pair_save(logits, target, temperature=1.0, top_p=1.0, top_k=-1, *, out_full=None,
                   out_restr=None, out_support=None, out_stats=None, err_count=None, stream=None):
    """logp_pair plus the per-row record for a later backward: returns
    (full, restricted, support, stats), stats a float32 [T, 4] tensor holding
    rlk_row_stats (column 3 is the int32 min_key, stored bitwise)."""
    lib = load_library()
    torch = _torch()
    a = make_args(logits, target, temperature, top_p, top_k, err_count)
    out_full = _empty(a.T, torch.float32, logits) if out_full is None else out_full
    out_restr = _empty(a.T, torch.float32, logits) if out_restr is None else out_restr
    out_support = _empty(a.T, torch.int32, logits) if out_support is None else out_support
    if out_stats is None:
        out_stats = torch.empty((a.T, 4), dtype=torch.float32, device=logits.device)
    check(lib.rlk_logp_pair_save(ctypes.byref(a), _ptr(out_full), _ptr(out_restr), _ptr(out_support),
                                 _ptr(out_stats), _stream(stream)))
    return out_full, out_restr, out_support, out_stats


def logp_backward_saved(logits, target, stats, temperature=1.0, *, grad_full=None, grad_restr=None,
                        dtype=None, out=None, stream=None):
    """The backward from a record saved by logp_pair_save (same logits, targets
    and temperatures): a streaming pass, bit-identical to logp_backward."""
    lib = load_library()
    torch = _torch()
    a = make_args(logits, target, temperature, 1.0, -1, None)
    if stats.dtype != torch.float32 or stats.shape != (a.T, 4) or not stats.is_contiguous():
        raise ValueError("stats must be the contiguous float32 [T, 4] record of logp_pair_save")
    for g, name in ((grad_full, "grad_full"), (grad_restr, "grad_restr")):
        if g is not None and (g.dtype != torch.float32 or g.shape != (a.T,) or not g.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous float32 tensor of shape [T]")
    if out is None:
        dtype = torch.bfloat16 if dtype is None else dtype
        out = torch.empty((a.T, VOCAB_PADDED), dtype=dtype, device=logits.device)
    if out.dtype not in (torch.bfloat16, torch.float32) or out.dim() != 2 or out.stride(1) != 1:
        raise ValueError("out must be a bf16 or float32 [T, >=152576] tensor with unit column stride")
    gd = RLK_GRAD_F32 if out.dtype == torch.float32 else RLK_GRAD_BF16
    check(lib.rlk_logp_backward_saved(ctypes.byref(a), _ptr(stats), _ptr(grad_full), _ptr(grad_restr),
                                      out.data_ptr() if a.T else None,
                                      out.stride(0) if a.T else VOCAB_PADDED, gd, _stream(stream)))
    return out


def _autograd_function():
    torch = _torch()

    class _Logp(torch.autograd.Function):
        """(full, restr) of each row's target, differentiable with respect to
        the logits.  The forward saves a 16-byte record per row; the backward
        is one streaming call of rlk_logp_backward_saved."""

        @staticmethod
        def forward(ctx, logits, target, temperature, top_p, top_k):
            full, restr, _, stats = logp_pair_save(logits, target, temperature, top_p, top_k)
            ctx.save_for_backward(logits, target, stats)
            ctx.temperature = temperature
            return full, restr

        @staticmethod
        def backward(ctx, g_full, g_restr):
            logits, target, stats = ctx.saved_tensors
            gf = None if g_full is None else g_full.float().contiguous()
            gr = None if g_restr is None else g_restr.float().contiguous()
            if gf is None and gr is None:
                return None, None, None, None, None
            grad = torch.empty_like(logits)
            if logits.shape[1] > VOCAB_PADDED:
                grad[:, VOCAB_PADDED:] = 0
            logp_backward_saved(logits, target, stats, ctx.temperature, grad_full=gf,
                                grad_restr=gr, out=grad)
            return grad, None, None, None, None

    return _Logp


_LOGP_FN = None


def logp_autograd(logits, target, temperature=1.0, top_p=1.0, top_k=-1):
    """(full, restr) as differentiable torch outputs (see logp_backward)."""
    global _LOGP_FN
    if _LOGP_FN is None:
        _LOGP_FN = _autograd_function()
    return _LOGP_FN.apply(logits, target, temperature, top_p, top_k)


# ------------------------------------------------------------ sampler

def sample_workspace_bytes(T: int) -> int:
    """RLK_SAMPLE_WORKSPACE_BYTES(T): a 16-byte record and a 2432-byte chunk bitmap per row."""
    return T * (16 + 2432)


def sample(logits, temperature=1.0, top_p=1.0, top_k=-1, *, seed=0, counter=None, uniform=None,
           out_token=None, out_restr=None, out_full=None, out_support=None, workspace=None,
           err_count=None, stream=None):
    """Draw one token per row from the restricted distribution (inverse CDF in
    column order).  Random words: ``uniform`` (uint32 bits in an int32 [T]
    tensor) or Philox4x32-10 of ``seed`` over ``counter`` (int64 [T]).
    ``workspace``: uint8 [sample_workspace_bytes(T)] scratch (allocated here
    if not given).  Returns (token, restricted logprob, full logprob, support)."""
    lib = load_library()
    torch = _torch()
    a = make_args(logits, None, temperature, top_p, top_k, err_count)
    T = a.T
    for v, name, dt in ((counter, "counter", torch.int64), (uniform, "uniform", torch.int32)):
        if v is not None and (v.dtype != dt or v.shape != (T,) or not v.is_contiguous() or not v.is_cuda):
            raise ValueError(f"{name} must be a contiguous {dt} CUDA tensor of shape [T]")
    if counter is None and uniform is None:
        raise ValueError("give counter (with seed) or uniform")
    out_token = _empty(T, torch.int32, logits) if out_token is None else out_token
    out_restr = _empty(T, torch.float32, logits) if out_restr is None else out_restr
    out_full = _empty(T, torch.float32, logits) if out_full is None else out_full
    out_support = _empty(T, torch.int32, logits) if out_support is None else out_support
    if workspace is None:
        workspace = torch.empty(sample_workspace_bytes(T), dtype=torch.uint8, device=logits.device)
    if workspace.numel() * workspace.element_size() < sample_workspace_bytes(T) or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor of at least sample_workspace_bytes(T) bytes")
    check(lib.rlk_sample(ctypes.byref(a), int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(counter), _ptr(uniform),
                         _ptr(out_token), _ptr(out_restr), _ptr(out_full), _ptr(out_support),
                         workspace.data_ptr() if T else None, _stream(stream)))
    return out_token, out_restr, out_full, out_support


# ------------------------------------------------------------ fused LM head

def linear_workspace_bytes(T: int) -> int:
    return T * (596 * 8 + 4)


def linear_logp(hidden, weight, target, temperature=1.0, *, out=None, workspace=None, err_count=None,
                stream=None):
    """Full-vocabulary logprob of each row's target with logits = hidden . weight^T
    formed on the tensor cores and never stored (hidden: bf16 [T, H]; weight:
    bf16 [152576, H], the padded LM head)."""
    lib = load_library()
    torch = _torch()
    T, H = hidden.shape
    for t, name in ((hidden, "hidden"), (weight, "weight")):
        if t.dtype != torch.bfloat16 or t.dim() != 2 or t.stride(1) != 1 or not t.is_cuda:
            raise ValueError(f"{name} must be a bf16 CUDA matrix with unit column stride")
    if weight.shape[0] != VOCAB_PADDED or weight.shape[1] != H:
        raise ValueError(f"weight must be [{VOCAB_PADDED}, {H}]")
    if target.dtype != torch.int32 or target.shape != (T,) or not target.is_contiguous():
        raise ValueError("target must be a contiguous int32 tensor of shape [T]")
    tp, ts = _param(temperature, T, torch.float32, "temperature")
    out = _empty(T, torch.float32, hidden) if out is None else out
    if workspace is None:
        workspace = torch.empty(max(1, linear_workspace_bytes(T)), dtype=torch.uint8, device=hidden.device)
    check(lib.rlk_linear_logp(hidden.data_ptr() if T else None, T, H, hidden.stride(0) if T else H,
                              weight.data_ptr(), weight.stride(0), _ptr(target), tp, ts, _ptr(out),
                              workspace.data_ptr(), _ptr(err_count), _stream(stream)))
    return out


def linear_pair_workspace_bytes(T: int) -> int:
    return T * 52640 + 4096


def linear_logp_pair(hidden, weight, target, temperature=1.0, top_p=1.0, top_k=-1, *, out_full=None,
                     out_restr=None, out_support=None, workspace=None, err_count=None, stream=None):
    """Full and restricted logprob of each row's target, and the support size,
    with logits = hidden . weight^T formed on the tensor cores and never
    stored; the support is selected exactly over the fp32 logits.  Returns
    (full, restr, support)."""
    lib = load_library()
    torch = _torch()
    T, H = hidden.shape
    for t, name in ((hidden, "hidden"), (weight, "weight")):
        if t.dtype != torch.bfloat16 or t.dim() != 2 or t.stride(1) != 1 or not t.is_cuda:
            raise ValueError(f"{name} must be a bf16 CUDA matrix with unit column stride")
    if weight.shape[0] != VOCAB_PADDED or weight.shape[1] != H:
        raise ValueError(f"weight must be [{VOCAB_PADDED}, {H}]")
    if target.dtype != torch.int32 or target.shape != (T,) or not target.is_contiguous():
        raise ValueError("target must be a contiguous int32 tensor of shape [T]")
    tp, ts = _param(temperature, T, torch.float32, "temperature")
    pp, ps = _param(top_p, T, torch.float32, "top_p")
    kp, ks = _param(top_k, T, torch.int32, "top_k")
    out_full = _empty(T, torch.float32, hidden) if out_full is None else out_full
    out_restr = _empty(T, torch.float32, hidden) if out_restr is None else out_restr
    out_support = _empty(T, torch.int32, hidden) if out_support is None else out_support
    if workspace is None:
        workspace = torch.empty(max(1, linear_pair_workspace_bytes(T)), dtype=torch.uint8,
                                device=hidden.device)
    elif workspace.numel() * workspace.element_size() < linear_pair_workspace_bytes(T):
        raise ValueError("workspace must hold at least linear_pair_workspace_bytes(T) bytes")
    check(lib.rlk_linear_logp_pair(hidden.data_ptr() if T else None, T, H, hidden.stride(0) if T else H,
                                   weight.data_ptr(), weight.stride(0), _ptr(target), tp, ts, pp, ps, kp,
                                   ks, _ptr(out_full), _ptr(out_restr), _ptr(out_support),
                                   workspace.data_ptr(), _ptr(err_count), _stream(stream)))
    return out_full, out_restr, out_support


# ----------------------------------------------------------------- gradient norm

NORM_BINS = 384
RLK_DT_F32, RLK_DT_BF16, RLK_DT_F16 = 0, 1, 2


def _norm_dtype(t) -> int:
    torch = _torch()
    codes = {torch.float32: RLK_DT_F32, torch.bfloat16: RLK_DT_BF16, torch.float16: RLK_DT_F16}
    if t.dtype not in codes:
        raise TypeError(f"gradient norm: dtype {t.dtype} is not float32, bfloat16 or float16")
    return codes[t.dtype]


def norm_bins(device=None):
    """A cleared bin vector for sqnorm_accumulate: the 384 uint64 words in int64 storage."""
    torch = _torch()
    return torch.zeros(NORM_BINS, dtype=torch.int64, device=device)


def sqnorm_accumulate(x, bins, stream=None):
    """Add the FP32 squares of the elements of x (contiguous) into bins."""
    lib = load_library()
    if not x.is_contiguous():
        raise ValueError("gradient norm: x must be contiguous")
    if bins.dtype != _torch().int64 or bins.numel() != NORM_BINS:
        raise ValueError("gradient norm: bins must be int64 [384] (see norm_bins)")
    n = x.numel()
    check(lib.rlk_sqnorm_accumulate(_ptr(x) if n else None, n, _norm_dtype(x), _ptr(bins),
                                    _stream(stream)))
    return bins


def sqnorm_finalize(bins, out=None, stream=None):
    """(sum of squares, norm) as a device float64 [2]."""
    lib = load_library()
    torch = _torch()
    out = torch.empty(2, dtype=torch.float64, device=bins.device) if out is None else out
    check(lib.rlk_sqnorm_finalize(_ptr(bins), _ptr(out), _stream(stream)))
    return out


def reduce_bins_(bins, group=None):
    """The distributed reduction: every rank's bins summed elementwise (integer
    adds, exact in any order), in place."""
    import torch.distributed as dist
    dist.all_reduce(bins, op=dist.ReduceOp.SUM, group=group)
    return bins


def grad_norm(tensors, *, distributed=False, group=None, bins=None, out=None, stream=None):
    """L2 norm of a list of gradient tensors, identical whatever their order,
    the launch shape, or (with ``distributed``) the split across the ranks
    of ``group``.  Returns the device float64 [2] (sum of squares, norm)."""
    torch = _torch()
    if isinstance(tensors, torch.Tensor):
        tensors = [tensors]
    tensors = list(tensors)
    if bins is None:
        if not tensors:
            raise ValueError("grad_norm: no tensors (pass bins to take the device from them)")
        bins = norm_bins(tensors[0].device)
    else:
        bins.zero_()
    for t in tensors:
        sqnorm_accumulate(t, bins, stream)
    if distributed:
        reduce_bins_(bins, group)
    return sqnorm_finalize(bins, out, stream)
