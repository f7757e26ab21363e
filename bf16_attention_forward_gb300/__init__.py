"""bf16 attention forward for GB300 (sm_103a): Python binding of the C-ABI library.

The binding only marshals arguments: every step of the computation runs in the library's
CUDA kernels (``csrc/attn_fwd.cu``, ABI in ``include/bf16_attn.h``).  PyTorch supplies
device memory and the current stream.  There is no CPU fallback: if the compiled library
is missing, importing the binding's entry points raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

LAYOUTS = {"bshd": 0, "bhsd": 1}
MODES = {"rtne": 0, "rtna": 1, "rtz": 2}
STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED",
          3: "ATTN_ERR_MISALIGNED", 4: "ATTN_ERR_ALIAS", 5: "ATTN_ERR_NO_DEVICE",
          6: "ATTN_ERR_WORKSPACE", 7: "ATTN_ERR_CUDA", 8: "ATTN_ERR_DEVICE_TIMEOUT"}
EXPORTS = ("attn_fwd", "attn_fwd_ws", "attn_fwd_noalloc", "attn_fwd_ex", "attn_fwd_workspace_size",
           "attn_fwd_workspace_size_opts", "attn_fwd_ex_workspace_size", "attn_plan",
           "attn_plan_ex", "attn_get_device_status", "attn_status_string", "attn_version",
           "attn_bwd", "attn_bwd_workspace_size", "attn_bwd_get_device_status",
           "attn_fwd_varlen", "attn_fwd_varlen_workspace_size", "attn_fwd_paged",
           "attn_fwd_paged_workspace_size", "attn_bwd_varlen", "attn_bwd_varlen_workspace_size")


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__("%s (%d): %s%s" % (STATUS.get(status, "?"), status,
                                            status_string(status), (" -- " + what) if what else ""))


class Options(ctypes.Structure):
    _fields_ = [("force_splits", ctypes.c_int32), ("max_ctas", ctypes.c_int32),
                ("wait_limit_ms", ctypes.c_uint32), ("test_hooks", ctypes.c_uint32),
                ("events", ctypes.c_void_p * 3)]


class Args(ctypes.Structure):
    """attn_args_t: the full argument set of attn_fwd_ex."""
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p)] + \
               [(n, ctypes.c_int64) for n in ("B", "H", "Hkv", "Sq", "Skv", "d")] + \
               [(n, ctypes.c_int32) for n in ("layout", "round_mode", "causal", "reserved")]


class BwdArgs(ctypes.Structure):
    """attn_bwd_args_t: the argument set of attn_bwd."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "v", "o", "dout", "lse", "dq", "dk", "dv")] + \
               [(n, ctypes.c_int64) for n in ("B", "H", "Hkv", "Sq", "Skv", "d")] + \
               [(n, ctypes.c_int32) for n in ("layout", "causal", "wait_limit_ms", "test_hooks",
                                              "deterministic", "reserved")]


class VarlenArgs(ctypes.Structure):
    """attn_varlen_args_t: the argument set of attn_fwd_varlen."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "v", "o", "lse", "cu_seqlens_q",
                                               "cu_seqlens_k")] + \
               [(n, ctypes.c_int64) for n in ("B", "H", "Hkv", "total_q", "total_k",
                                              "max_seqlen_q", "d")] + \
               [(n, ctypes.c_int32) for n in ("round_mode", "causal", "pack_heads", "max_splits")]


class PagedArgs(ctypes.Structure):
    """attn_paged_args_t: the argument set of attn_fwd_paged."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k_cache", "v_cache", "o", "lse", "cu_seqlens_q",
                                               "seqlens_k", "block_table")] + \
               [(n, ctypes.c_int64) for n in ("B", "H", "Hkv", "total_q", "num_pages", "page_size",
                                              "max_pages", "max_seqlen_q", "d")] + \
               [(n, ctypes.c_int32) for n in ("round_mode", "causal", "pack_heads", "max_splits")]


class BwdVarlenArgs(ctypes.Structure):
    """attn_bwd_varlen_args_t: the argument set of attn_bwd_varlen."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "v", "o", "dout", "lse", "dq", "dk", "dv",
                                               "cu_seqlens_q", "cu_seqlens_k")] + \
               [(n, ctypes.c_int64) for n in ("B", "H", "Hkv", "total_q", "total_k", "d")] + \
               [(n, ctypes.c_int32) for n in ("causal", "wait_limit_ms", "reserved", "reserved2")]


class Plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("units", "kv_tiles", "full_items", "split_units",
                                              "splits", "items", "grid", "workspace_bytes")]

    def as_dict(self) -> dict:
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Load the compiled library (it must already be built: ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB_PATH
        if not os.path.exists(p):
            raise ImportError("bf16 attention library not built: %s is missing "
                              "(run __graft_entry__.build())" % p)
        lib = ctypes.CDLL(p)
        i64, vp, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        lib.attn_fwd.restype = i32
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i32, i32, vp]
        lib.attn_fwd_ws.restype = i32
        lib.attn_fwd_ws.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i32, i32,
                                    ctypes.POINTER(Options), vp, ctypes.c_size_t, vp]
        lib.attn_fwd_noalloc.restype = i32
        lib.attn_fwd_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i32, i32, vp]
        lib.attn_fwd_workspace_size.restype = ctypes.c_size_t
        lib.attn_fwd_workspace_size.argtypes = [i64] * 5
        lib.attn_fwd_workspace_size_opts.restype = ctypes.c_size_t
        lib.attn_fwd_workspace_size_opts.argtypes = [i64] * 5 + [ctypes.POINTER(Options)]
        lib.attn_fwd_ex.restype = i32
        lib.attn_fwd_ex.argtypes = [ctypes.POINTER(Args), ctypes.POINTER(Options), vp,
                                    ctypes.c_size_t, vp]
        lib.attn_fwd_ex_workspace_size.restype = ctypes.c_size_t
        lib.attn_fwd_ex_workspace_size.argtypes = [ctypes.POINTER(Args), ctypes.POINTER(Options)]
        lib.attn_plan_ex.restype = i32
        lib.attn_plan_ex.argtypes = [ctypes.POINTER(Args), i64, ctypes.POINTER(Options),
                                     ctypes.POINTER(Plan)]
        lib.attn_bwd.restype = i32
        lib.attn_bwd.argtypes = [ctypes.POINTER(BwdArgs), vp, ctypes.c_size_t, vp]
        lib.attn_bwd_workspace_size.restype = ctypes.c_size_t
        lib.attn_bwd_workspace_size.argtypes = [ctypes.POINTER(BwdArgs)]
        lib.attn_bwd_get_device_status.restype = i32
        lib.attn_bwd_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
        lib.attn_fwd_varlen.restype = i32
        lib.attn_fwd_varlen.argtypes = [ctypes.POINTER(VarlenArgs), ctypes.POINTER(Options), vp,
                                        ctypes.c_size_t, vp]
        lib.attn_fwd_varlen_workspace_size.restype = ctypes.c_size_t
        lib.attn_fwd_varlen_workspace_size.argtypes = [ctypes.POINTER(VarlenArgs)]
        lib.attn_fwd_paged.restype = i32
        lib.attn_fwd_paged.argtypes = [ctypes.POINTER(PagedArgs), ctypes.POINTER(Options), vp,
                                       ctypes.c_size_t, vp]
        lib.attn_fwd_paged_workspace_size.restype = ctypes.c_size_t
        lib.attn_fwd_paged_workspace_size.argtypes = [ctypes.POINTER(PagedArgs)]
        lib.attn_bwd_varlen.restype = i32
        lib.attn_bwd_varlen.argtypes = [ctypes.POINTER(BwdVarlenArgs), vp, ctypes.c_size_t, vp]
        lib.attn_bwd_varlen_workspace_size.restype = ctypes.c_size_t
        lib.attn_bwd_varlen_workspace_size.argtypes = [ctypes.POINTER(BwdVarlenArgs)]
        lib.attn_plan.restype = i32
        lib.attn_plan.argtypes = [i64] * 6 + [ctypes.POINTER(Options), ctypes.POINTER(Plan)]
        lib.attn_get_device_status.restype = i32
        lib.attn_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_status_string.argtypes = [i32]
        lib.attn_version.restype = i32
        lib.attn_version.argtypes = []
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().attn_status_string(int(status)).decode()


def _dims(q, k, v, layout, grouped=False):
    """(B, H, Hkv, Sq, Skv, d) from the tensors' shapes, checking that they agree."""
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D (BSHD or BHSD)")
    if tuple(k.shape) != tuple(v.shape):
        raise ValueError("k and v must have the same shape")
    if layout == "bshd":
        (B, Sq, H, d), (Bk, Skv, Hkv, dk) = q.shape, k.shape
    else:
        (B, H, Sq, d), (Bk, Hkv, Skv, dk) = q.shape, k.shape
    if Bk != B or dk != d:
        raise ValueError("q and k/v differ in batch or head dimension")
    if (Hkv != H) if not grouped else (Hkv < 1 or H % Hkv != 0):
        raise ValueError("k/v heads (%d) must %s the query heads (%d)"
                         % (Hkv, "divide" if grouped else "equal", H))
    return int(B), int(H), int(Hkv), int(Sq), int(Skv), int(d)


def _check_tensors(q, k, v):
    import torch
    for t in (q, k, v):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError("q, k, v must be CUDA bf16 tensors")
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous")


def _check_out(o, q):
    import torch
    if (not isinstance(o, torch.Tensor) or o.dtype != torch.bfloat16 or not o.is_cuda
            or not o.is_contiguous() or tuple(o.shape) != tuple(q.shape)):
        raise ValueError("o must be a contiguous CUDA bf16 tensor shaped like q")


def _stream_ptr(stream, device):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream if hasattr(s, "cuda_stream") else int(s))


def _opts(force_splits=0, max_ctas=0, wait_limit_ms=0, events=None, test_hooks=0):
    if not (force_splits or max_ctas or wait_limit_ms or events or test_hooks):
        return None
    o = Options(int(force_splits), int(max_ctas), int(wait_limit_ms), int(test_hooks))
    if events:
        for i, e in enumerate(events[:3]):
            o.events[i] = None if e is None else int(e.cuda_event)
    return o


def plan(B, H, Sq, Skv, d=128, num_sms=152, force_splits=0, max_ctas=0) -> dict:
    """The work split the library would launch for this shape (host only)."""
    pl = Plan()
    o = _opts(force_splits, max_ctas)
    st = load().attn_plan(B, H, Sq, Skv, d, num_sms, ctypes.byref(o) if o else None,
                          ctypes.byref(pl))
    if st != 0:
        raise AttnError(st, "attn_plan")
    return pl.as_dict()


def workspace_size(B, H, Sq, Skv, d=128, force_splits=0, max_ctas=0) -> int:
    o = _opts(force_splits, max_ctas)
    return int(load().attn_fwd_workspace_size_opts(B, H, Sq, Skv, d,
                                                   ctypes.byref(o) if o else None))


def attn_fwd(q, k, v, o=None, layout: str = "bshd", round: str = "rtne", stream=None,
             workspace=None, force_splits: int = 0, max_ctas: int = 0, wait_limit_ms: int = 0,
             events=None, test_hooks: int = 0):
    """O = softmax(Q K^T / sqrt(d)) V on CUDA tensors (bf16, contiguous, same layout; d is
    the head dimension, 128 or 64).

    ``workspace``: optional caller tensor (any dtype, CUDA) used through ``attn_fwd_ws``;
    with the knobs set and no workspace, one is allocated here with torch.  ``events``: up to
    three ``torch.cuda.Event`` recorded around the attention and combine kernels on the
    launching stream.  ``test_hooks``: 0 for normal use (ATTN_TEST_WITHHOLD_O_READY = 1 makes a
    bounded wait expire, to test that path).  Returns ``o``.
    """
    import torch
    if layout not in LAYOUTS or round not in MODES:
        raise ValueError("layout must be bshd/bhsd and round rtne/rtna/rtz")
    _check_tensors(q, k, v)
    B, H, _, Sq, Skv, d = _dims(q, k, v, layout)
    if o is None:
        o = torch.empty_like(q)
    _check_out(o, q)
    sp = _stream_ptr(stream, q.device)
    lib = load()
    opts = _opts(force_splits, max_ctas, wait_limit_ms, events, test_hooks)
    if workspace is None and opts is None:
        st = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, H, Sq,
                          Skv, d, LAYOUTS[layout], MODES[round], sp)
    else:
        need = workspace_size(B, H, Sq, Skv, d, force_splits, max_ctas)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
        nbytes = workspace.numel() * workspace.element_size()
        st = lib.attn_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, H, Sq,
                             Skv, d, LAYOUTS[layout], MODES[round],
                             ctypes.byref(opts) if opts else None, workspace.data_ptr(),
                             nbytes, sp)
    if st != 0:
        raise AttnError(st, "attn_fwd")
    return o


def _args(q, k, v, o, lse, layout, round, causal) -> Args:
    B, H, Hkv, Sq, Skv, d = _dims(q, k, v, layout, grouped=True)
    a = Args()
    a.q, a.k, a.v, a.o = q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr()
    a.lse = None if lse is None else lse.data_ptr()
    a.B, a.H, a.Hkv, a.Sq, a.Skv, a.d = B, H, Hkv, Sq, Skv, d
    a.layout, a.round_mode, a.causal, a.reserved = LAYOUTS[layout], MODES[round], int(causal), 0
    return a


def plan_ex(B, H, Sq, Skv, Hkv=None, d=128, causal=False, num_sms=152, force_splits=0,
            max_ctas=0) -> dict:
    """attn_plan_ex: the work split for the full argument set (host only)."""
    a = Args()
    a.B, a.H, a.Hkv, a.Sq, a.Skv, a.d = B, H, H if Hkv is None else Hkv, Sq, Skv, d
    a.causal = int(causal)
    pl = Plan()
    o = _opts(force_splits, max_ctas)
    st = load().attn_plan_ex(ctypes.byref(a), num_sms, ctypes.byref(o) if o else None,
                             ctypes.byref(pl))
    if st != 0:
        raise AttnError(st, "attn_plan_ex")
    return pl.as_dict()


def attn_fwd_ex(q, k, v, o=None, lse=None, layout: str = "bshd", round: str = "rtne",
                causal: bool = False, return_lse: bool = False, stream=None, workspace=None,
                force_splits: int = 0, max_ctas: int = 0, wait_limit_ms: int = 0, events=None):
    """attn_fwd with grouped K/V heads (k, v carry Hkv heads, Hkv dividing H), the causal mask
    (key j visible to query i iff j <= i + Skv - Sq) and the fp32 row log-sum-exp.

    ``lse``: optional CUDA fp32 tensor of B*H*Sq elements laid out [B][H][Sq]; with
    ``return_lse`` and no ``lse`` one is allocated.  Returns ``o`` or ``(o, lse)``.
    ``workspace``: optional caller tensor; without it the library-owned workspace is used.
    """
    import torch
    if layout not in LAYOUTS or round not in MODES:
        raise ValueError("layout must be bshd/bhsd and round rtne/rtna/rtz")
    _check_tensors(q, k, v)
    B, H, _, Sq, _, _ = _dims(q, k, v, layout, grouped=True)
    if o is None:
        o = torch.empty_like(q)
    _check_out(o, q)
    if lse is None and return_lse:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous()
                            or lse.numel() != B * H * Sq):
        raise ValueError("lse must be a contiguous CUDA fp32 tensor of B*H*Sq elements")
    a = _args(q, k, v, o, lse, layout, round, causal)
    opts = _opts(force_splits, max_ctas, wait_limit_ms, events)
    lib = load()
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = lib.attn_fwd_ex(ctypes.byref(a), ctypes.byref(opts) if opts else None, ws_ptr, ws_bytes,
                         _stream_ptr(stream, q.device))
    if st != 0:
        raise AttnError(st, "attn_fwd_ex")
    return (o, lse) if (return_lse or lse is not None) else o


def _varlen_args(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, round, causal, pack_heads=False,
                 max_splits=0):
    import torch
    _check_tensors(q, k, v)
    if q.dim() != 3 or k.dim() != 3 or tuple(k.shape) != tuple(v.shape) or q.shape[2] != k.shape[2]:
        raise ValueError("q must be [total_q, H, d] and k, v [total_k, Hkv, d]")
    H, Hkv, d = q.shape[1], k.shape[1], q.shape[2]
    for c in (cu_seqlens_q, cu_seqlens_k):
        if (not isinstance(c, torch.Tensor) or c.dtype != torch.int32 or not c.is_cuda
                or not c.is_contiguous() or c.dim() != 1):
            raise ValueError("cu_seqlens_q and cu_seqlens_k must be contiguous CUDA int32 vectors")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both hold B + 1 >= 2 offsets")
    a = VarlenArgs()
    a.q, a.k, a.v, a.o = q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr()
    a.lse = None if lse is None else lse.data_ptr()
    a.cu_seqlens_q, a.cu_seqlens_k = cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr()
    a.B, a.H, a.Hkv = cu_seqlens_q.numel() - 1, H, Hkv
    a.total_q, a.total_k, a.max_seqlen_q, a.d = q.shape[0], k.shape[0], int(max_seqlen_q), d
    a.round_mode, a.causal, a.pack_heads = MODES[round], int(causal), int(bool(pack_heads))
    a.max_splits = int(max_splits)
    return a


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int = 0, o=None, lse=None,
                    round: str = "rtne", causal: bool = False, return_lse: bool = False,
                    stream=None, workspace=None, max_ctas: int = 0, wait_limit_ms: int = 0,
                    events=None, pack_heads: bool = False, max_splits: int = 0):
    """Attention over a variable-length batch packed along the token axis.

    ``q``: [total_q, H, d], ``k``/``v``: [total_k, Hkv, d] (CUDA bf16, contiguous);
    ``cu_seqlens_q``/``cu_seqlens_k``: CUDA int32 [B + 1] row offsets of each sequence's
    queries and keys (checked on the device: bad offsets write nothing and are reported by
    :func:`device_status` as ATTN_ERR_INVALID_ARG).  Every sequence attends only to its own
    keys, with the causal mask (if asked) aligned at its own last query and key.
    ``max_seqlen_q``: an upper bound on any sequence's query length, used to size the grid
    (0: unknown).  ``lse``: optional fp32 [H, total_q].  ``pack_heads``: the query heads of
    each K/V head share one tile's rows (H / Hkv a power of two up to 32): same results, faster
    for short query chunks.  ``max_splits`` >= 2: when the items number fewer than the CTAs
    (a few long sequences, decoding), split each query block's keys into up to that many parts
    and merge them (deterministic; differs from the unsplit result by rounding).  Returns ``o``
    or ``(o, lse)``.
    """
    import torch
    if round not in MODES:
        raise ValueError("round must be rtne/rtna/rtz")
    if o is None:
        o = torch.empty_like(q)
    _check_out(o, q)
    if lse is None and return_lse:
        lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous()
                            or lse.numel() != q.shape[0] * q.shape[1]):
        raise ValueError("lse must be a contiguous CUDA fp32 tensor of H*total_q elements")
    a = _varlen_args(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, round, causal, pack_heads,
                     max_splits)
    opts = _opts(0, max_ctas, wait_limit_ms, events)
    lib = load()
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = lib.attn_fwd_varlen(ctypes.byref(a), ctypes.byref(opts) if opts else None, ws_ptr,
                             ws_bytes, _stream_ptr(stream, q.device))
    if st != 0:
        raise AttnError(st, "attn_fwd_varlen")
    return (o, lse) if (return_lse or lse is not None) else o


def _int32_cuda(t, name, dim):
    import torch
    if (not isinstance(t, torch.Tensor) or t.dtype != torch.int32 or not t.is_cuda
            or not t.is_contiguous() or t.dim() != dim):
        raise ValueError("%s must be a contiguous CUDA int32 tensor of %d dimension(s)" % (name, dim))


def attn_fwd_paged(q, k_cache, v_cache, cu_seqlens_q, seqlens_k, block_table, max_seqlen_q: int = 0,
                   o=None, lse=None, round: str = "rtne", causal: bool = False,
                   return_lse: bool = False, stream=None, workspace=None, max_ctas: int = 0,
                   wait_limit_ms: int = 0, events=None, pack_heads: bool = False, max_splits: int = 0):
    """Attention of packed queries over a paged K/V cache (``pack_heads`` and ``max_splits``
    as in :func:`attn_fwd_varlen`).

    ``q``: [total_q, H, d]; ``k_cache``/``v_cache``: [num_pages, page_size, Hkv, d] (CUDA bf16,
    contiguous; page_size a multiple of 128); ``cu_seqlens_q``: CUDA int32 [B + 1];
    ``seqlens_k``: CUDA int32 [B] keys per sequence; ``block_table``: CUDA int32
    [B, max_pages], the physical page of each sequence's page (entries past its last used
    page are not read).  Key j of sequence b is slot j % page_size of page
    block_table[b, j // page_size].  Causal: aligned at each sequence's last query and key.
    Bad offsets, lengths or page indices write nothing and are reported by
    :func:`device_status`.  Returns ``o`` or ``(o, lse)`` (lse: fp32 [H, total_q]).
    """
    import torch
    if round not in MODES:
        raise ValueError("round must be rtne/rtna/rtz")
    _check_tensors(q, k_cache, v_cache)
    if (q.dim() != 3 or k_cache.dim() != 4 or tuple(k_cache.shape) != tuple(v_cache.shape)
            or q.shape[2] != k_cache.shape[3]):
        raise ValueError("q must be [total_q, H, d] and k_cache, v_cache [num_pages, page_size, Hkv, d]")
    _int32_cuda(cu_seqlens_q, "cu_seqlens_q", 1)
    _int32_cuda(seqlens_k, "seqlens_k", 1)
    _int32_cuda(block_table, "block_table", 2)
    B = cu_seqlens_q.numel() - 1
    if B < 1 or seqlens_k.numel() != B or block_table.shape[0] != B:
        raise ValueError("cu_seqlens_q needs B + 1 offsets, seqlens_k B lengths, block_table B rows")
    if o is None:
        o = torch.empty_like(q)
    _check_out(o, q)
    if lse is None and return_lse:
        lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous()
                            or lse.numel() != q.shape[0] * q.shape[1]):
        raise ValueError("lse must be a contiguous CUDA fp32 tensor of H*total_q elements")
    a = PagedArgs()
    a.q, a.k_cache, a.v_cache, a.o = q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), o.data_ptr()
    a.lse = None if lse is None else lse.data_ptr()
    a.cu_seqlens_q, a.seqlens_k, a.block_table = (cu_seqlens_q.data_ptr(), seqlens_k.data_ptr(),
                                                  block_table.data_ptr())
    a.B, a.H, a.Hkv, a.total_q = B, q.shape[1], k_cache.shape[2], q.shape[0]
    a.num_pages, a.page_size, a.max_pages = k_cache.shape[0], k_cache.shape[1], block_table.shape[1]
    a.max_seqlen_q, a.d = int(max_seqlen_q), q.shape[2]
    a.round_mode, a.causal, a.pack_heads = MODES[round], int(causal), int(bool(pack_heads))
    a.max_splits = int(max_splits)
    opts = _opts(0, max_ctas, wait_limit_ms, events)
    lib = load()
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = lib.attn_fwd_paged(ctypes.byref(a), ctypes.byref(opts) if opts else None, ws_ptr,
                            ws_bytes, _stream_ptr(stream, q.device))
    if st != 0:
        raise AttnError(st, "attn_fwd_paged")
    return (o, lse) if (return_lse or lse is not None) else o


def workspace_size_ex(q, k, v, layout="bshd", causal=False, force_splits=0, max_ctas=0) -> int:
    """attn_fwd_ex_workspace_size for tensors shaped like q, k, v."""
    B, H, Hkv, Sq, Skv, d = _dims(q, k, v, layout, grouped=True)
    a = Args()
    a.B, a.H, a.Hkv, a.Sq, a.Skv, a.d, a.causal = B, H, Hkv, Sq, Skv, d, int(causal)
    a.layout = LAYOUTS[layout]
    o = _opts(force_splits, max_ctas)
    return int(load().attn_fwd_ex_workspace_size(ctypes.byref(a), ctypes.byref(o) if o else None))


def device_status(stream=None) -> tuple:
    """Synchronize and read/clear the device status word: (status, wait site)."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    site = ctypes.c_int32(0)
    st = load().attn_get_device_status(ctypes.c_void_p(s.cuda_stream), ctypes.byref(site))
    return int(st), int(site.value)


def attn_bwd(q, k, v, o, dout, lse, layout: str = "bshd", causal: bool = False, dq=None, dk=None,
             dv=None, workspace=None, stream=None, wait_limit_ms: int = 0, test_hooks: int = 0,
             deterministic: bool = False):
    """Gradients (dq, dk, dv) of softmax(Q K^T / sqrt(d)) V for the upstream gradient ``dout``,
    from the forward's inputs, output ``o`` and fp32 row log-sum-exp ``lse`` ([B][H][Sq], as
    returned by :func:`attn_fwd_ex` with ``return_lse``).  d = 128 or 64.  ``wait_limit_ms``
    bounds each wait in the kernel (0: 2000 ms); ``test_hooks`` is 0 for normal use (1 makes a
    bounded wait expire, to test that path).  ``deterministic``: dq bitwise reproducible too
    (dk and dv always are), at the cost of one fp32 dQ-sized workspace slice per 128-key tile.
    Returns (dq, dk, dv)."""
    import torch
    if layout not in LAYOUTS:
        raise ValueError("layout must be bshd or bhsd")
    _check_tensors(q, k, v)
    _check_tensors(o, dout, dout)
    B, H, Hkv, Sq, Skv, d = _dims(q, k, v, layout, grouped=True)
    for t in (o, dout):
        if tuple(t.shape) != tuple(q.shape):
            raise ValueError("o and dout must be shaped like q")
    if (lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous()
            or lse.numel() != B * H * Sq):
        raise ValueError("lse must be a contiguous CUDA fp32 tensor of B*H*Sq elements")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for g, ref in ((dq, q), (dk, k), (dv, v)):
        _check_out(g, ref)
    a = BwdArgs()
    a.q, a.k, a.v, a.o, a.dout = q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr()
    a.lse, a.dq, a.dk, a.dv = lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr()
    a.B, a.H, a.Hkv, a.Sq, a.Skv, a.d = B, H, Hkv, Sq, Skv, d
    a.layout, a.causal = LAYOUTS[layout], int(causal)
    a.wait_limit_ms, a.test_hooks = int(wait_limit_ms), int(test_hooks)
    a.deterministic = int(bool(deterministic))
    lib = load()
    need = int(lib.attn_bwd_workspace_size(ctypes.byref(a)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    nbytes = workspace.numel() * workspace.element_size()
    st = lib.attn_bwd(ctypes.byref(a), workspace.data_ptr(), nbytes, _stream_ptr(stream, q.device))
    if st != 0:
        raise AttnError(st, "attn_bwd")
    return dq, dk, dv


def attn_bwd_varlen(q, k, v, o, dout, lse, cu_seqlens_q, cu_seqlens_k, causal: bool = False, dq=None,
                    dk=None, dv=None, workspace=None, stream=None, wait_limit_ms: int = 0):
    """Gradients (dq, dk, dv) of :func:`attn_fwd_varlen`: q, o, dout [total_q, H, d]; k, v
    [total_k, Hkv, d]; lse fp32 [H, total_q] (attn_fwd_varlen's); cu_seqlens_q/k CUDA int32
    [B + 1].  Bad offsets write nothing and are reported by :func:`bwd_device_status`."""
    import torch
    _check_tensors(q, k, v)
    _check_tensors(o, dout, dout)
    if q.dim() != 3 or k.dim() != 3 or tuple(k.shape) != tuple(v.shape) or q.shape[2] != k.shape[2]:
        raise ValueError("q must be [total_q, H, d] and k, v [total_k, Hkv, d]")
    for t in (o, dout):
        if tuple(t.shape) != tuple(q.shape):
            raise ValueError("o and dout must be shaped like q")
    if (lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous()
            or lse.numel() != q.shape[0] * q.shape[1]):
        raise ValueError("lse must be a contiguous CUDA fp32 tensor of H*total_q elements")
    _int32_cuda(cu_seqlens_q, "cu_seqlens_q", 1)
    _int32_cuda(cu_seqlens_k, "cu_seqlens_k", 1)
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both hold B + 1 >= 2 offsets")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for g, ref in ((dq, q), (dk, k), (dv, v)):
        _check_out(g, ref)
    a = BwdVarlenArgs()
    a.q, a.k, a.v, a.o, a.dout = q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr()
    a.lse, a.dq, a.dk, a.dv = lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr()
    a.cu_seqlens_q, a.cu_seqlens_k = cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr()
    a.B, a.H, a.Hkv = cu_seqlens_q.numel() - 1, q.shape[1], k.shape[1]
    a.total_q, a.total_k, a.d = q.shape[0], k.shape[0], q.shape[2]
    a.causal, a.wait_limit_ms = int(causal), int(wait_limit_ms)
    lib = load()
    need = int(lib.attn_bwd_varlen_workspace_size(ctypes.byref(a)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    nbytes = workspace.numel() * workspace.element_size()
    st = lib.attn_bwd_varlen(ctypes.byref(a), workspace.data_ptr(), nbytes, _stream_ptr(stream, q.device))
    if st != 0:
        raise AttnError(st, "attn_bwd_varlen")
    return dq, dk, dv


def bwd_device_status(stream=None) -> tuple:
    """Synchronize and read/clear the backward kernel's status word: (status, wait site)."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    site = ctypes.c_int32(0)
    st = load().attn_bwd_get_device_status(ctypes.c_void_p(s.cuda_stream), ctypes.byref(site))
    return int(st), int(site.value)
