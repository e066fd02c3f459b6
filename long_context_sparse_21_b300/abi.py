"""ctypes binding of libcsa (include/csa.h): structs that mirror the C ABI and
one Python function per entry point, with the same name.

The binding only marshals arguments: it turns torch tensors into device
pointers, allocates outputs and workspaces with torch when the caller does not
pass them, and raises on a non-zero status.  Every step of the hot path runs in
the library's CUDA kernels; there is no Python or CPU fallback, and a missing
library is an error.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass, field

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa.so")

# enums (include/csa.h)
OK, ERR_INVALID_ARG, ERR_SHAPE, ERR_ALIGN, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = range(8)
F32, BF16, E4M3, E2M1 = range(4)
FMT_DENSE_F32, FMT_DENSE_BF16, FMT_KV_POOL_FP8, FMT_INDEX_POOL_BF16, FMT_INDEX_POOL_E2M1 = range(5)
COMPRESS_DENSE, COMPRESS_APPEND, COMPRESS_WINDOW, COMPRESS_DENSE_AB, COMPRESS_APPEND_AB = 0, 1, 2, 3, 4
ATTEND_BATCH_INVARIANT, ATTEND_WINDOW_ONLY = 1, 2
FLAG_OVERLAP_PREVIOUS = 0x100
FLAG_AFTER_APPEND = 0x200
ABI_VERSION = 2

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32


class CStore(ctypes.Structure):
    _fields_ = [("format", _i32), ("dim", _i32), ("base", _vp), ("capacity", _i32), ("page_entries", _i32),
                ("page_table", _vp), ("max_pages", _i32), ("num_pages", _i32)]


class CCacheWriteParams(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32), ("batch", _i32), ("n", _i32), ("first", _i32), ("src", _vp),
                ("dst", CStore), ("status", _vp)]


class CCompressParams(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32), ("mode", _i32), ("batch", _i32), ("m", _i32), ("dim", _i32),
                ("bias", _vp), ("n_tokens", _i32), ("k", _vp), ("k_dtype", _i32), ("g", _vp), ("g_dtype", _i32),
                ("seq_len", _vp), ("k_new", _vp), ("g_new", _vp), ("ring", _vp), ("ring_size", _i32),
                ("tail_gate", _vp), ("dst", CStore), ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t),
                ("norm", _vp), ("norm_eps", ctypes.c_float), ("rope_base", ctypes.c_float), ("flags", _i32),
                ("bias_b", _vp), ("k_b", _vp), ("g_b", _vp), ("k_new_b", _vp), ("g_new_b", _vp), ("tail_b", _vp),
                ("tail_gate_b", _vp)]


class CIndexParams(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32), ("num_queries", _i32), ("batch", _i32), ("heads", _i32),
                ("dim", _i32), ("m", _i32), ("max_pos", _i32), ("q", _vp), ("q_dtype", _i32), ("w", _vp),
                ("w_shared", _i32), ("pos", _vp), ("seq", _vp), ("keys", CStore), ("top_k", _i32),
                ("score_dtype", _i32), ("idx", _vp), ("cnt", _vp), ("scores_out", _vp), ("score_capacity", _i32),
                ("flags", _i32)]


class CAttendParams(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32), ("num_queries", _i32), ("batch", _i32), ("heads", _i32),
                ("dim", _i32), ("m", _i32), ("max_pos", _i32), ("q", _vp), ("q_dtype", _i32), ("pos", _vp),
                ("seq", _vp), ("idx", _vp), ("cnt", _vp), ("top_k", _i32), ("kv", CStore), ("window", _i32),
                ("win", _vp), ("win_dtype", _i32), ("win_ring", _i32), ("scale", ctypes.c_float), ("sink", _vp),
                ("out", _vp), ("out_dtype", _i32), ("lse", _vp), ("flags", _i32), ("q_norm", _vp), ("win_norm", _vp),
                ("norm_eps", ctypes.c_float), ("rope_base", ctypes.c_float)]


class CsaError(RuntimeError):
    def __init__(self, fn, status):
        detail = f"; CUDA: {lib().csa_last_cuda_error().decode()}" if status == ERR_CUDA else ""
        super().__init__(f"{fn}: status {status} ({status_string(status)}){detail}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libcsa; raises if it has not been built (no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libcsa.so not found at {LIB_PATH}; build it with "
                               "`python -m long_context_sparse_21_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        L.csa_abi_version.restype = ctypes.c_int
        L.csa_status_string.restype = ctypes.c_char_p
        L.csa_status_string.argtypes = [ctypes.c_int]
        L.csa_last_cuda_error.restype = ctypes.c_char_p
        L.csa_last_cuda_error.argtypes = []
        L.csa_page_bytes.restype = ctypes.c_size_t
        L.csa_page_bytes.argtypes = [_i32, _i32]
        for name, ptype in [("csa_cache_write", CCacheWriteParams), ("csa_compress", CCompressParams)]:
            f = getattr(L, name)
            f.restype = ctypes.c_int
            f.argtypes = [ctypes.POINTER(ptype), _vp]
        for name, ptype in [("csa_index_topk", CIndexParams), ("csa_index_score", CIndexParams),
                            ("csa_index_select", CIndexParams), ("csa_attend", CAttendParams),
                            ("hca_attend", CAttendParams)]:
            f = getattr(L, name)
            f.restype = ctypes.c_int
            f.argtypes = [ctypes.POINTER(ptype), _vp, ctypes.c_size_t, _vp]
        for name, ptype in [("csa_compress_workspace_size", CCompressParams),
                            ("csa_index_topk_workspace_size", CIndexParams),
                            ("csa_attend_workspace_size", CAttendParams),
                            ("hca_attend_workspace_size", CAttendParams)]:
            f = getattr(L, name)
            f.restype = ctypes.c_size_t
            f.argtypes = [ctypes.POINTER(ptype)]
        L.csa_index_topk_noalloc.restype = ctypes.c_int
        L.csa_index_topk_noalloc.argtypes = [ctypes.POINTER(CIndexParams), _vp]
        L.csa_index_topk_noalloc_status.restype = ctypes.c_int
        L.csa_index_topk_noalloc_status.argtypes = [ctypes.POINTER(_i32), _vp]
        L.csa_attend_plan.restype = ctypes.c_int
        L.csa_attend_plan.argtypes = [ctypes.POINTER(CAttendParams), _i32, ctypes.POINTER(_i32), ctypes.POINTER(_i32)]
        L.csa_workspace_status.restype = ctypes.c_int
        L.csa_workspace_status.argtypes = [_vp, ctypes.POINTER(_i32), _vp]
        L.csa_workspace_clear_status.restype = ctypes.c_int
        L.csa_workspace_clear_status.argtypes = [_vp, _vp]
        if L.csa_abi_version() != ABI_VERSION:
            raise RuntimeError("libcsa ABI version mismatch")
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().csa_status_string(status).decode()


def _check(fn, status):
    if status != OK:
        raise CsaError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t):
    return {torch.float32: F32, torch.bfloat16: BF16}[t.dtype]


# ------------------------------------------------------------------ stores (cache layouts)

def page_bytes(fmt: int, page_entries: int) -> int:
    return int(lib().csa_page_bytes(fmt, page_entries))


@dataclass
class Store:
    """A dense array or a paged pool of compressed entries (csa_store)."""
    fmt: int
    dim: int
    tensor: torch.Tensor              # owns the memory
    offset: int = 0                   # byte offset of the 1024-aligned base
    capacity: int = 0
    page_entries: int = 0
    page_table: torch.Tensor | None = None
    num_pages: int = 0                # pages the pool holds (page ids must be below it)
    keep: list = field(default_factory=list)

    @property
    def base_ptr(self) -> int:
        return self.tensor.data_ptr() + self.offset

    def c(self) -> CStore:
        return CStore(self.fmt, self.dim, self.base_ptr, self.capacity, self.page_entries,
                      None if self.page_table is None else self.page_table.data_ptr(),
                      0 if self.page_table is None else self.page_table.shape[1], self.num_pages)


def dense_store(t: torch.Tensor) -> Store:
    """t: [B, capacity, dim] float32 or bfloat16."""
    fmt = FMT_DENSE_F32 if t.dtype == torch.float32 else FMT_DENSE_BF16
    return Store(fmt, t.shape[2], t, 0, t.shape[1])


def make_pool(fmt: int, batch: int, entries: int, dim: int, page_entries: int = 2048, device="cuda",
              shuffle_seed: int | None = 0) -> Store:
    """Allocate a paged pool holding `entries` compressed entries for each of
    `batch` sequences, with a page table that (when shuffle_seed is given)
    scatters pages over the pool in a seeded random order."""
    P = page_entries
    per_seq = max(1, math.ceil(entries / P))
    n_pages = batch * per_seq
    nbytes = n_pages * page_bytes(fmt, P)
    raw = torch.empty(nbytes + 1024, dtype=torch.uint8, device=device)
    off = (-raw.data_ptr()) % 1024
    order = torch.arange(n_pages, dtype=torch.int32)
    if shuffle_seed is not None:
        g = torch.Generator().manual_seed(shuffle_seed)
        order = order[torch.randperm(n_pages, generator=g)]
    table = order.reshape(batch, per_seq).to(device)
    return Store(fmt, dim, raw, off, 0, P, table, n_pages)


def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A 1024-byte aligned uint8 workspace view of at least nbytes."""
    raw = torch.empty(nbytes + 1024, dtype=torch.uint8, device=device)
    off = (-raw.data_ptr()) % 1024
    return raw[off:off + nbytes]


# ------------------------------------------------------------------ entry points

def csa_cache_write(src: torch.Tensor, dst: Store, first: int = 0, stream=None, status=None):
    """Quantize float32 entries src [B, n, dim] into dst entries [first, first+n).
    status (optional): a workspace whose status word records a page id outside
    the pool."""
    assert src.dtype == torch.float32 and src.is_contiguous()
    p = CCacheWriteParams(ctypes.sizeof(CCacheWriteParams), src.shape[0], src.shape[1], first,
                          src.data_ptr(), dst.c(), None if status is None else status.data_ptr())
    _check("csa_cache_write", lib().csa_cache_write(ctypes.byref(p), _stream(stream)))


def compress_workspace(batch: int, dim: int, device="cuda") -> torch.Tensor:
    """A workspace for csa_compress (the library reports that no mode needs
    scratch; a minimal buffer is returned so callers can pass one uniformly)."""
    p = CCompressParams()
    p.struct_size = ctypes.sizeof(CCompressParams)
    p.mode, p.batch, p.dim, p.m = COMPRESS_APPEND, batch, dim, 1
    ws = alloc_workspace(max(int(lib().csa_compress_workspace_size(ctypes.byref(p))), 1024), device)
    ws.zero_()
    return ws


def csa_compress(dst: Store, bias: torch.Tensor, m: int, *, k=None, g=None, seq_len=None, k_new=None,
                 g_new=None, ring=None, tail_gate=None, workspace=None, stream=None, norm=None, norm_eps=0.0,
                 rope_base=0.0, overlap=False, bias_b=None, k_b=None, g_b=None, k_new_b=None, g_new_b=None,
                 tail_b=None, tail_gate_b=None):
    """Dense mode when k/g are given (k, g: [B, n, dim]); append mode when
    seq_len/k_new/g_new/ring/tail_gate are given (with a workspace from
    compress_workspace(); one is made on the fly when none is passed).
    norm (f32 [dim]) / norm_eps / rope_base: RMSNorm and RoPE of every pooled
    entry before it is stored.  bias_b with k_b/g_b (dense) or with
    k_new_b/g_new_b/tail_b/tail_gate_b (append; tails [B, 2m, dim]):
    overlapping compression, the b stream pooled over the previous block."""
    p = CCompressParams()
    p.struct_size = ctypes.sizeof(CCompressParams)
    p.m = m
    p.dim = dst.dim
    p.bias = bias.data_ptr()
    p.dst = dst.c()
    p.norm = None if norm is None else norm.data_ptr()
    p.norm_eps, p.rope_base = norm_eps, rope_base
    # overlap: may run alongside the previous kernel of the stream (csa.h states the condition)
    p.flags = FLAG_OVERLAP_PREVIOUS if overlap else 0
    if k is not None:
        p.mode = COMPRESS_DENSE
        p.batch = k.shape[0]
        p.n_tokens = k.shape[1]
        p.k, p.k_dtype = k.data_ptr(), _dtype_code(k)
        p.g, p.g_dtype = g.data_ptr(), _dtype_code(g)
        if bias_b is not None:
            p.mode, p.bias_b, p.k_b, p.g_b = COMPRESS_DENSE_AB, bias_b.data_ptr(), k_b.data_ptr(), g_b.data_ptr()
    else:
        p.mode = COMPRESS_APPEND
        if bias_b is not None:
            p.mode, p.bias_b = COMPRESS_APPEND_AB, bias_b.data_ptr()
            p.k_new_b, p.g_new_b = k_new_b.data_ptr(), g_new_b.data_ptr()
            p.tail_b, p.tail_gate_b = tail_b.data_ptr(), tail_gate_b.data_ptr()
        p.batch = k_new.shape[0]
        p.seq_len = seq_len.data_ptr()
        p.k_new = k_new.data_ptr()
        p.g_new = g_new.data_ptr()
        p.ring = ring.data_ptr()
        p.ring_size = ring.shape[1]
        p.tail_gate = tail_gate.data_ptr()
        if workspace is None:
            workspace = compress_workspace(p.batch, dst.dim, k_new.device)
        p.workspace, p.workspace_bytes = workspace.data_ptr(), workspace.numel()
    _check("csa_compress", lib().csa_compress(ctypes.byref(p), _stream(stream)))


def csa_window_append(seq_len, k_new, ring, stream=None, overlap=False):
    """Window-only decode append (a layer without a compressed branch): ring
    slot seq_len[b] % R <- k_new[b]."""
    p = CCompressParams()
    p.struct_size = ctypes.sizeof(CCompressParams)
    p.mode, p.batch, p.m, p.dim = COMPRESS_WINDOW, k_new.shape[0], 1, k_new.shape[1]
    p.seq_len, p.k_new, p.ring, p.ring_size = seq_len.data_ptr(), k_new.data_ptr(), ring.data_ptr(), ring.shape[1]
    p.bias = ring.data_ptr()  # not read in this mode (any aligned pointer)
    p.flags = FLAG_OVERLAP_PREVIOUS if overlap else 0
    _check("csa_compress", lib().csa_compress(ctypes.byref(p), _stream(stream)))


class IndexCall:
    """A prepared csa_index_topk call: outputs and workspace allocated once, so
    repeated launches (and CUDA-graph capture) allocate nothing."""

    def __init__(self, q, w, pos, keys: Store, top_k: int, m: int, max_pos: int, batch: int, seq=None,
                 score_dtype=F32, w_shared=False, scores_out=None, ws=None, idx=None, cnt=None, overlap=False,
                 after_append=False):
        T = q.shape[0]
        self.idx = idx if idx is not None else torch.empty((T, top_k), dtype=torch.int32, device=q.device)
        self.cnt = cnt if cnt is not None else torch.empty((T,), dtype=torch.int32, device=q.device)
        self._keep = (q, w, pos, keys, seq, scores_out)
        p = CIndexParams()
        p.struct_size = ctypes.sizeof(CIndexParams)
        p.num_queries, p.batch, p.heads, p.dim = T, batch, q.shape[1], q.shape[2]
        p.m, p.max_pos = m, max_pos
        p.q, p.q_dtype = q.data_ptr(), _dtype_code(q)
        p.w, p.w_shared = w.data_ptr(), int(w_shared)
        p.pos = pos.data_ptr()
        p.seq = None if seq is None else seq.data_ptr()
        p.keys = keys.c()
        p.top_k = top_k
        p.score_dtype = score_dtype
        p.idx, p.cnt = self.idx.data_ptr(), self.cnt.data_ptr()
        if scores_out is not None:
            p.scores_out, p.score_capacity = scores_out.data_ptr(), scores_out.shape[1]
        # overlap: the kernels may start before the previous kernel of the
        # stream ends; it must not write q, w, pos or seq (csa.h)
        # after_append: the previous kernel is the decode append of `keys`,
        # which writes at most each query's last visible key (csa.h)
        p.flags = (FLAG_OVERLAP_PREVIOUS if overlap else 0) | (FLAG_AFTER_APPEND if after_append else 0)
        self.p = p
        nbytes = lib().csa_index_topk_workspace_size(ctypes.byref(p))
        if nbytes == 0 and T > 0:
            # surface the validation status
            _check("csa_index_topk", lib().csa_index_topk(ctypes.byref(p), None, 0, _stream(None)))
        if ws is not None and ws.numel() >= nbytes:
            self.ws = ws  # a caller-owned workspace (shared between calls that run in order)
        else:
            self.ws = alloc_workspace(max(int(nbytes), 1024), q.device)
        lib().csa_workspace_clear_status(_ptr(self.ws), _stream(None))

    @staticmethod
    def workspace_bytes(T, heads, dim, m, max_pos, keys: "Store", score_dtype=F32) -> int:
        """csa_index_topk_workspace_size for a call of this shape."""
        p = CIndexParams(struct_size=ctypes.sizeof(CIndexParams), num_queries=T, batch=1, heads=heads, dim=dim, m=m,
                         max_pos=max_pos, q=16, q_dtype=BF16 if keys.fmt == FMT_INDEX_POOL_BF16 else F32, w=16,
                         pos=16, keys=keys.c(), top_k=1, score_dtype=score_dtype, idx=16, cnt=16)
        return int(lib().csa_index_topk_workspace_size(ctypes.byref(p)))

    def __call__(self, stream=None):
        _check("csa_index_topk", lib().csa_index_topk(ctypes.byref(self.p), _ptr(self.ws), self.ws.numel(),
                                                      _stream(stream)))
        return self.idx, self.cnt

    def score(self, stream=None):
        """Step 2 only (scores into the workspace)."""
        _check("csa_index_score", lib().csa_index_score(ctypes.byref(self.p), _ptr(self.ws), self.ws.numel(),
                                                        _stream(stream)))

    def select(self, stream=None):
        """Step 3 only (selection from the workspace scores)."""
        _check("csa_index_select", lib().csa_index_select(ctypes.byref(self.p), _ptr(self.ws), self.ws.numel(),
                                                          _stream(stream)))
        return self.idx, self.cnt

    def status(self) -> int:
        out = _i32(0)
        _check("csa_workspace_status", lib().csa_workspace_status(_ptr(self.ws), ctypes.byref(out), _stream(None)))
        return out.value


def csa_index_topk_noalloc(p: CIndexParams, stream=None):
    """The no-allocation indexer + top-k on a prepared parameter struct."""
    _check("csa_index_topk_noalloc", lib().csa_index_topk_noalloc(ctypes.byref(p), _stream(stream)))


def csa_index_topk_noalloc_status(stream=None) -> int:
    """Status word of the last csa_index_topk_noalloc call on this device."""
    out = _i32(0)
    _check("csa_index_topk_noalloc_status", lib().csa_index_topk_noalloc_status(ctypes.byref(out), _stream(stream)))
    return out.value


def workspace_status(ws: torch.Tensor, stream=None) -> int:
    """Status word of a workspace (csa_workspace_status)."""
    out = _i32(0)
    _check("csa_workspace_status", lib().csa_workspace_status(_ptr(ws), ctypes.byref(out), _stream(stream)))
    return out.value


def csa_index_topk(q, w, pos, keys: Store, top_k: int, m: int, max_pos: int, batch: int, **kw):
    """One-shot lightning indexer + top-k; returns (idx [T, top_k], cnt [T])."""
    return IndexCall(q, w, pos, keys, top_k, m, max_pos, batch, **kw)()


class AttendCall:
    """A prepared csa_attend / hca_attend call (outputs and workspace owned)."""

    def __init__(self, sparse: bool, q, pos, kv: Store, window: int, win, scale: float, m: int, max_pos: int,
                 batch: int, idx=None, cnt=None, seq=None, sink=None, out_dtype=None, with_lse=True, out=None,
                 batch_invariant: bool = False, q_norm=None, win_norm=None, norm_eps: float = 0.0,
                 rope_base: float = 0.0, overlap: bool = False, window_only: bool = False):
        T, H, D = q.shape
        self.sparse = sparse
        out_dtype = out_dtype or q.dtype
        self.out = out if out is not None else torch.empty((T, H, D), dtype=out_dtype, device=q.device)
        self.lse = torch.empty((T, H), dtype=torch.float32, device=q.device) if with_lse else None
        self._keep = (q, pos, kv, win, idx, cnt, seq, sink, q_norm, win_norm)
        p = CAttendParams()
        p.struct_size = ctypes.sizeof(CAttendParams)
        p.num_queries, p.batch, p.heads, p.dim = T, batch, H, D
        p.m, p.max_pos = m, max_pos
        p.q, p.q_dtype = q.data_ptr(), _dtype_code(q)
        p.pos = pos.data_ptr()
        p.seq = None if seq is None else seq.data_ptr()
        if sparse:
            p.idx, p.cnt, p.top_k = idx.data_ptr(), cnt.data_ptr(), idx.shape[1]
        if kv is not None:
            p.kv = kv.c()
        p.window = window
        p.win, p.win_dtype, p.win_ring = win.data_ptr(), _dtype_code(win), win.shape[1]
        p.scale = scale
        p.sink = None if sink is None else sink.data_ptr()
        p.out, p.out_dtype = self.out.data_ptr(), _dtype_code(self.out)
        p.lse = None if self.lse is None else self.lse.data_ptr()
        # overlap: the kernel may start before the previous kernel of the
        # stream ends; it must not write q or seq (csa.h)
        p.flags = (ATTEND_BATCH_INVARIANT if batch_invariant else 0) | (FLAG_OVERLAP_PREVIOUS if overlap else 0) | \
            (ATTEND_WINDOW_ONLY if window_only else 0)
        p.q_norm = None if q_norm is None else q_norm.data_ptr()
        p.win_norm = None if win_norm is None else win_norm.data_ptr()
        p.norm_eps, p.rope_base = norm_eps, rope_base
        self.p = p
        fn = lib().csa_attend_workspace_size if sparse else lib().hca_attend_workspace_size
        nbytes = fn(ctypes.byref(p))
        if nbytes == 0 and T > 0:
            self.ws = alloc_workspace(1024, q.device)
            self()  # raises with the validation status
        self.ws = alloc_workspace(max(int(nbytes), 1024), q.device)
        lib().csa_workspace_clear_status(_ptr(self.ws), _stream(None))

    def plan(self):
        """(splits per query, merge): merge 0 = one split, 1 = in a cluster
        inside the kernel, 2 = a second (combine) kernel."""
        sp, mg = _i32(0), _i32(0)
        _check("csa_attend_plan", lib().csa_attend_plan(ctypes.byref(self.p), int(self.sparse), ctypes.byref(sp),
                                                        ctypes.byref(mg)))
        return sp.value, mg.value

    def launches(self) -> int:
        """Kernel launches of one call."""
        return 2 if self.plan()[1] == 2 else 1

    def __call__(self, stream=None):
        fn = lib().csa_attend if self.sparse else lib().hca_attend
        name = "csa_attend" if self.sparse else "hca_attend"
        _check(name, fn(ctypes.byref(self.p), _ptr(self.ws), self.ws.numel(), _stream(stream)))
        return self.out, self.lse

    def status(self) -> int:
        out = _i32(0)
        _check("csa_workspace_status", lib().csa_workspace_status(_ptr(self.ws), ctypes.byref(out), _stream(None)))
        return out.value


def csa_attend(q, pos, idx, cnt, kv: Store, window: int, win, scale: float, m: int, max_pos: int, batch: int,
               **kw):
    return AttendCall(True, q, pos, kv, window, win, scale, m, max_pos, batch, idx=idx, cnt=cnt, **kw)()


def hca_attend(q, pos, kv: Store, window: int, win, scale: float, m: int, max_pos: int, batch: int, **kw):
    return AttendCall(False, q, pos, kv, window, win, scale, m, max_pos, batch, **kw)()
