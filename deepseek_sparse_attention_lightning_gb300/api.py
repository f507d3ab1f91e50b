"""ctypes binding of libdsa.so: the C ABI of include/dsa.h, same names.

Argument marshalling only: every step of the decode path runs in the
library's CUDA kernels.  Tensors are torch CUDA tensors (torch provides device
memory and streams); each wrapper checks dtype, device and contiguity, passes
raw pointers, and raises ``DSAError`` on a non-zero status.  There is no CPU
fallback: without the built library every call raises.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import c_float, c_int32, c_int64, c_size_t, c_void_p

import torch

from . import build as _build

DSA_OK = 0
STATUS_NAMES = {0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_UNSUPPORTED",
                3: "DSA_ERR_WORKSPACE", 4: "DSA_ERR_CUDA", 5: "DSA_ERR_DEVICE_CHECK",
                6: "DSA_ERR_TIMEOUT"}
PAGE_SIZE = 64


class DSAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class DecodeDesc(ctypes.Structure):
    _fields_ = [("batch", c_int32), ("q_per_req", c_int32), ("num_heads", c_int32),
                ("topk", c_int32), ("page_size", c_int32), ("max_pages", c_int32),
                ("num_pages", c_int32), ("seqlens", c_void_p), ("page_table", c_void_p)]


class StepRing(ctypes.Structure):
    """The caller-owned resources of a ring of decode steps (dsa_step_ring)."""
    _fields_ = [("dev_in", c_void_p * 2), ("out", c_void_p * 2), ("ws", c_void_p),
                ("ws_bytes", c_size_t), ("copy_in_stream", c_void_p), ("copy_out_stream", c_void_p),
                ("ev_in", c_void_p * 2), ("ev_done", c_void_p * 2), ("ev_out", c_void_p * 2),
                ("step", c_int64)]


class StepLayout(ctypes.Structure):
    """Byte offsets of a decode step's inputs in one host/device block."""
    _fields_ = [("q_fp8", c_size_t), ("q_scale", c_size_t), ("w", c_size_t), ("q", c_size_t),
                ("seqlens", c_size_t), ("page_table", c_size_t), ("bytes", c_size_t)]


_SIGS = {
    "dsa_indexer_logits": (c_int32, [ctypes.POINTER(DecodeDesc), c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_void_p, c_int64, c_void_p]),
    "dsa_topk": (c_int32, [ctypes.POINTER(DecodeDesc), c_void_p, c_int64, c_void_p, c_void_p,
                           c_size_t, c_void_p]),
    "dsa_topk_workspace_bytes": (c_size_t, [ctypes.POINTER(DecodeDesc), c_int64]),
    "dsa_topk_noalloc": (c_int32, [ctypes.POINTER(DecodeDesc), c_void_p, c_int64, c_void_p,
                                   c_void_p]),
    "dsa_sparse_mla_decode_split": (c_int32, [ctypes.POINTER(DecodeDesc), c_void_p, c_void_p,
                                              c_void_p, c_int32, c_float, c_void_p, c_void_p,
                                              c_void_p]),
    "dsa_merge": (c_int32, [c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "dsa_cache_write": (c_int32, [ctypes.POINTER(DecodeDesc), c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_void_p, c_void_p]),
    "dsa_decode_fused": (c_int32, [ctypes.POINTER(DecodeDesc), c_void_p, c_void_p, c_void_p,
                                   c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                   c_float, c_int32, c_int32, c_void_p, c_void_p, c_size_t,
                                   c_void_p]),
    "dsa_decode_fused_timed": (c_int32, [ctypes.POINTER(DecodeDesc), c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_float, c_int32, c_int32, c_void_p, c_void_p,
                                         c_size_t, c_void_p, ctypes.POINTER(c_void_p)]),
    "dsa_decode_fused_write": (c_int32, [ctypes.POINTER(DecodeDesc), c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_void_p, c_void_p, c_float, c_int32, c_int32,
                                         c_void_p, c_void_p, c_size_t, c_void_p]),
    "dsa_latent_to_fp8": (c_int32, [c_void_p, c_int64, c_void_p, c_void_p]),
    "dsa_sparse_mla_decode_split_fp8": (c_int32, [ctypes.POINTER(DecodeDesc), c_void_p, c_void_p,
                                                  c_void_p, c_int32, c_float, c_void_p, c_void_p,
                                                  c_void_p]),
    "dsa_decode_fused_fp8kv": (c_int32, [ctypes.POINTER(DecodeDesc), c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_float, c_int32, c_int32, c_void_p, c_void_p,
                                         c_size_t, c_void_p]),
    "dsa_decode_mli": (c_int32, [ctypes.POINTER(DecodeDesc), c_void_p, c_void_p, c_void_p,
                                 c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                 c_float, c_int32, c_int32, c_void_p, c_void_p, c_size_t,
                                 c_void_p]),
    "dsa_num_splits_mli": (c_int32, [ctypes.POINTER(DecodeDesc)]),
    "dsa_step_layout_get": (c_int32, [c_int32, c_int32, c_int32, c_int32,
                                      ctypes.POINTER(StepLayout)]),
    "dsa_decode_step_host": (c_int32, [ctypes.POINTER(DecodeDesc), c_void_p, c_void_p, c_void_p,
                                       c_void_p, c_void_p, c_float, c_int32, c_int32, c_void_p,
                                       c_void_p, c_void_p, c_size_t, c_void_p]),
    "dsa_decode_step_ring": (c_int32, [ctypes.POINTER(DecodeDesc), ctypes.POINTER(StepRing),
                                       c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_float,
                                       c_int32, c_int32, c_void_p]),
    "dsa_workspace_bytes": (c_size_t, [ctypes.POINTER(DecodeDesc), c_int32, c_int32]),
    "dsa_num_splits_auto": (c_int32, [ctypes.POINTER(DecodeDesc)]),
    "dsa_status_str": (ctypes.c_char_p, [c_int32]),
    "dsa_get_device_error": (c_int32, [c_void_p]),
    "dsa_version": (ctypes.c_char_p, []),
    "dsa_debug_set_wait_cycles": (c_int32, [c_int64]),
}

_lib = None


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Loads libdsa.so (built in-tree by ``build.build()``); raises if absent."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libdsa.so not built at {path}: run "
                               "`python -c 'import __graft_entry__ as g; g.build()'` first")
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status: int, where: str):
    if status != DSA_OK:
        raise DSAError(status, where)


def _ptr(t, dtype, name, ndim=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name}: expected {ndim} dims, got {t.dim()}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _u16(t: torch.Tensor, name):
    if t.dtype == torch.bfloat16:
        return _ptr(t, torch.bfloat16, name)
    return _ptr(t, torch.int16, name)


def make_desc(seqlens: torch.Tensor, page_table: torch.Tensor, q_per_req: int, num_heads: int,
              topk: int, num_pages: int) -> DecodeDesc:
    """Descriptor of one decode batch (keeps no reference to the tensors)."""
    B = int(seqlens.shape[0])
    return DecodeDesc(batch=B, q_per_req=int(q_per_req), num_heads=int(num_heads),
                      topk=int(topk), page_size=PAGE_SIZE, max_pages=int(page_table.shape[1]),
                      num_pages=int(num_pages),
                      seqlens=_ptr(seqlens, torch.int32, "seqlens", 1),
                      page_table=_ptr(page_table, torch.int32, "page_table", 2))


def dsa_indexer_logits(desc, q_fp8, q_scale, w, k_fp8, k_scale, logits, ld=None, stream=None):
    ld = int(logits.shape[-1]) if ld is None else int(ld)
    _check(lib().dsa_indexer_logits(
        ctypes.byref(desc), _ptr(q_fp8, torch.uint8, "q_fp8"), _ptr(q_scale, torch.float32, "q_scale"),
        _ptr(w, torch.float32, "w"), _ptr(k_fp8, torch.uint8, "k_fp8"),
        _ptr(k_scale, torch.float32, "k_scale"), _ptr(logits, torch.float32, "logits"), ld,
        _stream(stream)), "dsa_indexer_logits")


def dsa_topk_workspace_bytes(desc, ld) -> int:
    return int(lib().dsa_topk_workspace_bytes(ctypes.byref(desc), int(ld)))


def dsa_topk(desc, logits, topk_idx, ws, ld=None, stream=None):
    ld = int(logits.shape[-1]) if ld is None else int(ld)
    _check(lib().dsa_topk(ctypes.byref(desc), _ptr(logits, torch.float32, "logits"), ld,
                          _ptr(topk_idx, torch.int32, "topk_idx"), _ptr(ws, torch.uint8, "ws"),
                          ws.numel(), _stream(stream)), "dsa_topk")


def dsa_topk_noalloc(desc, logits, topk_idx, ld=None, stream=None):
    """dsa_topk with the library's fixed device scratch instead of a workspace
    (for callers that cannot allocate device memory; see include/dsa.h)."""
    ld = int(logits.shape[-1]) if ld is None else int(ld)
    _check(lib().dsa_topk_noalloc(ctypes.byref(desc), _ptr(logits, torch.float32, "logits"), ld,
                                  _ptr(topk_idx, torch.int32, "topk_idx"), _stream(stream)),
           "dsa_topk_noalloc")


def dsa_sparse_mla_decode_split(desc, q, kv, topk_idx, num_splits, sm_scale, mid_o, mid_lse,
                                stream=None):
    _check(lib().dsa_sparse_mla_decode_split(
        ctypes.byref(desc), _u16(q, "q"), _u16(kv, "kv"), _ptr(topk_idx, torch.int32, "topk_idx"),
        int(num_splits), float(sm_scale), _ptr(mid_o, torch.float32, "mid_o"),
        _ptr(mid_lse, torch.float32, "mid_lse"), _stream(stream)), "dsa_sparse_mla_decode_split")


def dsa_cache_write(desc, new_latent, new_index_k, kv, k_fp8, k_scale, stream=None):
    _check(lib().dsa_cache_write(ctypes.byref(desc), _ptr(new_latent, torch.bfloat16, "new_latent"),
                                 _ptr(new_index_k, torch.bfloat16, "new_index_k"),
                                 _ptr(kv, torch.bfloat16, "kv"), _ptr(k_fp8, torch.uint8, "k_fp8"),
                                 _ptr(k_scale, torch.float32, "k_scale"), _stream(stream)),
           "dsa_cache_write")


def dsa_merge(num_rows, num_splits, mid_o, mid_lse, out, out_lse=None, stream=None):
    _check(lib().dsa_merge(int(num_rows), int(num_splits), _ptr(mid_o, torch.float32, "mid_o"),
                           _ptr(mid_lse, torch.float32, "mid_lse"), _ptr(out, torch.float32, "out"),
                           _ptr(out_lse, torch.float32, "out_lse"), _stream(stream)), "dsa_merge")


def dsa_workspace_bytes(desc, max_seqlen, num_splits=0) -> int:
    return int(lib().dsa_workspace_bytes(ctypes.byref(desc), int(max_seqlen), int(num_splits)))


def dsa_num_splits_auto(desc) -> int:
    return int(lib().dsa_num_splits_auto(ctypes.byref(desc)))


def dsa_decode_fused(desc, q_fp8, q_scale, w, k_fp8, k_scale, q, kv, out, ws, max_seqlen,
                     sm_scale, num_splits=0, topk_in=None, topk_out=None, stream=None,
                     stage_events=None):
    """``stage_events``: optional list of 5 torch.cuda.Event (timing enabled)."""
    if stage_events is not None:
        arr = (c_void_p * 5)(*[ev.cuda_event if ev is not None else None for ev in stage_events])
        _check(lib().dsa_decode_fused_timed(
            ctypes.byref(desc), _ptr(q_fp8, torch.uint8, "q_fp8"),
            _ptr(q_scale, torch.float32, "q_scale"), _ptr(w, torch.float32, "w"),
            _ptr(k_fp8, torch.uint8, "k_fp8"), _ptr(k_scale, torch.float32, "k_scale"),
            _u16(q, "q"), _u16(kv, "kv"), _ptr(topk_in, torch.int32, "topk_in"),
            _ptr(topk_out, torch.int32, "topk_out"), float(sm_scale), int(num_splits),
            int(max_seqlen), _ptr(out, torch.float32, "out"), _ptr(ws, torch.uint8, "ws"),
            ws.numel(), _stream(stream), arr), "dsa_decode_fused_timed")
        return
    _check(lib().dsa_decode_fused(
        ctypes.byref(desc), _ptr(q_fp8, torch.uint8, "q_fp8"), _ptr(q_scale, torch.float32, "q_scale"),
        _ptr(w, torch.float32, "w"), _ptr(k_fp8, torch.uint8, "k_fp8"),
        _ptr(k_scale, torch.float32, "k_scale"), _u16(q, "q"), _u16(kv, "kv"),
        _ptr(topk_in, torch.int32, "topk_in"), _ptr(topk_out, torch.int32, "topk_out"),
        float(sm_scale), int(num_splits), int(max_seqlen), _ptr(out, torch.float32, "out"),
        _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)), "dsa_decode_fused")


def dsa_decode_fused_write(desc, new_latent, new_index_k, q_fp8, q_scale, w, k_fp8, k_scale, q,
                           kv, out, ws, max_seqlen, sm_scale, num_splits=0, topk_in=None,
                           topk_out=None, stream=None):
    _check(lib().dsa_decode_fused_write(
        ctypes.byref(desc), _ptr(new_latent, torch.bfloat16, "new_latent"),
        _ptr(new_index_k, torch.bfloat16, "new_index_k"), _ptr(q_fp8, torch.uint8, "q_fp8"),
        _ptr(q_scale, torch.float32, "q_scale"), _ptr(w, torch.float32, "w"),
        _ptr(k_fp8, torch.uint8, "k_fp8"), _ptr(k_scale, torch.float32, "k_scale"), _u16(q, "q"),
        _u16(kv, "kv"), _ptr(topk_in, torch.int32, "topk_in"),
        _ptr(topk_out, torch.int32, "topk_out"), float(sm_scale), int(num_splits),
        int(max_seqlen), _ptr(out, torch.float32, "out"), _ptr(ws, torch.uint8, "ws"),
        ws.numel(), _stream(stream)), "dsa_decode_fused_write")


def dsa_latent_to_fp8(kv, kv8, stream=None):
    rows = int(kv.shape[0])
    if kv8.shape != (rows, 656):
        raise ValueError("kv8 must be [rows, 656]")
    _check(lib().dsa_latent_to_fp8(_u16(kv, "kv"), rows, _ptr(kv8, torch.uint8, "kv8"),
                                   _stream(stream)), "dsa_latent_to_fp8")


def dsa_sparse_mla_decode_split_fp8(desc, q, kv8, topk_idx, num_splits, sm_scale, mid_o, mid_lse,
                                    stream=None):
    _check(lib().dsa_sparse_mla_decode_split_fp8(
        ctypes.byref(desc), _u16(q, "q"), _ptr(kv8, torch.uint8, "kv8"),
        _ptr(topk_idx, torch.int32, "topk_idx"), int(num_splits), float(sm_scale),
        _ptr(mid_o, torch.float32, "mid_o"), _ptr(mid_lse, torch.float32, "mid_lse"),
        _stream(stream)), "dsa_sparse_mla_decode_split_fp8")


def dsa_decode_fused_fp8kv(desc, q_fp8, q_scale, w, k_fp8, k_scale, q, kv8, out, ws, max_seqlen,
                           sm_scale, num_splits=0, topk_in=None, topk_out=None, stream=None):
    _check(lib().dsa_decode_fused_fp8kv(
        ctypes.byref(desc), _ptr(q_fp8, torch.uint8, "q_fp8"), _ptr(q_scale, torch.float32, "q_scale"),
        _ptr(w, torch.float32, "w"), _ptr(k_fp8, torch.uint8, "k_fp8"),
        _ptr(k_scale, torch.float32, "k_scale"), _u16(q, "q"), _ptr(kv8, torch.uint8, "kv8"),
        _ptr(topk_in, torch.int32, "topk_in"), _ptr(topk_out, torch.int32, "topk_out"),
        float(sm_scale), int(num_splits), int(max_seqlen), _ptr(out, torch.float32, "out"),
        _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)), "dsa_decode_fused_fp8kv")


def dsa_decode_mli(desc, q_fp8, q_scale, w, k_fp8, k_scale, q, kv, topk_prev, topk_next, out, ws,
                   max_seqlen, sm_scale, num_splits=0, stream=None):
    """One layer of the Multi-layer Indexer schedule: attention over
    ``topk_prev`` while this layer's indexer and top-k write ``topk_next``
    (see include/dsa.h)."""
    _check(lib().dsa_decode_mli(
        ctypes.byref(desc), _ptr(q_fp8, torch.uint8, "q_fp8"), _ptr(q_scale, torch.float32, "q_scale"),
        _ptr(w, torch.float32, "w"), _ptr(k_fp8, torch.uint8, "k_fp8"),
        _ptr(k_scale, torch.float32, "k_scale"), _u16(q, "q"), _u16(kv, "kv"),
        _ptr(topk_prev, torch.int32, "topk_prev"), _ptr(topk_next, torch.int32, "topk_next"),
        float(sm_scale), int(num_splits), int(max_seqlen), _ptr(out, torch.float32, "out"),
        _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)), "dsa_decode_mli")


def dsa_num_splits_mli(desc) -> int:
    return int(lib().dsa_num_splits_mli(ctypes.byref(desc)))


def dsa_step_layout_get(batch, q_per_req, num_heads, max_pages) -> StepLayout:
    lay = StepLayout()
    _check(lib().dsa_step_layout_get(int(batch), int(q_per_req), int(num_heads), int(max_pages),
                                     ctypes.byref(lay)), "dsa_step_layout_get")
    return lay


def step_views(block: torch.Tensor, layout: StepLayout, batch, q_per_req, num_heads, max_pages):
    """Typed views of each step input inside a uint8 block (host or device)
    laid out by ``dsa_step_layout_get``."""
    if block.dtype != torch.uint8 or block.dim() != 1 or block.numel() < layout.bytes:
        raise ValueError("block must be a 1-D uint8 tensor of at least layout.bytes")
    T = int(batch) * int(q_per_req)
    parts = (("q_fp8", torch.uint8, (T, 64, 128)), ("q_scale", torch.float32, (T,)),
             ("w", torch.float32, (T, 64)), ("q", torch.bfloat16, (T, int(num_heads), 576)),
             ("seqlens", torch.int32, (int(batch),)),
             ("page_table", torch.int32, (int(batch), int(max_pages))))
    views = {}
    for name, dtype, shape in parts:
        off = getattr(layout, name)
        n = 1
        for x in shape:
            n *= x
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        views[name] = block[off:off + nbytes].view(dtype).view(shape)
    return views


class HostStepPipeline:
    """Decode layers whose per-step inputs start in host memory and whose
    outputs end there, with the copies of one step overlapping the layers of
    its neighbours: the resources of a ``dsa_decode_step_ring`` (two device
    input blocks laid out by ``dsa_step_layout_get``, two device outputs, the
    workspace, a copy-in and a copy-out stream, six events), and one library
    call per step.  Step i (slot i % 2) copies its block in once the layer of
    step i - 2 is done reading that slot, its layer waits for that copy and
    for the output copy of step i - 2, and its output is copied out after its
    layer; so while layer i runs, the inputs of step i + 1 come in and the
    output of step i - 1 goes out.  The caches and the workspace stay in
    device memory.  A host block may be rewritten once the copy of the step
    that read it is done (``input_copied(i)``); ``host_out`` of step i is
    valid once ``output_copied(i)`` (or ``drain``) has been waited on.  Every
    step of one pipeline runs its layer on the same stream (the steps share
    one workspace); another stream raises.
    """

    def __init__(self, batch, q_per_req, num_heads, topk, max_pages, num_pages, max_seqlen,
                 sm_scale, num_splits=0, device=None):
        device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        self.layout = dsa_step_layout_get(batch, q_per_req, num_heads, max_pages)
        self.dims = (batch, q_per_req, num_heads, max_pages)
        self.dev_in = [torch.empty(self.layout.bytes, dtype=torch.uint8, device=device)
                       for _ in range(2)]
        self.views = [step_views(d, self.layout, *self.dims) for d in self.dev_in]
        T = batch * q_per_req
        self.out = [torch.empty((T, num_heads, 512), dtype=torch.float32, device=device)
                    for _ in range(2)]
        self.desc = make_desc(self.views[0]["seqlens"], self.views[0]["page_table"], q_per_req,
                              num_heads, topk, num_pages)
        self.splits = num_splits if num_splits else dsa_num_splits_auto(self.desc)
        self.ws = torch.empty(dsa_workspace_bytes(self.desc, max_seqlen, self.splits),
                              dtype=torch.uint8, device=device)
        self.max_seqlen, self.sm_scale = int(max_seqlen), float(sm_scale)
        self.h2d = torch.cuda.Stream(device)
        self.d2h = torch.cuda.Stream(device)
        mk = lambda: [torch.cuda.Event() for _ in range(2)]
        self.ev_in, self.ev_done, self.ev_out = mk(), mk(), mk()
        with torch.cuda.device(device):
            for e in self.ev_in + self.ev_done + self.ev_out:
                e.record()   # creates the event (torch creates them on first record)
            torch.cuda.current_stream().synchronize()
        r = StepRing()
        for b in range(2):
            r.dev_in[b] = _ptr(self.dev_in[b], torch.uint8, "dev_in")
            r.out[b] = _ptr(self.out[b], torch.float32, "out")
            r.ev_in[b], r.ev_done[b], r.ev_out[b] = (self.ev_in[b].cuda_event,
                                                     self.ev_done[b].cuda_event,
                                                     self.ev_out[b].cuda_event)
        r.ws, r.ws_bytes = _ptr(self.ws, torch.uint8, "ws"), self.ws.numel()
        r.copy_in_stream, r.copy_out_stream = self.h2d.cuda_stream, self.d2h.cuda_stream
        r.step = 0
        self.ring = r
        self._ring_fn = lib().dsa_decode_step_ring
        self._calls = {}
        self._stream = None

    @property
    def steps(self) -> int:
        return int(self.ring.step)

    def submit(self, host_in, host_out, k_fp8, k_scale, kv, stream=None):
        """Queues one step: host_in (a pinned uint8 block) -> layer over the
        given caches -> host_out (pinned float32 [T, H, 512])."""
        comp = torch.cuda.current_stream() if stream is None else stream
        sid = _stream(comp)
        if self._stream is None:
            self._stream = sid
        elif sid != self._stream:
            raise ValueError("every step of a HostStepPipeline runs on the same stream")
        # The call's arguments are checked and packed once per host buffer
        # pair, cache set and stream; later steps only issue the call.
        key = (host_in.data_ptr(), host_out.data_ptr(), k_fp8.data_ptr(), k_scale.data_ptr(),
               kv.data_ptr(), k_fp8.dtype, k_scale.dtype, kv.dtype, sid)
        args = self._calls.get(key)
        if args is None:
            if host_in.dtype != torch.uint8 or host_in.is_cuda or host_in.numel() < self.layout.bytes:
                raise ValueError("host_in: a host uint8 block of at least layout.bytes")
            if host_out.is_cuda or host_out.dtype != torch.float32 or host_out.shape != self.out[0].shape:
                raise ValueError("host_out: a host float32 tensor shaped like the output")
            args = (ctypes.byref(self.desc), ctypes.byref(self.ring),
                    _host_ptr(host_in, torch.uint8, "host_in"),
                    _host_ptr(host_out, torch.float32, "host_out"),
                    _ptr(k_fp8, torch.uint8, "k_fp8"), _ptr(k_scale, torch.float32, "k_scale"),
                    _u16(kv, "kv"), self.sm_scale, self.splits, self.max_seqlen, sid)
            self._calls[key] = args
        _check(self._ring_fn(*args), "dsa_decode_step_ring")

    def input_copied(self, step):
        """Event after which the host block of `step` may be rewritten (valid
        until step + 2 is submitted)."""
        return self.ev_in[step % 2]

    def output_copied(self, step):
        """Event after which host_out of `step` holds its output (valid until
        step + 2 is submitted)."""
        return self.ev_out[step % 2]

    def drain(self, stream=None):
        """Makes `stream` (default: the current one) wait for every queued copy."""
        comp = torch.cuda.current_stream() if stream is None else stream
        comp.wait_stream(self.h2d)
        comp.wait_stream(self.d2h)


def _host_ptr(t, dtype, name):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.is_cuda:
        raise ValueError(f"{name}: expected a host tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    return t.data_ptr()


def dsa_decode_step_host(desc, host_in, dev_in, k_fp8, k_scale, kv, out, host_out, ws, max_seqlen,
                         sm_scale, num_splits=0, stream=None):
    """One decode layer from a host input block to a host output (see
    include/dsa.h): one host-to-device copy, the fused layer, one
    device-to-host copy, all queued on ``stream``."""
    _check(lib().dsa_decode_step_host(
        ctypes.byref(desc), _host_ptr(host_in, torch.uint8, "host_in"),
        _ptr(dev_in, torch.uint8, "dev_in"), _ptr(k_fp8, torch.uint8, "k_fp8"),
        _ptr(k_scale, torch.float32, "k_scale"), _u16(kv, "kv"), float(sm_scale),
        int(num_splits), int(max_seqlen), _ptr(out, torch.float32, "out"),
        _host_ptr(host_out, torch.float32, "host_out"), _ptr(ws, torch.uint8, "ws"), ws.numel(),
        _stream(stream)), "dsa_decode_step_host")


def dsa_get_device_error(stream=None) -> int:
    return int(lib().dsa_get_device_error(_stream(stream)))


def dsa_status_str(status: int) -> str:
    return lib().dsa_status_str(int(status)).decode()


def dsa_version() -> str:
    return lib().dsa_version().decode()


def dsa_debug_set_wait_cycles(cycles: int):
    """Bound of the indexer's pipeline waits in SM cycles (0: the default);
    a test hook for the timeout path (see include/dsa.h)."""
    _check(lib().dsa_debug_set_wait_cycles(int(cycles)), "dsa_debug_set_wait_cycles")


# ---------------------------------------------------------------------------
# Convenience layer over a synthetic ``workloads.Workload`` (allocates outputs
# with torch, then calls the ABI above).
# ---------------------------------------------------------------------------

def workload_desc(wl) -> DecodeDesc:
    s = wl.spec
    return make_desc(wl.seqlens, wl.page_table, s.q_per_req, s.num_heads, s.topk, wl.num_pages)


def logits_ld(wl) -> int:
    return wl.max_pages * PAGE_SIZE


def run_indexer(wl, layer: int = 0, stream=None) -> torch.Tensor:
    lc = wl.layers[layer]
    T = wl.spec.num_tokens
    ld = logits_ld(wl)
    logits = torch.full((T, ld), float("nan"), device=wl.q_fp8.device, dtype=torch.float32)
    dsa_indexer_logits(workload_desc(wl), wl.q_fp8, wl.q_scale, wl.w, lc.k_fp8, lc.k_scale,
                       logits, ld, stream)
    return logits


def run_topk(wl, logits: torch.Tensor, stream=None) -> torch.Tensor:
    desc = workload_desc(wl)
    ld = int(logits.shape[1])
    ws = torch.empty(dsa_topk_workspace_bytes(desc, ld), dtype=torch.uint8, device=logits.device)
    out = torch.empty((wl.spec.num_tokens, wl.spec.topk), dtype=torch.int32, device=logits.device)
    dsa_topk(desc, logits, out, ws, ld, stream)
    return out


def run_sparse_mla_split(wl, topk_idx, num_splits=0, layer: int = 0, stream=None):
    lc = wl.layers[layer]
    desc = workload_desc(wl)
    S = dsa_num_splits_auto(desc) if num_splits == 0 else num_splits
    T, H = wl.spec.num_tokens, wl.spec.num_heads
    mid_o = torch.empty((T, H, S, 512), dtype=torch.float32, device=lc.q.device)
    mid_lse = torch.empty((T, H, S), dtype=torch.float32, device=lc.q.device)
    dsa_sparse_mla_decode_split(desc, lc.q, lc.kv, topk_idx, S, wl.spec.sm_scale, mid_o, mid_lse,
                                stream)
    return mid_o, mid_lse


def run_merge(mid_o, mid_lse, stream=None):
    T, H, S, _ = mid_o.shape
    out = torch.empty((T, H, 512), dtype=torch.float32, device=mid_o.device)
    lse = torch.empty((T, H), dtype=torch.float32, device=mid_o.device)
    dsa_merge(T * H, S, mid_o, mid_lse, out, lse, stream)
    return out, lse


def alloc_workspace(wl, num_splits=0) -> torch.Tensor:
    desc = workload_desc(wl)
    n = dsa_workspace_bytes(desc, wl.max_seqlen, num_splits)
    return torch.empty(n, dtype=torch.uint8, device=wl.q_fp8.device)


def run_decode(wl, ws=None, num_splits=0, layer: int = 0, topk_in=None, topk_out=None,
               out=None, stream=None, stage_events=None) -> torch.Tensor:
    lc = wl.layers[layer]
    T, H = wl.spec.num_tokens, wl.spec.num_heads
    if ws is None:
        ws = alloc_workspace(wl, num_splits)
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.float32, device=lc.q.device)
    dsa_decode_fused(workload_desc(wl), wl.q_fp8, wl.q_scale, wl.w, lc.k_fp8, lc.k_scale, lc.q,
                     lc.kv, out, ws, wl.max_seqlen, wl.spec.sm_scale, num_splits, topk_in,
                     topk_out, stream, stage_events)
    return out
