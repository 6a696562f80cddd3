"""ctypes binding of libbsa (include/bsa.h).  Argument marshalling only: every
step of planning and attention runs in the library's CUDA kernels.  PyTorch
supplies device memory and streams."""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbsa.so")

BSA_OK = 0
STATUS_NAMES = {
    0: "BSA_OK", -1: "BSA_ERR_INVALID_ARG", -2: "BSA_ERR_UNSUPPORTED", -3: "BSA_ERR_ARCH",
    -4: "BSA_ERR_CUDA", -5: "BSA_ERR_WORKSPACE", -6: "BSA_ERR_TIMEOUT", -7: "BSA_ERR_PLAN_MISMATCH",
}
PLAN_NO_UNION = 0x1
PLAN_REMAP = 0x2
PLAN_Q64 = 0x4
STAGE_PREPARE, STAGE_BOUNDED, STAGE_EXACT, STAGE_ALL = 0x1, 0x2, 0x4, 0x7
STAGE_KNORM, STAGE_ROWBOUND = 0x8, 0x10
FWD_CAUSAL = 0x1
FWD_SPLIT_P = 0x2


class KVPagesC(ctypes.Structure):
    """Mirror of bsa_kv_pages (include/bsa.h)."""
    _fields_ = [("block_table", ctypes.c_void_p), ("max_pages", ctypes.c_int),
                ("page_size", ctypes.c_int), ("num_pages", ctypes.c_int)]


class BsaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


class Layout(ctypes.Structure):
    """Mirror of ``bsa_plan_layout``."""
    _fields_ = [(n, ctypes.c_int32) for n in (
        "B", "H", "Hkv", "NQB", "NKB", "bq", "bk", "gqa_group",
        "qu", "rq", "sq", "ku", "rk", "sk",
        "NQT", "NKU", "rows", "urows", "max_row_slots", "groups")] + [
        ("slot_capacity", ctypes.c_int64), ("union_capacity", ctypes.c_int64)] + [
        (n, ctypes.c_uint64) for n in (
            "off_row_ptr", "off_slot_ku", "off_slot_mask", "off_urow_ptr", "off_ukb",
            "off_order", "off_totals", "off_control", "off_scratch", "workspace_bytes", "off_sigma")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class PlanArraysC(ctypes.Structure):
    """Mirror of ``bsa_plan_arrays`` (host buffers for bsa_plan_export)."""
    _fields_ = []
    for _n, _t in (("row_ptr", ctypes.c_void_p), ("slot_ku", ctypes.c_void_p),
                   ("slot_mask", ctypes.c_void_p), ("urow_ptr", ctypes.c_void_p),
                   ("ukb", ctypes.c_void_p), ("order", ctypes.c_void_p),
                   ("plane_sigma", ctypes.c_void_p)):
        _fields_ += [(_n, _t), (_n + "_cap", ctypes.c_size_t)]
    _fields_ += [("totals", ctypes.c_int64 * 4)]


_lib = None


def library() -> ctypes.CDLL:
    """Load libbsa.so (built in-tree by ``block_sparse_attention_plan_gb300.build``).
    Raises if it is missing: there is no fallback path."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run block_sparse_attention_plan_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, U8P, VP = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p
    lib.bsa_version.restype = I
    lib.bsa_version.argtypes = []
    lib.bsa_status_string.restype = ctypes.c_char_p
    lib.bsa_status_string.argtypes = [I]
    lib.bsa_plan_layout_query.restype = I
    lib.bsa_plan_layout_query.argtypes = [I, I, I, I, I, I, I, I, ctypes.POINTER(Layout)]
    lib.bsa_plan_create.restype = I
    lib.bsa_plan_create.argtypes = [U8P, I, I, I, I, I, I, I, VP, ctypes.c_size_t, I, VP,
                                    ctypes.POINTER(P)]
    lib.bsa_plan_select_flags.restype = I
    lib.bsa_plan_select_flags.argtypes = [I, I, I, I, I, I, I, I]
    lib.bsa_plan_workspace_bytes.restype = ctypes.c_size_t
    lib.bsa_plan_workspace_bytes.argtypes = [I, I, I, I, I, I, I]
    lib.bsa_plan_export.restype = I
    lib.bsa_plan_export.argtypes = [P, VP, ctypes.POINTER(PlanArraysC)]
    lib.bsa_plan_get_layout.restype = I
    lib.bsa_plan_get_layout.argtypes = [P, ctypes.POINTER(Layout)]
    lib.bsa_plan_workspace.restype = VP
    lib.bsa_plan_workspace.argtypes = [P]
    lib.bsa_plan_destroy.restype = None
    lib.bsa_plan_destroy.argtypes = [P]
    lib.bsa_forward.restype = I
    lib.bsa_forward.argtypes = [P, VP, VP, VP, VP, VP, I, F, VP]
    lib.bsa_forward_ex.restype = I
    lib.bsa_forward_ex.argtypes = [P, VP, VP, VP, ctypes.POINTER(KVPagesC), VP, I, VP, VP, I, F, VP]
    lib.bsa_forward_stage.restype = I
    lib.bsa_forward_stage.argtypes = [P, VP, VP, VP, ctypes.POINTER(KVPagesC), VP, I, VP, VP, I, F, I, VP]
    lib.bsa_sync_status.restype = I
    lib.bsa_sync_status.argtypes = [P, VP, ctypes.POINTER(ctypes.c_int32)]
    lib.bsa_plan_check.restype = I
    lib.bsa_plan_check.argtypes = [P, VP]
    lib.bsa_watchdog_selftest.restype = I
    lib.bsa_watchdog_selftest.argtypes = [VP, I, VP]
    lib.bsa_attention_static.restype = I
    lib.bsa_attention_static.argtypes = [U8P, I, I, I, I, I, I, I, VP, VP, VP, VP, VP, I, F, VP]
    lib.bsa_attention_static_status.restype = I
    lib.bsa_attention_static_status.argtypes = [VP, ctypes.POINTER(ctypes.c_int32)]
    lib.bsa_plan_create_affine.restype = I
    lib.bsa_plan_create_affine.argtypes = [U8P, VP, VP, I, I, I, I, I, I, I, I, VP, ctypes.c_size_t,
                                           I, VP, ctypes.POINTER(P)]
    lib.bsa_attention_host_buffer_bytes.restype = I
    lib.bsa_attention_host_buffer_bytes.argtypes = [I, I, I, I, I, I, I, I, I,
                                                    ctypes.POINTER(ctypes.c_size_t)]
    lib.bsa_attention_host.restype = I
    lib.bsa_attention_host.argtypes = [U8P, I, I, I, I, I, I, I, VP, VP, VP, VP, VP, I, F, I, VP,
                                       ctypes.c_size_t, VP]
    _lib = lib
    return lib


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int, what: str):
    if status != BSA_OK:
        raise BsaError(status, what)


def select_flags(B: int, H: int, NQB: int, NKB: int, bq: int, bk: int, gqa_group: int, d: int) -> int:
    """Plan flags chosen from the library's measured table (bsa_plan_select_flags)."""
    f = int(library().bsa_plan_select_flags(B, H, NQB, NKB, bq, bk, gqa_group, d))
    _check(min(f, 0), "bsa_plan_select_flags")
    return f


def plan_workspace_bytes(B: int, H: int, NQB: int, NKB: int, bq: int, bk: int,
                         gqa_group: int = 1) -> int:
    """Workspace bytes of a plan (bsa_plan_workspace_bytes; 0 for bad arguments)."""
    return int(library().bsa_plan_workspace_bytes(B, H, NQB, NKB, bq, bk, gqa_group))


def plan_layout(B: int, H: int, NQB: int, NKB: int, bq: int, bk: int, gqa_group: int = 1,
                flags: int = 0) -> Layout:
    L = Layout()
    _check(library().bsa_plan_layout_query(B, H, NQB, NKB, bq, bk, gqa_group, flags, ctypes.byref(L)),
           "bsa_plan_layout_query")
    return L


class Plan:
    """A plan built on the GPU.  Holds the caller-side workspace tensor (which
    owns every plan array) and the library's host handle."""

    def __init__(self, handle: ctypes.c_void_p, workspace: torch.Tensor, layout: Layout,
                 mask: torch.Tensor):
        self._handle = handle
        self.workspace = workspace
        self.layout = layout
        self.mask = mask  # keeps the mask alive while the plan kernels may still read it

    @property
    def handle(self) -> ctypes.c_void_p:
        if self._handle is None:
            raise RuntimeError("plan destroyed")
        return self._handle

    def _view(self, off: int, count: int, dtype: torch.dtype) -> torch.Tensor:
        nbytes = count * torch.empty(0, dtype=dtype).element_size()
        return self.workspace[off:off + nbytes].view(dtype)

    def arrays(self) -> dict:
        """Device views of the plan arrays (sliced to their used lengths where
        the totals are needed: that read synchronises)."""
        L = self.layout
        totals = self._view(L.off_totals, 4, torch.int64).cpu()
        S = int(totals[0])
        U = int(totals[2])
        return {
            "row_ptr": self._view(L.off_row_ptr, L.rows + 1, torch.int32),
            "slot_ku": self._view(L.off_slot_ku, S * L.rk, torch.int32),
            "slot_mask": self._view(L.off_slot_mask, S, torch.int32),
            "urow_ptr": self._view(L.off_urow_ptr, L.urows + 1, torch.int32),
            "ukb": self._view(L.off_ukb, U, torch.int32),
            "order": self._view(L.off_order, L.rows, torch.int32),
            "totals": totals,
            "plane_sigma": self._view(L.off_sigma, L.B * L.H, torch.int32),
        }

    def export(self, stream: Optional[torch.cuda.Stream] = None) -> dict:
        """Host copies of the plan arrays through bsa_plan_export (synchronises):
        int32 numpy arrays (slot_mask as uint32) and the int64 totals."""
        import numpy as np
        L = self.layout
        c = PlanArraysC()
        _check(library().bsa_plan_export(self.handle, _stream_ptr(stream), ctypes.byref(c)),
               "bsa_plan_export")
        tot = np.array(list(c.totals), dtype=np.int64)
        S, U = int(tot[0]), int(tot[2])
        out = {"row_ptr": np.empty(L.rows + 1, np.int32), "slot_ku": np.empty(S * L.rk, np.int32),
               "slot_mask": np.empty(S, np.uint32), "urow_ptr": np.empty(L.urows + 1, np.int32),
               "ukb": np.empty(U, np.int32), "order": np.empty(L.rows, np.int32),
               "plane_sigma": np.empty(L.B * L.H, np.int32)}
        for k, a in out.items():
            setattr(c, k, ctypes.c_void_p(a.ctypes.data))
            setattr(c, k + "_cap", a.size)
        _check(library().bsa_plan_export(self.handle, _stream_ptr(stream), ctypes.byref(c)),
               "bsa_plan_export")
        out["totals"] = tot
        return out

    def control(self) -> torch.Tensor:
        return self._view(self.layout.off_control, 16, torch.int32)

    def destroy(self):
        if self._handle is not None:
            library().bsa_plan_destroy(self._handle)
            self._handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def plan(mask: torch.Tensor, bq: int, bk: int, gqa_group: int = 1, flags: int = 0,
         stream: Optional[torch.cuda.Stream] = None,
         workspace: Optional[torch.Tensor] = None) -> Plan:
    """Build the plan of a device u8 mask [B, H, Nq/bq, Nk/bk] (bsa_plan_create)."""
    if mask.dtype != torch.uint8 or not mask.is_cuda or mask.dim() != 4:
        raise ValueError("mask must be a CUDA uint8 tensor [B, H, NQB, NKB]")
    mask = mask.contiguous()
    B, H, NQB, NKB = mask.shape
    L = plan_layout(B, H, NQB, NKB, bq, bk, gqa_group, flags)
    if workspace is None:
        workspace = torch.empty(int(L.workspace_bytes), dtype=torch.uint8, device=mask.device)
    h = ctypes.c_void_p()
    _check(library().bsa_plan_create(
        ctypes.c_void_p(mask.data_ptr()), B, H, NQB, NKB, bq, bk, gqa_group,
        ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), flags, _stream_ptr(stream),
        ctypes.byref(h)), "bsa_plan_create")
    return Plan(h, workspace, L, mask)


def affine_segments(segments, device="cuda"):
    """Device arrays (segments int32 [nseg, 4], seg_ptr int32 [H + 1]) of a
    per-head list of (a, b, stride, count) segments."""
    flat = [tuple(int(x) for x in sg) for head in segments for sg in head]
    ptr = [0]
    for head in segments:
        ptr.append(ptr[-1] + len(head))
    seg = torch.tensor(flat if flat else [(0, 0, 0, 0)], dtype=torch.int32).reshape(-1, 4)
    return seg.to(device).contiguous(), torch.tensor(ptr, dtype=torch.int32, device=device), len(flat)


def plan_affine(segments, B: int, NQB: int, NKB: int, bq: int, bk: int, gqa_group: int = 1,
                mask: Optional[torch.Tensor] = None, flags: int = 0,
                stream: Optional[torch.cuda.Stream] = None,
                workspace: Optional[torch.Tensor] = None, device="cuda") -> Plan:
    """Build the plan of affine row segments (bsa_plan_create_affine):
    ``segments[h]`` lists the (a, b, stride, count) of query head h, or
    ``segments`` is the (seg, seg_ptr, nseg) device triple of
    ``affine_segments`` (nothing copied per call); ``mask`` (optional device
    u8 [B, H, NQB, NKB]) is OR-ed in."""
    if isinstance(segments, tuple) and len(segments) == 3 and torch.is_tensor(segments[0]):
        seg, ptr, nseg = segments
    else:
        seg, ptr, nseg = affine_segments(segments, device)
    H = ptr.numel() - 1
    if mask is not None:
        if mask.dtype != torch.uint8 or not mask.is_cuda or tuple(mask.shape) != (B, H, NQB, NKB):
            raise ValueError("mask must be a CUDA uint8 tensor [B, H, NQB, NKB]")
        mask = mask.contiguous()
    L = plan_layout(B, H, NQB, NKB, bq, bk, gqa_group, flags)
    if workspace is None:
        workspace = torch.empty(int(L.workspace_bytes), dtype=torch.uint8, device=device)
    h = ctypes.c_void_p()
    _check(library().bsa_plan_create_affine(
        ctypes.c_void_p(mask.data_ptr() if mask is not None else None), ctypes.c_void_p(seg.data_ptr()),
        ctypes.c_void_p(ptr.data_ptr()), nseg, B, H, NQB, NKB, bq, bk, gqa_group,
        ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), flags, _stream_ptr(stream),
        ctypes.byref(h)), "bsa_plan_create_affine")
    return Plan(h, workspace, L, (mask, seg, ptr))


def forward(p: Plan, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
            out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
            scale: Optional[float] = None,
            stream: Optional[torch.cuda.Stream] = None,
            block_table: Optional[torch.Tensor] = None,
            kv_lens: Optional[torch.Tensor] = None,
            causal: bool = False, stages: Optional[int] = None,
            split: bool = False) -> Tuple[torch.Tensor, torch.Tensor]:
    """Block-sparse attention over plan ``p``.  Returns (O, LSE).

    Contiguous K/V: k, v [B, Hkv, Nk, d].  Paged K/V (``block_table`` given,
    int32 CUDA [B, max_pages]): k, v are pools [num_pages, Hkv, page_size, d].
    ``kv_lens`` (int32 CUDA [B]) and ``causal`` mask keys inside the selected
    blocks (bsa_forward_ex); ``split`` applies every row's weights as two bf16
    terms (BSA_FWD_SPLIT_P).  ``stages`` (STAGE_* bits) enqueues only those
    stages of the forward (bsa_forward_stage); O and LSE are complete once
    all three have run, in order."""
    L = p.layout
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor with 4 dimensions")
    B, Hq, Nq, d = q.shape
    if (B, Hq, Nq) != (L.B, L.H, L.NQB * L.bq):
        raise ValueError("q shape does not match the plan")
    if k.shape != v.shape:
        raise ValueError("k and v shapes differ")
    pages = None
    if block_table is None:
        if tuple(k.shape) != (L.B, L.Hkv, L.NKB * L.bk, d):
            raise ValueError("k/v shape does not match the plan")
    else:
        if (block_table.dtype != torch.int32 or not block_table.is_cuda or block_table.dim() != 2
                or not block_table.is_contiguous() or block_table.shape[0] != L.B):
            raise ValueError("block_table must be a contiguous CUDA int32 tensor [B, max_pages]")
        if k.shape[1] != L.Hkv or k.shape[3] != d:
            raise ValueError("k/v pools must be [num_pages, Hkv, page_size, d]")
        pages = KVPagesC(block_table.data_ptr(), block_table.shape[1], k.shape[2], k.shape[0])
    if kv_lens is not None and (kv_lens.dtype != torch.int32 or not kv_lens.is_cuda
                                or tuple(kv_lens.shape) != (L.B,)):
        raise ValueError("kv_lens must be a CUDA int32 tensor [B]")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, Hq, Nq, dtype=torch.float32, device=q.device)
    sc = 0.0 if scale is None else float(scale)
    flags = (FWD_CAUSAL if causal else 0) | (FWD_SPLIT_P if split else 0)
    if stages is not None:
        _check(library().bsa_forward_stage(
            p.handle, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
            ctypes.c_void_p(v.data_ptr()), ctypes.byref(pages) if pages is not None else None,
            ctypes.c_void_p(kv_lens.data_ptr()) if kv_lens is not None else None,
            flags, ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(lse.data_ptr()), d, sc, int(stages), _stream_ptr(stream)), "bsa_forward_stage")
    elif pages is None and kv_lens is None and flags == 0:
        _check(library().bsa_forward(
            p.handle, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
            ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(lse.data_ptr()), d, sc, _stream_ptr(stream)), "bsa_forward")
    else:
        _check(library().bsa_forward_ex(
            p.handle, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
            ctypes.c_void_p(v.data_ptr()), ctypes.byref(pages) if pages is not None else None,
            ctypes.c_void_p(kv_lens.data_ptr()) if kv_lens is not None else None,
            flags, ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(lse.data_ptr()), d, sc, _stream_ptr(stream)), "bsa_forward_ex")
    return out, lse


def sync_status(p: Plan, stream: Optional[torch.cuda.Stream] = None) -> Tuple[int, int]:
    """(status, detail) the last forward on this plan left (synchronises)."""
    det = ctypes.c_int32(0)
    st = library().bsa_sync_status(p.handle, _stream_ptr(stream), ctypes.byref(det))
    return st, det.value


def plan_check(p: Plan, stream: Optional[torch.cuda.Stream] = None) -> int:
    return library().bsa_plan_check(p.handle, _stream_ptr(stream))


def watchdog_selftest(limit_us: int = 20000, device: Optional[torch.device] = None) -> int:
    buf = torch.zeros(4, dtype=torch.int32, device=device or "cuda")
    return library().bsa_watchdog_selftest(ctypes.c_void_p(buf.data_ptr()), limit_us,
                                           _stream_ptr(None))


_host_buffers = {}


def host_buffer_bytes(B: int, H: int, NQB: int, NKB: int, bq: int, bk: int, gqa_group: int, d: int,
                      chunks: int) -> int:
    n = ctypes.c_size_t(0)
    _check(library().bsa_attention_host_buffer_bytes(B, H, NQB, NKB, bq, bk, gqa_group, d, chunks,
                                                     ctypes.byref(n)), "bsa_attention_host_buffer_bytes")
    return int(n.value)


def attention(mask: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, bq: int,
              bk: int, scale: Optional[float] = None, device: str = "cuda",
              stream: Optional[torch.cuda.Stream] = None, chunks: int = 8,
              out: Optional[torch.Tensor] = None, lse_out: Optional[torch.Tensor] = None):
    """One call from host or device tensors.  Host tensors go through
    bsa_attention_host (chunks copied in, computed and copied out on
    overlapping streams; pinned memory keeps the copies asynchronous), with a
    device scratch buffer cached per shape; O and LSE come back in pinned host
    tensors (or ``out`` / ``lse_out``).  Device tensors: plan + forward.
    Device plans take the flags of the library's measured table
    (bsa_plan_select_flags: q-tile height, regrouping).
    Returns (O, LSE) on the inputs' device."""
    host = not q.is_cuda
    g = q.shape[1] // k.shape[1]
    if not host:
        flags = select_flags(*mask.shape, bq, bk, g, q.shape[3])
        pl = plan(mask, bq, bk, g, flags=flags, stream=stream)
        return forward(pl, q, k, v, scale=scale, stream=stream)
    B, H, NQB, NKB = mask.shape
    d = q.shape[3]
    for name, t in (("mask", mask), ("q", q), ("k", k), ("v", v)):
        if not t.is_contiguous() or t.is_cuda:
            raise ValueError(f"{name} must be a contiguous host tensor")
    key = (torch.device(device).index, B, H, NQB, NKB, bq, bk, g, d, chunks)
    buf = _host_buffers.get(key)
    if buf is None:
        nbytes = host_buffer_bytes(B, H, NQB, NKB, bq, bk, g, d, chunks)
        _host_buffers.clear()  # one cached buffer at a time
        buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _host_buffers[key] = buf
    o_h = out if out is not None else torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    l_h = lse_out if lse_out is not None else torch.empty(q.shape[:3], dtype=torch.float32,
                                                          pin_memory=True)
    _check(library().bsa_attention_host(
        ctypes.c_void_p(mask.data_ptr()), B, H, NQB, NKB, bq, bk, g,
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(o_h.data_ptr()), ctypes.c_void_p(l_h.data_ptr()), d,
        0.0 if scale is None else float(scale), chunks, ctypes.c_void_p(buf.data_ptr()), buf.numel(),
        _stream_ptr(stream)), "bsa_attention_host")
    return o_h, l_h


def attention_static(mask: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                     bq: int, bk: int, out: Optional[torch.Tensor] = None,
                     lse: Optional[torch.Tensor] = None, scale: Optional[float] = None,
                     stream: Optional[torch.cuda.Stream] = None):
    """Plan + forward in one call with the library's built-in scratch area
    (bsa_attention_static): for callers that cannot allocate device memory.
    ``out`` and ``lse`` may be supplied so that nothing is allocated here."""
    B, H, NQB, NKB = mask.shape
    d = q.shape[3]
    g = q.shape[1] // k.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    _check(library().bsa_attention_static(
        ctypes.c_void_p(mask.data_ptr()), B, H, NQB, NKB, bq, bk, g,
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()), d,
        0.0 if scale is None else float(scale), _stream_ptr(stream)), "bsa_attention_static")
    return out, lse


def attention_static_status(stream: Optional[torch.cuda.Stream] = None) -> Tuple[int, int]:
    """(status, detail) the kernels of the last attention_static call on the
    current device recorded (bsa_attention_static_status; synchronises)."""
    det = ctypes.c_int32(0)
    st = library().bsa_attention_static_status(_stream_ptr(stream), ctypes.byref(det))
    return st, det.value

